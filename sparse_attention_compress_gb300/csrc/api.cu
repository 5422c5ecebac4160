// C ABI of libnsa.so: argument checks, layout bookkeeping and dispatch to the kernels.
// Every check runs before any launch; nothing here allocates device memory.
#include <stdarg.h>
#include <stdio.h>

#include "nsa.h"
#include <algorithm>

#include "launch.h"

// NVTX ranges name every entry point in a profiler's timeline (nvtx3 is header-only: with
// no tool attached a range costs one pointer check).
#include <nvtx3/nvToolsExt.h>

using namespace nsa;

namespace {

thread_local char g_err[512] = "";

nsa_status fail(nsa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

nsa_status cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) {
    g_err[0] = 0;
    return NSA_OK;
  }
  return fail(NSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
};
#define NSA_RANGE() const Range nsa_range_(__func__)

#define NSA_REQUIRE(cond, st, ...)     \
  do {                                 \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

#define NSA_PTR(p)                                                                     \
  do {                                                                                 \
    if ((p) == nullptr) return fail(NSA_ERR_INVALID, "%s: null pointer " #p, __func__); \
    if (!aligned16(p)) return fail(NSA_ERR_INVALID, "%s: " #p " not 16-byte aligned", __func__); \
  } while (0)

// Validate the common shape and build the kernel-side sequence description.
nsa_status make_seqs(const nsa_shape* s, Seqs* out, const char* fn) {
  if (!s) return fail(NSA_ERR_INVALID, "%s: null shape", fn);
  if (s->h <= 0 || s->h_kv <= 0 || s->d <= 0) return fail(NSA_ERR_INVALID, "%s: h, h_kv, d must be positive", fn);
  if (s->h % s->h_kv) return fail(NSA_ERR_INVALID, "%s: h (%d) not a multiple of h_kv (%d)", fn, s->h, s->h_kv);
  if (s->dtype != NSA_F32 && s->dtype != NSA_BF16) return fail(NSA_ERR_INVALID, "%s: unknown dtype", fn);
  if (s->seqlen < 0) return fail(NSA_ERR_INVALID, "%s: negative seqlen", fn);
  Seqs q{};
  if (s->cu_seqlens) {
    if (s->n_seqs < 1) return fail(NSA_ERR_INVALID, "%s: varlen needs n_seqs >= 1", fn);
    if (s->total_tokens < 0) return fail(NSA_ERR_INVALID, "%s: negative total_tokens", fn);
    q.cu = s->cu_seqlens;
    q.n_seqs = s->n_seqs;
    q.T = 0;
    q.tokens = s->total_tokens;
    q.max_len = s->seqlen;
  } else {
    if (s->batch < 0) return fail(NSA_ERR_INVALID, "%s: negative batch", fn);
    q.cu = nullptr;
    q.n_seqs = s->batch;
    q.T = s->seqlen;
    q.tokens = (int64_t)s->batch * s->seqlen;
    q.max_len = s->seqlen;
  }
  *out = q;
  return NSA_OK;
}

bool pow2_le16(int r) { return r == 1 || r == 2 || r == 4 || r == 8 || r == 16; }
int num_cmp_host(int L, int kernel, int stride) { return L >= kernel ? (L - kernel) / stride + 1 : 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

void nsa::set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

nsa_status nsa::decode_check_sizes(int batch, int max_len, int h, int h_kv, int d, int kernel, int stride,
                                   int block_size, int n_init, int n_local, int k) {
  NSA_REQUIRE(batch >= 0 && max_len >= 1 && h > 0 && h_kv > 0 && h % h_kv == 0, NSA_ERR_INVALID,
              "nsa_sparse_decode: bad sizes");
  NSA_REQUIRE(kernel == 32 && stride == 16 && block_size == 64, NSA_ERR_UNSUPPORTED,
              "nsa_sparse_decode: supports kernel 32, stride 16, block_size 64");
  NSA_REQUIRE(d == 128, NSA_ERR_UNSUPPORTED, "nsa_sparse_decode: d must be 128");
  NSA_REQUIRE(pow2_le16(h / h_kv), NSA_ERR_UNSUPPORTED, "nsa_sparse_decode: h/h_kv must be 1, 2, 4, 8 or 16");
  NSA_REQUIRE(k >= 1 && k <= 64, NSA_ERR_UNSUPPORTED, "nsa_sparse_decode: k must be in [1, 64]");
  NSA_REQUIRE(n_init >= 0 && n_local >= 0, NSA_ERR_INVALID, "nsa_sparse_decode: negative n_init/n_local");
  NSA_REQUIRE(max_len <= 65536, NSA_ERR_UNSUPPORTED, "nsa_sparse_decode: max_len must be <= 65536");
  return NSA_OK;
}

extern "C" {

const char* nsa_version(void) { return "nsa-gb300 0.1 (sm_103a)"; }

const char* nsa_last_error(void) { return g_err; }

nsa_status nsa_device_status(int32_t* status, int reset) {
  NSA_RANGE();
  NSA_REQUIRE(status != nullptr, NSA_ERR_INVALID, "nsa_device_status: status is NULL");
  int32_t a = 0, b = 0, c = 0, f = 0, k = 0;
  cudaError_t e = status_word_dense_tc(&a, reset != 0);
  if (e == cudaSuccess) e = status_word_decode(&b, reset != 0);
  if (e == cudaSuccess) e = status_word_decode_nosa(&c, reset != 0);
  if (e == cudaSuccess) e = status_word_sparse_fwd(&f, reset != 0);
  if (e == cudaSuccess) e = status_word_sparse_bwd_tc(&k, reset != 0);
  *status = a ? a : b ? b : c ? c : f ? f : k;
  return cuda_status(e, "nsa_device_status");
}

nsa_status nsa_set_wait_limit_ns(uint64_t ns) {
  NSA_RANGE();
  const unsigned long long v = ns ? (unsigned long long)ns : 1000000000ull;
  cudaError_t e = wait_limit_dense_tc(v);
  if (e == cudaSuccess) e = wait_limit_decode(v);
  if (e == cudaSuccess) e = wait_limit_decode_nosa(v);
  if (e == cudaSuccess) e = wait_limit_sparse_fwd(v);
  if (e == cudaSuccess) e = wait_limit_sparse_bwd_tc(v);
  return cuda_status(e, "nsa_set_wait_limit_ns");
}

nsa_status nsa_compress_k(const nsa_shape* shape, const void* k, void* k_cmp, int kernel, int stride,
                          cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(kernel > 0 && stride > 0, NSA_ERR_INVALID, "nsa_compress_k: kernel and stride must be positive");
  NSA_REQUIRE(kernel % stride == 0 && kernel / stride <= 4, NSA_ERR_UNSUPPORTED,
              "nsa_compress_k: needs kernel %% stride == 0 and kernel/stride <= 4 (got %d/%d)", kernel, stride);
  const int vec = shape->dtype == NSA_BF16 ? 8 : 4;
  NSA_REQUIRE((shape->h_kv * shape->d) % vec == 0, NSA_ERR_UNSUPPORTED,
              "nsa_compress_k: h_kv*d must be a multiple of %d", vec);
  if (s.tokens == 0 || s.max_len < kernel) return NSA_OK;
  NSA_PTR(k);
  NSA_PTR(k_cmp);
  return cuda_status(launch_compress(s, k, k_cmp, shape->h_kv, shape->d, shape->dtype, kernel, stride, stream),
                     "nsa_compress_k");
}

nsa_status nsa_cmp_scores_pool(const nsa_shape* shape, const void* q, const void* k_cmp, int kernel,
                               int stride, int block_size, float scale, const float* lse_in,
                               float* block_scores, int nb_stride, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(kernel == 32 && stride == 16 && block_size == 64, NSA_ERR_UNSUPPORTED,
              "nsa_cmp_scores_pool: supports kernel 32, stride 16, block_size 64");
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "nsa_cmp_scores_pool: bf16 only");
  NSA_REQUIRE(shape->d == 64 || shape->d == 128, NSA_ERR_UNSUPPORTED, "nsa_cmp_scores_pool: d must be 64 or 128");
  NSA_REQUIRE(pow2_le16(shape->h / shape->h_kv), NSA_ERR_UNSUPPORTED,
              "nsa_cmp_scores_pool: h/h_kv must be 1, 2, 4, 8 or 16");
  NSA_REQUIRE(nb_stride >= (s.max_len + block_size - 1) / block_size, NSA_ERR_INVALID,
              "nsa_cmp_scores_pool: nb_stride %d < blocks of the longest sequence", nb_stride);
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(block_scores);
  if (s.max_len >= kernel) NSA_PTR(k_cmp);
  if (lse_in && (reinterpret_cast<uintptr_t>(lse_in) & 3u))
    return fail(NSA_ERR_INVALID, "nsa_cmp_scores_pool: lse_in misaligned");
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  return cuda_status(launch_scores_pool(s, q, k_cmp, shape->h, shape->h_kv, shape->d, scale, lse_in, block_scores,
                                        nb_stride, stream),
                     "nsa_cmp_scores_pool");
}

nsa_status nsa_topk_select(const nsa_shape* shape, const float* block_scores, int nb_stride,
                           int block_size, int n_init, int n_local, int k, int32_t* block_indices,
                           cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(block_size > 0 && n_init >= 0 && n_local >= 0, NSA_ERR_INVALID,
              "nsa_topk_select: block_size > 0, n_init >= 0, n_local >= 0");
  NSA_REQUIRE(k >= 1 && k <= 64, NSA_ERR_UNSUPPORTED, "nsa_topk_select: k must be in [1, 64]");
  NSA_REQUIRE(nb_stride >= (s.max_len + block_size - 1) / block_size, NSA_ERR_INVALID,
              "nsa_topk_select: nb_stride %d < blocks of the longest sequence", nb_stride);
  NSA_REQUIRE(nb_stride <= 2048, NSA_ERR_UNSUPPORTED, "nsa_topk_select: nb_stride must be <= 2048");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(block_scores);
  NSA_PTR(block_indices);
  return cuda_status(launch_topk(s, block_scores, nb_stride, shape->h_kv, block_size, n_init, n_local, k,
                                 block_indices, stream),
                     "nsa_topk_select");
}

nsa_status nsa_cis_block_scores(const nsa_shape* shape, const float* cis, int kernel, int stride, int block_size,
                                int nb_stride, float* out, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(kernel > 0 && stride > 0 && block_size > 0, NSA_ERR_INVALID,
              "nsa_cis_block_scores: kernel, stride and block_size must be positive");
  NSA_REQUIRE(nb_stride >= (s.max_len + block_size - 1) / block_size, NSA_ERR_INVALID,
              "nsa_cis_block_scores: nb_stride %d < blocks of the longest sequence", nb_stride);
  if (s.n_seqs == 0 || nb_stride == 0) return NSA_OK;
  NSA_PTR(out);
  if (s.tokens > 0) NSA_PTR(cis);
  return cuda_status(launch_cis_block_scores(s, cis, shape->h_kv, kernel, stride, block_size, nb_stride, out, stream),
                     "nsa_cis_block_scores");
}

nsa_status nsa_topk_two_stage(const nsa_shape* shape, const float* block_scores, int nb_stride,
                              const float* cis_block_scores, int block_size, int n_init, int n_local, int qk_select,
                              int k, int32_t* block_indices, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(block_size > 0 && n_init >= 0 && n_local >= 0, NSA_ERR_INVALID,
              "nsa_topk_two_stage: block_size > 0, n_init >= 0, n_local >= 0");
  NSA_REQUIRE(k >= 1 && k <= qk_select && qk_select <= 64, NSA_ERR_UNSUPPORTED,
              "nsa_topk_two_stage: need 1 <= k <= qk_select <= 64");
  NSA_REQUIRE(nb_stride >= (s.max_len + block_size - 1) / block_size, NSA_ERR_INVALID,
              "nsa_topk_two_stage: nb_stride %d < blocks of the longest sequence", nb_stride);
  NSA_REQUIRE(nb_stride <= 2048, NSA_ERR_UNSUPPORTED, "nsa_topk_two_stage: nb_stride must be <= 2048");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(block_scores);
  NSA_PTR(cis_block_scores);
  NSA_PTR(block_indices);
  return cuda_status(launch_topk_two_stage(s, block_scores, nb_stride, cis_block_scores, shape->h_kv, block_size,
                                           n_init, n_local, qk_select, k, block_indices, stream),
                     "nsa_topk_two_stage");
}

nsa_status nsa_sparse_cis_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v, const float* cis,
                              const int32_t* block_indices, int S, int block_size, float scale, void* o, float* lse,
                              cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  const int r = shape->h / shape->h_kv;
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "nsa_sparse_cis_fwd: bf16 only");
  NSA_REQUIRE(shape->d == 64 || shape->d == 128, NSA_ERR_UNSUPPORTED, "nsa_sparse_cis_fwd: d must be 64 or 128");
  NSA_REQUIRE(block_size == 64, NSA_ERR_UNSUPPORTED, "nsa_sparse_cis_fwd: block_size must be 64");
  NSA_REQUIRE(S >= 1 && S <= 64, NSA_ERR_UNSUPPORTED, "nsa_sparse_cis_fwd: S must be in [1, 64]");
  NSA_REQUIRE(r <= 16 || r % 16 == 0, NSA_ERR_UNSUPPORTED,
              "nsa_sparse_cis_fwd: h/h_kv must be <= 16 or a multiple of 16");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(block_indices);
  NSA_PTR(o);
  NSA_REQUIRE(cis != nullptr && (reinterpret_cast<uintptr_t>(cis) & 3u) == 0, NSA_ERR_INVALID,
              "nsa_sparse_cis_fwd: cis must be non-null and 4-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(NSA_ERR_INVALID, "nsa_sparse_cis_fwd: lse misaligned");
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  return cuda_status(launch_sparse_fwd(s, q, k, v, block_indices, S, block_size, shape->h, shape->h_kv, shape->d,
                                       shape->dtype, scale, o, lse, stream, cis),
                     "nsa_sparse_cis_fwd");
}

static nsa_status check_cmp_bwd(const nsa_shape* shape, int kernel, int stride, Seqs* s, const char* fn) {
  if (nsa_status st = make_seqs(shape, s, fn)) return st;
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "%s: bf16 only", fn);
  NSA_REQUIRE(shape->d == 128, NSA_ERR_UNSUPPORTED, "%s: d must be 128", fn);
  NSA_REQUIRE(kernel >= 1 && stride >= 1 && kernel <= 1024 && stride <= kernel, NSA_ERR_UNSUPPORTED,
              "%s: needs 1 <= stride <= kernel <= 1024", fn);
  NSA_REQUIRE(shape->h / shape->h_kv <= 16, NSA_ERR_UNSUPPORTED, "%s: h/h_kv must be <= 16", fn);
  NSA_REQUIRE(num_cmp_host(s->max_len, kernel, stride) <= 4096, NSA_ERR_UNSUPPORTED,
              "%s: at most 4096 compressed keys per sequence", fn);
  NSA_REQUIRE(s->max_len <= (1 << 24), NSA_ERR_UNSUPPORTED, "%s: sequences must be <= 2^24 tokens", fn);
  return NSA_OK;
}

size_t nsa_cmp_attn_bwd_workspace_size(const nsa_shape* shape, int kernel, int stride) {
  Seqs s;
  if (check_cmp_bwd(shape, kernel, stride, &s, "nsa_cmp_attn_bwd_workspace_size") != NSA_OK) return 0;
  return cmp_attn_bwd_workspace_bytes(s, shape->h, shape->h_kv, kernel, stride);
}

nsa_status nsa_cmp_attn_bwd(const nsa_shape* shape, const void* q, const void* k_cmp, const void* v_cmp, int kernel,
                            int stride, float scale, const void* o, const float* lse, const void* d_o, void* dq,
                            void* dk_cmp, void* dv_cmp, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = check_cmp_bwd(shape, kernel, stride, &s, __func__)) return st;
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(o);
  NSA_PTR(d_o);
  NSA_PTR(dq);
  if (num_cmp_host(s.max_len, kernel, stride) > 0) {
    NSA_PTR(k_cmp);
    NSA_PTR(v_cmp);
    NSA_PTR(dk_cmp);
    NSA_PTR(dv_cmp);
  }
  NSA_REQUIRE(lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) == 0, NSA_ERR_INVALID,
              "nsa_cmp_attn_bwd: lse must be non-null and 4-byte aligned");
  const size_t need = cmp_attn_bwd_workspace_bytes(s, shape->h, shape->h_kv, kernel, stride);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_cmp_attn_bwd: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= need, NSA_ERR_INVALID, "nsa_cmp_attn_bwd: workspace %zu < %zu bytes",
              workspace_bytes, need);
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  return cuda_status(launch_cmp_attn_bwd(s, q, k_cmp, v_cmp, shape->h, shape->h_kv, kernel, stride, scale, o, lse,
                                         d_o, dq, dk_cmp, dv_cmp, workspace, stream),
                     "nsa_cmp_attn_bwd");
}

nsa_status nsa_compress_bwd(const nsa_shape* shape, const void* dk_cmp, int kernel, int stride, void* dk,
                            cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "nsa_compress_bwd: bf16 only");
  NSA_REQUIRE(shape->d % 8 == 0, NSA_ERR_UNSUPPORTED, "nsa_compress_bwd: d must be a multiple of 8");
  NSA_REQUIRE(kernel >= 1 && stride >= 1, NSA_ERR_INVALID, "nsa_compress_bwd: kernel and stride must be positive");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(dk);
  if (num_cmp_host(s.max_len, kernel, stride) > 0) NSA_PTR(dk_cmp);
  return cuda_status(launch_compress_bwd(s, dk_cmp, shape->h_kv, shape->d, kernel, stride, dk, stream),
                     "nsa_compress_bwd");
}

size_t nsa_swa_bwd_workspace_size(const nsa_shape* shape, int window) {
  Seqs s;
  if (make_seqs(shape, &s, "nsa_swa_bwd_workspace_size") != NSA_OK || window < 1 || window > 1984) return 0;
  return swa_bwd_workspace_bytes(s, shape->h, shape->h_kv, window);
}

nsa_status nsa_swa_bwd(const nsa_shape* shape, const void* q, const void* k, const void* v, int window, float scale,
                       const void* o, const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "nsa_swa_bwd: bf16 only");
  NSA_REQUIRE(shape->d == 128, NSA_ERR_UNSUPPORTED, "nsa_swa_bwd: d must be 128");
  NSA_REQUIRE(shape->h / shape->h_kv <= 16, NSA_ERR_UNSUPPORTED, "nsa_swa_bwd: h/h_kv must be <= 16");
  NSA_REQUIRE(window >= 1 && window <= 1984, NSA_ERR_UNSUPPORTED, "nsa_swa_bwd: window must be in [1, 1984]");
  NSA_REQUIRE(s.max_len <= (1 << 24), NSA_ERR_UNSUPPORTED, "nsa_swa_bwd: sequences must be <= 2^24 tokens");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(o);
  NSA_PTR(d_o);
  NSA_PTR(dq);
  NSA_PTR(dk);
  NSA_PTR(dv);
  NSA_REQUIRE(lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) == 0, NSA_ERR_INVALID,
              "nsa_swa_bwd: lse must be non-null and 4-byte aligned");
  const size_t need = swa_bwd_workspace_bytes(s, shape->h, shape->h_kv, window);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_swa_bwd: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= need, NSA_ERR_INVALID, "nsa_swa_bwd: workspace %zu < %zu bytes", workspace_bytes,
              need);
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  return cuda_status(launch_swa_bwd(s, q, k, v, shape->h, shape->h_kv, window, scale, o, lse, d_o, dq, dk, dv,
                                    workspace, stream),
                     "nsa_swa_bwd");
}

nsa_status nsa_gate_combine_bwd(int64_t tokens, int h, int d, const void* d_o, const void* o_cmp, const void* o_slc,
                                const void* o_swa, const float* gate_logits, void* d_cmp, void* d_slc, void* d_swa,
                                float* d_gate_logits, cudaStream_t stream) {
  NSA_RANGE();
  NSA_REQUIRE(tokens >= 0 && h > 0 && d > 0, NSA_ERR_INVALID, "nsa_gate_combine_bwd: bad sizes");
  NSA_REQUIRE(d % 8 == 0 && d <= 256, NSA_ERR_UNSUPPORTED, "nsa_gate_combine_bwd: d must be a multiple of 8, <= 256");
  if (tokens == 0) return NSA_OK;
  NSA_PTR(d_o);
  NSA_PTR(o_cmp);
  NSA_PTR(o_slc);
  NSA_PTR(o_swa);
  NSA_PTR(gate_logits);
  NSA_PTR(d_cmp);
  NSA_PTR(d_slc);
  NSA_PTR(d_swa);
  NSA_PTR(d_gate_logits);
  return cuda_status(launch_gate_bwd(tokens * h, d, d_o, o_cmp, o_slc, o_swa, gate_logits, d_cmp, d_slc, d_swa,
                                     d_gate_logits, stream),
                     "nsa_gate_combine_bwd");
}

static nsa_status check_sparse_bwd(const nsa_shape* shape, int S, int block_size, Seqs* s, const char* fn) {
  if (nsa_status st = make_seqs(shape, s, fn)) return st;
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "%s: bf16 only", fn);
  NSA_REQUIRE(shape->d == 128, NSA_ERR_UNSUPPORTED, "%s: d must be 128", fn);
  NSA_REQUIRE(block_size == 64, NSA_ERR_UNSUPPORTED, "%s: block_size must be 64", fn);
  NSA_REQUIRE(S >= 1 && S <= 64, NSA_ERR_UNSUPPORTED, "%s: S must be in [1, 64]", fn);
  NSA_REQUIRE(shape->h / shape->h_kv <= 16, NSA_ERR_UNSUPPORTED, "%s: h/h_kv must be <= 16", fn);
  NSA_REQUIRE(s->max_len <= (1 << 24), NSA_ERR_UNSUPPORTED, "%s: sequences must be <= 2^24 tokens", fn);
  return NSA_OK;
}

size_t nsa_sparse_bwd_workspace_size(const nsa_shape* shape, int S, int block_size) {
  Seqs s;
  if (check_sparse_bwd(shape, S, block_size, &s, "nsa_sparse_bwd_workspace_size") != NSA_OK) return 0;
  return sparse_bwd_workspace_bytes(s, shape->h, shape->h_kv, S);
}

nsa_status nsa_sparse_bwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                          const int32_t* block_indices, int S, int block_size, float scale, const void* o,
                          const float* lse, const void* d_o, void* dq, void* dk, void* dv, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = check_sparse_bwd(shape, S, block_size, &s, __func__)) return st;
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(block_indices);
  NSA_PTR(o);
  NSA_PTR(d_o);
  NSA_PTR(dq);
  NSA_PTR(dk);
  NSA_PTR(dv);
  NSA_REQUIRE(lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) == 0, NSA_ERR_INVALID,
              "nsa_sparse_bwd: lse must be non-null and 4-byte aligned");
  const size_t need = sparse_bwd_workspace_bytes(s, shape->h, shape->h_kv, S);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_sparse_bwd: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= need, NSA_ERR_INVALID, "nsa_sparse_bwd: workspace %zu < %zu bytes",
              workspace_bytes, need);
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  return cuda_status(launch_sparse_bwd(s, q, k, v, block_indices, S, shape->h, shape->h_kv, scale, o, lse, d_o, dq,
                                       dk, dv, workspace, stream),
                     "nsa_sparse_bwd");
}

size_t nsa_block_sparse_workspace_size(const nsa_shape* shape) {
  Seqs s;
  if (make_seqs(shape, &s, __func__) != NSA_OK) return 0;
  return align256((size_t)shape->h * shape->d * tc_vt_pad(s.tokens > 0 ? s.tokens : 1) * 2);
}

nsa_status nsa_block_sparse_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                                const uint8_t* block_mask, int block_size, int causal, float scale, void* o,
                                float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(shape->cu_seqlens == nullptr, NSA_ERR_UNSUPPORTED, "nsa_block_sparse_fwd: dense layout only");
  NSA_REQUIRE(shape->dtype == NSA_BF16 && shape->d == 128, NSA_ERR_UNSUPPORTED,
              "nsa_block_sparse_fwd: bf16 with d = 128 only");
  NSA_REQUIRE(shape->h == shape->h_kv, NSA_ERR_UNSUPPORTED, "nsa_block_sparse_fwd: needs h_kv == h");
  NSA_REQUIRE(block_size == 64, NSA_ERR_UNSUPPORTED, "nsa_block_sparse_fwd: block_size must be 64");
  NSA_REQUIRE(shape->seqlen % 64 == 0 && shape->seqlen <= 65536, NSA_ERR_UNSUPPORTED,
              "nsa_block_sparse_fwd: seqlen must be a multiple of 64, at most 65536");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(o);
  NSA_REQUIRE(block_mask != nullptr, NSA_ERR_INVALID, "nsa_block_sparse_fwd: block_mask is NULL");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(NSA_ERR_INVALID, "nsa_block_sparse_fwd: lse misaligned");
  const size_t need = nsa_block_sparse_workspace_size(shape);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_block_sparse_fwd: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= need, NSA_ERR_INVALID, "nsa_block_sparse_fwd: workspace %zu < %zu bytes",
              workspace_bytes, need);
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  cudaError_t e = launch_transpose_v(s, v, workspace, s.tokens, shape->h, false, 32, 16, stream);
  if (e) return cuda_status(e, "nsa_block_sparse_fwd/transpose v");
  return cuda_status(launch_block_sparse_tc(s, q, k, workspace, shape->h, block_mask, causal ? 1 : 0, scale, o, lse,
                                            stream),
                     "nsa_block_sparse_fwd");
}

size_t nsa_select_workspace_size(const nsa_shape* shape, int block_size) {
  Seqs s;
  if (make_seqs(shape, &s, __func__) != NSA_OK || block_size <= 0) return 0;
  const int nb = (s.max_len + block_size - 1) / block_size;
  return align256((size_t)s.tokens * shape->h_kv * (nb > 0 ? nb : 1) * 4);
}

nsa_status nsa_select(const nsa_shape* shape, const void* q, const void* k_cmp, int kernel, int stride,
                      int block_size, float scale, int n_init, int n_local, int k, int32_t* block_indices,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  NSA_REQUIRE(kernel == 32 && stride == 16 && block_size == 64, NSA_ERR_UNSUPPORTED,
              "nsa_select: supports kernel 32, stride 16, block_size 64");
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "nsa_select: bf16 only");
  NSA_REQUIRE(shape->d == 64 || shape->d == 128, NSA_ERR_UNSUPPORTED, "nsa_select: d must be 64 or 128");
  NSA_REQUIRE(pow2_le16(shape->h / shape->h_kv), NSA_ERR_UNSUPPORTED, "nsa_select: h/h_kv must be 1, 2, 4, 8 or 16");
  NSA_REQUIRE(n_init >= 0 && n_local >= 0, NSA_ERR_INVALID, "nsa_select: negative n_init/n_local");
  NSA_REQUIRE(k >= 1 && k <= 64, NSA_ERR_UNSUPPORTED, "nsa_select: k must be in [1, 64]");
  const int nb = (s.max_len + block_size - 1) / block_size;
  NSA_REQUIRE(nb <= 2048, NSA_ERR_UNSUPPORTED, "nsa_select: sequences longer than 131072 tokens");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(block_indices);
  if (s.max_len >= kernel) NSA_PTR(k_cmp);
  const size_t need = nsa_select_workspace_size(shape, block_size);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_select: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= need, NSA_ERR_INVALID, "nsa_select: workspace %zu < %zu bytes", workspace_bytes,
              need);
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  float* scores = static_cast<float*>(workspace);
  cudaError_t e = launch_scores_pool(s, q, k_cmp, shape->h, shape->h_kv, shape->d, scale, nullptr, scores,
                                     nb > 0 ? nb : 1, stream);
  if (e) return cuda_status(e, "nsa_select/block scores");
  return cuda_status(launch_topk(s, scores, nb > 0 ? nb : 1, shape->h_kv, block_size, n_init, n_local, k,
                                 block_indices, stream),
                     "nsa_select/top-k");
}

nsa_status nsa_sparse_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                          const int32_t* block_indices, int S, int block_size, float scale, void* o,
                          float* lse, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = make_seqs(shape, &s, __func__)) return st;
  const int r = shape->h / shape->h_kv;
  NSA_REQUIRE(S >= 1 && block_size >= 1, NSA_ERR_INVALID, "nsa_sparse_fwd: S and block_size must be positive");
  if (shape->dtype == NSA_BF16) {
    NSA_REQUIRE(shape->d == 64 || shape->d == 128, NSA_ERR_UNSUPPORTED, "nsa_sparse_fwd: bf16 needs d 64 or 128");
    NSA_REQUIRE(block_size == 16 || block_size == 32 || block_size == 64, NSA_ERR_UNSUPPORTED,
                "nsa_sparse_fwd: bf16 needs block_size 16, 32 or 64");
    NSA_REQUIRE(S <= 64, NSA_ERR_UNSUPPORTED, "nsa_sparse_fwd: S must be <= 64");
    NSA_REQUIRE(r <= 16 || r % 16 == 0, NSA_ERR_UNSUPPORTED,
                "nsa_sparse_fwd: h/h_kv must be <= 16 or a multiple of 16");
  } else {
    NSA_REQUIRE(shape->d <= 256, NSA_ERR_UNSUPPORTED, "nsa_sparse_fwd: fp32 needs d <= 256");
    NSA_REQUIRE((int64_t)S * block_size <= 4096, NSA_ERR_UNSUPPORTED, "nsa_sparse_fwd: fp32 needs S*block_size <= 4096");
  }
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(block_indices);
  NSA_PTR(o);
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(NSA_ERR_INVALID, "nsa_sparse_fwd: lse misaligned");
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  return cuda_status(launch_sparse_fwd(s, q, k, v, block_indices, S, block_size, shape->h, shape->h_kv, shape->d,
                                       shape->dtype, scale, o, lse, stream),
                     "nsa_sparse_fwd");
}

static nsa_status dense_common(const nsa_shape* shape, Seqs* s, const char* fn) {
  if (nsa_status st = make_seqs(shape, s, fn)) return st;
  const int r = shape->h / shape->h_kv;
  NSA_REQUIRE(shape->dtype == NSA_BF16, NSA_ERR_UNSUPPORTED, "%s: bf16 only", fn);
  NSA_REQUIRE(shape->d == 64 || shape->d == 128, NSA_ERR_UNSUPPORTED, "%s: d must be 64 or 128", fn);
  NSA_REQUIRE((r <= 16 && 16 % r == 0) || (r % 16 == 0 && r <= 128), NSA_ERR_UNSUPPORTED,
              "%s: h/h_kv must divide 16 or be a multiple of 16 up to 128", fn);
  return NSA_OK;
}

// Scratch of the tensor-core dense branches: V transposed per kv-head ([h_kv, d, rows
// padded to 64]), the K-major B operand of the PV product.  Rows: the caller's value rows
// (tokens), or for the compressed branch a bound on the packed compressed rows.
static int64_t cmp_rows_bound(const Seqs& s, int kernel, int stride) {
  return s.cu ? s.tokens / stride + s.n_seqs : (int64_t)s.n_seqs * num_cmp_host(s.T, kernel, stride);
}

size_t nsa_cmp_attn_fwd_workspace_size(const nsa_shape* shape, int kernel, int stride) {
  Seqs s;
  if (make_seqs(shape, &s, __func__) != NSA_OK || kernel <= 0 || stride <= 0) return 0;
  if (shape->dtype != NSA_BF16 || !dense_tc_supported(shape->h, shape->h_kv, shape->d)) return 0;
  return align256((size_t)tc_vt_pad(cmp_rows_bound(s, kernel, stride)) * shape->h_kv * shape->d * 2);
}

size_t nsa_swa_fwd_workspace_size(const nsa_shape* shape) {
  Seqs s;
  if (make_seqs(shape, &s, __func__) != NSA_OK) return 0;
  if (shape->dtype != NSA_BF16 || !dense_tc_supported(shape->h, shape->h_kv, shape->d)) return 0;
  return align256((size_t)tc_vt_pad(s.tokens) * shape->h_kv * shape->d * 2);
}

nsa_status nsa_cmp_attn_fwd(const nsa_shape* shape, const void* q, const void* k_cmp,
                            const void* v_cmp, int kernel, int stride, float scale, void* o, float* lse,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = dense_common(shape, &s, __func__)) return st;
  NSA_REQUIRE(kernel > 0 && stride > 0, NSA_ERR_INVALID, "nsa_cmp_attn_fwd: kernel and stride must be positive");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(o);
  if (s.max_len >= kernel) {
    NSA_PTR(k_cmp);
    NSA_PTR(v_cmp);
  }
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(NSA_ERR_INVALID, "nsa_cmp_attn_fwd: lse misaligned");
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  const size_t need = nsa_cmp_attn_fwd_workspace_size(shape, kernel, stride);
  // d 64, a group size the tensor-core kernel does not take, or no sequence with a
  // compressed key (k_cmp / v_cmp may then be NULL): the mma.sync kernel
  if (need == 0 || s.max_len < kernel)
    return cuda_status(launch_dense_attn(0, s, q, k_cmp, v_cmp, shape->h, shape->h_kv, shape->d, kernel, stride, 0,
                                         scale, o, lse, stream),
                       "nsa_cmp_attn_fwd");
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_cmp_attn_fwd: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= need, NSA_ERR_INVALID, "nsa_cmp_attn_fwd: workspace %zu < %zu bytes", workspace_bytes,
              need);
  const int64_t rows = cmp_rows_bound(s, kernel, stride);
  cudaError_t e = launch_transpose_v(s, v_cmp, workspace, rows, shape->h_kv, true, kernel, stride, stream);
  if (e == cudaSuccess)  // the caller's k_cmp holds exactly the packed compressed rows: tiles past them are bounds-checked
    e = launch_dense_attn_tc(0, s, q, k_cmp, workspace, rows, shape->h, shape->h_kv, kernel, stride, 0, scale, o, lse,
                             nullptr, 0, stream, -1);
  return cuda_status(e, "nsa_cmp_attn_fwd");
}

nsa_status nsa_swa_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v, int window,
                       float scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = dense_common(shape, &s, __func__)) return st;
  NSA_REQUIRE(window >= 1, NSA_ERR_INVALID, "nsa_swa_fwd: window must be >= 1");
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(o);
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(NSA_ERR_INVALID, "nsa_swa_fwd: lse misaligned");
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  const size_t need = nsa_swa_fwd_workspace_size(shape);
  if (need == 0)  // d 64 or a group size the tensor-core kernel does not take
    return cuda_status(launch_dense_attn(1, s, q, k, v, shape->h, shape->h_kv, shape->d, 0, 1, window, scale, o, lse,
                                         stream),
                       "nsa_swa_fwd");
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_swa_fwd: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= need, NSA_ERR_INVALID, "nsa_swa_fwd: workspace %zu < %zu bytes", workspace_bytes,
              need);
  cudaError_t e = launch_transpose_v(s, v, workspace, s.tokens, shape->h_kv, false, 0, 1, stream);
  if (e == cudaSuccess)
    e = launch_dense_attn_tc(1, s, q, k, workspace, s.tokens, shape->h, shape->h_kv, 0, 1, window, scale, o, lse,
                             nullptr, 0, stream);
  return cuda_status(e, "nsa_swa_fwd");
}

nsa_status nsa_gate_combine(int64_t tokens, int h, int d, const void* o_cmp, const void* o_slc,
                            const void* o_swa, const float* gate_logits, void* o, cudaStream_t stream) {
  NSA_RANGE();
  NSA_REQUIRE(tokens >= 0 && h > 0 && d > 0, NSA_ERR_INVALID, "nsa_gate_combine: bad sizes");
  NSA_REQUIRE(d % 8 == 0, NSA_ERR_UNSUPPORTED, "nsa_gate_combine: d must be a multiple of 8");
  if (tokens == 0) return NSA_OK;
  NSA_PTR(o_cmp);
  NSA_PTR(o_slc);
  NSA_PTR(o_swa);
  NSA_PTR(gate_logits);
  NSA_PTR(o);
  return cuda_status(launch_gate_combine(tokens, h, d, o_cmp, o_slc, o_swa, gate_logits, o, stream),
                     "nsa_gate_combine");
}

// The address a kernel uses for a K/V cache that may sit in device memory or in
// page-locked host memory.  [NOSA-Parts] "core idea": the whole KV cache is offloaded to
// host memory and only the chosen blocks travel back to the GPU; on a Grace-Blackwell
// node host memory is reachable from the SMs over the coherent chip-to-chip link, so the
// decode kernel's gather reads the chosen blocks straight from it into shared memory.
// Pageable host memory is rejected: only allocations known to the CUDA runtime
// (cudaHostAlloc, cudaHostRegister) have a device address here.
static nsa_status gpu_address(const void* p, const void** out, const char* what) {
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(NSA_ERR_INVALID, "nsa_sparse_decode: %s: pointer query failed (%s)", what, cudaGetErrorString(e));
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return NSA_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
    *out = a.devicePointer;
    return NSA_OK;
  }
  return fail(NSA_ERR_INVALID, "nsa_sparse_decode: %s must be device memory or page-locked host memory", what);
}

size_t nsa_sparse_decode_workspace_size(int batch, int max_len, int h, int h_kv, int d, int kernel,
                                        int stride, int block_size, int k) {
  if (batch <= 0 || max_len <= 0 || h <= 0 || h_kv <= 0 || h % h_kv || k <= 0 || kernel <= 0 || stride <= 0)
    return 0;
  return decode_layout(batch, max_len, h, h_kv, d, kernel, stride, block_size, k).total;
}

static nsa_status decode_call(int batch, const int32_t* seqlens, int max_len, int h, int h_kv, int d, const void* q,
                              const void* k_cache, const void* v_cache, const void* k_cmp_cache, int kernel,
                              int stride, int block_size, int n_init, int n_local, int k, float scale,
                              int32_t* idx_out, void* o, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                              const float* cis_cache, const float* cis_block, int cis_nb_stride, int qk_select) {
  if (nsa_status st = decode_check_sizes(batch, max_len, h, h_kv, d, kernel, stride, block_size, n_init, n_local, k))
    return st;
  if (batch == 0) return NSA_OK;
  NSA_PTR(seqlens);
  NSA_PTR(q);
  NSA_PTR(k_cache);
  NSA_PTR(v_cache);
  NSA_PTR(o);
  if (max_len >= kernel) NSA_PTR(k_cmp_cache);
  if (idx_out) NSA_PTR(idx_out);
  const DecodeLayout l = decode_layout(batch, max_len, h, h_kv, d, kernel, stride, block_size, k);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_sparse_decode: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= l.total, NSA_ERR_INVALID, "nsa_sparse_decode: workspace %zu < %zu bytes",
              workspace_bytes, l.total);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  DecodeArgs a{};
  a.batch = batch;
  a.max_len = max_len;
  a.h = h;
  a.hkv = h_kv;
  a.d = d;
  a.kernel = kernel;
  a.stride = stride;
  a.block_size = block_size;
  a.n_init = n_init;
  a.n_local = n_local;
  a.k = k;
  a.scale = scale > 0.f ? scale : 1.f / sqrtf((float)d);
  a.seqlens = seqlens;
  a.q = q;
  nsa_status ps = gpu_address(k_cache, &a.k_cache, "k_cache");
  if (ps == NSA_OK) ps = gpu_address(v_cache, &a.v_cache, "v_cache");
  if (ps == NSA_OK && max_len >= kernel) ps = gpu_address(k_cmp_cache, &a.kc_cache, "k_cmp_cache");
  if (ps != NSA_OK) return ps;
  a.idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(w + l.idx);
  a.o = o;
  a.z = reinterpret_cast<float*>(w + l.z);
  a.unit_ml = reinterpret_cast<float*>(w + l.unit_ml);
  a.part_o = reinterpret_cast<float*>(w + l.part_o);
  a.part_ml = reinterpret_cast<float*>(w + l.part_ml);
  a.counters = reinterpret_cast<int*>(w + l.counters);
  a.n_split = l.n_split;
  if (cis_cache) {
    const void* cp = nullptr;
    if (nsa_status st = gpu_address(cis_cache, &cp, "cis_cache")) return st;
    a.cis = static_cast<const float*>(cp);
    a.cis_block = cis_block;
    a.cis_nb_stride = cis_nb_stride;
    a.qk = qk_select;
  }
  return cuda_status(launch_decode(a, stream), "nsa_sparse_decode");
}

nsa_status nsa_sparse_decode(int batch, const int32_t* seqlens, int max_len, int h, int h_kv, int d,
                             const void* q, const void* k_cache, const void* v_cache,
                             const void* k_cmp_cache, int kernel, int stride, int block_size,
                             int n_init, int n_local, int k, float scale, int32_t* idx_out, void* o,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  return decode_call(batch, seqlens, max_len, h, h_kv, d, q, k_cache, v_cache, k_cmp_cache, kernel, stride,
                     block_size, n_init, n_local, k, scale, idx_out, o, workspace, workspace_bytes, stream, nullptr,
                     nullptr, 0, 0);
}

nsa_status nsa_sparse_decode_cis(int batch, const int32_t* seqlens, int max_len, int h, int h_kv, int d,
                                 const void* q, const void* k_cache, const void* v_cache, const void* k_cmp_cache,
                                 const float* cis_cache, const float* cis_block_scores, int nb_stride,
                                 int qk_select, int kernel, int stride, int block_size, int n_init, int n_local,
                                 int k, float scale, int32_t* idx_out, void* o, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  NSA_REQUIRE(cis_cache != nullptr && (reinterpret_cast<uintptr_t>(cis_cache) & 3u) == 0, NSA_ERR_INVALID,
              "nsa_sparse_decode_cis: cis_cache must be non-null and 4-byte aligned");
  if (cis_block_scores) {
    NSA_REQUIRE((reinterpret_cast<uintptr_t>(cis_block_scores) & 3u) == 0, NSA_ERR_INVALID,
                "nsa_sparse_decode_cis: cis_block_scores misaligned");
    NSA_REQUIRE(qk_select >= k && qk_select <= 64, NSA_ERR_UNSUPPORTED,
                "nsa_sparse_decode_cis: needs k <= qk_select <= 64");
    NSA_REQUIRE(nb_stride >= (max_len + block_size - 1) / (block_size > 0 ? block_size : 1), NSA_ERR_INVALID,
                "nsa_sparse_decode_cis: nb_stride < blocks of max_len");
  }
  return decode_call(batch, seqlens, max_len, h, h_kv, d, q, k_cache, v_cache, k_cmp_cache, kernel, stride,
                     block_size, n_init, n_local, k, scale, idx_out, o, workspace, workspace_bytes, stream, cis_cache,
                     cis_block_scores, nb_stride, qk_select);
}

// Layer workspace: compressed K and V, V^T of the compressed and of the full values
// (K-major operands of the tensor-core branches), the compressed and sliding branch
// outputs, the compressed normaliser, the block scores and (when idx_out is NULL) the
// block lists.
struct LayerLayout {
  size_t kc, vc, vtc, vt, o_cmp, o_swa, lse, scores, idx, total;
  int64_t ncr;
  int nb_stride;
};

static LayerLayout layer_layout(const Seqs& s, int h, int hkv, int d, int esz, int kernel, int stride,
                                int block_size, int S) {
  LayerLayout l{};
  // packed compressed rows: sum of n_c(L_i) <= tokens/stride + n_seqs
  const int64_t ncr = s.cu ? s.tokens / stride + s.n_seqs : (int64_t)s.n_seqs * num_cmp_host(s.T, kernel, stride);
  l.nb_stride = ((s.max_len + block_size - 1) / block_size + 3) / 4 * 4;
  if (l.nb_stride == 0) l.nb_stride = 4;
  size_t off = 0;
  l.kc = off;
  off = align256(off + (size_t)ncr * hkv * d * esz);
  l.vc = off;
  off = align256(off + (size_t)ncr * hkv * d * esz);
  l.ncr = ncr;
  l.vtc = off;
  off = align256(off + (size_t)tc_vt_pad(ncr) * hkv * d * esz);
  l.vt = off;
  off = align256(off + (size_t)tc_vt_pad(s.tokens) * hkv * d * esz);
  l.o_cmp = off;
  off = align256(off + (size_t)s.tokens * h * d * esz);
  l.o_swa = off;
  off = align256(off + (size_t)s.tokens * h * d * esz);
  l.lse = off;
  off = align256(off + (size_t)s.tokens * h * 4);
  l.scores = off;
  off = align256(off + (size_t)s.tokens * hkv * l.nb_stride * 4);
  l.idx = off;
  off = align256(off + (size_t)s.tokens * hkv * S * 4);
  l.total = off;
  return l;
}

size_t nsa_layer_fwd_workspace_size(const nsa_shape* shape, int kernel, int stride, int block_size, int S) {
  Seqs s;
  if (make_seqs(shape, &s, __func__) != NSA_OK || kernel <= 0 || stride <= 0 || block_size <= 0 || S <= 0) return 0;
  return layer_layout(s, shape->h, shape->h_kv, shape->d, shape->dtype == NSA_BF16 ? 2 : 4, kernel, stride,
                      block_size, S)
      .total;
}

// Layer forward; with `saved`, the compressed keys and values, each branch's output and
// normaliser and the block lists go to the caller's buffers for nsa_layer_bwd.
static nsa_status layer_forward(const nsa_shape* shape, const void* q, const void* k, const void* v,
                                const float* gate_logits, int kernel, int stride, int block_size, int S, int n_init,
                                int n_local, int window, float scale, void* o, int32_t* idx_out,
                                const nsa_layer_saved* saved, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream, const char* fn) {
  Seqs s;
  if (nsa_status st = dense_common(shape, &s, fn)) return st;
  NSA_REQUIRE(kernel == 32 && stride == 16 && block_size == 64, NSA_ERR_UNSUPPORTED,
              "%s: supports kernel 32, stride 16, block_size 64", fn);
  NSA_REQUIRE(pow2_le16(shape->h / shape->h_kv), NSA_ERR_UNSUPPORTED, "%s: h/h_kv must be 1, 2, 4, 8 or 16", fn);
  NSA_REQUIRE(S >= 1 && S <= 64, NSA_ERR_UNSUPPORTED, "%s: S must be in [1, 64]", fn);
  NSA_REQUIRE(window >= 1 && n_init >= 0 && n_local >= 0, NSA_ERR_INVALID, "%s: bad window/n_init/n_local", fn);
  if (s.tokens == 0) return NSA_OK;
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(gate_logits);
  NSA_PTR(o);
  if (idx_out) NSA_PTR(idx_out);
  if (saved) {
    NSA_PTR(saved->k_cmp);
    NSA_PTR(saved->v_cmp);
    NSA_PTR(saved->o_cmp);
    NSA_PTR(saved->o_slc);
    NSA_PTR(saved->o_swa);
    NSA_PTR(saved->lse_cmp);
    NSA_PTR(saved->lse_slc);
    NSA_PTR(saved->lse_swa);
    NSA_PTR(saved->idx);
  }
  const LayerLayout l = layer_layout(s, shape->h, shape->h_kv, shape->d, 2, kernel, stride, block_size, S);
  NSA_REQUIRE(l.nb_stride <= 2048, NSA_ERR_UNSUPPORTED, "%s: sequences longer than 131072 tokens", fn);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "%s: workspace must be non-null and 256-byte aligned", fn);
  NSA_REQUIRE(workspace_bytes >= l.total, NSA_ERR_INVALID, "%s: workspace %zu < %zu bytes", fn, workspace_bytes,
              l.total);
  if (scale <= 0.f) scale = 1.f / sqrtf((float)shape->d);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  void* kc = saved ? saved->k_cmp : w + l.kc;
  void* vc = saved ? saved->v_cmp : w + l.vc;
  void* o_cmp = saved ? saved->o_cmp : w + l.o_cmp;
  void* o_swa = saved ? saved->o_swa : w + l.o_swa;
  void* o_slc = saved ? saved->o_slc : o;  // without saved, the selected branch writes o and the gate runs in place
  float* lse = saved ? saved->lse_cmp : reinterpret_cast<float*>(w + l.lse);
  float* scores = reinterpret_cast<float*>(w + l.scores);
  int32_t* idx = saved ? saved->idx : idx_out ? idx_out : reinterpret_cast<int32_t*>(w + l.idx);
  const int h = shape->h, hkv = shape->h_kv, d = shape->d;
  cudaError_t e;
  if ((e = launch_compress(s, k, kc, hkv, d, kBF16, kernel, stride, stream))) return cuda_status(e, "layer/compress k");
  if ((e = launch_compress(s, v, vc, hkv, d, kBF16, kernel, stride, stream))) return cuda_status(e, "layer/compress v");
  const bool tc = d == 128;
  void* vtc = w + l.vtc;
  void* vt = w + l.vt;
  if (tc) {
    if ((e = launch_transpose_v(s, vc, vtc, l.ncr, hkv, true, kernel, stride, stream)))
      return cuda_status(e, "layer/transpose compressed v");
    if ((e = launch_transpose_v(s, v, vt, s.tokens, hkv, false, kernel, stride, stream)))
      return cuda_status(e, "layer/transpose v");
    // the compressed branch also writes the block scores (second pass over its keys)
    e = launch_dense_attn_tc(0, s, q, kc, vtc, l.ncr, h, hkv, kernel, stride, 0, scale, o_cmp,
                             saved ? saved->lse_cmp : nullptr, scores, l.nb_stride, stream);
    if (e) return cuda_status(e, "layer/compressed branch and block scores");
  } else {
    e = launch_dense_attn(0, s, q, kc, vc, h, hkv, d, kernel, stride, 0, scale, o_cmp, lse, stream);
    if (e) return cuda_status(e, "layer/compressed branch");
    if ((e = launch_scores_pool(s, q, kc, h, hkv, d, scale, lse, scores, l.nb_stride, stream)))
      return cuda_status(e, "layer/block scores");
  }
  if ((e = launch_topk(s, scores, l.nb_stride, hkv, block_size, n_init, n_local, S, idx, stream)))
    return cuda_status(e, "layer/top-k");
  if (saved && idx_out && (e = cudaMemcpyAsync(idx_out, idx, (size_t)s.tokens * hkv * S * 4, cudaMemcpyDeviceToDevice,
                                                stream)))
    return cuda_status(e, "layer/copy block lists");
  if ((e = launch_sparse_fwd(s, q, k, v, idx, S, block_size, h, hkv, d, kBF16, scale, o_slc,
                             saved ? saved->lse_slc : nullptr, stream)))
    return cuda_status(e, "layer/selected branch");
  e = tc ? launch_dense_attn_tc(1, s, q, k, vt, s.tokens, h, hkv, kernel, stride, window, scale, o_swa,
                                 saved ? saved->lse_swa : nullptr, nullptr, 0, stream)
         : launch_dense_attn(1, s, q, k, v, h, hkv, d, kernel, stride, window, scale, o_swa,
                             saved ? saved->lse_swa : nullptr, stream);
  if (e) return cuda_status(e, "layer/sliding branch");
  return cuda_status(launch_gate_combine(s.tokens, h, d, o_cmp, o_slc, o_swa, gate_logits, o, stream),
                     "layer/gate combine");
}

nsa_status nsa_layer_fwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                         const float* gate_logits, int kernel, int stride, int block_size, int S,
                         int n_init, int n_local, int window, float scale, void* o, int32_t* idx_out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  return layer_forward(shape, q, k, v, gate_logits, kernel, stride, block_size, S, n_init, n_local, window, scale, o,
                       idx_out, nullptr, workspace, workspace_bytes, stream, __func__);
}

nsa_status nsa_layer_fwd_train(const nsa_shape* shape, const void* q, const void* k, const void* v,
                               const float* gate_logits, int kernel, int stride, int block_size, int S, int n_init,
                               int n_local, int window, float scale, void* o, const nsa_layer_saved* saved,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  NSA_REQUIRE(saved != nullptr, NSA_ERR_INVALID, "nsa_layer_fwd_train: saved is NULL");
  return layer_forward(shape, q, k, v, gate_logits, kernel, stride, block_size, S, n_init, n_local, window, scale, o,
                       nullptr, saved, workspace, workspace_bytes, stream, __func__);
}

// Layer backward workspace: the three branch gradients of dO, each branch's dq, dk, dv,
// the compressed-key gradients, and one branch-backward scratch (used in turn).
struct LayerBwdLayout {
  size_t d_br, dq3, dk3, dv3, dkc, dvc, scratch, total;
};

static LayerBwdLayout layer_bwd_layout(const Seqs& s, int h, int hkv, int d, int kernel, int stride, int window,
                                       int S) {
  LayerBwdLayout l{};
  const int64_t ncr = s.cu ? s.tokens / stride + s.n_seqs : (int64_t)s.n_seqs * num_cmp_host(s.T, kernel, stride);
  const size_t qsz = (size_t)s.tokens * h * d * 2, ksz = (size_t)s.tokens * hkv * d * 2;
  size_t off = 0;
  l.d_br = off;
  off = align256(off + 3 * qsz);
  l.dq3 = off;
  off = align256(off + 3 * qsz);
  l.dk3 = off;
  off = align256(off + 3 * ksz);
  l.dv3 = off;
  off = align256(off + 3 * ksz);
  l.dkc = off;
  off = align256(off + (size_t)ncr * hkv * d * 2);
  l.dvc = off;
  off = align256(off + (size_t)ncr * hkv * d * 2);
  l.scratch = off;
  size_t sc = sparse_bwd_workspace_bytes(s, h, hkv, S);
  sc = std::max(sc, cmp_attn_bwd_workspace_bytes(s, h, hkv, kernel, stride));
  sc = std::max(sc, swa_bwd_workspace_bytes(s, h, hkv, window));
  l.total = align256(off + sc);
  return l;
}

static nsa_status check_layer_bwd(const nsa_shape* shape, int kernel, int stride, int block_size, int S, int window,
                                  Seqs* s, const char* fn) {
  if (nsa_status st = make_seqs(shape, s, fn)) return st;
  NSA_REQUIRE(shape->dtype == NSA_BF16 && shape->d == 128, NSA_ERR_UNSUPPORTED, "%s: bf16 and d 128 only", fn);
  NSA_REQUIRE(kernel == 32 && stride == 16 && block_size == 64, NSA_ERR_UNSUPPORTED,
              "%s: supports kernel 32, stride 16, block_size 64", fn);
  NSA_REQUIRE(pow2_le16(shape->h / shape->h_kv), NSA_ERR_UNSUPPORTED, "%s: h/h_kv must be 1, 2, 4, 8 or 16", fn);
  NSA_REQUIRE(S >= 1 && S <= 64, NSA_ERR_UNSUPPORTED, "%s: S must be in [1, 64]", fn);
  NSA_REQUIRE(window >= 1 && window <= 1984, NSA_ERR_UNSUPPORTED, "%s: window must be in [1, 1984]", fn);
  NSA_REQUIRE(num_cmp_host(s->max_len, kernel, stride) <= 4096, NSA_ERR_UNSUPPORTED,
              "%s: at most 4096 compressed keys per sequence", fn);
  return NSA_OK;
}

size_t nsa_layer_bwd_workspace_size(const nsa_shape* shape, int kernel, int stride, int block_size, int S,
                                    int window) {
  Seqs s;
  if (check_layer_bwd(shape, kernel, stride, block_size, S, window, &s, "nsa_layer_bwd_workspace_size") != NSA_OK)
    return 0;
  if (s.tokens == 0) return 0;
  return layer_bwd_layout(s, shape->h, shape->h_kv, shape->d, kernel, stride, window, S).total;
}

nsa_status nsa_layer_bwd(const nsa_shape* shape, const void* q, const void* k, const void* v,
                         const float* gate_logits, int kernel, int stride, int block_size, int S, int window,
                         float scale, const nsa_layer_saved* saved, const void* d_o, void* dq, void* dk, void* dv,
                         float* d_gate_logits, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NSA_RANGE();
  Seqs s;
  if (nsa_status st = check_layer_bwd(shape, kernel, stride, block_size, S, window, &s, __func__)) return st;
  if (s.tokens == 0) return NSA_OK;
  NSA_REQUIRE(saved != nullptr, NSA_ERR_INVALID, "nsa_layer_bwd: saved is NULL");
  NSA_PTR(q);
  NSA_PTR(k);
  NSA_PTR(v);
  NSA_PTR(gate_logits);
  NSA_PTR(d_o);
  NSA_PTR(dq);
  NSA_PTR(dk);
  NSA_PTR(dv);
  NSA_PTR(d_gate_logits);
  NSA_PTR(saved->k_cmp);
  NSA_PTR(saved->v_cmp);
  NSA_PTR(saved->o_cmp);
  NSA_PTR(saved->o_slc);
  NSA_PTR(saved->o_swa);
  NSA_PTR(saved->lse_cmp);
  NSA_PTR(saved->lse_slc);
  NSA_PTR(saved->lse_swa);
  NSA_PTR(saved->idx);
  const int h = shape->h, hkv = shape->h_kv, d = shape->d;
  const LayerBwdLayout l = layer_bwd_layout(s, h, hkv, d, kernel, stride, window, S);
  NSA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, NSA_ERR_INVALID,
              "nsa_layer_bwd: workspace must be non-null and 256-byte aligned");
  NSA_REQUIRE(workspace_bytes >= l.total, NSA_ERR_INVALID, "nsa_layer_bwd: workspace %zu < %zu bytes",
              workspace_bytes, l.total);
  if (scale <= 0.f) scale = 1.f / sqrtf((float)d);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t qsz = (size_t)s.tokens * h * d * 2, ksz = (size_t)s.tokens * hkv * d * 2;
  uint8_t* d_cmp = w + l.d_br;
  uint8_t* d_slc = d_cmp + qsz;
  uint8_t* d_swa = d_slc + qsz;
  uint8_t* dq3 = w + l.dq3;
  uint8_t* dk3 = w + l.dk3;
  uint8_t* dv3 = w + l.dv3;
  void* scratch = w + l.scratch;
  cudaError_t e;
  if ((e = launch_gate_bwd(s.tokens * h, d, d_o, saved->o_cmp, saved->o_slc, saved->o_swa, gate_logits, d_cmp, d_slc,
                           d_swa, d_gate_logits, stream)))
    return cuda_status(e, "layer bwd/gate");
  if ((e = launch_cmp_attn_bwd(s, q, saved->k_cmp, saved->v_cmp, h, hkv, kernel, stride, scale, saved->o_cmp,
                               saved->lse_cmp, d_cmp, dq3, w + l.dkc, w + l.dvc, scratch, stream)))
    return cuda_status(e, "layer bwd/compressed branch");
  if ((e = launch_compress_bwd(s, w + l.dkc, hkv, d, kernel, stride, dk3, stream)) ||
      (e = launch_compress_bwd(s, w + l.dvc, hkv, d, kernel, stride, dv3, stream)))
    return cuda_status(e, "layer bwd/pooling");
  if ((e = launch_sparse_bwd(s, q, k, v, saved->idx, S, h, hkv, scale, saved->o_slc, saved->lse_slc, d_slc,
                             dq3 + qsz, dk3 + ksz, dv3 + ksz, scratch, stream)))
    return cuda_status(e, "layer bwd/selected branch");
  if ((e = launch_swa_bwd(s, q, k, v, h, hkv, window, scale, saved->o_swa, saved->lse_swa, d_swa, dq3 + 2 * qsz,
                          dk3 + 2 * ksz, dv3 + 2 * ksz, scratch, stream)))
    return cuda_status(e, "layer bwd/sliding branch");
  if ((e = launch_add3(dq3, dq3 + qsz, dq3 + 2 * qsz, dq, s.tokens * h * d, stream)) ||
      (e = launch_add3(dk3, dk3 + ksz, dk3 + 2 * ksz, dk, s.tokens * hkv * d, stream)) ||
      (e = launch_add3(dv3, dv3 + ksz, dv3 + 2 * ksz, dv, s.tokens * hkv * d, stream)))
    return cuda_status(e, "layer bwd/sum over branches");
  return NSA_OK;
}

}  // extern "C"
