// Block scores from the compressed keys, and top-k block selection.
//
// [NSA-Triton] "DeepSeek NSA ... with Triton", sec. 1.1: selection reuses the scores of
// the compressed attention.  [NOSA-Parts] "NOSA-1B core components", core component 3,
// stage 1: a light attention of the query against the compressed keys gives block-level
// scores.  [NOSA-Triton] mechanisms 2 and 3: a window of scores is summed and divided
// by the number of valid entries (validity from the sequence length).
//
// GB300 design of the scorer.  A CTA takes a run of consecutive query tokens of one
// sequence and one kv-group; its 8 warps hold 16 (token, head) rows each as mma.sync A
// fragments, and every 64-key tile of compressed keys is staged once in shared memory
// (cp.async, double buffered) for all of them.  Pass 1 runs the online max/sum of each
// row (skipped when the caller passes the normaliser); pass 2 recomputes the scores,
// turns them into probabilities, pools the three windows of each 64-token block inside
// the quad of lanes that holds them, sums the heads of a group with lane shuffles and
// writes one fp32 score per (token, kv-head, block).  Nothing but the block scores
// touches HBM.
#include "launch.h"
#include "topk.cuh"

namespace nsa {

constexpr int kSPWarps = 8;
constexpr int kCmpKernel = 32, kCmpStride = 16;

struct ScoresParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const float* lse_in;
  float* scores;
  Seqs seqs;
  int h, hkv, nb_stride;
  float scale_log2;
};

template <int D, int R, bool HAS_LSE>
__global__ void __launch_bounds__(kSPWarps * 32) scores_pool_kernel(const ScoresParams p) {
  constexpr int TPW = 16 / R;
  constexpr int TPC = kSPWarps * TPW;
  constexpr int TILE = 64;
  constexpr int TILE_BYTES = TILE * D * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const int sq = blockIdx.y, g = blockIdx.z;
  const int L = seq_len(p.seqs, sq);
  const int n_tok_tiles = (L + TPC - 1) / TPC;
  const int tile = n_tok_tiles - 1 - (int)blockIdx.x;  // longest rows first
  if (tile < 0) return;
  const int t0 = tile * TPC;
  const int64_t start = seq_start(p.seqs, sq);
  const int n_c = num_cmp(L, kCmpKernel, kCmpStride);
  const int64_t kc0 = cmp_offset(p.seqs, sq, kCmpKernel, kCmpStride);
  const int t_last = min(t0 + TPC, L) - 1;
  const int n_kt = (num_causal_cmp(t_last, n_c, kCmpKernel, kCmpStride) + TILE - 1) / TILE;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rlo = lane >> 2, rhi = rlo + 8;
  const int t_lo = t0 + warp * TPW + rlo / R, t_hi = t0 + warp * TPW + rhi / R;
  const int hd_lo = rlo % R, hd_hi = rhi % R;
  const bool v_lo = t_lo < L, v_hi = t_hi < L;
  const int nca_lo = v_lo ? num_causal_cmp(t_lo, n_c, kCmpKernel, kCmpStride) : 0;
  const int nca_hi = v_hi ? num_causal_cmp(t_hi, n_c, kCmpKernel, kCmpStride) : 0;

  uint32_t qa[D / 16][4];
  load_a_frags<D>(qa, v_lo ? p.q + ((start + t_lo) * p.h + g * R + hd_lo) * D : nullptr,
                  v_hi ? p.q + ((start + t_hi) * p.h + g * R + hd_hi) * D : nullptr, lane);

  const uint32_t sbase = smem_u32(smem);
  const int64_t row_stride = (int64_t)p.hkv * D;
  const __nv_bfloat16* kbase = p.kc + (kc0 * p.hkv + g) * D;
  auto load = [&](int kt) {
    load_tile_async<D, TILE, kSPWarps * 32>(sbase + (kt & 1) * TILE_BYTES, threadIdx.x, p.kc,
                                            [&](int row) -> const __nv_bfloat16* {
                                              const int c = kt * TILE + row;
                                              return c < n_c ? kbase + c * row_stride : nullptr;
                                            });
  };
  auto scores_tile = [&](int kt, float (*s)[4]) {
    const uint32_t b = sbase + (kt & 1) * TILE_BYTES;
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int k16 = 0; k16 < 4; ++k16) qk_16keys<D>(&s[2 * k16], qa, b, k16 * 16, lane);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = kt * TILE + nt * 8 + (lane & 3) * 2 + (j & 1);
        const int lim = j < 2 ? nca_lo : nca_hi;
        s[nt][j] = c < lim ? s[nt][j] * p.scale_log2 : kNegInf;
      }
  };

  float lse_lo, lse_hi;  // base-2 normalisers
  if (HAS_LSE) {
    lse_lo = v_lo ? p.lse_in[(start + t_lo) * p.h + g * R + hd_lo] * kLog2e : kNegInf;
    lse_hi = v_hi ? p.lse_in[(start + t_hi) * p.h + g * R + hd_hi] * kLog2e : kNegInf;
  } else {
    float m_lo = kNegInf, m_hi = kNegInf, l_lo = 0.f, l_hi = 0.f;
    if (n_kt > 0) load(0);
    cp_async_commit();
    for (int kt = 0; kt < n_kt; ++kt) {
      if (kt + 1 < n_kt) load(kt + 1);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      float s[8][4];
      scores_tile(kt, s);
      float x_lo = kNegInf, x_hi = kNegInf;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        x_lo = fmaxf(x_lo, fmaxf(s[nt][0], s[nt][1]));
        x_hi = fmaxf(x_hi, fmaxf(s[nt][2], s[nt][3]));
      }
      const float mn_lo = fmaxf(m_lo, quad_max(x_lo)), mn_hi = fmaxf(m_hi, quad_max(x_hi));
      const float mu_lo = mn_lo == kNegInf ? 0.f : mn_lo, mu_hi = mn_hi == kNegInf ? 0.f : mn_hi;
      float a_lo = 0.f, a_hi = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        a_lo += ex2(s[nt][0] - mu_lo) + ex2(s[nt][1] - mu_lo);
        a_hi += ex2(s[nt][2] - mu_hi) + ex2(s[nt][3] - mu_hi);
      }
      l_lo = l_lo * ex2(m_lo - mu_lo) + a_lo;
      l_hi = l_hi * ex2(m_hi - mu_hi) + a_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
      __syncthreads();
    }
    l_lo = quad_sum(l_lo);
    l_hi = quad_sum(l_hi);
    lse_lo = l_lo > 0.f ? m_lo + __log2f(l_lo) : kNegInf;
    lse_hi = l_hi > 0.f ? m_hi + __log2f(l_hi) : kNegInf;
  }
  const float sub_lo = lse_lo == kNegInf ? 0.f : lse_lo;
  const float sub_hi = lse_hi == kNegInf ? 0.f : lse_hi;

  const int q4 = lane & 3;
  const bool writer = (q4 & 1) == 0 && (R == 16 ? rlo == 0 : (rlo % R) == 0);
  float* out_lo = p.scores + ((start + t_lo) * p.hkv + g) * p.nb_stride;
  float* out_hi = p.scores + ((start + t_hi) * p.hkv + g) * p.nb_stride;

  if (n_kt > 0) load(0);
  cp_async_commit();
  for (int kt = 0; kt < n_kt; ++kt) {
    if (kt + 1 < n_kt) load(kt + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    float s[8][4];
    scores_tile(kt, s);
    float b_lo[8], b_hi[8];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      // keys nt*8 + 2*q4 + {0,1}: windows 4j, 4j+1, 4j+2 of blocks 2nt (q4 0,1) and 2nt+1 (q4 2,3)
      const float p0 = ex2(s[nt][0] - sub_lo), p1 = ex2(s[nt][1] - sub_lo);
      const float p2 = ex2(s[nt][2] - sub_hi), p3 = ex2(s[nt][3] - sub_hi);
      float x = (q4 & 1) ? p0 : p0 + p1;
      float y = (q4 & 1) ? p2 : p2 + p3;
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      y += __shfl_xor_sync(0xffffffffu, y, 1);
      b_lo[nt] = x;
      b_hi[nt] = y;
    }
    // sum over the heads of each token (rows sharing lane bits 2.. of one token)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      if (R == 16) {
        float x = b_lo[nt] + b_hi[nt];
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        b_lo[nt] = x;
      } else {
#pragma unroll
        for (int off = 4; off < 4 * R; off <<= 1) {
          b_lo[nt] += __shfl_xor_sync(0xffffffffu, b_lo[nt], off);
          b_hi[nt] += __shfl_xor_sync(0xffffffffu, b_hi[nt], off);
        }
      }
    }
    if (writer) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int j = kt * 16 + 2 * nt + (q4 >> 1);
        if (j >= p.nb_stride) continue;
        const int c0 = 4 * j;
        const int cnt = (c0 < n_c) + (c0 + 1 < n_c) + (c0 + 2 < n_c);
        const float inv = cnt ? 1.f / (float)cnt : 0.f;
        if (v_lo) out_lo[j] = b_lo[nt] * inv;
        if (R < 16 && v_hi) out_hi[j] = b_hi[nt] * inv;
      }
    }
    __syncthreads();
  }
  // blocks past the last processed tile get no probability mass
  for (int tl = 0; tl < TPW; ++tl) {
    const int t = t0 + warp * TPW + tl;
    if (t >= L) break;
    float* out = p.scores + ((start + t) * p.hkv + g) * p.nb_stride;
    for (int j = n_kt * 16 + lane; j < p.nb_stride; j += 32) out[j] = 0.f;
  }
}

template <int D, int R>
static cudaError_t run_scores(const ScoresParams& p, dim3 grid, cudaStream_t st, bool has_lse) {
  constexpr int bytes = 2 * 64 * D * 2;
  if (has_lse) {
    scores_pool_kernel<D, R, true><<<grid, kSPWarps * 32, bytes, st>>>(p);
  } else {
    scores_pool_kernel<D, R, false><<<grid, kSPWarps * 32, bytes, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_scores_pool(const Seqs& s, const void* q, const void* k_cmp, int h, int hkv, int d,
                               float scale, const float* lse_in, float* scores, int nb_stride,
                               cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  if (k_cmp && scores_tc_supported(h, hkv, d, kCmpKernel, kCmpStride, 64)) {
    // packed compressed rows: exact for the dense layout, an upper bound otherwise
    const int64_t exact = s.cu ? -1 : (int64_t)s.n_seqs * (s.T >= kCmpKernel ? (s.T - kCmpKernel) / kCmpStride + 1 : 0);
    const int64_t bound = s.cu ? s.tokens / kCmpStride + s.n_seqs : exact;
    return launch_scores_tc(s, q, k_cmp, bound, exact, h, hkv, scale, lse_in, scores, nb_stride, st);
  }
  ScoresParams p{};
  p.q = (const __nv_bfloat16*)q;
  p.kc = (const __nv_bfloat16*)k_cmp;
  p.lse_in = lse_in;
  p.scores = scores;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.nb_stride = nb_stride;
  p.scale_log2 = scale * kLog2e;
  const int R = h / hkv;
  const int tpc = kSPWarps * (16 / R);
  dim3 grid((s.max_len + tpc - 1) / tpc, s.n_seqs, hkv);
  const bool hl = lse_in != nullptr;
#define NSA_SCORES_R(DD)                               \
  switch (R) {                                         \
    case 1: return run_scores<DD, 1>(p, grid, st, hl); \
    case 2: return run_scores<DD, 2>(p, grid, st, hl); \
    case 4: return run_scores<DD, 4>(p, grid, st, hl); \
    case 8: return run_scores<DD, 8>(p, grid, st, hl); \
    default: return run_scores<DD, 16>(p, grid, st, hl); \
  }
  if (d == 128) {
    NSA_SCORES_R(128)
  } else {
    NSA_SCORES_R(64)
  }
#undef NSA_SCORES_R
}

// ---------------------------------------------------------------------------
// Top-k selection: one warp per (token, kv-head) row.
template <int NPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ scores, int nb_stride, int32_t* out,
                                                  Seqs s, int hkv, int block_size, int n_init, int n_local,
                                                  int k) {
  __shared__ uint32_t s_key[8][64];
  __shared__ int s_idx[8][64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= s.tokens * hkv) return;
  const int64_t tok = row / hkv;
  const int sq = seq_of_token(s, tok);
  const int t = (int)(tok - seq_start(s, sq));
  warp_topk<NPL>(scores + row * nb_stride, nb_stride, t / block_size, n_init, n_local, k, out + row * k,
                 s_key[warp], s_idx[warp], lane);
}

cudaError_t launch_topk(const Seqs& s, const float* scores, int nb_stride, int hkv, int block_size,
                        int n_init, int n_local, int k, int32_t* idx, cudaStream_t st) {
  const int64_t rows = s.tokens * hkv;
  if (rows == 0) return cudaSuccess;
  dim3 grid((unsigned)((rows + 7) / 8));
  const int npl = (nb_stride + 31) / 32;
#define NSA_TOPK(N)                                                                                        \
  if (npl <= N) {                                                                                          \
    topk_kernel<N><<<grid, 256, 0, st>>>(scores, nb_stride, idx, s, hkv, block_size, n_init, n_local, k); \
    return cudaGetLastError();                                                                             \
  }
  NSA_TOPK(1)
  NSA_TOPK(2)
  NSA_TOPK(4)
  NSA_TOPK(8)
  NSA_TOPK(16)
  NSA_TOPK(32)
  NSA_TOPK(64)
#undef NSA_TOPK
  return cudaErrorInvalidValue;
}

}  // namespace nsa
