// Internal launchers (host side) of the sm_103a kernels.  Arguments are validated by
// the C ABI layer before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"
#include "nsa.h"

namespace nsa {

enum DType { kF32 = 0, kBF16 = 1 };

// Record the message returned by nsa_last_error() for the calling thread.
void set_error(const char* fmt, ...);

// Size checks of the decode step (kernel/stride/block, d, group size, k, max_len), the
// first checks of nsa_sparse_decode; NSA_OK or the status with nsa_last_error() set.
nsa_status decode_check_sizes(int batch, int max_len, int h, int h_kv, int d, int kernel, int stride,
                              int block_size, int n_init, int n_local, int k);

cudaError_t launch_compress(const Seqs& s, const void* k, void* k_cmp, int hkv, int d, int dtype,
                            int kernel, int stride, cudaStream_t st);

cudaError_t launch_scores_pool(const Seqs& s, const void* q, const void* k_cmp, int h, int hkv, int d,
                               float scale, const float* lse_in, float* scores, int nb_stride,
                               cudaStream_t st);

cudaError_t launch_topk(const Seqs& s, const float* scores, int nb_stride, int hkv, int block_size,
                        int n_init, int n_local, int k, int32_t* idx, cudaStream_t st);

// cis (nullable, bf16 path, block 64): per-key weights [tokens, hkv] fp32 (NOSA CIS).
cudaError_t launch_sparse_fwd(const Seqs& s, const void* q, const void* k, const void* v,
                              const int32_t* idx, int S, int block_size, int h, int hkv, int d,
                              int dtype, float scale, void* o, float* lse, cudaStream_t st,
                              const float* cis = nullptr);

// NOSA stage 2 (csrc/nosa.cu): block CIS scores [n_seqs, hkv, nb_stride] from per-key
// CIS [tokens, hkv]; two-stage selection (top qk by attention score, then top k by CIS).
cudaError_t launch_cis_block_scores(const Seqs& s, const float* cis, int hkv, int kernel, int stride, int block_size,
                                    int nb_stride, float* out, cudaStream_t st);
cudaError_t launch_topk_two_stage(const Seqs& s, const float* scores, int nb_stride, const float* cis_scores, int hkv,
                                  int block_size, int n_init, int n_local, int qk, int k, int32_t* idx,
                                  cudaStream_t st);

// Backward of selected attention (bf16, d 128, block 64, h/hkv <= 16): dq [tokens,h,d],
// dk/dv [tokens,hkv,d] from q, k, v, the block lists, the forward's o and lse and dO.
size_t sparse_bwd_workspace_bytes(const Seqs& s, int h, int hkv, int S);
cudaError_t launch_sparse_bwd(const Seqs& s, const void* q, const void* k, const void* v, const int32_t* idx, int S,
                              int h, int hkv, float scale, const void* o, const float* lse, const void* dout,
                              void* dq, void* dk, void* dv, void* workspace, cudaStream_t st);
// Backward of the compressed branch (same kernels over the packed compressed keys):
// dq [tokens,h,d], dk_cmp/dv_cmp [n_cmp,hkv,d]; and of the mean pooling (bf16, d % 8 == 0).
size_t cmp_attn_bwd_workspace_bytes(const Seqs& s, int h, int hkv, int kernel, int stride);
cudaError_t launch_cmp_attn_bwd(const Seqs& s, const void* q, const void* k_cmp, const void* v_cmp, int h, int hkv,
                                int kernel, int stride, float scale, const void* o, const float* lse,
                                const void* dout, void* dq, void* dk_cmp, void* dv_cmp, void* workspace,
                                cudaStream_t st);
cudaError_t launch_compress_bwd(const Seqs& s, const void* dk_cmp, int hkv, int d, int kernel, int stride, void* dk,
                                cudaStream_t st);
// out = a + b + c (bf16, n a multiple of 8).
cudaError_t launch_add3(const void* a, const void* b, const void* c, void* out, int64_t n, cudaStream_t st);
// Backward of the sigmoid gate combine over rows = tokens * h (bf16, d % 8 == 0).
cudaError_t launch_gate_bwd(int64_t rows, int d, const void* dout, const void* o_cmp, const void* o_slc,
                            const void* o_swa, const float* logits, void* d_cmp, void* d_slc, void* d_swa,
                            float* d_logits, cudaStream_t st);
// Backward of the sliding window (same kernels; keys max(0, t-window+1) .. t).
size_t swa_bwd_workspace_bytes(const Seqs& s, int h, int hkv, int window);
cudaError_t launch_swa_bwd(const Seqs& s, const void* q, const void* k, const void* v, int h, int hkv, int window,
                           float scale, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* workspace, cudaStream_t st);

// mode 0: compressed-attention branch (keys/values are packed compressed rows)
// mode 1: sliding-window branch
cudaError_t launch_dense_attn(int mode, const Seqs& s, const void* q, const void* k, const void* v,
                              int h, int hkv, int d, int kernel, int stride, int window, float scale,
                              void* o, float* lse, cudaStream_t st);

// Tensor-core (tcgen05) versions of the two dense branches for d = 128, bf16.  They take
// V transposed per kv-head, [hkv, 128, tc_vt_pad(kv_rows)], written by launch_transpose_v
// (compressed = true: valid rows are the packed compressed rows of all sequences).
// mode 0 with scores != nullptr also writes the pooled block scores [tokens, hkv,
// nb_stride] (h / hkv must then be 1, 2, 4, 8 or 16).
int64_t tc_vt_pad(int64_t rows);
cudaError_t launch_transpose_v(const Seqs& s, const void* v, void* vt, int64_t rows, int hkv, bool compressed,
                               int kernel, int stride, cudaStream_t st);
// kv_total (mode 0): key rows the k buffer holds; tiles reaching past them are read with
// bounds-checked copies (-1: the packed compressed rows of all sequences, computed on the
// device; 0: the buffer extends past every tile, as in the layer's workspace).
cudaError_t launch_dense_attn_tc(int mode, const Seqs& s, const void* q, const void* k, const void* vt,
                                 int64_t kv_rows, int h, int hkv, int kernel, int stride, int window, float scale,
                                 void* o, float* lse, float* scores, int nb_stride, cudaStream_t st,
                                 int64_t kv_total = 0);
// Whether the tensor-core dense branches take this shape (d 128 and a group size that is
// a power of two up to 128).
bool dense_tc_supported(int h, int hkv, int d);
// Block-mask sparse attention on the tensor cores: dense layout, seqlen % 64 == 0,
// multi-head K/V (h_kv == h), d = 128, bf16; vt = V transposed as for the dense branches;
// mask uint8 [batch, h, n_qb, n_qb] over 64 x 64 tiles.
cudaError_t launch_block_sparse_tc(const Seqs& s, const void* q, const void* k, const void* vt, int h,
                                   const uint8_t* mask, int causal, float scale, void* o, float* lse,
                                   cudaStream_t st);

// Block scores (S2 + S3) on the tensor cores, d = 128, kernel 32 / stride 16 / block 64,
// group size 1..16 (power of two).  kv_rows: rows the key tensor map spans (an upper
// bound is fine); kv_total: rows the k_cmp buffer holds, or -1 for the packed compressed
// rows of all sequences (computed on the device).  Tiles reaching past kv_total are
// read with bounds-checked copies.
bool scores_tc_supported(int h, int hkv, int d, int kernel, int stride, int block_size);
cudaError_t launch_scores_tc(const Seqs& s, const void* q, const void* k_cmp, int64_t kv_rows, int64_t kv_total,
                             int h, int hkv, float scale, const float* lse_in, float* scores, int nb_stride,
                             cudaStream_t st);

// Status words of the units with bounded waits (NSA_ERR_TIMEOUT once a wait ran out);
// optionally cleared.
cudaError_t status_word_dense_tc(int32_t* out, bool reset);
cudaError_t status_word_decode(int32_t* out, bool reset);
cudaError_t status_word_decode_nosa(int32_t* out, bool reset);
cudaError_t status_word_sparse_fwd(int32_t* out, bool reset);
cudaError_t status_word_sparse_bwd_tc(int32_t* out, bool reset);
// Limit (ns) of the first-level bounded waits of each of those units.
cudaError_t wait_limit_dense_tc(unsigned long long ns);
cudaError_t wait_limit_decode(unsigned long long ns);
cudaError_t wait_limit_decode_nosa(unsigned long long ns);
cudaError_t wait_limit_sparse_fwd(unsigned long long ns);
cudaError_t wait_limit_sparse_bwd_tc(unsigned long long ns);

cudaError_t launch_gate_combine(int64_t tokens, int h, int d, const void* o_cmp, const void* o_slc,
                                const void* o_swa, const float* gates, void* o, cudaStream_t st);

struct DecodeArgs {
  int batch, max_len, h, hkv, d, kernel, stride, block_size, n_init, n_local, k;
  float scale;
  const int32_t* seqlens;
  const void *q, *k_cache, *v_cache, *kc_cache;
  int32_t* idx;  // [batch, hkv, k]
  void* o;
  // scratch
  float* z;        // [batch, hkv, n_units, 8, r]
  float* unit_ml;  // [batch, hkv, n_units, r, 2]
  float* part_o;   // [batch, hkv * rtiles, n_split, 16, d]
  float* part_ml;  // [batch, hkv * rtiles, n_split, 16, 2]
  int* counters;  // DecodeLayout::counter_bytes: queue head, arrivals, ready flags (zeroed per call)
  int n_split;
  // NOSA decode (optional; null = plain decode): per-key CIS [batch, max_len, hkv] fp32 and
  // block CIS scores [batch, hkv, cis_nb_stride] fp32 with stage-1 size qk (k <= qk <= 64)
  const float* cis = nullptr;
  const float* cis_block = nullptr;
  int cis_nb_stride = 0, qk = 0;
};
struct DecodeLayout {
  size_t z, unit_ml, idx, part_o, part_ml, counters, counter_bytes, total;
  int n_units, n_split;
};
DecodeLayout decode_layout(int batch, int max_len, int h, int hkv, int d, int kernel, int stride,
                           int block_size, int k);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
// The NOSA variant (a.cis set): decode_nosa.cu; launch_decode calls it after the memset.
cudaError_t launch_decode_nosa(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st);

}  // namespace nsa
