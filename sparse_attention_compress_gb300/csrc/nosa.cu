// NOSA stage 2: pooled importance scores (CIS) per block and the two-stage selection.
//
// [NOSA-Parts] "NOSA-1B core components", core component 2: a scorer gives every key
// position an importance score (CIS; an input here, since the scorer is learned);
// [NOSA-Triton] "NOSA-1B source walk-through #3", mechanisms 1-3: the scores are
// mean-pooled over windows of 32 positions at step 16, aligned with the key compressor;
// [NOSA-Parts] core component 3: the pooled scores are brought to block granularity
// (block_score_cis) and merged with the stage-1 candidates chosen by attention score,
// and the final top-k is taken from those.
//
// cis_block_kernel: one thread per (sequence, kv-head, block): the mean, over the
// compressor windows lying inside the block, of each window's mean CIS (the rule the
// attention scores use, S3).  The CIS array is read about twice in all: HBM bound and
// small beside the attention.
//
// topk_two_stage_kernel: one warp per (token, kv-head): warp_topk keeps the forced
// blocks and the best qk_select blocks by attention score (stage 1) in shared memory,
// then the kept blocks are ranked by their block CIS score (forced ones first, ties to
// the lower block) and the best k are written in ascending order, -1 padded.
#include "common.cuh"
#include "launch.h"
#include "topk.cuh"

namespace nsa {

namespace {

__global__ void __launch_bounds__(256) cis_block_kernel(const float* __restrict__ cis, float* __restrict__ out,
                                                        Seqs s, int hkv, int kernel, int stride, int block_size,
                                                        int nb_stride) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)s.n_seqs * hkv * nb_stride) return;
  const int j = (int)(i % nb_stride);
  const int64_t sg = i / nb_stride;
  const int g = (int)(sg % hkv), sq = (int)(sg / hkv);
  const int L = seq_len(s, sq);
  const int64_t base = seq_start(s, sq);
  const int n_c = num_cmp(L, kernel, stride);
  float acc = 0.f;
  int cnt = 0;
  if (j < (L + block_size - 1) / block_size) {
    const int first = j * block_size, last_start = (j + 1) * block_size - kernel;
    if (last_start >= first) {
      for (int c = (first + stride - 1) / stride; c <= last_start / stride && c < n_c; ++c) {
        float w = 0.f;
        const float* src = cis + (base + (int64_t)c * stride) * hkv + g;
        for (int e = 0; e < kernel; ++e) w += src[(int64_t)e * hkv];
        acc += w / (float)kernel;
        ++cnt;
      }
    }
  }
  out[i] = cnt ? acc / (float)cnt : 0.f;
}

template <int NPL>
__global__ void __launch_bounds__(256) topk_two_stage_kernel(const float* __restrict__ scores, int nb_stride,
                                                             const float* __restrict__ cis_scores,
                                                             int32_t* __restrict__ out, Seqs s, int hkv,
                                                             int block_size, int n_init, int n_local, int qk, int k) {
  __shared__ uint32_t s_key[8][64];
  __shared__ int s_idx[8][64];
  __shared__ int s_first[8][64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= s.tokens * hkv) return;
  const int64_t tok = row / hkv;
  const int g = (int)(row % hkv);
  const int sq = seq_of_token(s, tok);
  const int t = (int)(tok - seq_start(s, sq));
  const int own = t / block_size;
  warp_topk<NPL>(scores + row * nb_stride, nb_stride, own, n_init, n_local, qk, s_first[warp], s_key[warp],
                 s_idx[warp], lane);
  __syncwarp();
  const float* cs = cis_scores + ((int64_t)sq * hkv + g) * nb_stride;
  int blk[2];
  uint32_t key[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = lane + 32 * h;
    blk[h] = e < qk ? s_first[warp][e] : -1;
    const bool forced = blk[h] < n_init || blk[h] > own - n_local;
    key[h] = blk[h] < 0 ? 0u : (forced ? 0xffffffffu : order_key(cs[blk[h]]));
    s_key[warp][e] = key[h];
    s_idx[warp][e] = blk[h];
  }
  __syncwarp();
  bool sel[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = lane + 32 * h;
    int rank = 0;
    for (int f = 0; f < qk; ++f) {
      const uint32_t kf = s_key[warp][f];
      rank += s_idx[warp][f] >= 0 && (kf > key[h] || (kf == key[h] && f < e));
    }
    sel[h] = blk[h] >= 0 && rank < k;
  }
  const unsigned lt = (1u << lane) - 1u;
  const unsigned m0 = __ballot_sync(0xffffffffu, sel[0]), m1 = __ballot_sync(0xffffffffu, sel[1]);
  int32_t* o = out + row * k;
  if (sel[0]) o[__popc(m0 & lt)] = blk[0];
  if (sel[1]) o[__popc(m0) + __popc(m1 & lt)] = blk[1];
  for (int q = __popc(m0) + __popc(m1) + lane; q < k; q += 32) o[q] = -1;
}

}  // namespace

cudaError_t launch_cis_block_scores(const Seqs& s, const float* cis, int hkv, int kernel, int stride, int block_size,
                                    int nb_stride, float* out, cudaStream_t st) {
  const int64_t n = (int64_t)s.n_seqs * hkv * nb_stride;
  if (n == 0) return cudaSuccess;
  cis_block_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(cis, out, s, hkv, kernel, stride, block_size,
                                                                  nb_stride);
  return cudaGetLastError();
}

cudaError_t launch_topk_two_stage(const Seqs& s, const float* scores, int nb_stride, const float* cis_scores, int hkv,
                                  int block_size, int n_init, int n_local, int qk, int k, int32_t* idx,
                                  cudaStream_t st) {
  const int64_t rows = s.tokens * hkv;
  if (rows == 0) return cudaSuccess;
  dim3 grid((unsigned)((rows + 7) / 8));
  const int npl = (nb_stride + 31) / 32;
#define NSA_TOPK2(N)                                                                                              \
  if (npl <= N) {                                                                                                 \
    topk_two_stage_kernel<N><<<grid, 256, 0, st>>>(scores, nb_stride, cis_scores, idx, s, hkv, block_size, n_init, \
                                                   n_local, qk, k);                                               \
    return cudaGetLastError();                                                                                    \
  }
  NSA_TOPK2(1)
  NSA_TOPK2(2)
  NSA_TOPK2(4)
  NSA_TOPK2(8)
  NSA_TOPK2(16)
  NSA_TOPK2(32)
  NSA_TOPK2(64)
#undef NSA_TOPK2
  return cudaErrorInvalidValue;
}

}  // namespace nsa
