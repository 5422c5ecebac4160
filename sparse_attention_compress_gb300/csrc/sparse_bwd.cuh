// Definitions shared by the backward kernels of selected-block attention (the
// cp.async / mma.sync kernels in sparse_bwd.cu and the tensor-core dK/dV kernel in
// sparse_bwd_tc.cu): the parameters, the three key spaces (selected blocks, compressed
// keys, sliding window) and the numbering of the dK/dV work items.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace nsa {
namespace bwd {

constexpr int kD = 128;
constexpr int kBS = 64;
constexpr int kChunk = 2048;              // query positions per dK/dV work item
constexpr int kGroup = kChunk / kBS;      // key blocks that share a first chunk
constexpr int kTileBytes = kBS * kD * 2;  // one 64 x 128 bf16 block
constexpr int kRowsBytes = 16 * kD * 2;   // 16 rows x 128 bf16

struct BwdParams {
  const __nv_bfloat16 *q, *k, *v, *o, *dout;
  const float* lse;
  const int32_t* idx;
  __nv_bfloat16 *dq, *dk, *dv;
  float* dsum;  // [tokens, h]: D = dO . o
  float* part;  // [n_seqs * hkv][items_per_bg][2][64][128] fp32 partial dK (unscaled), dV
  Seqs seqs;
  int h, hkv, S, r;
  float scale, scale_log2;
  int n_chunks, nb, items_per_bg;
  // compressed branch (cmp_kernel > 0): the keys are the packed compressed rows, query t
  // reaches the compressed keys c < n_causal(t) and its list is every such block (idx is
  // unused); otherwise the keys are the tokens and query t reaches keys <= t of its list.
  int cmp_kernel, cmp_stride;
  // sliding window (window > 0): query t reaches keys max(0, t-window+1) .. t (idx unused);
  // one work item per key block covers every query that reaches it.
  int window;
  // selected blocks with the tensor-core dK/dV kernel: the chunk-wise inverted lists
  // (invert_kernel): per (sequence and kv-head, query chunk) kChunk * S token slots, and
  // per (sequence and kv-head, chunk, key block) the (offset, count) of the block's tokens
  int32_t* inv_list;
  int2* inv_tab;
};

// First key query t may attend.
__device__ __forceinline__ int key_lo(const BwdParams& p, int t) { return p.window ? max(0, t - p.window + 1) : 0; }

// Key rows of sequence b start here; the sequence has key_len(L) of them.
__device__ __forceinline__ int64_t key_base(const BwdParams& p, int b) {
  return p.cmp_kernel ? cmp_offset(p.seqs, b, p.cmp_kernel, p.cmp_stride) : (int64_t)seq_start(p.seqs, b);
}
__device__ __forceinline__ int key_len(const BwdParams& p, int L) {
  return p.cmp_kernel ? num_cmp(L, p.cmp_kernel, p.cmp_stride) : L;
}
// Last key query t may attend (-1: none).
__device__ __forceinline__ int key_bound(const BwdParams& p, int t, int Lk) {
  return p.cmp_kernel ? num_causal_cmp(t, Lk, p.cmp_kernel, p.cmp_stride) - 1 : t;
}
// First query position that reaches key block j.
__device__ __forceinline__ int first_query(const BwdParams& p, int j) {
  return p.cmp_kernel ? p.cmp_stride * kBS * j + p.cmp_kernel - 1 : kBS * j;
}

__device__ __forceinline__ float dot_bf16x2(uint32_t a, uint32_t b) {
  const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a));
  const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b));
  return x.x * y.x + x.y * y.y;
}

// P and dS enter the dV, dQ and dK products as bf16.  Where a warp's 16 x 16 tile holds
// a |value| above the threshold (rows with few keys, where p is large and a bf16 rounding
// of it is not small beside the gradient), the bf16 remainder x - bf16(x) goes through a
// second product, so the operand is carried to about 16 bits.  The threshold for P is
// low: with a nearly uniform softmax (the compressed branch's logits are small, since
// compressed keys are means) p ~ 1/n rounds alike on every row of the same length, and
// those errors add up over the thousands of rows that reach a key.
constexpr float kSplitAbove = 0.0625f;   // dS
constexpr float kSplitPAbove = 0.00390625f;  // P (1/256)

__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
  lo = pack_bf16(a - h.x, b - h.y);
}

// base-2 log-sum-exp of a row from the forward's natural-log lse; rows without keys
// (lse = -inf) give +inf so that every exponential of that row is 0.
__device__ __forceinline__ float lse_to_log2(float l) { return l == kNegInf ? __builtin_inff() : l * kLog2e; }

// 4-byte global->shared copy (zero-fill when src_bytes == 0).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Item index (within one sequence / kv-head) -> (key block j, chunk c).  Blocks
// j = m*kGroup .. m*kGroup+kGroup-1 have their first query chunk at m and one item for
// each chunk m .. n_chunks-1.
__device__ __forceinline__ void item_to_block(const BwdParams& p, int item, int& j, int& c, int& m) {
  const int n_chunks = p.n_chunks, nb = p.nb;
  int rem = item;
  if (p.window) {
    j = item;
    c = m = 0;
    return;
  }
  if (p.cmp_kernel) {  // block j has chunks first_query(j) / kChunk .. n_chunks-1
    for (j = 0; j < nb; ++j) {
      m = first_query(p, j) / kChunk;
      if (rem < n_chunks - m) {
        c = m + rem;
        return;
      }
      rem -= n_chunks - m;
    }
    c = n_chunks;
    return;
  }
  for (m = 0; m < n_chunks; ++m) {
    const int blocks = min(kGroup, nb - m * kGroup);
    const int per = n_chunks - m;
    if (rem < blocks * per) {
      j = m * kGroup + rem / per;
      c = m + rem % per;
      return;
    }
    rem -= blocks * per;
  }
  j = nb;  // not reached for item < items_per_bg
  c = n_chunks;
}

// The tensor-core dK/dV kernel (sparse_bwd_tc.cu): the same work items and fp32 partials
// as sparse_bwd_dkv, for group sizes r = 8 and 16 (d = 128, blocks of 64).
bool dkv_tc_supported(const BwdParams& p);
// The same test from the shape alone (group size r, key blocks per sequence nb).
inline bool dkv_tc_shape(int r, bool cmp_or_window, int nb) {
  return (r == 8 || r == 16) && (cmp_or_window || nb <= 1024);
}
cudaError_t launch_dkv_tc(const BwdParams& p, int64_t items, int64_t q_rows, cudaStream_t st);
// Selected blocks: the inverted lists the tensor-core kernel reads (p.inv_list, p.inv_tab).
cudaError_t launch_invert(const BwdParams& p, cudaStream_t st);
// The tensor-core dQ kernel (sparse_bwd_tc.cu) of the compressed and window key spaces,
// group sizes 8 and 16; like sparse_bwd_dq it also stores D = dO . o (p.dsum).  kv_rows:
// the rows of p.k and p.v (for the compressed keys, a bound on the packed rows).
bool dq_tc_supported(const BwdParams& p);
cudaError_t launch_dq_tc(const BwdParams& p, int64_t kv_rows, cudaStream_t st);

}  // namespace bwd
}  // namespace nsa
