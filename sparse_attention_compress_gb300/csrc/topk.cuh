// Warp-level top-k over one row of block scores, shared by the prefill selection
// kernel and the decode selection kernel.
//
// [NOSA-Triton] "NOSA-1B source walk-through #3", beyond the kernel: the fused block
// scores keep init_blocks + local_blocks + selected candidates, the rest are filled
// with -inf, top-k picks the blocks and the indices are handed on sorted.
//
// Each lane owns NPL consecutive blocks.  Scores become order-preserving 32-bit keys
// (forced blocks take the largest key, blocks after the query are not candidates).
// The k-th largest key is found by a 32-step bitwise search with warp-wide counts
// (__reduce_add_sync), so the cost is independent of k; keys equal to the threshold
// are taken in ascending block order, which breaks ties toward the lower index.  The
// chosen blocks are written in ascending order by a warp prefix count; -1 pads the tail.
#pragma once

#include "common.cuh"

namespace nsa {

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (f == 0.f) u = 0u;  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int warp_excl_scan(int x, int lane) {
  int inc = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  return inc - x;
}

// row: scores of blocks 0..nb-1 (generic pointer: global or shared).  own = t / block_size.
// VEC: row is 16-byte aligned and NPL % 4 == 0.
template <int NPL, bool VEC>
__device__ __forceinline__ void warp_topk(const float* row, int nb, int own, int n_init, int n_local, int k,
                                          int32_t* out, int lane) {
  uint32_t key[NPL];
  bool valid[NPL];
  const int j0 = lane * NPL;
  float sc[NPL];
  if (VEC) {
#pragma unroll
    for (int i = 0; i < NPL; i += 4) {
      if (j0 + i < nb && j0 + i <= own) {
        const float4 f = *reinterpret_cast<const float4*>(row + j0 + i);
        sc[i] = f.x;
        sc[i + 1] = f.y;
        sc[i + 2] = f.z;
        sc[i + 3] = f.w;
      } else {
        sc[i] = sc[i + 1] = sc[i + 2] = sc[i + 3] = 0.f;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NPL; ++i) sc[i] = (j0 + i < nb && j0 + i <= own) ? row[j0 + i] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int j = j0 + i;
    valid[i] = j <= own && j < nb;
    const bool forced = j < n_init || j > own - n_local;
    key[i] = forced ? 0xffffffffu : order_key(sc[i]);
  }
  const int ncand = min(own + 1, nb);
  uint32_t P = 0u;
  int need = k;
  if (ncand > k) {
#pragma unroll 1
    for (int b = 31; b >= 0; --b) {
      const uint32_t trial = P | (1u << b);
      int c = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i) c += (valid[i] && key[i] >= trial) ? 1 : 0;
      c = (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
      if (c >= k) P = trial;
    }
    int gt = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) gt += (valid[i] && key[i] > P) ? 1 : 0;
    need = k - (int)__reduce_add_sync(0xffffffffu, (unsigned)gt);
  }
  // ties at the threshold: rank them in block order
  int tie = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) tie += (ncand > k && valid[i] && key[i] == P) ? 1 : 0;
  int rank = warp_excl_scan(tie, lane);
  bool sel[NPL];
  int nsel = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (ncand <= k) {
      sel[i] = valid[i];
    } else if (valid[i] && key[i] == P) {
      sel[i] = rank < need;
      ++rank;
    } else {
      sel[i] = valid[i] && key[i] > P;
    }
    nsel += sel[i] ? 1 : 0;
  }
  int pos = warp_excl_scan(nsel, lane);
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (sel[i]) out[pos++] = j0 + i;
  const int total = min(k, ncand);
  for (int p = total + lane; p < k; p += 32) out[p] = -1;
}

// The same selection spread over a whole CTA of NT threads (each owns E consecutive
// blocks), for rows whose latency matters more than throughput: one barrier per search
// step, with per-warp counts double buffered in shared memory.  scratch: 2*(NT/32)+NT/32
// ints of shared memory.  Every thread of the CTA must call it.
template <int E, int NT>
__device__ __forceinline__ void block_topk(const float* row, int nb, int own, int n_init, int n_local, int k,
                                           int32_t* out, int* scratch) {
  constexpr int NWARP = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* s_cnt = scratch;              // [2][NWARP]
  int* s_tot = scratch + 2 * NWARP;  // [NWARP]
  uint32_t key[E];
  bool valid[E];
  const int j0 = tid * E;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int j = j0 + i;
    valid[i] = j <= own && j < nb;
    const bool forced = j < n_init || j > own - n_local;
    key[i] = forced ? 0xffffffffu : order_key(valid[i] ? row[j] : 0.f);
  }
  const int ncand = min(own + 1, nb);
  auto block_sum = [&](int c, int buf) {  // c summed over the CTA (one barrier)
    c = (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
    if (lane == 0) s_cnt[buf * NWARP + warp] = c;
    __syncthreads();
    int tot = 0;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) tot += s_cnt[buf * NWARP + w];
    return tot;
  };
  uint32_t P = 0u;
  int need = k;
  if (ncand > k) {
#pragma unroll 1
    for (int b = 31; b >= 0; --b) {
      const uint32_t trial = P | (1u << b);
      int c = 0;
#pragma unroll
      for (int i = 0; i < E; ++i) c += (valid[i] && key[i] >= trial) ? 1 : 0;
      if (block_sum(c, b & 1) >= k) P = trial;
    }
    int gt = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) gt += (valid[i] && key[i] > P) ? 1 : 0;
    need = k - block_sum(gt, 1);  // buffer 1: its last readers passed the b = 0 barrier
  }
  // exclusive prefix over the CTA, in block order (threads own consecutive blocks)
  auto block_scan = [&](int x) {
    const int incl = warp_excl_scan(x, lane) + x;
    __syncthreads();  // s_tot may still be read by a previous scan
    if (lane == 31) s_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_tot[w];
    return before + incl - x;
  };
  int tie = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) tie += (ncand > k && valid[i] && key[i] == P) ? 1 : 0;
  int rank = block_scan(tie);
  bool sel[E];
  int nsel = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    if (ncand <= k) {
      sel[i] = valid[i];
    } else if (valid[i] && key[i] == P) {
      sel[i] = rank < need;
      ++rank;
    } else {
      sel[i] = valid[i] && key[i] > P;
    }
    nsel += sel[i] ? 1 : 0;
  }
  int pos = block_scan(nsel);
#pragma unroll
  for (int i = 0; i < E; ++i)
    if (sel[i]) out[pos++] = j0 + i;
  const int total = min(k, ncand);
  for (int q = total + tid; q < k; q += NT) out[q] = -1;
}

}  // namespace nsa
