// Warp-level top-k over one row of block scores, shared by the prefill selection
// kernel and the decode selection kernel.
//
// [NOSA-Triton] "NOSA-1B source walk-through #3", beyond the kernel: the fused block
// scores keep init_blocks + local_blocks + selected candidates, the rest are filled
// with -inf, top-k picks the blocks and the indices are handed on sorted.
//
// Scores become order-preserving 32-bit keys (forced blocks take the largest key,
// blocks after the query are not candidates).  Keys equal to the k-th largest are taken
// in ascending block order, which breaks ties toward the lower index; the chosen blocks
// are written in ascending order; -1 pads the tail when a row has fewer than k
// candidates.
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

// k-th largest (1-based) of the 32 lanes' values, by a bitonic sort across the warp.
__device__ __forceinline__ uint32_t warp_kth_largest(uint32_t v, int k, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool desc = (lane & size) == 0 || size == 32;  // the final order is descending
      const bool lower = (lane & stride) == 0;
      v = (lower == desc) ? max(v, o) : min(v, o);
    }
  }
  return __shfl_sync(0xffffffffu, v, k - 1);
}

// row: scores of blocks 0..nb-1 (global or shared).  own = t / block_size.  Lane owns
// blocks lane, lane + 32, ... (coalesced loads).  cand_key / cand_idx: 64 entries of
// warp-private shared memory.
//
// For k <= 32 a lower bound of the k-th largest key is the k-th largest of the lanes'
// maxima (k lanes hold a key at least that large), so the top k lie among the keys at or
// above it; those candidates (usually a few more than k) are ranked exactly by (key
// descending, block ascending).  With more than 64 candidates, or k > 32, the k-th
// largest key is found by a 32-step bitwise search with warp-wide counts instead.
template <int NPL>
__device__ __forceinline__ void warp_topk(const float* row, int nb, int own, int n_init, int n_local, int k,
                                          int32_t* out, uint32_t* cand_key, int* cand_idx, int lane) {
  const int ncand = min(own + 1, nb);
  if (ncand <= k) {  // every candidate is chosen
    for (int q = lane; q < k; q += 32) out[q] = q < ncand ? q : -1;
    return;
  }
  const unsigned lt = (1u << lane) - 1u;
  uint32_t key[NPL];
  uint32_t lmax = 0u;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int j = i * 32 + lane;
    key[i] = 0u;
    if (j < ncand) {
      const bool forced = j < n_init || j > own - n_local;
      key[i] = forced ? 0xffffffffu : order_key(row[j]);
      lmax = max(lmax, key[i]);
    }
  }
  const int n_it = (ncand + 31) / 32;
  if (k <= 32) {
    const uint32_t tau = warp_kth_largest(lmax, k, lane);
    int c = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (i < n_it) c += __popc(__ballot_sync(0xffffffffu, i * 32 + lane < ncand && key[i] >= tau));
    if (c <= 64) {
      int base = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        if (i < n_it) {
          const bool in = i * 32 + lane < ncand && key[i] >= tau;
          const unsigned m = __ballot_sync(0xffffffffu, in);
          if (in) {
            cand_key[base + __popc(m & lt)] = key[i];
            cand_idx[base + __popc(m & lt)] = i * 32 + lane;
          }
          base += __popc(m);
        }
      }
      __syncwarp();
      // candidates are in ascending block order: rank by key, ties by position
      bool sel[2];
      int idx[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ci = lane + 32 * h;
        sel[h] = false;
        idx[h] = -1;
        if (ci < c) {
          const uint32_t kc = cand_key[ci];
          int rank = 0;
          for (int j = 0; j < c; ++j) {
            const uint32_t kj = cand_key[j];
            rank += (kj > kc) || (kj == kc && j < ci);
          }
          sel[h] = rank < k;
          idx[h] = cand_idx[ci];
        }
      }
      const unsigned m0 = __ballot_sync(0xffffffffu, sel[0]), m1 = __ballot_sync(0xffffffffu, sel[1]);
      if (sel[0]) out[__popc(m0 & lt)] = idx[0];
      if (sel[1]) out[__popc(m0) + __popc(m1 & lt)] = idx[1];
      __syncwarp();  // cand_* may be reused by the next row of this warp
      return;
    }
  }
  // exact k-th largest key P by bitwise search
  uint32_t P = 0u;
#pragma unroll 1
  for (int b = 31; b >= 0; --b) {
    const uint32_t trial = P | (1u << b);
    int c = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) c += (i * 32 + lane < ncand && key[i] >= trial) ? 1 : 0;
    c = (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
    if (c >= k) P = trial;
  }
  int gt = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) gt += (i * 32 + lane < ncand && key[i] > P) ? 1 : 0;
  const int need = k - (int)__reduce_add_sync(0xffffffffu, (unsigned)gt);
  // keys above P, and the first `need` keys equal to P in block order
  int taken = 0, pos = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (i < n_it) {
      const bool v = i * 32 + lane < ncand;
      const bool eq = v && key[i] == P;
      const unsigned me = __ballot_sync(0xffffffffu, eq);
      const bool s = (v && key[i] > P) || (eq && taken + __popc(me & lt) < need);
      taken += __popc(me);
      const unsigned ms = __ballot_sync(0xffffffffu, s);
      if (s) out[pos + __popc(ms & lt)] = i * 32 + lane;
      pos += __popc(ms);
    }
  }
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
