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

// Exact k-th largest of the warp's candidate keys (lane owns keys[i] for block
// i*32 + lane < ncand) by a radix select on 4-bit digits.  Bits shared by every
// candidate (found with a warp AND / OR) take no pass; each pass counts the digits of
// the keys that match the digits fixed so far in sixteen 8-bit counters per lane
// (registers, no shared-memory atomics) and sums each counter over the warp.
// Returns the key; *need = how many keys equal to it belong to the top k.
template <int NPL>
__device__ __forceinline__ uint32_t warp_radix_kth(const uint32_t (&key)[NPL], int ncand, int k, int* need,
                                                   int lane) {
  const int n_it = (ncand + 31) / 32;
  uint32_t all_and = 0xffffffffu, all_or = 0u;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (i >= n_it) break;  // warp-uniform: rows shorter than NPL * 32 skip the rest
    if (i * 32 + lane < ncand) {
      all_and &= key[i];
      all_or |= key[i];
    }
  }
  all_and = __reduce_and_sync(0xffffffffu, all_and);
  all_or = __reduce_or_sync(0xffffffffu, all_or);
  const uint32_t varying = all_and ^ all_or;
  if (varying == 0u) {  // every candidate key is the same
    *need = k;
    return all_and;
  }
  int shift = ((31 - __clz(varying)) / 4) * 4;  // lowest bit of the highest varying digit
  uint32_t pmask = shift + 4 >= 32 ? 0u : (0xffffffffu << (shift + 4));
  uint32_t prefix = all_and & pmask;
  int left = k;
#pragma unroll 1
  for (; shift >= 0; shift -= 4) {
    unsigned long long lo = 0ull, hi = 0ull;  // digits 0..7 and 8..15, 8 bits each
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if (i >= n_it) break;
      if (i * 32 + lane < ncand && (key[i] & pmask) == prefix) {
        const uint32_t d = (key[i] >> shift) & 15u;
        const unsigned long long inc = 1ull << ((d & 7u) * 8u);
        if (d < 8u) lo += inc; else hi += inc;
      }
    }
    // from the top digit down: the digit where the count of larger-or-equal keys reaches left
    int run = 0, dsel = 0, above = 0;
    bool found = false;
#pragma unroll
    for (int q = 15; q >= 0; --q) {
      const unsigned f = (unsigned)(((q < 8 ? lo : hi) >> ((q & 7) * 8)) & 0xffull);
      const int c = (int)__reduce_add_sync(0xffffffffu, f);
      if (!found && run + c >= left) {
        found = true;
        dsel = q;
        above = run;
      }
      run += c;
    }
    left -= above;
    prefix |= (uint32_t)dsel << shift;
    pmask |= 15u << shift;
  }
  *need = left;
  return prefix;
}

// row: scores of blocks 0..nb-1 (global or shared).  own = t / block_size.  Lane owns
// blocks lane, lane + 32, ... (coalesced loads).  cand_key / cand_idx: 64 entries of
// warp-private shared memory.
//
// For k <= 32 a lower bound of the k-th largest key is the k-th largest of the lanes'
// maxima (k lanes hold a key at least that large), so the top k lie among the keys at or
// above it; those candidates (usually a few more than k) are ranked exactly by (key
// descending, block ascending).  With more than 64 candidates, or k > 32, the k-th
// largest key is found by a radix select instead.
template <int NPL>
__device__ __forceinline__ void warp_topk(const float* row, int nb, int own, int n_init, int n_local, int k,
                                          int32_t* out, uint32_t* cand_key, int* cand_idx, int lane) {
  const int ncand = min(own + 1, nb);
  if (ncand <= k) {  // every candidate is chosen
    for (int q = lane; q < k; q += 32) out[q] = q < ncand ? q : -1;
    return;
  }
  const unsigned lt = (1u << lane) - 1u;
  const int n_it = (ncand + 31) / 32;
  uint32_t key[NPL];
  uint32_t lmax = 0u;
  // every loop over the lane's blocks stops at the row's own length (a warp-uniform
  // exit), so a short row costs its length, not NPL * 32; the loads of the row are all
  // issued before the first of them is used
  float sv[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (i >= n_it) break;
    const int j = i * 32 + lane;
    sv[i] = j < ncand ? row[j] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (i >= n_it) break;
    const int j = i * 32 + lane;
    key[i] = 0u;
    if (j < ncand) {
      const bool forced = j < n_init || j > own - n_local;
      key[i] = forced ? 0xffffffffu : order_key(sv[i]);
      lmax = max(lmax, key[i]);
    }
  }
  if (k <= 32) {
    const uint32_t tau = warp_kth_largest(lmax, k, lane);
    unsigned in_mask[NPL];  // the ballots of the candidate test, kept for the compaction
    int c = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if (i >= n_it) break;
      in_mask[i] = __ballot_sync(0xffffffffu, i * 32 + lane < ncand && key[i] >= tau);
      c += __popc(in_mask[i]);
    }
    if (c <= 64) {
      int base = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        if (i >= n_it) break;
        const unsigned m = in_mask[i];
        if ((m >> lane) & 1u) {
          cand_key[base + __popc(m & lt)] = key[i];
          cand_idx[base + __popc(m & lt)] = i * 32 + lane;
        }
        base += __popc(m);
      }
      __syncwarp();
      if (c <= 32) {
        // one candidate per lane: a bitonic sort of (key descending, list position
        // ascending) puts the chosen blocks in lanes 0 .. k-1; the positions, being in
        // ascending block order, then give each chosen block its output slot
        uint32_t ck = lane < c ? cand_key[lane] : 0u;
        int cp = lane < c ? lane : 0x7fffffff;
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
          for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t ok = __shfl_xor_sync(0xffffffffu, ck, stride);
            const int op = __shfl_xor_sync(0xffffffffu, cp, stride);
            const bool mine_first = ck > ok || (ck == ok && cp < op);
            const bool desc = (lane & size) == 0 || size == 32;  // the final order is descending
            const bool lower = (lane & stride) == 0;
            if ((lower == desc) != mine_first) {
              ck = ok;
              cp = op;
            }
          }
        }
        const bool chosen = lane < k && cp < c;
        const unsigned pos_mask = __reduce_or_sync(0xffffffffu, chosen ? 1u << cp : 0u);
        if (chosen) out[__popc(pos_mask & ((1u << cp) - 1u))] = cand_idx[cp];
        __syncwarp();  // cand_* may be reused by the next row of this warp
        return;
      }
      // 33 .. 64 candidates: rank each by key, ties by position
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
  // exact k-th largest key P by radix select
  int need;
  const uint32_t P = warp_radix_kth<NPL>(key, ncand, k, &need, lane);
  // keys above P, and the first `need` keys equal to P in block order
  int taken = 0, pos = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (i >= n_it) break;
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

// The same selection spread over a CTA of NT threads, each owning E consecutive blocks
// of a row (global or shared memory): the radix passes count digits in registers, sum
// them per warp and combine the warps through shared memory, one barrier per pass; the
// chosen blocks are written in block order through a CTA prefix count.  For rows whose
// latency matters (the decode selection): a single warp's chain of dependent
// reductions is what this avoids.  scratch: 2 * 16 * (NT / 32) + 2 * (NT / 32) ints.
// Every thread of the CTA must call it.
template <int E, int NT>
__device__ __forceinline__ void block_topk(const float* row, int nb, int own, int n_init, int n_local, int k,
                                           int32_t* out, int* scratch) {
  constexpr int NWARP = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* s_cnt = scratch;                   // [2][NWARP][16]
  int* s_red = scratch + 2 * NWARP * 16;  // [2][NWARP]
  const int ncand = min(own + 1, nb);
  if (ncand <= k) {
    for (int q = tid; q < k; q += NT) out[q] = q < ncand ? q : -1;
    return;
  }
  uint32_t key[E];
  bool valid[E];
  const int j0 = tid * E;
  uint32_t all_and = 0xffffffffu, all_or = 0u;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int j = j0 + i;
    valid[i] = j < ncand;
    const bool forced = j < n_init || j > own - n_local;
    key[i] = valid[i] ? (forced ? 0xffffffffu : order_key(row[j])) : 0u;
    if (valid[i]) {
      all_and &= key[i];
      all_or |= key[i];
    }
  }
  // bits shared by every candidate take no pass
  all_and = __reduce_and_sync(0xffffffffu, all_and);
  all_or = __reduce_or_sync(0xffffffffu, all_or);
  if (lane == 0) {
    s_red[warp] = (int)all_and;
    s_red[NWARP + warp] = (int)all_or;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    all_and &= (uint32_t)s_red[w];
    all_or |= (uint32_t)s_red[NWARP + w];
  }
  const uint32_t varying = all_and ^ all_or;
  uint32_t P = all_and;
  int left = k;
  if (varying != 0u) {
    int shift = ((31 - __clz(varying)) / 4) * 4;
    uint32_t pmask = shift + 4 >= 32 ? 0u : (0xffffffffu << (shift + 4));
    uint32_t prefix = all_and & pmask;
    int buf = 0;
#pragma unroll 1
    for (; shift >= 0; shift -= 4, buf ^= 1) {
      unsigned long long lo = 0ull, hi = 0ull;  // 16 digit counters of this thread, 8 bits each
#pragma unroll
      for (int i = 0; i < E; ++i)
        if (valid[i] && (key[i] & pmask) == prefix) {
          const uint32_t d = (key[i] >> shift) & 15u;
          const unsigned long long inc = 1ull << ((d & 7u) * 8u);
          if (d < 8u) lo += inc; else hi += inc;
        }
      int* cnt = s_cnt + buf * NWARP * 16 + warp * 16;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const unsigned f = (unsigned)(((q < 8 ? lo : hi) >> ((q & 7) * 8)) & 0xffull);
        const int c = (int)__reduce_add_sync(0xffffffffu, f);
        if (lane == 0) cnt[q] = c;
      }
      __syncthreads();  // the other buffer is rewritten only after the next barrier
      int run = 0, dsel = 0, above = 0;
      bool found = false;
#pragma unroll
      for (int q = 15; q >= 0; --q) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) c += s_cnt[buf * NWARP * 16 + w * 16 + q];
        if (!found && run + c >= left) {
          found = true;
          dsel = q;
          above = run;
        }
        run += c;
      }
      left -= above;
      prefix |= (uint32_t)dsel << shift;
      pmask |= 15u << shift;
    }
    P = prefix;
  }
  // exclusive prefix over the CTA, in block order (threads own consecutive blocks)
  int* s_tot = s_red;  // reused: its last readers passed at least one barrier since
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
  for (int i = 0; i < E; ++i) tie += (valid[i] && key[i] == P) ? 1 : 0;
  int rank = block_scan(tie);
  bool sel[E];
  int nsel = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    if (valid[i] && key[i] == P) {
      sel[i] = rank < left;
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
}

}  // namespace nsa
