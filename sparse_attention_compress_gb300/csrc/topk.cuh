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

// Exclusive prefix of x over the CTA in thread order; tot: NW ints of shared scratch
// that no thread reads or writes around the call.  Every thread must call it.
template <int NW>
__device__ __forceinline__ int block_excl_scan(int x, int* tot, int lane, int warp) {
  const int incl = warp_excl_scan(x, lane) + x;
  if (lane == 31) tot[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += tot[w];
  __syncthreads();  // tot may be rewritten after this
  return before + incl - x;
}

// The same selection spread over a CTA of NT = 128 threads, each owning E consecutive
// blocks of a row (global or shared memory), for rows whose latency matters (the decode
// selection, k <= NT).  The steps are chosen for few dependent CTA-wide exchanges:
//  1. the forced blocks are counted apart (always kept; if they alone reach k, the k
//     lowest are kept), and the bits shared by every other candidate's key are found
//     with one reduction, so no pass spends itself on them;
//  2. radix passes over 8 bits at a time: a shared-memory histogram of the candidates
//     that match the prefix so far, and a suffix count over the bins that finds the bin
//     holding the remaining k-th best; its bits join the prefix.  One pass usually
//     leaves a handful of keys in that bin;
//  3. once the bin holds at most NT candidates, they are ranked exactly against each
//     other by (key descending, block ascending), one candidate per thread, and the
//     winners are marked in a per-block table; if a bin is still larger when every bit is
//     used, its keys are equal and the lowest blocks win.
// The chosen blocks are written in block order through a CTA prefix count.
// scratch: block_topk_scratch_ints<NT>() ints, 8-byte aligned.  Every thread of the CTA
// must call it.
template <int NT>
constexpr int block_topk_scratch_ints() {
  return 2 * 256 + 2 * NT + 32 + 1024 / 4;
}

template <int E, int NT>
__device__ __forceinline__ void block_topk(const float* row, int nb, int own, int n_init, int n_local, int k,
                                           int32_t* out, int* scratch) {
  static_assert(NT == 128, "four warps: two histogram bins per thread");
  constexpr int NWARP = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* hist = scratch;                                              // [2][256]
  uint64_t* cand = reinterpret_cast<uint64_t*>(scratch + 512);      // [NT]
  int* misc = scratch + 512 + 2 * NT;                               // [32]
  uint8_t* won = reinterpret_cast<uint8_t*>(scratch + 512 + 2 * NT + 32);  // [1024] bin winners
  const int ncand = min(own + 1, nb);
  if (ncand <= k) {
    for (int q = tid; q < k; q += NT) out[q] = q < ncand ? q : -1;
    return;
  }
  uint32_t key[E];
  bool norm[E], forced[E];
  int nf = 0;
  uint32_t all_and = 0xffffffffu, all_or = 0u;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int j = tid * E + i;
    const bool valid = j < ncand;
    forced[i] = valid && (j < n_init || j > own - n_local);
    norm[i] = valid && !forced[i];
    key[i] = norm[i] ? order_key(row[j]) : 0u;
    nf += forced[i];
    if (norm[i]) {
      all_and &= key[i];
      all_or |= key[i];
    }
  }
  // step 1: forced count and the bits shared by the other candidates
  {
    const int f = (int)__reduce_add_sync(0xffffffffu, (unsigned)nf);
    const uint32_t a = __reduce_and_sync(0xffffffffu, all_and), o = __reduce_or_sync(0xffffffffu, all_or);
    for (int q = tid; q < 256; q += NT) hist[q] = 0;
    if (lane == 0) {
      misc[warp] = f;
      misc[NWARP + warp] = (int)a;
      misc[2 * NWARP + warp] = (int)o;
    }
  }
  __syncthreads();
  int n_forced = 0;
  all_and = 0xffffffffu;
  all_or = 0u;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    n_forced += misc[w];
    all_and &= (uint32_t)misc[NWARP + w];
    all_or |= (uint32_t)misc[2 * NWARP + w];
  }
  bool sel[E];
  int left = k - n_forced;
  if (left <= 0) {
    // the forced blocks alone fill the list: the k lowest of them
    int rank = block_excl_scan<NWARP>(nf, misc + 16, lane, warp);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      sel[i] = forced[i] && rank < k;
      rank += forced[i];
    }
  } else {
    const uint32_t varying = all_and ^ all_or;
    int shift = varying ? 31 - __clz(varying) + 1 : 0;  // bits [shift, 32) are settled
    uint32_t mask = shift >= 32 ? 0u : (0xffffffffu << shift);
    uint32_t prefix = all_and & mask;
    int buf = 0, in_bin = ncand - n_forced;
    // step 2: radix passes while the k-th best's bin is larger than NT
    while (shift > 0 && in_bin > NT) {
      const int w = shift < 8 ? shift : 8;
      shift -= w;
      int* h = hist + buf * 256;
      int* h_next = hist + (buf ^ 1) * 256;
      for (int q = tid; q < 256; q += NT) h_next[q] = 0;  // read-free until the next pass
#pragma unroll
      for (int i = 0; i < E; ++i)
        if (norm[i] && (key[i] & mask) == prefix) atomicAdd(&h[(key[i] >> shift) & ((1u << w) - 1u)], 1);
      __syncthreads();
      // suffix counts: thread t owns bins 2t and 2t+1; counts above a bin are those of
      // higher bins
      const int b0 = h[2 * tid], b1 = h[2 * tid + 1], c = b0 + b1;
      int sfx = c;  // inclusive suffix sum within the warp (higher lanes hold higher bins)
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, sfx, off);
        if (lane + off < 32) sfx += y;
      }
      if (lane == 0) misc[16 + warp] = sfx;
      __syncthreads();
      int higher = sfx - c;  // count in bins above this thread's two
      for (int w2 = warp + 1; w2 < NWARP; ++w2) higher += misc[16 + w2];
      if (higher < left && left <= higher + c) {  // the k-th best lies in one of this thread's bins
        const bool top = left <= higher + b1;
        misc[20] = top ? 2 * tid + 1 : 2 * tid;
        misc[21] = top ? higher : higher + b1;
        misc[22] = top ? b1 : b0;
      }
      __syncthreads();
      const uint32_t d = (uint32_t)misc[20];
      left -= misc[21];
      in_bin = misc[22];
      prefix |= d << shift;
      mask |= ((1u << w) - 1u) << shift;
      buf ^= 1;
      __syncthreads();  // misc is rewritten by the next pass
    }
    // step 3: the k-th best's bin (keys equal to prefix on the settled bits)
    int rank_tie = 0;
    if (in_bin > NT) {  // every bit settled: equal keys, the lowest blocks win
      int eq = 0;
#pragma unroll
      for (int i = 0; i < E; ++i) eq += norm[i] && key[i] == prefix;
      rank_tie = block_excl_scan<NWARP>(eq, misc + 16, lane, warp);
    } else {
      if (tid == 0) misc[23] = 0;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < E; ++i)
        if (norm[i] && (key[i] & mask) == prefix)
          cand[atomicAdd(&misc[23], 1)] = ((uint64_t)key[i] << 32) | (uint32_t)~(uint32_t)(tid * E + i);
      __syncthreads();
      const int nc = in_bin;
      if (tid < nc) {  // candidate tid's rank in the bin: the candidates above it
        const uint64_t me = cand[tid];
        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        int q = 0;
        for (; q + 4 <= nc; q += 4) {
          r0 += cand[q] > me;
          r1 += cand[q + 1] > me;
          r2 += cand[q + 2] > me;
          r3 += cand[q + 3] > me;
        }
        for (; q < nc; ++q) r0 += cand[q] > me;
        won[~(uint32_t)me] = (r0 + r1) + (r2 + r3) < left;
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const bool inb = norm[i] && (key[i] & mask) == prefix;
      bool s = forced[i] || (norm[i] && (key[i] & mask) > prefix);
      if (inb) {
        if (in_bin > NT) {
          s = rank_tie < left;
          ++rank_tie;
        } else {
          s = won[tid * E + i] != 0;
        }
      }
      sel[i] = s;
    }
  }
  int nsel = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) nsel += sel[i];
  int pos = block_excl_scan<NWARP>(nsel, misc + 24, lane, warp);
#pragma unroll
  for (int i = 0; i < E; ++i)
    if (sel[i]) out[pos++] = tid * E + i;
}

}  // namespace nsa
