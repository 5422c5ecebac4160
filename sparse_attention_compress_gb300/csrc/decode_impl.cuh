// Kernels of the decode step (see decode.cu), templated on W: the NOSA variant, whose
// attention weights each key by its CIS and whose selection can re-rank the kept blocks by
// their CIS block score.  decode.cu instantiates W = false and decode_nosa.cu W = true, in
// separate translation units so that the two builds run in parallel.
#pragma once

#include "attend.cuh"
#include "launch.h"
#include "sm100.cuh"
#include "topk.cuh"

namespace nsa {

constexpr int kUnit = 32;        // compressed keys per score unit
constexpr int kMaxUnits = 128;   // units per row: max_len <= 65536
constexpr int kNW = 4;           // warps per CTA
constexpr int kDecodeStages = 3;  // ring stages per warp (score units and attention slices)
constexpr int kUnitBytes = kUnit * 128 * 2;

struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* seqlens;
  int h, hkv, max_len, nc_stride, n_units, n_init, n_local, k, n_split, eps;
  float scale_log2;
  float* z;        // pooled block partials [rows, n_units * 8 blocks, r]
  float* unit_ml;  // per unit and head (max, sum) [rows, n_units, r, 2]
  float* part_o;
  float* part_ml;
  int32_t* idx;
  __nv_bfloat16* o;
  int* queue;        // [1]
  int* score_count;  // [rows]
  int* merge_count;  // [rows]
  int* ready;        // [rows]
  // NOSA decode (optional): per-key CIS [batch, max_len, hkv] weighting the attention, and
  // block CIS scores [batch, hkv, cis_nb_stride] for the two-stage selection (stage 1 keeps
  // qk blocks by attention score, stage 2 keeps k of them by CIS score).
  const float* cis;
  const float* cis_block;
  int cis_nb_stride, qk;
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_add(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Cross-CTA hand-offs follow one pattern: the writers' stores, a CTA barrier, then a
// release (store, reduction or read-modify-write) by one thread; the reader's acquire by
// one thread, then a CTA barrier, then the reads.  The barrier orders every thread's
// accesses with the one thread's release or acquire, and release and acquire carry that
// order across CTAs.

// Thread 0 waits (bounded) until *f >= v (an acquire load), then every thread learns the
// outcome; on a timeout the device status records it.
__device__ __forceinline__ bool cta_wait_ge(const int* f, int v, int* s_flag) {
  if (threadIdx.x == 0) {
    int ok = 1;
    if (ld_acquire(f) < v) {
      const unsigned long long t0 = tc::globaltimer(), lim = tc::wait_limit();
      while (ld_acquire(f) < v) {
        if (tc::device_status_set() || lim < tc::kQuickNs || tc::globaltimer() - t0 >= lim) {
          atomicExch(&g_device_status, (int)NSA_ERR_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(128);
      }
    }
    *s_flag = ok;
  }
  __syncthreads();
  const bool ok = *s_flag;
  __syncthreads();  // s_flag is rewritten only after every thread has read it
  return ok;
}

// Causal compressed keys of the newest query of sequence b.
__device__ __forceinline__ int decode_nca(const DecodeParams& p, int b) {
  const int L = p.seqlens[b];
  return num_causal_cmp(L - 1, num_cmp(L, 32, 16), 32, 16);
}

// Score phase of one CTA: units [u0, u1) of the flattened (row, unit) space, unit u of a
// row being its compressed keys 32u .. 32u+31.  Warp w takes units u0 + w, u0 + w + 4, ...
// and streams them through its own cp.async ring, so every load of the phase is issued
// at once and the next unit's keys arrive while the current one is scored.  For each
// unit and head the warp writes the (max, sum) of its probabilities relative to the
// unit's own max, and the pooled partials of its 8 blocks (block jl of the unit sums the
// windows 4jl, 4jl+1, 4jl+2).  Units past a row's causal keys are skipped; the first
// stages are issued before the row's length is known (bounded only by the cache
// extent), so the phase's loads start at once, and scoring masks them.
template <int D, int R>
__device__ __forceinline__ void score_units(const DecodeParams& p, int u0, int u1, uint8_t* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int U = p.n_units;
  const int first = u0 + warp;
  const int n = first < u1 ? (u1 - first + kNW - 1) / kNW : 0;
  const uint32_t ring = smem_u32(smem) + warp * kDecodeStages * kUnitBytes;
  const int64_t row_stride = (int64_t)p.hkv * D;
  int c_row = -1, c_nca = 0;  // row of the last issued unit and its causal key count
  auto issue = [&](int i, bool early) {
    if (i < n) {
      const int u = first + i * kNW;
      const int row = u / U, uu = u - row * U;
      const int b = row / p.hkv, g = row % p.hkv;
      if (early) {
        c_row = -1;
        c_nca = p.nc_stride;  // every cached compressed row; scoring masks the row's own length
      } else if (row != c_row) {
        c_row = row;
        c_nca = decode_nca(p, b);
      }
      if (uu * kUnit < c_nca) {
        const __nv_bfloat16* kbase = p.kc + (((int64_t)b * p.nc_stride) * p.hkv + g) * D;
        const int nca = c_nca;
        load_tile_async<D, kUnit, 32>(ring + (i % kDecodeStages) * kUnitBytes, lane, p.kc,
                                      [&](int rr) -> const __nv_bfloat16* {
                                        const int c = uu * kUnit + rr;
                                        return c < nca ? kbase + c * row_stride : nullptr;
                                      });
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < kDecodeStages - 1; ++i) issue(i, true);
  const int rlo = lane >> 2, rhi = rlo + 8, q4 = lane & 3;
  int q_row = -1, nca = 0;
  uint32_t qa[D / 16][4];
  for (int i = 0; i < n; ++i) {
    issue(i + kDecodeStages - 1, false);
    const int u = first + i * kNW;
    const int row = u / U, uu = u - row * U;
    if (row != q_row) {  // a warp's units cross at most a few row boundaries
      q_row = row;
      const int b = row / p.hkv, g = row % p.hkv;
      nca = decode_nca(p, b);
      const __nv_bfloat16* qb = p.q + ((int64_t)b * p.h + g * R) * D;
      load_a_frags<D>(qa, rlo < R ? qb + rlo * D : nullptr, rhi < R ? qb + rhi * D : nullptr, lane);
    }
    cp_async_wait<kDecodeStages - 1>();
    __syncwarp();
    if (uu * kUnit < nca) {
      const uint32_t sb = ring + (i % kDecodeStages) * kUnitBytes;
      float s[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a) s[a][0] = s[a][1] = s[a][2] = s[a][3] = 0.f;
      qk_16keys<D>(&s[0], qa, sb, 0, lane);
      qk_16keys<D>(&s[2], qa, sb, 16, lane);
      float x_lo = kNegInf, x_hi = kNegInf;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = uu * kUnit + nt * 8 + q4 * 2 + (j & 1);
          s[nt][j] = c < nca ? s[nt][j] * p.scale_log2 : kNegInf;
          if (j < 2) x_lo = fmaxf(x_lo, s[nt][j]); else x_hi = fmaxf(x_hi, s[nt][j]);
        }
      const float mx_lo = quad_max(x_lo), mx_hi = quad_max(x_hi);
      const float m_lo = mx_lo == kNegInf ? 0.f : mx_lo, m_hi = mx_hi == kNegInf ? 0.f : mx_hi;
      float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        s[nt][0] = ex2(s[nt][0] - m_lo);
        s[nt][1] = ex2(s[nt][1] - m_lo);
        s[nt][2] = ex2(s[nt][2] - m_hi);
        s[nt][3] = ex2(s[nt][3] - m_hi);
        l_lo += s[nt][0] + s[nt][1];
        l_hi += s[nt][2] + s[nt][3];
      }
      l_lo = quad_sum(l_lo);
      l_hi = quad_sum(l_hi);
      float* zt = p.z + ((int64_t)row * U + uu) * 8 * R;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {  // n-tile nt holds blocks 2nt and 2nt+1 of the unit
        float x = (q4 & 1) ? s[nt][0] : s[nt][0] + s[nt][1];
        float y = (q4 & 1) ? s[nt][2] : s[nt][2] + s[nt][3];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        y += __shfl_xor_sync(0xffffffffu, y, 1);
        if ((q4 & 1) == 0) {
          const int jl = 2 * nt + (q4 >> 1);
          if (rlo < R) zt[jl * R + rlo] = x;
          if (rhi < R) zt[jl * R + rhi] = y;
        }
      }
      if (q4 == 0) {
        float* um = p.unit_ml + (((int64_t)row * U + uu) * R) * 2;
        if (rlo < R) {
          um[rlo * 2] = m_lo;
          um[rlo * 2 + 1] = l_lo;
        }
        if (rhi < R) {
          um[rhi * 2] = m_hi;
          um[rhi * 2 + 1] = l_hi;
        }
      }
    }
    __syncwarp();  // the stage is refilled by the next iteration's issue
  }
  cp_async_wait<0>();
}

// Selection of one row (b, g), run by the CTA that completed the row's score units:
// the normaliser per head from the units' (max, sum), the pooled block scores, the
// top-k, and the release of the row's block list.  Every thread of the CTA calls it.
template <int D, int R, int NPL, bool W>
__device__ __forceinline__ void select_row(const DecodeParams& p, int row, uint8_t* smem, int* s_topk,
                                           int (*s_two)[64]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = row / p.hkv;
  const int L = p.seqlens[b];
  const int n_c = num_cmp(L, 32, 16);
  const int nca = num_causal_cmp(L - 1, n_c, 32, 16);
  const int n_u = (nca + kUnit - 1) / kUnit;
  const int U = p.n_units;
  // Every global load of the selection is issued in one batch (data written by other
  // SMs costs a full L2 round trip each time): the row's unit (max, sum) pairs go to
  // shared memory, this thread's pooled block partials to registers.
  constexpr int JPT = NPL * 32 / 128;                     // blocks per thread
  constexpr int ZB = JPT * R <= 64 ? JPT : (64 / R > 0 ? 64 / R : 1);  // blocks per batch
  float* red_m = reinterpret_cast<float*>(smem);  // [R][kMaxUnits]
  float* red_l = red_m + R * kMaxUnits;           // [R][kMaxUnits]
  float* sc = red_l + R * kMaxUnits;              // [NPL*32]
  float* fac = sc + NPL * 32;                     // [kMaxUnits][R]
  const int nb = (L + 63) / 64;
  const float* zr = p.z + (int64_t)row * U * 8 * R;
  float zreg[ZB][R];
  auto load_z = [&](int j0) {  // blocks j0 + 128*i, i < ZB
#pragma unroll
    for (int i = 0; i < ZB; ++i) {
      const int j = j0 + 128 * i;
      const bool ok = j < nb && j / 8 < n_u;
#pragma unroll
      for (int hh = 0; hh < R; ++hh) zreg[i][hh] = ok ? __ldcg(zr + (int64_t)j * R + hh) : 0.f;
    }
  };
  for (int i = threadIdx.x; i < R * n_u; i += blockDim.x) {
    const int hh = i / n_u, ul = i % n_u;
    const float* um = p.unit_ml + (((int64_t)row * U + ul) * R + hh) * 2;
    red_m[hh * kMaxUnits + ul] = __ldcg(um);
    red_l[hh * kMaxUnits + ul] = __ldcg(um + 1);
  }
  load_z(threadIdx.x);
  __syncthreads();
  // per-head normaliser: one warp per head folds the unit pairs with shuffles, then
  // writes the factor 2^(m_unit - lse) that turns a unit's partials into probabilities
  for (int hh = warp; hh < R; hh += kNW) {
    float mv[kMaxUnits / 32], lv[kMaxUnits / 32];
    float M = kNegInf;
#pragma unroll
    for (int i = 0; i < kMaxUnits / 32; ++i) {
      const int ul = lane + 32 * i;
      mv[i] = ul < n_u ? red_m[hh * kMaxUnits + ul] : kNegInf;
      lv[i] = ul < n_u ? red_l[hh * kMaxUnits + ul] : 0.f;
      M = fmaxf(M, mv[i]);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mu = M == kNegInf ? 0.f : M;
    float S = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxUnits / 32; ++i) S += lv[i] * ex2(mv[i] - Mu);
#pragma unroll
    for (int off = 16; off; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    const float lse = S > 0.f ? Mu + __log2f(S) : 0.f;
#pragma unroll
    for (int i = 0; i < kMaxUnits / 32; ++i) {
      const int ul = lane + 32 * i;
      if (ul < n_u) fac[ul * R + hh] = ex2(mv[i] - lse);
    }
  }
  __syncthreads();
  // pooled block scores: mean over the windows inside each block
  for (int j0 = threadIdx.x; j0 < NPL * 32; j0 += 128 * ZB) {
    if (j0 != (int)threadIdx.x) load_z(j0);  // only for the largest shapes
#pragma unroll
    for (int i = 0; i < ZB; ++i) {
      const int j = j0 + 128 * i;
      if (j >= NPL * 32) break;
      const int c0 = 4 * j;
      const int cnt = (c0 < n_c) + (c0 + 1 < n_c) + (c0 + 2 < n_c);
      float acc = 0.f;
      if (j < nb && j / 8 < n_u) {
        const float* fj = fac + (j / 8) * R;
#pragma unroll
        for (int hh = 0; hh < R; ++hh) acc += zreg[i][hh] * fj[hh];
      }
      sc[j] = cnt ? acc / (float)cnt : 0.f;
    }
  }
  __syncthreads();
  // the whole CTA runs the top-k (radix select, one barrier per pass), then publishes
  // the list: every thread's writes, the barrier, and one release store
  const int own = (L - 1) / 64;
  if (!W || !p.cis_block) {
    block_topk<NPL * 32 / (kNW * 32), kNW * 32>(sc, nb, own, p.n_init, p.n_local, p.k, p.idx + row * p.k, s_topk);
  } else {
    // stage 1: the forced blocks and the best qk by attention score
    block_topk<NPL * 32 / (kNW * 32), kNW * 32>(sc, nb, own, p.n_init, p.n_local, p.qk, s_two[0], s_topk);
    __syncthreads();
    // stage 2: rank the kept blocks by CIS score (forced first, ties to the lower block)
    const float* cs = p.cis_block + (int64_t)row * p.cis_nb_stride;
    const int e = threadIdx.x;
    int blk = -1;
    uint32_t key = 0u;
    if (e < p.qk) {
      blk = s_two[0][e];
      if (blk >= 0) key = (blk < p.n_init || blk > own - p.n_local) ? 0xffffffffu : order_key(__ldg(cs + blk));
    }
    if (e < 64) {
      s_two[1][e] = (int)key;
      s_two[2][e] = blk;
    }
    __syncthreads();
    bool sel = false;
    if (blk >= 0) {
      int rank = 0;
      for (int f = 0; f < p.qk; ++f) {
        const uint32_t kf = (uint32_t)s_two[1][f];
        rank += s_two[2][f] >= 0 && (kf > key || (kf == key && f < e));
      }
      sel = rank < p.k;
    }
    if (e < 64) s_two[3][e] = sel;
    const int nsel = __syncthreads_count(sel);
    if (sel) {
      int pos = 0;
      for (int f = 0; f < e; ++f) pos += s_two[3][f];
      p.idx[row * p.k + pos] = blk;
    }
    for (int q = nsel + e; q < p.k; q += blockDim.x) p.idx[row * p.k + q] = -1;
  }
  __syncthreads();
  if (threadIdx.x == 0) st_release(&p.ready[row], 1);
}

// Attention item: split `sp` of row (b, g).  Four warps each own a 16-key slice of every
// block in the split's part of the list (warp_attend); the CTA merges the warps, writes
// the split's state O * 2^-M, (M, L); the last split of the row merges all of them.
template <int D, int R, int NSTAGE, bool W>
__device__ __forceinline__ void attn_item(const DecodeParams& p, int b, int g, int sp, uint8_t* smem, int* s_flag,
                                          int (*s_list)[64]) {
  constexpr int BS = 64;
  constexpr int STAGE_BYTES = attend_stage_bytes<D, W>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = warp;  // four warps, four 16-key slices of a 64-key block
  const int row = b * p.hkv + g;
  const int t = p.seqlens[b] - 1;
  const int64_t kv_base = (int64_t)b * p.max_len;
  const int e0 = sp * p.eps, e1 = min(p.k, e0 + p.eps);
  const int hbase = g * R;
  const int rlo = lane >> 2, rhi = rlo + 8;
  const __nv_bfloat16* qb = p.q + ((int64_t)b * p.h + hbase) * D;
  uint32_t qa[D / 16][4];
  load_a_frags<D>(qa, rlo < R ? qb + rlo * D : nullptr, rhi < R ? qb + rhi * D : nullptr, lane);
  // the row's block list is ready once its selecting CTA has released the flag
  if (!cta_wait_ge(&p.ready[row], 1, s_flag)) return;
  // this warp's work list: the split's blocks whose slice starts at or before t
  const int32_t* il = p.idx + (int64_t)row * p.k;
  int cnt = 0;
  for (int base = e0; base < e1; base += 32) {
    const int e = base + lane;
    int blk = -1;
    bool ok = false;
    if (e < e1) {
      blk = __ldcg(il + e);
      ok = blk >= 0 && (int64_t)blk * BS + slice * 16 <= t;
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (ok) s_list[warp][cnt + __popc(m & ((1u << lane) - 1u))] = blk;
    cnt += __popc(m);
  }
  __syncwarp();
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  const uint32_t ring = smem_u32(smem) + warp * NSTAGE * STAGE_BYTES;
  WarpState st = warp_attend<D, BS, NSTAGE, W>(s_list[warp], cnt, slice, p.k_cache + (kv_base * p.hkv + g) * D,
                                               p.v_cache + (kv_base * p.hkv + g) * D, (int64_t)p.hkv * D, t,
                                               p.scale_log2, qa, ring, p.k_cache, o, lane,
                                               W ? p.cis + kv_base * p.hkv + g : nullptr, p.hkv);
  __syncthreads();  // every warp is done with its ring: the merge reuses the shared memory
  cta_merge<D, kNW>(reinterpret_cast<float*>(smem), o, st, warp, lane);
  const int64_t slot = ((int64_t)row * p.n_split + sp) * 16;
  if (warp == 0) {
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(p.part_o + (slot + rlo) * D + col) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(p.part_o + (slot + rhi) * D + col) = make_float2(o[nt][2], o[nt][3]);
    }
    if ((lane & 3) == 0) {
      p.part_ml[(slot + rlo) * 2] = st.m0;
      p.part_ml[(slot + rlo) * 2 + 1] = st.l0;
      p.part_ml[(slot + rhi) * 2] = st.m1;
      p.part_ml[(slot + rhi) * 2 + 1] = st.l1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *s_flag = atom_acq_rel_add(&p.merge_count[row], 1) == p.n_split - 1;
  __syncthreads();
  if (!*s_flag) return;
  const int hr = threadIdx.x >> 3;  // head row of the group, 8 threads per row
  if (hr >= R) return;
  const int64_t base = (int64_t)row * p.n_split;
  float M = kNegInf;
  for (int s2 = 0; s2 < p.n_split; ++s2) M = fmaxf(M, __ldcg(p.part_ml + ((base + s2) * 16 + hr) * 2));
  const float Mu = M == kNegInf ? 0.f : M;
  float L = 0.f;
  float acc[D / 8];
#pragma unroll
  for (int c = 0; c < D / 8; ++c) acc[c] = 0.f;
  const int cl = threadIdx.x & 7;  // columns cl, cl+8, ... : 8 lanes read 32 contiguous bytes
  for (int s2 = 0; s2 < p.n_split; ++s2) {
    const int64_t sl = (base + s2) * 16 + hr;
    const float f = ex2(__ldcg(p.part_ml + sl * 2) - Mu);
    L += f * __ldcg(p.part_ml + sl * 2 + 1);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) acc[c] += f * __ldcg(p.part_o + sl * D + cl + 8 * c);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* dst = p.o + ((int64_t)b * p.h + hbase + hr) * D;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) dst[cl + 8 * c] = __float2bfloat16_rn(acc[c] * inv);
}

// 96 KB of rings: two CTAs per SM
template <bool W>
constexpr int decode_smem() {
  return kNW * kDecodeStages * attend_stage_bytes<128, W>();
}

// The step.  Phase 1: every CTA scores a contiguous run of the (row, unit) space and
// adds its unit count to each row it touched (it waits on nothing).  Phase 2: the CTAs
// take items from the queue, first one selection per row, then the attention items
// (row, split).  A selection waits (bounded) until all of its row's units have arrived,
// an attention item until its row's list is released.  Every CTA is resident
// (cooperative launch) and finishes phase 1 before it takes an item, and the queue
// hands out every selection before any attention item, so every awaited count or list
// is being made by a running CTA.
template <int R, int NPL, bool W>
__global__ void __launch_bounds__(kNW * 32, 2) decode_step(const DecodeParams p, int rows) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_item, s_flag;
  __shared__ __align__(16) int s_topk[block_topk_scratch_ints<kNW * 32>()];  // top-k scratch
  __shared__ int s_list[kNW][64];
  __shared__ int s_two[W ? 4 : 1][64];  // two-stage selection: kept list, keys, blocks, chosen flags
  const int U = p.n_units;
  const int64_t total = (int64_t)rows * U;  // < 2^31 (checked by the launcher)
  const int u0 = (int)(total * blockIdx.x / gridDim.x), u1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  score_units<128, R>(p, u0, u1, smem);
  __syncthreads();
  if (u0 < u1) {
    const int r_first = u0 / U, r_last = (u1 - 1) / U;
    for (int r = r_first + (int)threadIdx.x; r <= r_last; r += kNW * 32) {
      const int lo = u0 > r * U ? u0 : r * U;
      const int hi = u1 < (r + 1) * U ? u1 : (r + 1) * U;
      red_release_add(&p.score_count[r], hi - lo);
    }
  }
  __syncthreads();  // the shared memory of the score rings is reused by the items
  const int n_items = rows + rows * p.n_split;
  for (;;) {
    if (threadIdx.x == 0) s_item = atomicAdd(p.queue, 1);
    __syncthreads();
    const int item = s_item;
    __syncthreads();  // s_item is rewritten only after every thread has read it
    if (item >= n_items || tc::device_status_set()) break;
    if (item < rows) {
      if (cta_wait_ge(&p.score_count[item], U, &s_flag)) {
        select_row<128, R, NPL, W>(p, item, smem, s_topk, s_two);
      }
    } else {
      const int a = item - rows, row = a / p.n_split;
      attn_item<128, R, kDecodeStages, W>(p, row / p.hkv, row % p.hkv, a % p.n_split, smem, &s_flag, s_list);
    }
    __syncthreads();
  }
}

template <int R, int NPL, bool W>
static cudaError_t run_decode(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  constexpr int kDecodeSmem = decode_smem<W>();
  static_assert(2 * R * kMaxUnits * 4 + NPL * 32 * 4 + kMaxUnits * R * 4 <= kDecodeSmem,
                "selection scratch must fit the rings");
  static_assert(kNW * kDecodeStages * kUnitBytes <= kDecodeSmem, "score rings must fit");
  auto kern = decode_step<R, NPL, W>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecodeSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNW * 32, kDecodeSmem)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  DecodeParams p{};
  p.q = (const __nv_bfloat16*)a.q;
  p.kc = (const __nv_bfloat16*)a.kc_cache;
  p.k_cache = (const __nv_bfloat16*)a.k_cache;
  p.v_cache = (const __nv_bfloat16*)a.v_cache;
  p.seqlens = a.seqlens;
  p.h = a.h;
  p.hkv = a.hkv;
  p.max_len = a.max_len;
  p.nc_stride = a.max_len >= a.kernel ? (a.max_len - a.kernel) / a.stride + 1 : 0;
  p.n_units = l.n_units;  // >= 1: a row without compressed keys still has a unit to complete
  p.n_init = a.n_init;
  p.n_local = a.n_local;
  p.k = a.k;
  p.n_split = l.n_split;
  p.eps = (a.k + l.n_split - 1) / l.n_split;
  p.scale_log2 = a.scale * kLog2e;
  p.z = a.z;
  p.unit_ml = a.unit_ml;
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.idx = a.idx;
  p.o = (__nv_bfloat16*)a.o;
  p.cis = a.cis;
  p.cis_block = a.cis_block;
  p.cis_nb_stride = a.cis_nb_stride;
  p.qk = a.qk;
  const int rows = a.batch * a.hkv;
  p.queue = a.counters;
  p.score_count = a.counters + 1;
  p.merge_count = p.score_count + rows;
  p.ready = p.merge_count + rows;
  if ((int64_t)rows * p.n_units >= (int64_t)1 << 31) return cudaErrorInvalidValue;
  const int64_t work = (int64_t)rows * (p.n_units > p.n_split ? p.n_units : p.n_split);
  // persistent: at most one CTA per resident slot (the cooperative launch checks it)
  const int grid = work < (int64_t)per_sm * sms ? (int)work : per_sm * sms;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kNW * 32);
  cfg.dynamicSmemBytes = kDecodeSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, rows);
}

template <int R, bool W>
static cudaError_t run_decode_r(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  const int nb_max = (a.max_len + 63) / 64;
  if (nb_max <= 4 * 32) return run_decode<R, 4, W>(a, l, st);
  if (nb_max <= 8 * 32) return run_decode<R, 8, W>(a, l, st);
  if (nb_max <= 16 * 32) return run_decode<R, 16, W>(a, l, st);
  return run_decode<R, 32, W>(a, l, st);
}

template <bool W>
static cudaError_t run_decode_all(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  switch (a.h / a.hkv) {
    case 1: return run_decode_r<1, W>(a, l, st);
    case 2: return run_decode_r<2, W>(a, l, st);
    case 4: return run_decode_r<4, W>(a, l, st);
    case 8: return run_decode_r<8, W>(a, l, st);
    default: return run_decode_r<16, W>(a, l, st);
  }
}

}  // namespace nsa
