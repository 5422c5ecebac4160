// One decode step: score the newest query against the compressed key cache, pick the
// top-k blocks, attend over them.
//
// [NOSA-Parts] "NOSA-1B core components", how decoding uses only 64 KV blocks: the
// selection picks topk = 64 blocks and the sparse attention runs over those blocks only.
//
// GB300 design.  A decode step has only batch * h_kv independent rows, far fewer than
// the 152 SMs, and the path is HBM bound (compressed keys plus the chosen K/V blocks),
// so both passes are split to fill the machine:
//   1. decode_score_select: one warp per 64-key tile of compressed keys, for every
//      (sequence, kv-head); it writes base-2 scaled scores and each tile's (max, sum) per
//      head.  The last CTA of a (sequence, kv-head) to finish (arrival counter) folds the
//      tile partials into the per-head normaliser, pools the group probabilities to
//      64-token blocks in shared memory and runs the warp top-k.
//   2. the selected-attention kernel in split mode (several CTAs per row, each over a
//      slice of the block list); the last split CTA merges the softmax states.
// A memset of the arrival counters and the two kernels are stream ordered and capture
// into one CUDA graph.
#include "launch.h"
#include "topk.cuh"

namespace nsa {

cudaError_t launch_decode_attn(const DecodeArgs& a, cudaStream_t st);

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

DecodeLayout decode_layout(int batch, int max_len, int h, int hkv, int d, int kernel, int stride,
                           int block_size, int k) {
  DecodeLayout l{};
  const int r = h / hkv;
  const int rtiles = (r + 15) / 16;
  const int nc_max = max_len >= kernel ? (max_len - kernel) / stride + 1 : 0;
  l.n_tiles = (nc_max + 63) / 64;
  l.nc_pad = l.n_tiles * 64;
#ifdef NSA_DECODE_SPLIT
  int ns = NSA_DECODE_SPLIT;
#else
  // as many splits as keep the attention grid within one resident wave (2 CTAs per SM)
  const int64_t units = (int64_t)batch * hkv * rtiles;
  int ns = (int)(2 * 152 / (units > 0 ? units : 1));
  ns = ns < 1 ? 1 : (ns > 16 ? 16 : ns);
#endif
  l.n_split = ns < k ? ns : k;
  size_t off = 0;
  l.z = off;  // per-tile pooled partial sums [batch, hkv, n_tiles, 16 blocks, r]
  off = align256(off + (size_t)batch * hkv * l.n_tiles * 16 * r * 4);
  l.tile_ml = off;
  off = align256(off + (size_t)batch * hkv * l.n_tiles * r * 2 * 4);
  l.idx = off;
  off = align256(off + (size_t)batch * hkv * k * 4);
  l.part_o = off;
  off = align256(off + (size_t)batch * hkv * rtiles * l.n_split * 16 * d * 4);
  l.part_ml = off;
  off = align256(off + (size_t)batch * hkv * rtiles * l.n_split * 16 * 2 * 4);
  l.counters = off;
  l.counter_bytes = (size_t)batch * hkv * (1 + rtiles) * 4;
  off = align256(off + l.counter_bytes);
  l.total = off;
  return l;
}

constexpr int kTile = 64;

// grid (ceil(n_tiles/4), batch, hkv), 4 warps; warp w scores compressed tile blockIdx.x*4+w;
// the last CTA of each (sequence, kv-head) then selects its blocks.
constexpr int kMaxTiles = 64;  // max_len <= 65536

struct ScoreSelectParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const int32_t* seqlens;
  int h, hkv, nc_stride, nc_pad, n_tiles, n_init, n_local, k;
  float scale_log2;
  float* z;
  float* tile_ml;
  int32_t* idx;
  int* count;
};

template <int D, int R, int NPL>
__global__ void __launch_bounds__(128) decode_score_select(const ScoreSelectParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y, g = blockIdx.z;
  const int tile = blockIdx.x * 4 + warp;
  const int L = p.seqlens[b];
  const int n_c = num_cmp(L, 32, 16);
  const int nca = num_causal_cmp(L - 1, n_c, 32, 16);
  const int n_tb = (nca + kTile - 1) / kTile;
  const int64_t row = (int64_t)b * p.hkv + g;
  if (tile < n_tb) {
    const uint32_t sb = smem_u32(smem) + warp * kTile * D * 2;
    const __nv_bfloat16* kbase = p.kc + (((int64_t)b * p.nc_stride) * p.hkv + g) * D;
    const int64_t row_stride = (int64_t)p.hkv * D;
    load_tile_async<D, kTile, 32>(sb, lane, p.kc, [&](int rr) -> const __nv_bfloat16* {
      const int c = tile * kTile + rr;
      return c < nca ? kbase + c * row_stride : nullptr;
    });
    cp_async_commit();
    const int rlo = lane >> 2, rhi = rlo + 8;
    const __nv_bfloat16* qb = p.q + ((int64_t)b * p.h + g * R) * D;
    uint32_t qa[D / 16][4];
    load_a_frags<D>(qa, rlo < R ? qb + rlo * D : nullptr, rhi < R ? qb + rhi * D : nullptr, lane);
    cp_async_wait<0>();
    __syncwarp();
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int k16 = 0; k16 < 4; ++k16) qk_16keys<D>(&s[2 * k16], qa, sb, k16 * 16, lane);
    float x_lo = kNegInf, x_hi = kNegInf;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = tile * kTile + nt * 8 + (lane & 3) * 2 + (j & 1);
        s[nt][j] = c < nca ? s[nt][j] * p.scale_log2 : kNegInf;
        if (j < 2) x_lo = fmaxf(x_lo, s[nt][j]); else x_hi = fmaxf(x_hi, s[nt][j]);
      }
    const float mx_lo = quad_max(x_lo), mx_hi = quad_max(x_hi);
    const float m_lo = mx_lo == kNegInf ? 0.f : mx_lo, m_hi = mx_hi == kNegInf ? 0.f : mx_hi;
    float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      l_lo += ex2(s[nt][0] - m_lo) + ex2(s[nt][1] - m_lo);
      l_hi += ex2(s[nt][2] - m_hi) + ex2(s[nt][3] - m_hi);
    }
    l_lo = quad_sum(l_lo);
    l_hi = quad_sum(l_hi);
    // pooled partials of this tile relative to its own row max: block jl (0..15) of the
    // tile sums the windows 4jl, 4jl+1, 4jl+2 (n-tile nt holds blocks 2nt and 2nt+1)
    float* zt = p.z + (row * p.n_tiles + tile) * 16 * R;
    const int q4 = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = ex2(s[nt][0] - m_lo), p1 = ex2(s[nt][1] - m_lo);
      const float p2 = ex2(s[nt][2] - m_hi), p3 = ex2(s[nt][3] - m_hi);
      float x = (q4 & 1) ? p0 : p0 + p1;
      float y = (q4 & 1) ? p2 : p2 + p3;
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      y += __shfl_xor_sync(0xffffffffu, y, 1);
      if ((q4 & 1) == 0) {
        const int jl = 2 * nt + (q4 >> 1);
        if (rlo < R) zt[jl * R + rlo] = x;
        if (rhi < R) zt[jl * R + rhi] = y;
      }
    }
    if ((lane & 3) == 0) {
      float* tm = p.tile_ml + ((row * p.n_tiles + tile) * R) * 2;
      if (rlo < R) {
        tm[rlo * 2] = m_lo;
        tm[rlo * 2 + 1] = l_lo;
      }
      if (rhi < R) {
        tm[rhi * 2] = m_hi;
        tm[rhi * 2 + 1] = l_hi;
      }
    }
  }
  // allow the dependent attention grid to start its prologue; it waits for this grid's
  // writes (griddepcontrol.wait) before reading the block lists
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // arrival: the last CTA of this (sequence, kv-head) runs the selection
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.count[row], 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Every global load of the selection is issued in one batch (data written by other
  // SMs costs a full L2 round trip each time): the row's tile (max, sum) pairs go to
  // shared memory, this thread's pooled block partials to registers.
  constexpr int JPT = NPL * 32 / 128;                     // blocks per thread
  constexpr int ZB = JPT * R <= 64 ? JPT : (64 / R > 0 ? 64 / R : 1);  // blocks per batch
  float* red_m = reinterpret_cast<float*>(smem);  // [R][kMaxTiles]
  float* red_l = red_m + R * kMaxTiles;           // [R][kMaxTiles]
  float* sc = red_l + R * kMaxTiles;              // [NPL*32]
  float* fac = sc + NPL * 32;                     // [kMaxTiles][R]
  const int nb = (L + 63) / 64;
  const float* zr = p.z + row * p.n_tiles * 16 * R;
  float zreg[ZB][R];
  auto load_z = [&](int j0) {  // blocks j0 + 128*i, i < ZB
#pragma unroll
    for (int i = 0; i < ZB; ++i) {
      const int j = j0 + 128 * i;
      const bool ok = j < nb && j / 16 < n_tb;
#pragma unroll
      for (int hh = 0; hh < R; ++hh) zreg[i][hh] = ok ? __ldcg(zr + (int64_t)j * R + hh) : 0.f;
    }
  };
  for (int i = threadIdx.x; i < R * n_tb; i += blockDim.x) {
    const int hh = i / n_tb, tl = i % n_tb;
    const float* tm = p.tile_ml + ((row * p.n_tiles + tl) * R + hh) * 2;
    red_m[hh * kMaxTiles + tl] = __ldcg(tm);
    red_l[hh * kMaxTiles + tl] = __ldcg(tm + 1);
  }
  load_z(threadIdx.x);
  __syncthreads();
  // per-head normaliser: one warp per head folds the tile pairs with shuffles, then
  // writes the factor 2^(m_tile - lse) that turns a tile's partials into probabilities
  for (int hh = warp; hh < R; hh += 4) {
    float mv[kMaxTiles / 32], lv[kMaxTiles / 32];
    float M = kNegInf;
#pragma unroll
    for (int i = 0; i < kMaxTiles / 32; ++i) {
      const int tl = lane + 32 * i;
      mv[i] = tl < n_tb ? red_m[hh * kMaxTiles + tl] : kNegInf;
      lv[i] = tl < n_tb ? red_l[hh * kMaxTiles + tl] : 0.f;
      M = fmaxf(M, mv[i]);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mu = M == kNegInf ? 0.f : M;
    float S = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxTiles / 32; ++i) S += lv[i] * ex2(mv[i] - Mu);
#pragma unroll
    for (int off = 16; off; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    const float lse = S > 0.f ? Mu + __log2f(S) : 0.f;
#pragma unroll
    for (int i = 0; i < kMaxTiles / 32; ++i) {
      const int tl = lane + 32 * i;
      if (tl < n_tb) fac[tl * R + hh] = ex2(mv[i] - lse);
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
      if (j < nb && j / 16 < n_tb) {
        const float* fj = fac + (j / 16) * R;
#pragma unroll
        for (int hh = 0; hh < R; ++hh) acc += zreg[i][hh] * fj[hh];
      }
      sc[j] = cnt ? acc / (float)cnt : 0.f;
    }
  }
  __syncthreads();
  // the whole CTA runs the top-k: this tail sits on the critical path of the step
  __shared__ int s_topk[3 * 4];
  block_topk<NPL * 32 / 128, 128>(sc, nb, (L - 1) / 64, p.n_init, p.n_local, p.k, p.idx + row * p.k, s_topk);
}

template <int R, int NPL>
static cudaError_t run_score_select(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  constexpr int bytes = 4 * kTile * 128 * 2;
  static_assert(2 * R * kMaxTiles * 4 + NPL * 32 * 4 + kMaxTiles * R * 4 <= bytes,
                "select scratch must fit the tile buffers");
  auto kern = decode_score_select<128, R, NPL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  ScoreSelectParams p{};
  p.q = (const __nv_bfloat16*)a.q;
  p.kc = (const __nv_bfloat16*)a.kc_cache;
  p.seqlens = a.seqlens;
  p.h = a.h;
  p.hkv = a.hkv;
  p.nc_stride = a.max_len >= a.kernel ? (a.max_len - a.kernel) / a.stride + 1 : 0;
  p.nc_pad = l.nc_pad;
  p.n_tiles = l.n_tiles;
  p.n_init = a.n_init;
  p.n_local = a.n_local;
  p.k = a.k;
  p.scale_log2 = a.scale * kLog2e;
  p.z = a.z;
  p.tile_ml = a.tile_ml;
  p.idx = a.idx;
  p.count = a.select_count;
  dim3 grid((l.n_tiles + 3) / 4 > 0 ? (l.n_tiles + 3) / 4 : 1, a.batch, a.hkv);
  kern<<<grid, 128, bytes, st>>>(p);
  return cudaGetLastError();
}

template <int R>
static cudaError_t run_decode_r(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  const int nb_max = (a.max_len + 63) / 64;
  cudaError_t e;
  if (nb_max <= 4 * 32) e = run_score_select<R, 4>(a, l, st);
  else if (nb_max <= 8 * 32) e = run_score_select<R, 8>(a, l, st);
  else if (nb_max <= 16 * 32) e = run_score_select<R, 16>(a, l, st);
  else e = run_score_select<R, 32>(a, l, st);
  if (e != cudaSuccess) return e;
  return launch_decode_attn(a, st);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  const DecodeLayout l = decode_layout(a.batch, a.max_len, a.h, a.hkv, a.d, a.kernel, a.stride, a.block_size, a.k);
  // arrival counters start at zero on every call (a memset, not an allocation)
  cudaError_t e = cudaMemsetAsync(a.select_count, 0, l.counter_bytes, st);
  if (e != cudaSuccess) return e;
  switch (a.h / a.hkv) {
    case 1: return run_decode_r<1>(a, l, st);
    case 2: return run_decode_r<2>(a, l, st);
    case 4: return run_decode_r<4>(a, l, st);
    case 8: return run_decode_r<8>(a, l, st);
    default: return run_decode_r<16>(a, l, st);
  }
}

}  // namespace nsa
