// One decode step: score the newest query against the compressed key cache, pick the
// top-k blocks, attend over them.
//
// [NOSA-Parts] "NOSA-1B core components", how decoding uses only 64 KV blocks: the
// selection picks topk = 64 blocks and the sparse attention runs over those blocks only.
//
// GB300 design.  A decode step has only batch * h_kv independent rows, far fewer than
// the 152 SMs, and the path is HBM bound (compressed keys plus the chosen K/V blocks),
// so every pass is split to fill the machine:
//   1. decode_score: one warp per 64-key tile of compressed keys, for every (sequence,
//      kv-head).  Writes base-2 scaled scores and each tile's (max, sum) per head.
//   2. decode_select: one CTA per (sequence, kv-head): folds the tile partials into the
//      per-head normaliser, pools the group probabilities to 64-token blocks in shared
//      memory and runs the warp top-k.
//   3. the selected-attention kernel in split mode (several CTAs per row, each over a
//      slice of the block list), then a merge of the split softmax states.
// The four launches are stream ordered and capture into one CUDA graph.
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
  int ns = 1;
  while (ns < 16 && (int64_t)batch * hkv * rtiles * ns < 2 * 152) ns *= 2;
  l.n_split = ns < k ? ns : k;
  size_t off = 0;
  l.z = off;
  off = align256(off + (size_t)batch * hkv * r * l.nc_pad * 4);
  l.tile_ml = off;
  off = align256(off + (size_t)batch * hkv * l.n_tiles * r * 2 * 4);
  l.idx = off;
  off = align256(off + (size_t)batch * hkv * k * 4);
  l.part_o = off;
  off = align256(off + (size_t)batch * hkv * rtiles * l.n_split * 16 * d * 4);
  l.part_ml = off;
  off = align256(off + (size_t)batch * hkv * rtiles * l.n_split * 16 * 2 * 4);
  l.total = off;
  return l;
}

constexpr int kTile = 64;

// grid (ceil(n_tiles/4), batch, hkv), 4 warps; warp w scores compressed tile blockIdx.x*4+w.
template <int D, int R>
__global__ void __launch_bounds__(128) decode_score(const __nv_bfloat16* __restrict__ q,
                                                   const __nv_bfloat16* __restrict__ kc, const int32_t* seqlens,
                                                   int h, int hkv, int nc_stride, int nc_pad, int n_tiles,
                                                   float scale_log2, float* z, float* tile_ml) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y, g = blockIdx.z;
  const int tile = blockIdx.x * 4 + warp;
  const int L = seqlens[b];
  const int n_c = num_cmp(L, 32, 16);
  const int nca = num_causal_cmp(L - 1, n_c, 32, 16);
  if (tile * kTile >= nca) return;
  const uint32_t sb = smem_u32(smem) + warp * kTile * D * 2;
  const __nv_bfloat16* kbase = kc + (((int64_t)b * nc_stride) * hkv + g) * D;
  const int64_t row_stride = (int64_t)hkv * D;
  load_tile_async<D, kTile, 32>(sb, lane, kc, [&](int row) -> const __nv_bfloat16* {
    const int c = tile * kTile + row;
    return c < nca ? kbase + c * row_stride : nullptr;
  });
  cp_async_commit();
  const int rlo = lane >> 2, rhi = rlo + 8;
  const __nv_bfloat16* qb = q + ((int64_t)b * h + g * R) * D;
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
      s[nt][j] = c < nca ? s[nt][j] * scale_log2 : kNegInf;
      if (j < 2) x_lo = fmaxf(x_lo, s[nt][j]); else x_hi = fmaxf(x_hi, s[nt][j]);
    }
  const float m_lo = quad_max(x_lo), m_hi = quad_max(x_hi);
  float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    l_lo += ex2(s[nt][0] - m_lo) + ex2(s[nt][1] - m_lo);
    l_hi += ex2(s[nt][2] - m_hi) + ex2(s[nt][3] - m_hi);
  }
  l_lo = quad_sum(l_lo);
  l_hi = quad_sum(l_hi);
  const int64_t zrow = ((int64_t)b * hkv + g) * R;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int c = tile * kTile + nt * 8 + (lane & 3) * 2;
    if (rlo < R) *reinterpret_cast<float2*>(z + (zrow + rlo) * nc_pad + c) = make_float2(s[nt][0], s[nt][1]);
    if (rhi < R) *reinterpret_cast<float2*>(z + (zrow + rhi) * nc_pad + c) = make_float2(s[nt][2], s[nt][3]);
  }
  if ((lane & 3) == 0) {
    float* tm = tile_ml + ((((int64_t)b * hkv + g) * n_tiles + tile) * R) * 2;
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

// grid (batch, hkv), 256 threads.
template <int R, int NPL>
__global__ void __launch_bounds__(256) decode_select(const float* __restrict__ z, const float* __restrict__ tile_ml,
                                                    const int32_t* seqlens, int hkv, int nc_pad, int n_tiles,
                                                    int n_init, int n_local, int k, int32_t* idx) {
  __shared__ float lse2[16];
  __shared__ __align__(16) float sc[NPL * 32];
  const int b = blockIdx.x, g = blockIdx.y;
  const int L = seqlens[b];
  const int t = L - 1;
  const int n_c = num_cmp(L, 32, 16);
  const int nca = num_causal_cmp(t, n_c, 32, 16);
  const int nt = (nca + kTile - 1) / kTile;
  const int nb = (L + 63) / 64;
  const int64_t row = (int64_t)b * hkv + g;
  if (threadIdx.x < R) {
    const float* tm = tile_ml + (row * n_tiles * R + threadIdx.x) * 2;
    float M = kNegInf;
    for (int i = 0; i < nt; ++i) M = fmaxf(M, tm[(int64_t)i * R * 2]);
    const float Mu = M == kNegInf ? 0.f : M;
    float S = 0.f;
    for (int i = 0; i < nt; ++i) S += tm[(int64_t)i * R * 2 + 1] * ex2(tm[(int64_t)i * R * 2] - Mu);
    lse2[threadIdx.x] = S > 0.f ? Mu + __log2f(S) : 0.f;
  }
  __syncthreads();
  const float* zr = z + row * R * nc_pad;
  for (int j = threadIdx.x; j < NPL * 32; j += blockDim.x) {
    float acc = 0.f;
    int cnt = 0;
    if (j < nb) {
#pragma unroll
      for (int w = 0; w < 3; ++w) {
        const int c = 4 * j + w;
        if (c >= n_c) continue;
        ++cnt;
        if (c >= nca) continue;
#pragma unroll
        for (int hh = 0; hh < R; ++hh) acc += ex2(zr[(int64_t)hh * nc_pad + c] - lse2[hh]);
      }
    }
    sc[j] = cnt ? acc / (float)cnt : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < 32)
    warp_topk<NPL, true>(sc, nb, t / 64, n_init, n_local, k, idx + row * k, threadIdx.x);
}

template <int R>
static cudaError_t run_decode_select(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  const int nb_max = (a.max_len + 63) / 64;
  dim3 grid(a.batch, a.hkv);
#define NSA_DSEL(N)                                                                                     \
  if (nb_max <= N * 32) {                                                                              \
    decode_select<R, N><<<grid, 256, 0, st>>>(a.z, a.tile_ml, a.seqlens, a.hkv, l.nc_pad, l.n_tiles,     \
                                              a.n_init, a.n_local, a.k, a.idx);                        \
    return cudaGetLastError();                                                                         \
  }
  NSA_DSEL(4)
  NSA_DSEL(8)
  NSA_DSEL(16)
  NSA_DSEL(32)
#undef NSA_DSEL
  return cudaErrorInvalidValue;
}

template <int R>
static cudaError_t run_decode_r(const DecodeArgs& a, const DecodeLayout& l, cudaStream_t st) {
  const int nc_stride = a.max_len >= a.kernel ? (a.max_len - a.kernel) / a.stride + 1 : 0;
  if (l.n_tiles > 0) {
    constexpr int bytes = 4 * kTile * 128 * 2;
    cudaError_t e = cudaFuncSetAttribute(decode_score<128, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((l.n_tiles + 3) / 4, a.batch, a.hkv);
    decode_score<128, R><<<grid, 128, bytes, st>>>((const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kc_cache,
                                                   a.seqlens, a.h, a.hkv, nc_stride, l.nc_pad, l.n_tiles,
                                                   a.scale * kLog2e, a.z, a.tile_ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = run_decode_select<R>(a, l, st);
  if (e != cudaSuccess) return e;
  return launch_decode_attn(a, st);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  const DecodeLayout l = decode_layout(a.batch, a.max_len, a.h, a.hkv, a.d, a.kernel, a.stride, a.block_size, a.k);
  switch (a.h / a.hkv) {
    case 1: return run_decode_r<1>(a, l, st);
    case 2: return run_decode_r<2>(a, l, st);
    case 4: return run_decode_r<4>(a, l, st);
    case 8: return run_decode_r<8>(a, l, st);
    default: return run_decode_r<16>(a, l, st);
  }
}

}  // namespace nsa
