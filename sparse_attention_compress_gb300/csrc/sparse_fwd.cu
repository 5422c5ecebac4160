// Selected-block attention (prefill and the split decode pass).
//
// [TileLang-NSA] "TileLang operator development: Native Sparse Attention", sec. 2:
// for each entry of a query's block list, the block starting at index*block_size is
// attended when it starts at or before the query; keys past the query are masked.
// [NSA-Triton] "DeepSeek NSA ... with Triton", sec. 1.2 (group-centric loading): all
// query heads of a GQA group share one K/V block fetch.
//
// GB300 design.  One CTA serves one (query token, kv-head) and every query head of the
// group (up to 16 rows: the M of one m16n8k16 tile).  Its four warps split each 64-key
// block into four 16-key slices; each warp streams its slice of every listed block
// through a private cp.async ring, runs its own online softmax (base-2 exponentials
// with scale*log2(e) folded in, [TileLang-NSA] sec. 3.1) and the warps merge their
// (max, sum, O) states once at the end.  Warps never wait on one another inside the
// loop, so no CTA-wide barrier sits on the gather path.
#include "launch.h"

namespace nsa {

struct SparseParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* idx;
  __nv_bfloat16* o;
  float* lse;
  Seqs seqs;
  int h, hkv, S;
  float scale_log2;
  // decode: query row b sits at t = seqlens[b]-1 over cache rows b*max_len ..
  const int32_t* seqlens;
  int max_len;
  int entries_per_split;
  float* part_o;
  float* part_ml;
  int* merge_count;  // decode: [batch, gridDim.y] split arrivals, zero at launch
};

#ifndef NSA_PREFILL_NSTAGE
#define NSA_PREFILL_NSTAGE 2
#endif
#ifndef NSA_PREFILL_MINBLOCKS
#define NSA_PREFILL_MINBLOCKS 3
#endif

#ifndef NSA_DECODE_NSTAGE
#define NSA_DECODE_NSTAGE 2
#endif

// Softmax state is rescaled lazily: the running max m only moves when a new score
// exceeds it by more than 2^kLazy in base 2, so exponentials stay below 2^kLazy and
// almost no iteration pays the O rescale (the final normalisation is unchanged).
constexpr float kLazy = 8.f;

template <int D, int BS, int NSTAGE, bool DECODE>
__global__ void __launch_bounds__(128, NSA_PREFILL_MINBLOCKS) sparse_fwd_mma(const SparseParams p) {
  constexpr int NW = 4;
  constexpr int NSLICE = BS / 16;
  constexpr int NGROUP = NW / NSLICE;
  constexpr int SLICE_BYTES = 16 * D * 2;
  constexpr int STAGE_BYTES = 2 * SLICE_BYTES;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_list[NW][64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = warp % NSLICE, grp = warp / NSLICE;
  const int r = p.h / p.hkv;
  const int rtiles = (r + 15) >> 4;
  const int g = blockIdx.y / rtiles, rt = blockIdx.y % rtiles;

  int64_t qrow = blockIdx.x, kv_base;
  int t;
  if (DECODE) {
    t = p.seqlens[qrow] - 1;
    kv_base = qrow * (int64_t)p.max_len;
  } else {
    int sq = seq_of_token(p.seqs, qrow);
    kv_base = seq_start(p.seqs, sq);
    t = (int)(qrow - kv_base);
  }
  const int e0 = DECODE ? blockIdx.z * p.entries_per_split : 0;
  const int e1 = DECODE ? min(p.S, e0 + p.entries_per_split) : p.S;

  // Q fragments of the group's heads (rows past the group read as zero)
  const int hbase = g * r + rt * 16;
  const int rlo = lane >> 2, rhi = rlo + 8;
  const __nv_bfloat16* qb = p.q + (qrow * p.h + hbase) * D;
  uint32_t qa[D / 16][4];
  load_a_frags<D>(qa, rt * 16 + rlo < r ? qb + rlo * D : nullptr, rt * 16 + rhi < r ? qb + rhi * D : nullptr,
                  lane);
  // decode runs as a programmatic dependent launch: everything above overlaps the
  // selection kernel; the block lists it writes are read only after this point
  if (DECODE) asm volatile("griddepcontrol.wait;\n" ::: "memory");

  // this warp's work list: listed blocks whose slice starts at or before t
  const int32_t* il = p.idx + (qrow * p.hkv + g) * p.S;
  int cnt = 0;
  for (int base = e0; base < e1; base += 32) {
    const int e = base + lane;
    int blk = -1;
    bool ok = false;
    if (e < e1) {
      blk = il[e];
      ok = ((e - e0) % NGROUP == grp) && blk >= 0 && (int64_t)blk * BS + slice * 16 <= t;
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (ok) s_list[warp][cnt + __popc(m & ((1u << lane) - 1u))] = blk;
    cnt += __popc(m);
  }
  __syncwarp();

  const uint32_t wbase = smem_u32(smem) + warp * NSTAGE * STAGE_BYTES;
  const int64_t row_stride = (int64_t)p.hkv * D;
  auto issue = [&](int i) {
    const int64_t key0 = (int64_t)s_list[warp][i] * BS + slice * 16;
    const uint32_t sb = wbase + (i % NSTAGE) * STAGE_BYTES;
    const __nv_bfloat16* kb = p.k + ((kv_base + key0) * p.hkv + g) * D;
    const __nv_bfloat16* vb = p.v + ((kv_base + key0) * p.hkv + g) * D;
    const bool full = key0 + 15 <= t;
    constexpr int CH = D / 8;
#pragma unroll
    for (int c = lane; c < 16 * CH; c += 32) {
      const int row = c / CH, ch = c % CH;
      const bool ok = full || key0 + row <= t;
      const int64_t off = row * row_stride + ch * 8;
      cp_async16(tile_addr<D>(sb, row, ch), ok ? kb + off : p.k, ok ? 16 : 0);
      cp_async16(tile_addr<D>(sb + SLICE_BYTES, row, ch), ok ? vb + off : p.v, ok ? 16 : 0);
    }
  };

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;

#pragma unroll
  for (int i = 0; i < NSTAGE - 1; ++i) {
    if (i < cnt) issue(i);
    cp_async_commit();
  }
  for (int i = 0; i < cnt; ++i) {
    if (i + NSTAGE - 1 < cnt) issue(i + NSTAGE - 1);
    cp_async_commit();
    cp_async_wait<NSTAGE - 1>();
    __syncwarp();
    const uint32_t sb = wbase + (i % NSTAGE) * STAGE_BYTES;
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    qk_16keys_2acc<D>(s, s2, qa, sb, 0, lane);
    const int64_t key0 = (int64_t)s_list[warp][i] * BS + slice * 16;
    if (key0 + 15 <= t) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[nt][j] = (s[nt][j] + s2[nt][j]) * p.scale_log2;
    } else {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t key = key0 + nt * 8 + (lane & 3) * 2 + (j & 1);
          s[nt][j] = key <= t ? (s[nt][j] + s2[nt][j]) * p.scale_log2 : kNegInf;
        }
    }
    const float mx0 = quad_max(fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1])));
    const float mx1 = quad_max(fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3])));
    if (!__all_sync(0xffffffffu, mx0 <= m0 + kLazy && mx1 <= m1 + kLazy)) {
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float a0 = ex2(m0 - (mn0 == kNegInf ? 0.f : mn0)), a1 = ex2(m1 - (mn1 == kNegInf ? 0.f : mn1));
      m0 = mn0;
      m1 = mn1;
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        o[nt][0] *= a0;
        o[nt][1] *= a0;
        o[nt][2] *= a1;
        o[nt][3] *= a1;
      }
    }
    const float mu0 = m0 == kNegInf ? 0.f : m0, mu1 = m1 == kNegInf ? 0.f : m1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = ex2(s[nt][0] - mu0);
      pr[nt][1] = ex2(s[nt][1] - mu0);
      pr[nt][2] = ex2(s[nt][2] - mu1);
      pr[nt][3] = ex2(s[nt][3] - mu1);
    }
    l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
    l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
    const uint32_t pa[4] = {pack_bf16(pr[0][0], pr[0][1]), pack_bf16(pr[0][2], pr[0][3]),
                            pack_bf16(pr[1][0], pr[1][1]), pack_bf16(pr[1][2], pr[1][3])};
    pv_16keys<D>(o, pa, sb + SLICE_BYTES, 0, lane);
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();  // every warp is done with its ring: reuse shared memory to merge

  // Warps 1..3 park their (m, l, O) fragments in shared memory; warp 0 merges them
  // into its own registers in the same fragment layout (rows padded by 8 floats so the
  // 8-byte fragment stores and loads are free of bank conflicts).
  constexpr int OS = D + 8;
  float* sm_o = reinterpret_cast<float*>(smem);  // [NW][16][OS]
  float* sm_m = sm_o + NW * 16 * OS;             // [NW][16]
  float* sm_l = sm_m + NW * 16;                  // [NW][16]
  l0 = quad_sum(l0);
  l1 = quad_sum(l1);
  if (warp > 0) {
    if ((lane & 3) == 0) {
      sm_m[warp * 16 + rlo] = m0;
      sm_m[warp * 16 + rhi] = m1;
      sm_l[warp * 16 + rlo] = l0;
      sm_l[warp * 16 + rhi] = l1;
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(&sm_o[(warp * 16 + rlo) * OS + col]) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(&sm_o[(warp * 16 + rhi) * OS + col]) = make_float2(o[nt][2], o[nt][3]);
    }
  }
  __syncthreads();
  if (warp > 0) {
    if (!DECODE) return;
  } else {
    float M0 = m0, M1 = m1;
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      M0 = fmaxf(M0, sm_m[w * 16 + rlo]);
      M1 = fmaxf(M1, sm_m[w * 16 + rhi]);
    }
    const float u0 = M0 == kNegInf ? 0.f : M0, u1 = M1 == kNegInf ? 0.f : M1;
    float f0[NW], f1[NW];
    f0[0] = ex2(m0 - u0);
    f1[0] = ex2(m1 - u1);
    float L0 = f0[0] * l0, L1 = f1[0] * l1;
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      f0[w] = ex2(sm_m[w * 16 + rlo] - u0);
      f1[w] = ex2(sm_m[w * 16 + rhi] - u1);
      L0 += f0[w] * sm_l[w * 16 + rlo];
      L1 += f1[w] * sm_l[w * 16 + rhi];
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      float a0 = f0[0] * o[nt][0], a1 = f0[0] * o[nt][1], a2 = f1[0] * o[nt][2], a3 = f1[0] * o[nt][3];
#pragma unroll
      for (int w = 1; w < NW; ++w) {
        const float2 x = *reinterpret_cast<const float2*>(&sm_o[(w * 16 + rlo) * OS + col]);
        const float2 y = *reinterpret_cast<const float2*>(&sm_o[(w * 16 + rhi) * OS + col]);
        a0 += f0[w] * x.x;
        a1 += f0[w] * x.y;
        a2 += f1[w] * y.x;
        a3 += f1[w] * y.y;
      }
      o[nt][0] = a0;
      o[nt][1] = a1;
      o[nt][2] = a2;
      o[nt][3] = a3;
    }
    if (!DECODE) {
      const float i0 = L0 > 0.f ? 1.f / L0 : 0.f, i1 = L1 > 0.f ? 1.f / L1 : 0.f;
      const bool w0 = rt * 16 + rlo < r, w1 = rt * 16 + rhi < r;
      __nv_bfloat16* d0 = p.o + (qrow * p.h + hbase + rlo) * D;
      __nv_bfloat16* d1 = p.o + (qrow * p.h + hbase + rhi) * D;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        const int col = nt * 8 + (lane & 3) * 2;
        if (w0) *reinterpret_cast<uint32_t*>(d0 + col) = pack_bf16(o[nt][0] * i0, o[nt][1] * i0);
        if (w1) *reinterpret_cast<uint32_t*>(d1 + col) = pack_bf16(o[nt][2] * i1, o[nt][3] * i1);
      }
      if (p.lse && (lane & 3) == 0) {
        if (w0) p.lse[qrow * p.h + hbase + rlo] = L0 > 0.f ? (u0 + __log2f(L0)) * kLn2 : kNegInf;
        if (w1) p.lse[qrow * p.h + hbase + rhi] = L1 > 0.f ? (u1 + __log2f(L1)) * kLn2 : kNegInf;
      }
      return;
    }
    // decode: unnormalised partial state of this split, O * 2^-u, (M, L)
    const int64_t slot = ((qrow * gridDim.y + blockIdx.y) * gridDim.z + blockIdx.z) * 16;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(p.part_o + (slot + rlo) * D + col) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(p.part_o + (slot + rhi) * D + col) = make_float2(o[nt][2], o[nt][3]);
    }
    if ((lane & 3) == 0) {
      p.part_ml[(slot + rlo) * 2] = M0;
      p.part_ml[(slot + rlo) * 2 + 1] = L0;
      p.part_ml[(slot + rhi) * 2] = M1;
      p.part_ml[(slot + rhi) * 2 + 1] = L1;
    }
  }
  if (DECODE) {
    // The last split CTA of this (sequence, row tile) merges every split's state.
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      s_last = atomicAdd(&p.merge_count[qrow * gridDim.y + blockIdx.y], 1) == (int)gridDim.z - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int row = threadIdx.x >> 3;
    if (rt * 16 + row >= r) return;
    const int64_t base = (qrow * gridDim.y + blockIdx.y) * gridDim.z;
    float M = kNegInf;
    for (int sp = 0; sp < (int)gridDim.z; ++sp) M = fmaxf(M, __ldcg(p.part_ml + ((base + sp) * 16 + row) * 2));
    const float Mu = M == kNegInf ? 0.f : M;
    float L = 0.f;
    float acc[D / 8];
#pragma unroll
    for (int c = 0; c < D / 8; ++c) acc[c] = 0.f;
    const int cl = threadIdx.x & 7;  // columns cl, cl+8, ... : 8 lanes read 32 contiguous bytes
    for (int sp = 0; sp < (int)gridDim.z; ++sp) {
      const int64_t sl = (base + sp) * 16 + row;
      const float f = ex2(__ldcg(p.part_ml + sl * 2) - Mu);
      L += f * __ldcg(p.part_ml + sl * 2 + 1);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) acc[c] += f * __ldcg(p.part_o + sl * D + cl + 8 * c);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* dst = p.o + (qrow * p.h + hbase + row) * D;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) dst[cl + 8 * c] = __float2bfloat16_rn(acc[c] * inv);
  }
}

// fp32 selected attention on CUDA cores (small problems; exact fp32 arithmetic).
// One CTA per (token, kv-head); warp w serves heads w, w+4, ... of the group.
__global__ void __launch_bounds__(128) sparse_fwd_f32(const float* __restrict__ q, const float* __restrict__ k,
                                                      const float* __restrict__ v, const int32_t* __restrict__ idx,
                                                      float* __restrict__ o, float* __restrict__ lse, Seqs seqs,
                                                      int h, int hkv, int d, int S, int bs, float scale) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int max_keys = S * bs;
  int* keys = reinterpret_cast<int*>(smem);
  float* sc = reinterpret_cast<float*>(keys + max_keys);  // [4][max_keys]
  __shared__ int s_n;
  const int64_t tok = blockIdx.x;
  const int g = blockIdx.y;
  const int r = h / hkv;
  const int sq = seq_of_token(seqs, tok);
  const int64_t start = seq_start(seqs, sq);
  const int t = (int)(tok - start);
  if (threadIdx.x == 0) {
    int n = 0;
    const int32_t* il = idx + (tok * hkv + g) * S;
    for (int e = 0; e < S; ++e) {
      const int64_t b = il[e];
      if (b < 0 || b * bs > t) continue;
      for (int64_t tau = b * bs; tau < (b + 1) * bs && tau <= t; ++tau) keys[n++] = (int)tau;
    }
    s_n = n;
  }
  __syncthreads();
  const int n = s_n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* my = sc + warp * max_keys;
  for (int j = warp; j < r; j += 4) {
    const int hh = g * r + j;
    const float* qr = q + (tok * h + hh) * d;
    float mx = -INFINITY;
    for (int e = lane; e < n; e += 32) {
      const float* kr = k + ((start + keys[e]) * hkv + g) * d;
      float acc = 0.f;
      for (int i = 0; i < d; ++i) acc = fmaf(qr[i], kr[i], acc);
      acc *= scale;
      my[e] = acc;
      mx = fmaxf(mx, acc);
    }
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float sum = 0.f;
    for (int e = lane; e < n; e += 32) {
      const float pe = expf(my[e] - mx);
      my[e] = pe;
      sum += pe;
    }
    for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    __syncwarp();
    const float inv = n > 0 ? 1.f / sum : 0.f;
    for (int i = lane; i < d; i += 32) {
      float acc = 0.f;
      for (int e = 0; e < n; ++e) acc = fmaf(my[e], v[((start + keys[e]) * hkv + g) * d + i], acc);
      o[(tok * h + hh) * d + i] = acc * inv;
    }
    if (lse && lane == 0) lse[tok * h + hh] = n > 0 ? mx + logf(sum) : -INFINITY;
    __syncwarp();
  }
}

template <int D, int BS, int NSTAGE, bool DECODE>
static cudaError_t run_mma(const SparseParams& p, dim3 grid, cudaStream_t st) {
  constexpr int pipe = 4 * NSTAGE * 2 * 16 * D * 2;
  constexpr int merge = 4 * 16 * (D + 8) * 4 + 2 * 4 * 16 * 4;
  constexpr int bytes = pipe > merge ? pipe : merge;
  auto kern = sparse_fwd_mma<D, BS, NSTAGE, DECODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (!DECODE) {
    kern<<<grid, 128, bytes, st>>>(p);
    return cudaGetLastError();
  }
  // decode: launched as a programmatic dependent of the selection kernel
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_sparse_fwd(const Seqs& s, const void* q, const void* k, const void* v,
                              const int32_t* idx, int S, int block_size, int h, int hkv, int d,
                              int dtype, float scale, void* o, float* lse, cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  if (dtype == kF32) {
    const int max_keys = S * block_size;
    const size_t bytes = (size_t)max_keys * 4 * 5;
    cudaError_t e = cudaFuncSetAttribute(sparse_fwd_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    sparse_fwd_f32<<<dim3((unsigned)s.tokens, hkv), 128, bytes, st>>>(
        (const float*)q, (const float*)k, (const float*)v, idx, (float*)o, lse, s, h, hkv, d, S, block_size,
        scale);
    return cudaGetLastError();
  }
  SparseParams p{};
  p.q = (const __nv_bfloat16*)q;
  p.k = (const __nv_bfloat16*)k;
  p.v = (const __nv_bfloat16*)v;
  p.idx = idx;
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.S = S;
  p.scale_log2 = scale * kLog2e;
  const int r = h / hkv;
  dim3 grid((unsigned)s.tokens, hkv * ((r + 15) / 16), 1);
  if (d == 128) {
    constexpr int NS = NSA_PREFILL_NSTAGE;
    if (block_size == 64) return run_mma<128, 64, NS, false>(p, grid, st);
    if (block_size == 32) return run_mma<128, 32, NS, false>(p, grid, st);
    return run_mma<128, 16, NS, false>(p, grid, st);
  }
  constexpr int NS = NSA_PREFILL_NSTAGE;
  if (block_size == 64) return run_mma<64, 64, NS, false>(p, grid, st);
  if (block_size == 32) return run_mma<64, 32, NS, false>(p, grid, st);
  return run_mma<64, 16, NS, false>(p, grid, st);
}

// Decode attention over the chosen blocks, split over the list, then merged.
cudaError_t launch_decode_attn(const DecodeArgs& a, cudaStream_t st) {
  SparseParams p{};
  p.q = (const __nv_bfloat16*)a.q;
  p.k = (const __nv_bfloat16*)a.k_cache;
  p.v = (const __nv_bfloat16*)a.v_cache;
  p.idx = a.idx;
  p.h = a.h;
  p.hkv = a.hkv;
  p.S = a.k;
  p.scale_log2 = a.scale * kLog2e;
  p.seqlens = a.seqlens;
  p.max_len = a.max_len;
  p.entries_per_split = (a.k + a.n_split - 1) / a.n_split;
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.merge_count = a.merge_count;
  p.o = (__nv_bfloat16*)a.o;  // the last split CTA writes the merged row here
  if (!p.o || !p.part_o || !p.part_ml || !p.merge_count || !p.idx) return cudaErrorInvalidValue;
  const int r = a.h / a.hkv;
  const int rtiles = (r + 15) / 16;
  dim3 grid(a.batch, a.hkv * rtiles, a.n_split);
  return run_mma<128, 64, NSA_DECODE_NSTAGE, true>(p, grid, st);
}

}  // namespace nsa
