// Selected-block attention (prefill).
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
// through a private cp.async ring and keeps its own online softmax (warp_attend), and
// the warps merge their (max, sum, O) states once at the end (cta_merge).  Warps never
// wait on one another inside the loop, so no CTA-wide barrier sits on the gather path.
#include "attend.cuh"
#include "launch.h"

namespace nsa {

struct SparseParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* idx;
  const float* w;  // per-key weights [tokens, hkv] (NOSA CIS), used when the kernel is weighted
  __nv_bfloat16* o;
  float* lse;
  Seqs seqs;
  int h, hkv, S;
  float scale_log2;
};

#ifndef NSA_PREFILL_NSTAGE
#define NSA_PREFILL_NSTAGE 2
#endif
#ifndef NSA_PREFILL_MINBLOCKS
#define NSA_PREFILL_MINBLOCKS 3
#endif


template <int D, int BS, int NSTAGE, bool W = false>
__global__ void __launch_bounds__(128, NSA_PREFILL_MINBLOCKS) sparse_fwd_mma(const SparseParams p) {
  constexpr int NW = 4;
  constexpr int NSLICE = BS / 16;
  constexpr int NGROUP = NW / NSLICE;
  constexpr int STAGE_BYTES = attend_stage_bytes<D, W>();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_list[NW][64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = warp % NSLICE, grp = warp / NSLICE;
  const int r = p.h / p.hkv;
  const int rtiles = (r + 15) >> 4;
  const int g = blockIdx.y / rtiles, rt = blockIdx.y % rtiles;

  const int64_t qrow = blockIdx.x;
  const int sq = seq_of_token(p.seqs, qrow);
  const int64_t kv_base = seq_start(p.seqs, sq);
  const int t = (int)(qrow - kv_base);

  // Q fragments of the group's heads (rows past the group read as zero)
  const int hbase = g * r + rt * 16;
  const int rlo = lane >> 2, rhi = rlo + 8;
  const __nv_bfloat16* qb = p.q + (qrow * p.h + hbase) * D;
  uint32_t qa[D / 16][4];
  load_a_frags<D>(qa, rt * 16 + rlo < r ? qb + rlo * D : nullptr, rt * 16 + rhi < r ? qb + rhi * D : nullptr,
                  lane);
  // this warp's work list: listed blocks whose slice starts at or before t
  const int32_t* il = p.idx + (qrow * p.hkv + g) * p.S;
  int cnt = 0;
  for (int base = 0; base < p.S; base += 32) {
    const int e = base + lane;
    int blk = -1;
    bool ok = false;
    if (e < p.S) {
      blk = il[e];
      ok = (e % NGROUP == grp) && blk >= 0 && (int64_t)blk * BS + slice * 16 <= t;
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (ok) s_list[warp][cnt + __popc(m & ((1u << lane) - 1u))] = blk;
    cnt += __popc(m);
  }
  __syncwarp();

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  WarpState st = warp_attend<D, BS, NSTAGE, W>(s_list[warp], cnt, slice, p.k + (kv_base * p.hkv + g) * D,
                                               p.v + (kv_base * p.hkv + g) * D, (int64_t)p.hkv * D, t,
                                               p.scale_log2, qa, smem_u32(smem) + warp * NSTAGE * STAGE_BYTES, p.k,
                                               o, lane, W ? p.w + kv_base * p.hkv + g : nullptr, p.hkv);
  __syncthreads();  // every warp is done with its ring: the merge reuses the shared memory
  cta_merge<D, NW>(reinterpret_cast<float*>(smem), o, st, warp, lane);

  if (warp != 0) return;
  {
    const float u0 = st.m0 == kNegInf ? 0.f : st.m0, u1 = st.m1 == kNegInf ? 0.f : st.m1;
    const float i0 = st.l0 > 0.f ? 1.f / st.l0 : 0.f, i1 = st.l1 > 0.f ? 1.f / st.l1 : 0.f;
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
      if (w0) p.lse[qrow * p.h + hbase + rlo] = st.l0 > 0.f ? (u0 + __log2f(st.l0)) * kLn2 : kNegInf;
      if (w1) p.lse[qrow * p.h + hbase + rhi] = st.l1 > 0.f ? (u1 + __log2f(st.l1)) * kLn2 : kNegInf;
    }
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

template <int D, int BS, int NSTAGE, bool W = false>
static cudaError_t run_mma(const SparseParams& p, dim3 grid, cudaStream_t st) {
  constexpr int pipe = 4 * NSTAGE * attend_stage_bytes<D, W>();
  constexpr int merge = merge_bytes<D, 4>();
  constexpr int bytes = pipe > merge ? pipe : merge;
  auto kern = sparse_fwd_mma<D, BS, NSTAGE, W>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, bytes, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sparse_fwd(const Seqs& s, const void* q, const void* k, const void* v,
                              const int32_t* idx, int S, int block_size, int h, int hkv, int d,
                              int dtype, float scale, void* o, float* lse, cudaStream_t st, const float* cis) {
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
  p.w = cis;
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.S = S;
  p.scale_log2 = scale * kLog2e;
  const int r = h / hkv;
  dim3 grid((unsigned)s.tokens, hkv * ((r + 15) / 16), 1);
  if (cis) {  // CIS-weighted variant: block 64 only (checked by the caller)
    constexpr int NS = NSA_PREFILL_NSTAGE;
    return d == 128 ? run_mma<128, 64, NS, true>(p, grid, st) : run_mma<64, 64, NS, true>(p, grid, st);
  }
  if (d == 128) {
    constexpr int NS = NSA_PREFILL_NSTAGE;
    if (block_size == 64) return run_mma<128, 64, NS>(p, grid, st);
    if (block_size == 32) return run_mma<128, 32, NS>(p, grid, st);
    return run_mma<128, 16, NS>(p, grid, st);
  }
  constexpr int NS = NSA_PREFILL_NSTAGE;
  if (block_size == 64) return run_mma<64, 64, NS>(p, grid, st);
  if (block_size == 32) return run_mma<64, 32, NS>(p, grid, st);
  return run_mma<64, 16, NS>(p, grid, st);
}
}  // namespace nsa
