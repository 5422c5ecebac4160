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
// through a private ring and keeps its own online softmax, and the warps merge their
// (max, sum, O) states once at the end (cta_merge).  Warps never wait on one another
// inside the loop, so no CTA-wide barrier sits on the gather path.  The ring is fed by
// TMA for d 128 with blocks of 64 (sparse_fwd_tma, below) and by cp.async otherwise
// (sparse_fwd_mma, through warp_attend).
#include "attend.cuh"
#include "launch.h"
#include "sm100.cuh"

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


// TMA-fed variant (d 128, block 64).  Each warp's 16-key slices of K and V arrive by
// tensor-memory copies: lane 0 issues four 16-row x 64-column boxes (128-byte swizzle)
// per slice onto the stage's mbarrier, instead of every lane issuing eight pairs of
// 16-byte cp.async with their address arithmetic, which took about half of a warp's
// instructions.  Rows past the tensor end arrive as zeros and keys past the query are
// masked as before, so a slice needs no per-row copy logic.  The ldmatrix addressing
// follows the copy's swizzle: row r, 16-byte chunk c of a 16-row tile lives in half
// c / 8 (2 KB apart) at r * 128 + ((c % 8) ^ (r % 8)) * 16.
__device__ __forceinline__ uint32_t tma_addr(uint32_t base, int row, int chunk) {
  return base + ((chunk >> 3) << 11) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// Distance (in query tokens, i.e. CTAs of one kv-head row) of the L2 prefetch of a later
// CTA's query rows and block list: about the number of CTAs resident on the GPU at once.
constexpr int kPrefetchTokens = 512;

// With W, each key's weight (NOSA CIS, p.w [tokens, hkv]) multiplies its softmax weight
// before the PV product and the normaliser; a stage's 16 weights arrive by 4-byte cp.async
// into a small array of their own (the TMA stages keep their 1 KB alignment).
template <int NSTAGE, bool W = false>
__global__ void __launch_bounds__(128, NSA_PREFILL_MINBLOCKS)
    sparse_fwd_tma(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const SparseParams p) {
  constexpr int D = 128, BS = 64, NW = 4;
  constexpr int SLICE = 16 * D * 2;  // 4 KB: two 2 KB halves
  constexpr int STAGE = 2 * SLICE;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_list[NW][64];
  __shared__ __align__(8) uint64_t s_bar[NW][NSTAGE];
  __shared__ float s_w[W ? NW : 1][W ? NSTAGE : 1][16];
  const uint32_t smem = (smem_u32(smem_raw) + 1023) & ~1023u;  // swizzle atoms need 1 KB alignment

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = warp;
  const int r = p.h / p.hkv;
  const int rtiles = (r + 15) >> 4;
  const int g = blockIdx.y / rtiles, rt = blockIdx.y % rtiles;
  const int64_t qrow = blockIdx.x;
  const int sq = seq_of_token(p.seqs, qrow);
  const int64_t kv_base = seq_start(p.seqs, sq);
  const int t = (int)(qrow - kv_base);
  const int hbase = g * r + rt * 16;
  const int rlo = lane >> 2, rhi = rlo + 8;
  const __nv_bfloat16* qb = p.q + (qrow * p.h + hbase) * D;
  // the CTA of token qrow + kPrefetchTokens starts about one resident wave later: bring
  // its query rows and block list into L2 now, so that its start does not wait on DRAM
  if (warp == NW - 1) {
    const int64_t fut = qrow + kPrefetchTokens;
    if (fut < gridDim.x) {
      const int row = lane >> 1;
      if (rt * 16 + row < r)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p.q + (fut * p.h + hbase + row) * D + (lane & 1) * 64));
      if (lane == 0) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p.idx + (fut * p.hkv + g) * p.S));
    }
  }
  uint32_t qa[D / 16][4];
  load_a_frags<D>(qa, rt * 16 + rlo < r ? qb + rlo * D : nullptr, rt * 16 + rhi < r ? qb + rhi * D : nullptr,
                  lane);
  const int32_t* il = p.idx + (qrow * p.hkv + g) * p.S;
  int cnt = 0;
  for (int base = 0; base < p.S; base += 32) {
    const int e = base + lane;
    int blk = -1;
    bool ok = false;
    if (e < p.S) {
      blk = il[e];
      ok = blk >= 0 && (int64_t)blk * BS + slice * 16 <= t;
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (ok) s_list[warp][cnt + __popc(m & ((1u << lane) - 1u))] = blk;
    cnt += __popc(m);
  }
  const uint32_t bar0 = smem_u32(&s_bar[warp][0]);
  if (lane == 0) {
    for (int st = 0; st < NSTAGE; ++st) tc::mbar_init(bar0 + st * 8, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  const uint32_t wbase = smem + warp * NSTAGE * STAGE;
  const int* list = s_list[warp];
  const int x0 = g * D;
  auto issue = [&](int i) {  // lane 0 only
    const int st = i % NSTAGE;
    const uint32_t sb = wbase + st * STAGE, bar = bar0 + st * 8;
    const int y = (int)(kv_base + (int64_t)list[i] * BS + slice * 16);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // earlier reads of the stage come first
    tc::mbar_expect_tx(bar, STAGE);
    tc::tma2d(sb, &tm_k, x0, y, bar);
    tc::tma2d(sb + 2048, &tm_k, x0 + 64, y, bar);
    tc::tma2d(sb + SLICE, &tm_v, x0, y, bar);
    tc::tma2d(sb + SLICE + 2048, &tm_v, x0 + 64, y, bar);
  };

  // weights of slice i (lanes 0-15, one key each; zero past the query); one commit group
  // per call so that the groups count like the stages
  auto issue_w = [&](int i) {
    if (W && lane < 16 && i < cnt) {
      const int64_t key = (int64_t)list[i] * BS + slice * 16 + lane;
      const bool kok = key <= t;
      const float* src = p.w + (kv_base + (kok ? key : 0)) * p.hkv + g;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(&s_w[W ? warp : 0][W ? i % NSTAGE : 0][lane])),
                   "l"(src), "r"(kok ? 4 : 0)
                   : "memory");
    }
    if (W) cp_async_commit();
  };

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  WarpState st{kNegInf, kNegInf, 0.f, 0.f};
  if (lane == 0)
    for (int i = 0; i < NSTAGE - 1 && i < cnt; ++i) issue(i);
  for (int i = 0; i < NSTAGE - 1; ++i) issue_w(i);
  int issued = min(cnt, NSTAGE - 1);
  bool ok = true;
  int i = 0;
  for (; i < cnt; ++i) {
    if (i + NSTAGE - 1 < cnt) {
      if (lane == 0) issue(i + NSTAGE - 1);
      ++issued;
    }
    issue_w(i + NSTAGE - 1);
    const uint32_t bar = bar0 + (i % NSTAGE) * 8;
    if (!tc::warp_wait(bar, (i / NSTAGE) & 1, nullptr)) {
      ok = false;
      break;
    }
    if (W) {
      cp_async_wait<NSTAGE - 1>();
      __syncwarp();
    }
    const uint32_t sb = wbase + (i % NSTAGE) * STAGE;
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int key = (lane & 7) + ((lane >> 4) << 3);
      const int csel = (lane >> 3) & 1;
#pragma unroll
      for (int kk = 0; kk < D / 16; kk += 2) {
        uint32_t b[4], c[4];
        ldsm_x4(b, tma_addr(sb, key, 2 * kk + csel));
        ldsm_x4(c, tma_addr(sb, key, 2 * kk + 2 + csel));
        mma_bf16(s[0], qa[kk], b[0], b[1]);
        mma_bf16(s[1], qa[kk], b[2], b[3]);
        mma_bf16(s2[0], qa[kk + 1], c[0], c[1]);
        mma_bf16(s2[1], qa[kk + 1], c[2], c[3]);
      }
    }
    const int64_t key0 = (int64_t)list[i] * BS + slice * 16;
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
    if (!__all_sync(0xffffffffu, mx0 <= st.m0 + kLazy && mx1 <= st.m1 + kLazy)) {
      const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
      const float a0 = ex2(st.m0 - (mn0 == kNegInf ? 0.f : mn0)), a1 = ex2(st.m1 - (mn1 == kNegInf ? 0.f : mn1));
      st.m0 = mn0;
      st.m1 = mn1;
      st.l0 *= a0;
      st.l1 *= a1;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        o[nt][0] *= a0;
        o[nt][1] *= a0;
        o[nt][2] *= a1;
        o[nt][3] *= a1;
      }
    }
    const float mu0 = st.m0 == kNegInf ? 0.f : st.m0, mu1 = st.m1 == kNegInf ? 0.f : st.m1;
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pr[nt][0] = ex2(s[nt][0] - mu0);
      pr[nt][1] = ex2(s[nt][1] - mu0);
      pr[nt][2] = ex2(s[nt][2] - mu1);
      pr[nt][3] = ex2(s[nt][3] - mu1);
    }
    if (W) {
      const float* sw = s_w[W ? warp : 0][W ? i % NSTAGE : 0];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float w0 = sw[nt * 8 + (lane & 3) * 2], w1 = sw[nt * 8 + (lane & 3) * 2 + 1];
        pr[nt][0] *= w0;
        pr[nt][1] *= w1;
        pr[nt][2] *= w0;
        pr[nt][3] *= w1;
      }
    }
    st.l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
    st.l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
    const uint32_t pa[4] = {pack_bf16(pr[0][0], pr[0][1]), pack_bf16(pr[0][2], pr[0][3]),
                            pack_bf16(pr[1][0], pr[1][1]), pack_bf16(pr[1][2], pr[1][3])};
    {
      const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int csel = lane >> 4;
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        uint32_t b[4];
        ldsm_x4_t(b, tma_addr(sb + SLICE, key, 2 * dn + csel));
        mma_bf16(o[2 * dn], pa, b[0], b[1]);
        mma_bf16(o[2 * dn + 1], pa, b[2], b[3]);
      }
    }
    __syncwarp();
  }
  if (!ok) {  // a copy never arrived (the status word is set): drain what is in flight
    for (int k = i; k < issued; ++k) tc::warp_drain(bar0 + (k % NSTAGE) * 8, (k / NSTAGE) & 1);
  }
  if (W) cp_async_wait<0>();
  st.l0 = quad_sum(st.l0);
  st.l1 = quad_sum(st.l1);
  __syncthreads();  // every warp is done with its ring: the merge reuses the shared memory
  cta_merge<D, NW>(reinterpret_cast<float*>(smem_raw + (smem - smem_u32(smem_raw))), o, st, warp, lane);

  if (warp != 0) return;
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

template <bool W>
static cudaError_t run_tma(const SparseParams& p, const Seqs& s, int hkv, dim3 grid, cudaStream_t st) {
  constexpr int NS = NSA_PREFILL_NSTAGE;
  constexpr int pipe = 4 * NS * 2 * 16 * 128 * 2 + 1024;
  constexpr int merge = merge_bytes<128, 4>() + 1024;
  constexpr int bytes = pipe > merge ? pipe : merge;
  CUtensorMap mk, mv;
  const uint64_t dims[2] = {(uint64_t)hkv * 128, (uint64_t)s.tokens};
  const uint64_t strides[1] = {(uint64_t)hkv * 128 * 2};
  const uint32_t box[2] = {64, 16};
  if (!tc::make_map(&mk, p.k, 2, dims, strides, box) || !tc::make_map(&mv, p.v, 2, dims, strides, box))
    return cudaErrorInvalidValue;
  auto kern = sparse_fwd_tma<NS, W>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, bytes, st>>>(mk, mv, p);
  return cudaGetLastError();
}

// fp32 selected attention on CUDA cores (small problems; exact fp32 arithmetic).
// One CTA per (token, kv-head); warp w serves heads w, w+4, ... of the group.
__global__ void __launch_bounds__(128) sparse_fwd_f32(const float* __restrict__ q, const float* __restrict__ k,
                                                      const float* __restrict__ v, const int32_t* __restrict__ idx,
                                                      float* __restrict__ o, float* __restrict__ lse, Seqs seqs,
                                                      int h, int hkv, int d, int S, int bs, float scale) {
  extern __shared__ __align__(128) uint8_t smem[];
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
  // d 128 with blocks of 64: the TMA-fed kernel (plain or CIS-weighted)
  if (d == 128 && block_size == 64) return cis ? run_tma<true>(p, s, hkv, grid, st) : run_tma<false>(p, s, hkv, grid, st);
  constexpr int NS = NSA_PREFILL_NSTAGE;
  if (cis) return run_mma<64, 64, NS, true>(p, grid, st);  // CIS-weighted, d 64 (block 64: checked by the caller)
  if (d == 128) {
    if (block_size == 32) return run_mma<128, 32, NS>(p, grid, st);
    return run_mma<128, 16, NS>(p, grid, st);
  }
  if (block_size == 64) return run_mma<64, 64, NS>(p, grid, st);
  if (block_size == 32) return run_mma<64, 32, NS>(p, grid, st);
  return run_mma<64, 16, NS>(p, grid, st);
}
NSA_STATUS_ACCESSOR(sparse_fwd)

}  // namespace nsa
