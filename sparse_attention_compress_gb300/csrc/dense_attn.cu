// Compressed-attention branch, sliding-window branch and the gated sum of the three
// branches of the NSA layer.
//
// [NSA-Triton] "DeepSeek NSA ... with Triton", sec. 1.1: three parallel branches
// (compressed / selected / sliding window) combined by gates
// gates[0]*compressed + gates[1]*selected + gates[2]*local; the sliding branch attends
// to the most recent tokens; sec. 2.2 (read as the definition of the compressed branch:
// softmax of q against the compressed keys, weighted sum of the compressed values).
//
// GB300 design.  Both branches attend to a contiguous key range per query, so a CTA
// takes a run of consecutive tokens of one sequence and one kv-group (8 warps x 16
// (token, head) rows) and streams the union of their key ranges through shared memory
// in 64-key K and V tiles (cp.async, double buffered), shared by all 128 rows.  Each
// row applies its own mask (compressed: window end <= t; sliding: t-w < tau <= t) and
// keeps an online softmax in registers; mma.sync m16n8k16 for QK^T and PV.
#include "launch.h"

namespace nsa {

constexpr int kDWarps = 8;

struct DenseParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  Seqs seqs;
  int h, hkv, R, kernel, stride, window;
  float scale_log2;
};

template <int D, int MODE>
__global__ void __launch_bounds__(kDWarps * 32) dense_attn_kernel(const DenseParams p) {
  constexpr int TILE = 64;
  constexpr int TILE_BYTES = TILE * D * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const int R = p.R;
  const int TPC = kDWarps * 16 / R;
  const int sq = blockIdx.y, g = blockIdx.z;
  const int L = seq_len(p.seqs, sq);
  const int n_tok_tiles = (L + TPC - 1) / TPC;
  const int tile = n_tok_tiles - 1 - (int)blockIdx.x;
  if (tile < 0) return;
  const int t0 = tile * TPC;
  const int t_last = min(t0 + TPC, L) - 1;
  const int64_t start = seq_start(p.seqs, sq);
  int n_c = 0;
  int64_t kv0;
  int key_lo, key_hi;
  if (MODE == 0) {
    n_c = num_cmp(L, p.kernel, p.stride);
    kv0 = cmp_offset(p.seqs, sq, p.kernel, p.stride);
    key_lo = 0;
    key_hi = num_causal_cmp(t_last, n_c, p.kernel, p.stride);
  } else {
    kv0 = start;
    key_lo = max(0, t0 - p.window + 1);
    key_hi = t_last + 1;
  }
  const int n_kt = key_hi > key_lo ? (key_hi - key_lo + TILE - 1) / TILE : 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rlo = lane >> 2, rhi = rlo + 8;
  const int gl = warp * 16 + rlo, gh = warp * 16 + rhi;
  const int t_lo = t0 + gl / R, t_hi = t0 + gh / R;
  const int hd_lo = gl % R, hd_hi = gh % R;
  // rows past the CTA's TPC tokens (a group size that does not divide 128) belong to the
  // next CTA: they take no part
  const int rows = TPC * R;
  const bool v_lo = gl < rows && t_lo < L, v_hi = gh < rows && t_hi < L;
  // per-row key bounds [a, b)
  int a_lo, b_lo, a_hi, b_hi;
  if (MODE == 0) {
    a_lo = a_hi = 0;
    b_lo = v_lo ? num_causal_cmp(t_lo, n_c, p.kernel, p.stride) : 0;
    b_hi = v_hi ? num_causal_cmp(t_hi, n_c, p.kernel, p.stride) : 0;
  } else {
    a_lo = max(0, t_lo - p.window + 1);
    a_hi = max(0, t_hi - p.window + 1);
    b_lo = v_lo ? t_lo + 1 : 0;
    b_hi = v_hi ? t_hi + 1 : 0;
  }
  // key range touched by this warp's rows
  const int tw0 = min(t0 + (warp * 16) / R, L - 1), tw1 = min(t0 + (min(warp * 16 + 15, rows - 1)) / R, L - 1);
  int w_lo, w_hi;
  if (MODE == 0) {
    w_lo = 0;
    w_hi = num_causal_cmp(tw1, n_c, p.kernel, p.stride);
  } else {
    w_lo = max(0, tw0 - p.window + 1);
    w_hi = tw1 + 1;
  }
  const bool warp_live = warp * 16 < rows && t0 + (warp * 16) / R < L;

  uint32_t qa[D / 16][4];
  load_a_frags<D>(qa, v_lo ? p.q + ((start + t_lo) * p.h + g * R + hd_lo) * D : nullptr,
                  v_hi ? p.q + ((start + t_hi) * p.h + g * R + hd_hi) * D : nullptr, lane);

  const uint32_t sbase = smem_u32(smem);
  const int64_t row_stride = (int64_t)p.hkv * D;
  const __nv_bfloat16* kb = p.k + (kv0 * p.hkv + g) * D;
  const __nv_bfloat16* vb = p.v + (kv0 * p.hkv + g) * D;
  auto load = [&](int kt) {
    const uint32_t st = sbase + (kt & 1) * 2 * TILE_BYTES;
    const int base = key_lo + kt * TILE;
    load_tile_async<D, TILE, kDWarps * 32>(st, threadIdx.x, p.k, [&](int row) -> const __nv_bfloat16* {
      return base + row < key_hi ? kb + (base + row) * row_stride : nullptr;
    });
    load_tile_async<D, TILE, kDWarps * 32>(st + TILE_BYTES, threadIdx.x, p.v, [&](int row) -> const __nv_bfloat16* {
      return base + row < key_hi ? vb + (base + row) * row_stride : nullptr;
    });
  };

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = kNegInf, m_hi = kNegInf, l_lo = 0.f, l_hi = 0.f;

  if (n_kt > 0) load(0);
  cp_async_commit();
  for (int kt = 0; kt < n_kt; ++kt) {
    if (kt + 1 < n_kt) load(kt + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int base = key_lo + kt * TILE;
    if (warp_live && base < w_hi && base + TILE > w_lo) {
      const uint32_t st = sbase + (kt & 1) * 2 * TILE_BYTES;
      float s[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int k16 = 0; k16 < 4; ++k16) qk_16keys<D>(&s[2 * k16], qa, st, k16 * 16, lane);
      float x_lo = kNegInf, x_hi = kNegInf;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int key = base + nt * 8 + (lane & 3) * 2 + (j & 1);
          const bool ok = j < 2 ? (key >= a_lo && key < b_lo) : (key >= a_hi && key < b_hi);
          s[nt][j] = ok ? s[nt][j] * p.scale_log2 : kNegInf;
          if (j < 2) x_lo = fmaxf(x_lo, s[nt][j]); else x_hi = fmaxf(x_hi, s[nt][j]);
        }
      const float mn_lo = fmaxf(m_lo, quad_max(x_lo)), mn_hi = fmaxf(m_hi, quad_max(x_hi));
      const float mu_lo = mn_lo == kNegInf ? 0.f : mn_lo, mu_hi = mn_hi == kNegInf ? 0.f : mn_hi;
      const float al = ex2(m_lo - mu_lo), ah = ex2(m_hi - mu_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      float sl = 0.f, sh = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = ex2(s[nt][0] - mu_lo);
        s[nt][1] = ex2(s[nt][1] - mu_lo);
        s[nt][2] = ex2(s[nt][2] - mu_hi);
        s[nt][3] = ex2(s[nt][3] - mu_hi);
        sl += s[nt][0] + s[nt][1];
        sh += s[nt][2] + s[nt][3];
      }
      l_lo = l_lo * al + sl;
      l_hi = l_hi * ah + sh;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        o[nt][0] *= al;
        o[nt][1] *= al;
        o[nt][2] *= ah;
        o[nt][3] *= ah;
      }
#pragma unroll
      for (int k16 = 0; k16 < 4; ++k16) {
        const uint32_t pa[4] = {pack_bf16(s[2 * k16][0], s[2 * k16][1]), pack_bf16(s[2 * k16][2], s[2 * k16][3]),
                                pack_bf16(s[2 * k16 + 1][0], s[2 * k16 + 1][1]),
                                pack_bf16(s[2 * k16 + 1][2], s[2 * k16 + 1][3])};
        pv_16keys<D>(o, pa, st + TILE_BYTES, k16 * 16, lane);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  l_lo = quad_sum(l_lo);
  l_hi = quad_sum(l_hi);
  const float il = l_lo > 0.f ? 1.f / l_lo : 0.f, ih = l_hi > 0.f ? 1.f / l_hi : 0.f;
  __nv_bfloat16* o_lo = p.o + ((start + t_lo) * p.h + g * R + hd_lo) * D;
  __nv_bfloat16* o_hi = p.o + ((start + t_hi) * p.h + g * R + hd_hi) * D;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + (lane & 3) * 2;
    if (v_lo) *reinterpret_cast<uint32_t*>(o_lo + col) = pack_bf16(o[nt][0] * il, o[nt][1] * il);
    if (v_hi) *reinterpret_cast<uint32_t*>(o_hi + col) = pack_bf16(o[nt][2] * ih, o[nt][3] * ih);
  }
  if (p.lse && (lane & 3) == 0) {
    if (v_lo) p.lse[(start + t_lo) * p.h + g * R + hd_lo] = l_lo > 0.f ? (m_lo + __log2f(l_lo)) * kLn2 : kNegInf;
    if (v_hi) p.lse[(start + t_hi) * p.h + g * R + hd_hi] = l_hi > 0.f ? (m_hi + __log2f(l_hi)) * kLn2 : kNegInf;
  }
}

cudaError_t launch_dense_attn(int mode, const Seqs& s, const void* q, const void* k, const void* v,
                              int h, int hkv, int d, int kernel, int stride, int window, float scale,
                              void* o, float* lse, cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  DenseParams p{};
  p.q = (const __nv_bfloat16*)q;
  p.k = (const __nv_bfloat16*)k;
  p.v = (const __nv_bfloat16*)v;
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.R = h / hkv;
  p.kernel = kernel;
  p.stride = stride;
  p.window = window;
  p.scale_log2 = scale * kLog2e;
  const int tpc = kDWarps * 16 / p.R;
  dim3 grid((s.max_len + tpc - 1) / tpc, s.n_seqs, hkv);
  const int bytes = 2 * 2 * 64 * d * 2;
  cudaError_t e = cudaSuccess;
#define NSA_DENSE(DD, MM)                                                                                      \
  e = cudaFuncSetAttribute(dense_attn_kernel<DD, MM>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);    \
  if (e != cudaSuccess) return e;                                                                              \
  dense_attn_kernel<DD, MM><<<grid, kDWarps * 32, bytes, st>>>(p);
  if (d == 128) {
    if (mode == 0) { NSA_DENSE(128, 0) } else { NSA_DENSE(128, 1) }
  } else {
    if (mode == 0) { NSA_DENSE(64, 0) } else { NSA_DENSE(64, 1) }
  }
#undef NSA_DENSE
  return cudaGetLastError();
}

// o = sigmoid(a0) * o_cmp + sigmoid(a1) * o_slc + sigmoid(a2) * o_swa, 8 elements per thread.
__global__ void gate_combine_kernel(const uint4* __restrict__ oc, const uint4* __restrict__ os,
                                    const uint4* __restrict__ ow, const float* __restrict__ gates,
                                    uint4* __restrict__ o, int64_t n_vec, int d8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t th = i / d8;
    const float g0 = 1.f / (1.f + expf(-gates[th * 3]));
    const float g1 = 1.f / (1.f + expf(-gates[th * 3 + 1]));
    const float g2 = 1.f / (1.f + expf(-gates[th * 3 + 2]));
    const uint4 a = oc[i], b = os[i], c = ow[i];
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
    const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c);
    uint4 r;
    uint32_t* pr = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 x = __bfloat1622float2(pa[u]), y = __bfloat1622float2(pb[u]), z = __bfloat1622float2(pc[u]);
      pr[u] = pack_bf16(g0 * x.x + g1 * y.x + g2 * z.x, g0 * x.y + g1 * y.y + g2 * z.y);
    }
    o[i] = r;
  }
}

cudaError_t launch_gate_combine(int64_t tokens, int h, int d, const void* o_cmp, const void* o_slc,
                                const void* o_swa, const float* gates, void* o, cudaStream_t st) {
  const int64_t n_vec = tokens * h * (d / 8);
  if (n_vec == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (n_vec + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  gate_combine_kernel<<<(unsigned)blocks, threads, 0, st>>>((const uint4*)o_cmp, (const uint4*)o_slc,
                                                            (const uint4*)o_swa, gates, (uint4*)o, n_vec, d / 8);
  return cudaGetLastError();
}

}  // namespace nsa
