// Warp-level selected-block attention shared by the prefill and decode kernels.
//
// [TileLang-NSA] "TileLang operator development: Native Sparse Attention", sec. 2: a
// listed block starting at index*block_size is attended when it starts at or before
// the query; keys past the query are masked.  Softmax with base-2 exponentials of
// scale*log2(e)-folded scores (sec. 3.1).
//
// With W, each key's softmax weight is multiplied by a per-key weight wb[key * w_stride]
// before both the PV product and the normaliser: the CIS weighting of NOSA's
// sparse_forward ([NOSA-Parts] "decoding over 64 KV blocks": values scaled by the CIS and
// the output divided by the same attention of all-ones values, i.e. weights p*c / sum p*c).
//
// A warp owns one 16-key slice of every block in its list and the 16 (head) rows of
// one query; it streams K and V slices through a private cp.async ring (swizzled rows,
// conflict-free ldmatrix), keeps an online softmax in registers and returns its
// (m, l, O) state.  cta_merge then folds the warps' states (slices of the same rows)
// into warp 0.
#pragma once

#include "common.cuh"

namespace nsa {

// The running max moves only when a score exceeds it by more than 2^kLazy in base 2,
// so exponentials stay below 2^kLazy and O is almost never rescaled; the final
// normalisation is unchanged.
constexpr float kLazy = 8.f;

struct WarpState {
  float m0, m1, l0, l1;
};

// Ring bytes of one stage of warp_attend (K and V slices, and the slice's 16 weights
// padded to 128 bytes when weighted).
template <int D, bool W = false>
constexpr int attend_stage_bytes() {
  return 2 * 16 * D * 2 + (W ? 128 : 0);
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float x;
  asm volatile("ld.shared.f32 %0, [%1];\n" : "=f"(x) : "r"(addr));
  return x;
}

// list[0..cnt): block indices (already filtered to slices starting at or before t).
// kb / vb: K / V row 0 of the sequence for this kv-head; row_stride in elements.
// wb (with W): weight of key row 0 of the sequence for this kv-head; w_stride in floats.

template <int D, int BS, int NSTAGE, bool W = false>
__device__ __forceinline__ WarpState warp_attend(const int* list, int cnt, int slice, const __nv_bfloat16* kb,
                                                 const __nv_bfloat16* vb, int64_t row_stride, int64_t t,
                                                 float scale_log2, const uint32_t (*qa)[4], uint32_t wbase,
                                                 const void* dummy, float (*o)[4], int lane,
                                                 const float* wb = nullptr, int64_t w_stride = 0) {
  constexpr int SLICE_BYTES = 16 * D * 2;
  constexpr int STAGE_BYTES = attend_stage_bytes<D, W>();
  constexpr int CH = D / 8;
  auto issue = [&](int i) {
    const int64_t key0 = (int64_t)list[i] * BS + slice * 16;
    const uint32_t sb = wbase + (i % NSTAGE) * STAGE_BYTES;
    const __nv_bfloat16* kp = kb + key0 * row_stride;
    const __nv_bfloat16* vp = vb + key0 * row_stride;
    const bool full = key0 + 15 <= t;
#pragma unroll
    for (int c = lane; c < 16 * CH; c += 32) {
      const int row = c / CH, ch = c % CH;
      const bool ok = full || key0 + row <= t;
      const int64_t off = row * row_stride + ch * 8;
      cp_async16(tile_addr<D>(sb, row, ch), ok ? kp + off : dummy, ok ? 16 : 0);
      cp_async16(tile_addr<D>(sb + SLICE_BYTES, row, ch), ok ? vp + off : dummy, ok ? 16 : 0);
    }
    if (W && lane < 16) {
      const bool ok = key0 + lane <= t;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(sb + 2 * SLICE_BYTES + lane * 4),
                   "l"(ok ? (const void*)(wb + (key0 + lane) * w_stride) : dummy), "r"(ok ? 4 : 0)
                   : "memory");
    }
  };

  WarpState st{kNegInf, kNegInf, 0.f, 0.f};
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
    const int64_t key0 = (int64_t)list[i] * BS + slice * 16;
    if (key0 + 15 <= t) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[nt][j] = (s[nt][j] + s2[nt][j]) * scale_log2;
    } else {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t key = key0 + nt * 8 + (lane & 3) * 2 + (j & 1);
          s[nt][j] = key <= t ? (s[nt][j] + s2[nt][j]) * scale_log2 : kNegInf;
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
      const uint32_t sw = sb + 2 * SLICE_BYTES + (lane & 3) * 8;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float w0 = lds_f32(sw + nt * 32), w1 = lds_f32(sw + nt * 32 + 4);
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
    pv_16keys<D>(o, pa, sb + SLICE_BYTES, 0, lane);
    __syncwarp();
  }
  cp_async_wait<0>();
  st.l0 = quad_sum(st.l0);
  st.l1 = quad_sum(st.l1);
  return st;
}

// Shared memory needed by cta_merge<D, NW> (bytes).
template <int D, int NW>
constexpr int merge_bytes() {
  return NW * 16 * (D + 8) * 4 + 2 * NW * 16 * 4;
}

// Fold the states of NW warps (same 16 rows, different keys) into warp 0: on return
// warp 0's o holds sum_w 2^(m_w - M) O_w and st holds (M, L) per row (M = -inf when
// no key was attended; then O = 0 and L = 0).  sm: merge_bytes<D, NW>() of shared
// memory that no warp is still writing.  Every thread of the NW warps must call it.
template <int D, int NW>
__device__ __forceinline__ void cta_merge(float* sm, float (*o)[4], WarpState& st, int warp, int lane) {
  constexpr int OS = D + 8;  // padded rows: 8-byte fragment stores/loads without bank conflicts
  float* sm_o = sm;                   // [NW][16][OS]
  float* sm_m = sm_o + NW * 16 * OS;  // [NW][16]
  float* sm_l = sm_m + NW * 16;       // [NW][16]
  const int rlo = lane >> 2, rhi = rlo + 8;
  if (warp > 0) {
    if ((lane & 3) == 0) {
      sm_m[warp * 16 + rlo] = st.m0;
      sm_m[warp * 16 + rhi] = st.m1;
      sm_l[warp * 16 + rlo] = st.l0;
      sm_l[warp * 16 + rhi] = st.l1;
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(&sm_o[(warp * 16 + rlo) * OS + col]) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(&sm_o[(warp * 16 + rhi) * OS + col]) = make_float2(o[nt][2], o[nt][3]);
    }
  }
  __syncthreads();
  if (warp == 0) {
    float M0 = st.m0, M1 = st.m1;
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      M0 = fmaxf(M0, sm_m[w * 16 + rlo]);
      M1 = fmaxf(M1, sm_m[w * 16 + rhi]);
    }
    const float u0 = M0 == kNegInf ? 0.f : M0, u1 = M1 == kNegInf ? 0.f : M1;
    const float g0 = ex2(st.m0 - u0), g1 = ex2(st.m1 - u1);
    float L0 = g0 * st.l0, L1 = g1 * st.l1;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      o[nt][0] *= g0;
      o[nt][1] *= g0;
      o[nt][2] *= g1;
      o[nt][3] *= g1;
    }
#pragma unroll 1
    for (int w = 1; w < NW; ++w) {
      const float f0 = ex2(sm_m[w * 16 + rlo] - u0), f1 = ex2(sm_m[w * 16 + rhi] - u1);
      L0 += f0 * sm_l[w * 16 + rlo];
      L1 += f1 * sm_l[w * 16 + rhi];
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        const int col = nt * 8 + (lane & 3) * 2;
        const float2 x = *reinterpret_cast<const float2*>(&sm_o[(w * 16 + rlo) * OS + col]);
        const float2 y = *reinterpret_cast<const float2*>(&sm_o[(w * 16 + rhi) * OS + col]);
        o[nt][0] += f0 * x.x;
        o[nt][1] += f0 * x.y;
        o[nt][2] += f1 * y.x;
        o[nt][3] += f1 * y.y;
      }
    }
    st.m0 = M0;
    st.m1 = M1;
    st.l0 = L0;
    st.l1 = L1;
  }
}

}  // namespace nsa
