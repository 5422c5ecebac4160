// Shared device helpers of the sm_103a kernels: sequence lookup, cp.async staging,
// ldmatrix / mma.sync fragments for bf16 16x8x16 tiles, swizzled shared-memory tiles.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nsa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_inff();

// ---------------------------------------------------------------------------
// Sequences.  Dense layout: cu == nullptr, every sequence has T tokens.
struct Seqs {
  const int32_t* cu;
  int n_seqs;
  int T;
  int64_t tokens;
  int max_len;
};

__device__ __forceinline__ int seq_start(const Seqs& s, int i) {
  return s.cu ? s.cu[i] : i * s.T;
}
__device__ __forceinline__ int seq_len(const Seqs& s, int i) {
  return s.cu ? s.cu[i + 1] - s.cu[i] : s.T;
}
// Sequence holding packed token `tok` (binary search over cu_seqlens).
__device__ __forceinline__ int seq_of_token(const Seqs& s, int64_t tok) {
  if (!s.cu) return (int)(tok / s.T);
  int lo = 0, hi = s.n_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s.cu[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ int num_cmp(int L, int kernel, int stride) {
  return L >= kernel ? (L - kernel) / stride + 1 : 0;
}
// First packed compressed row of sequence i (sum of n_c over the sequences before it).
__device__ __forceinline__ int64_t cmp_offset(const Seqs& s, int i, int kernel, int stride) {
  if (!s.cu) return (int64_t)i * num_cmp(s.T, kernel, stride);
  int64_t off = 0;
  for (int j = 0; j < i; ++j) off += num_cmp(s.cu[j + 1] - s.cu[j], kernel, stride);
  return off;
}
// Number of compressed keys causal for position t (window end <= t).
__device__ __forceinline__ int num_causal_cmp(int t, int n_c, int kernel, int stride) {
  if (t < kernel - 1) return 0;
  int n = (t - (kernel - 1)) / stride + 1;
  return n < n_c ? n : n_c;
}

// ---------------------------------------------------------------------------
// PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte global->shared copy; src_bytes == 0 zero-fills without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Hardware base-2 exponential (ex2.approx; ex2(-inf) = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// Swizzled tile of ROWS x D bf16 in shared memory: row r, 16-byte chunk c lives at
// chunk (c ^ (r & 7)) of the row, so eight rows read at one logical chunk hit eight
// different bank groups (conflict-free ldmatrix).
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk) {
  return base + row * (D * 2) + ((chunk ^ (row & 7)) << 4);
}

// Issue cp.async for rows [0, ROWS) of a tile; row r comes from src(r) or is zero-filled
// when src(r) == nullptr (the copy then names `dummy`, a valid address, and reads 0
// bytes).  Threads [0, NT) take part.
template <int D, int ROWS, int NT, typename SrcFn>
__device__ __forceinline__ void load_tile_async(uint32_t base, int tid, const void* dummy, SrcFn src) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  constexpr int TOTAL = ROWS * CH;
#pragma unroll
  for (int i = tid; i < TOTAL; i += NT) {
    int r = i / CH, c = i % CH;
    const __nv_bfloat16* p = src(r);
    uint32_t dst = tile_addr<D>(base, r, c);
    if (p)
      cp_async16(dst, p + c * 8, 16);
    else
      cp_async16(dst, dummy, 0);
  }
}

// A fragments (m16n8k16, row-major A) of a 16-row x D bf16 block read from global
// memory: rows whose pointer is null read as zeros.  qa[kk][0..3] for k-step kk.
template <int D>
__device__ __forceinline__ void load_a_frags(uint32_t (*qa)[4], const __nv_bfloat16* row_lo,
                                             const __nv_bfloat16* row_hi, int lane) {
  const int c = (lane & 3) * 2;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    qa[kk][0] = row_lo ? *reinterpret_cast<const uint32_t*>(row_lo + kk * 16 + c) : 0u;
    qa[kk][1] = row_hi ? *reinterpret_cast<const uint32_t*>(row_hi + kk * 16 + c) : 0u;
    qa[kk][2] = row_lo ? *reinterpret_cast<const uint32_t*>(row_lo + kk * 16 + 8 + c) : 0u;
    qa[kk][3] = row_hi ? *reinterpret_cast<const uint32_t*>(row_hi + kk * 16 + 8 + c) : 0u;
  }
}

// S[16 x 16 keys] = A[16 x D] * K_tile[key0 .. key0+15]^T from a swizzled tile.
// s[0] covers keys key0..key0+7, s[1] keys key0+8..key0+15 (C fragment layout).
template <int D>
__device__ __forceinline__ void qk_16keys(float (*s)[4], const uint32_t (*qa)[4], uint32_t kbase,
                                          int key0, int lane) {
  const int key = key0 + (lane & 7) + ((lane >> 4) << 3);
  const int csel = (lane >> 3) & 1;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t b[4];
    ldsm_x4(b, tile_addr<D>(kbase, key, 2 * kk + csel));
    mma_bf16(s[0], qa[kk], b[0], b[1]);
    mma_bf16(s[1], qa[kk], b[2], b[3]);
  }
}

// Same product with the k-steps split over two accumulators (even / odd k-steps), so
// four independent mma chains are in flight instead of two; the caller adds them.
template <int D>
__device__ __forceinline__ void qk_16keys_2acc(float (*s)[4], float (*s2)[4], const uint32_t (*qa)[4],
                                               uint32_t kbase, int key0, int lane) {
  const int key = key0 + (lane & 7) + ((lane >> 4) << 3);
  const int csel = (lane >> 3) & 1;
#pragma unroll
  for (int kk = 0; kk < D / 16; kk += 2) {
    uint32_t b[4], c[4];
    ldsm_x4(b, tile_addr<D>(kbase, key, 2 * kk + csel));
    ldsm_x4(c, tile_addr<D>(kbase, key, 2 * kk + 2 + csel));
    mma_bf16(s[0], qa[kk], b[0], b[1]);
    mma_bf16(s[1], qa[kk], b[2], b[3]);
    mma_bf16(s2[0], qa[kk + 1], c[0], c[1]);
    mma_bf16(s2[1], qa[kk + 1], c[2], c[3]);
  }
}

// O[16 x D] += P[16 x 16 keys] * V_tile[key0 .. key0+15] from a swizzled tile.
// pa is the A fragment of P (bf16).  o[nt] is the C fragment of d-columns nt*8..nt*8+7.
template <int D>
__device__ __forceinline__ void pv_16keys(float (*o)[4], const uint32_t* pa, uint32_t vbase, int key0,
                                          int lane) {
  const int key = key0 + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int csel = lane >> 4;
#pragma unroll
  for (int dn = 0; dn < D / 16; ++dn) {
    uint32_t b[4];
    ldsm_x4_t(b, tile_addr<D>(vbase, key, 2 * dn + csel));
    mma_bf16(o[2 * dn], pa, b[0], b[1]);
    mma_bf16(o[2 * dn + 1], pa, b[2], b[3]);
  }
}

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

}  // namespace nsa
