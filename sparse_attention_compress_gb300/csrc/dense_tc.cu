// Compressed and sliding-window branches on the 5th-generation tensor cores.
//
// [NSA-Triton] "DeepSeek NSA ... with Triton", sec. 1.1: the compressed branch attends
// to the mean-pooled keys/values, the sliding branch to the most recent tokens; both
// are dense attention over a contiguous key range per query.
//
// GB300 design.  A CTA takes 128 (token, head) rows of one kv-group (8 tokens x 16 heads
// at the layer's group size): they share every K/V tile, so the contraction is a real
// M=128 GEMM.  Per 64-key tile:
//   S[128 x 64]  = Q K^T  : tcgen05.mma kind::f16, A = Q tile, B = K tile, both K-major
//                           in 128B-swizzled shared memory, D in TMEM (columns 0..63);
//   softmax      : thread i owns row i (TMEM lane i): tcgen05.ld of its 64 scores, mask,
//                  running max with lazy rescale, base-2 exponentials, P (bf16) written
//                  in the 128B-swizzled layout over the K tile it no longer needs;
//   O[128 x 128] += P V   : tcgen05.mma, A = P, B = V^T tile (V transposed once per call
//                           so that this operand is K-major too), D in TMEM (cols 128..255).
// cp.async double-buffers the K / V^T tiles; tcgen05.commit signals mbarriers whose
// waits are bounded (a timeout sets the library's device status and the CTA leaves after
// draining its copies and freeing its TMEM).  Two CTAs share an SM (96 KB shared memory,
// 256 TMEM columns each), so one CTA's softmax overlaps the other's MMAs.
#include "nsa.h"
#include "launch.h"

namespace nsa {

__device__ int g_device_status = 0;  // NSA_ERR_TIMEOUT when a bounded wait ran out

namespace tc {

constexpr int D = 128;
constexpr int ROWS = 128;  // query rows per CTA (= tcgen05 M)
constexpr int KT = 64;     // keys per tile (= N of S, K of PV)
constexpr int Q_BYTES = ROWS * D * 2;         // 32 KB: two 64-column halves
constexpr int K_BYTES = KT * D * 2;           // 16 KB: two halves; reused for P (128 x 64)
constexpr int V_BYTES = D * KT * 2;           // 16 KB: V^T tile, 128 rows of 64 keys
constexpr int SMEM_BYTES = Q_BYTES + 2 * K_BYTES + 2 * V_BYTES + 1024;  // + alignment
constexpr int TMEM_COLS = 256;  // S: 0..63, O: 128..255
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s: an mbarrier wait longer than this is stuck

// 128B-swizzled K-major tile of R rows x 64 bf16: row r, 16-byte chunk c at
// base + r*128 + ((c ^ (r & 7)) << 4); 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int chunk) {
  return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Shared-memory matrix descriptor: 128B swizzle, K-major, 1024-byte atom stride.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;              // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, A and B K-major, M x N.
__host__ __device__ constexpr uint32_t idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}
// Wait for phase `parity` of an mbarrier for at most kWaitNs; false (and the device
// status set to NSA_ERR_TIMEOUT) when the limit ran out.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitNs) break;
  }
  atomicExch(&g_device_status, (int)NSA_ERR_TIMEOUT);
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  return mbar_try(bar, parity) || mbar_wait_slow(bar, parity);
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;   // [kv_rows, hkv, D]
  const __nv_bfloat16* vt;  // [hkv, D, kv_pad]: V transposed, zero past kv_rows
  __nv_bfloat16* o;
  float* lse;
  Seqs seqs;
  int h, hkv, R, kernel, stride, window;
  int64_t kv_rows, kv_pad;
  float scale_log2;
};

template <int MODE>
__global__ void __launch_bounds__(128, 2) attn_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];  // 0: S tile ready, 1: O update done
  __shared__ uint32_t tmem_holder;
  const uint32_t base = (smem_u32(smem_raw) + 1023) & ~1023u;  // 128B-swizzle atoms need 1 KB alignment
  const uint32_t q_s = base, k_s = base + Q_BYTES, v_s = k_s + 2 * K_BYTES;
  const uint32_t bar_s = smem_u32(&bars[0]), bar_o = smem_u32(&bars[1]);
  const int tid = threadIdx.x, warp = tid >> 5;

  const int R = p.R;
  const int TPC = ROWS / R;  // tokens per CTA
  const int sq = blockIdx.y, g = blockIdx.z;
  const int L = seq_len(p.seqs, sq);
  const int tile = (L + TPC - 1) / TPC - 1 - (int)blockIdx.x;  // longest key ranges first
  if (tile < 0) return;
  const int t0 = tile * TPC;
  const int t_last = min(t0 + TPC, L) - 1;
  const int64_t start = seq_start(p.seqs, sq);
  int n_c = 0, key_lo, key_hi;
  int64_t kv0;  // key row of the sequence's first key
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
  // 64-key tiles in absolute key rows, so every V^T tile starts 128-byte aligned
  const int64_t a_lo = (kv0 + key_lo) / KT;
  const int n_kt = key_hi > key_lo ? (int)((kv0 + key_hi + KT - 1) / KT - a_lo) : 0;

  // this thread's row (TMEM lane = tid)
  const int row = tid;
  const int tl = row / R, hd = row % R;
  const int t_row = t0 + tl;
  const bool valid = tl < TPC && t_row < L;
  int b_lo = 0, b_hi = 0;  // attended keys [b_lo, b_hi), relative to kv0
  if (valid) {
    if (MODE == 0) {
      b_hi = num_causal_cmp(t_row, n_c, p.kernel, p.stride);
    } else {
      b_lo = max(0, t_row - p.window + 1);
      b_hi = t_row + 1;
    }
  }

  if (tid == 0) {
    mbar_init(bar_s);
    mbar_init(bar_o);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&tmem_holder)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    fence_before();
  }

  // Q: 128 rows x 128 d as two 64-column swizzled halves; rows past the tile are zero
  const int64_t q_row_stride = (int64_t)p.h * D;
  for (int c = tid; c < ROWS * (D / 8); c += 128) {
    const int r = c / (D / 8), ch = c % (D / 8);
    const int rt = t0 + r / R;
    const bool ok = r / R < TPC && rt < L;
    const __nv_bfloat16* src = p.q + (start + rt) * q_row_stride + (g * R + r % R) * D + ch * 8;
    cp_async16(sw128(q_s + (ch >> 3) * (ROWS * 128), r, ch & 7), ok ? src : (const void*)p.q, ok ? 16 : 0);
  }
  const int64_t k_row_stride = (int64_t)p.hkv * D;
  auto load_tile = [&](int kt, int stage) {
    const int64_t a0 = (a_lo + kt) * KT;
    const uint32_t ks = k_s + stage * K_BYTES, vs = v_s + stage * V_BYTES;
    for (int c = tid; c < KT * (D / 8); c += 128) {  // K: 64 key rows x 16 chunks, two halves
      const int r = c / (D / 8), ch = c % (D / 8);
      const bool ok = a0 + r < p.kv_rows;
      const __nv_bfloat16* src = p.k + (a0 + r) * k_row_stride + g * D + ch * 8;
      cp_async16(sw128(ks + (ch >> 3) * (KT * 128), r, ch & 7), ok ? src : (const void*)p.k, ok ? 16 : 0);
    }
    for (int c = tid; c < D * (KT / 8); c += 128) {  // V^T: 128 d rows x 8 chunks of 8 keys
      const int r = c / (KT / 8), ch = c % (KT / 8);
      cp_async16(sw128(vs, r, ch), p.vt + ((int64_t)g * D + r) * p.kv_pad + a0 + ch * 8, 16);
    }
  };
  if (n_kt > 0) load_tile(0, 0);
  cp_async_commit();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_holder;
  const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's 32 TMEM lanes

  float m = kNegInf, l = 0.f;
  bool bad = false, s_pending = false, o_pending = false;
  int kt = 0;
  for (; kt < n_kt; ++kt) {
    const int stage = kt & 1;
    // PV(kt-1) read the other stage: wait for it before refilling that stage
    if (o_pending) {
      bad |= !mbar_wait(bar_o, (kt - 1) & 1);
      o_pending = bad;
    }
    if (kt + 1 < n_kt && !bad) load_tile(kt + 1, stage ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    fence_async_smem();
    if (__syncthreads_or(bad)) break;
    if (tid == 0) {
      fence_after();
      const uint32_t ks = k_s + stage * K_BYTES;
#pragma unroll
      for (int s = 0; s < D / 16; ++s)
        mma(tmem, sdesc(q_s + (s >> 2) * (ROWS * 128) + (s & 3) * 32), sdesc(ks + (s >> 2) * (KT * 128) + (s & 3) * 32),
            idesc(ROWS, KT), s > 0);
      commit(bar_s);
    }
    s_pending = true;
    bad |= !mbar_wait(bar_s, kt & 1);
    s_pending = bad;
    fence_after();
    float sv[KT];
    tmem_ld32(t_lane + 0, sv);
    tmem_ld32(t_lane + 32, sv + 32);
    // key row a0 + j is key a0 + j - kv0 of the sequence: attended when in [b_lo, b_hi)
    const int64_t rel0 = (a_lo + kt) * KT - kv0;
    const int64_t jl = b_lo - rel0, jh = b_hi - rel0;
    const int j_lo = jl < 0 ? 0 : (jl > KT ? KT : (int)jl);
    const int j_hi = jh < 0 ? 0 : (jh > KT ? KT : (int)jh);
    float mx = kNegInf;
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      sv[j] = (j >= j_lo && j < j_hi) ? sv[j] * p.scale_log2 : kNegInf;
      mx = fmaxf(mx, sv[j]);
    }
    // lazy rescale: the running max moves only when a score exceeds it by 2^8
    const bool need = mx > m + 8.f;
    if (__any_sync(0xffffffffu, need)) {
      const float m_new = need ? mx : m;  // need implies mx > m
      const float alpha = need ? ex2(m - m_new) : 1.f;
      if (kt > 0) {
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float ov[32];
          tmem_ld32(t_lane + 128 + cc, ov);
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] *= alpha;
          tmem_st32(t_lane + 128 + cc, ov);
        }
      }
      l *= alpha;
      m = m_new;
    }
    const float mu = m == kNegInf ? 0.f : m;
    // P (bf16) goes over this stage's K tile, which S(kt) no longer reads
    const uint32_t ps = k_s + stage * K_BYTES;
#pragma unroll
    for (int ch = 0; ch < KT / 8; ++ch) {
      float e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        e[j] = ex2(sv[ch * 8 + j] - mu);
        l += e[j];
      }
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(sw128(ps, row, ch)), "r"(pack_bf16(e[0], e[1])),
                   "r"(pack_bf16(e[2], e[3])), "r"(pack_bf16(e[4], e[5])), "r"(pack_bf16(e[6], e[7]))
                   : "memory");
    }
    fence_async_smem();
    fence_before();
    if (__syncthreads_or(bad)) break;
    if (tid == 0) {
      fence_after();
      const uint32_t vs = v_s + stage * V_BYTES;
#pragma unroll
      for (int s = 0; s < KT / 16; ++s)
        mma(tmem + 128, sdesc(ps + s * 32), sdesc(vs + s * 32), idesc(ROWS, D), (kt > 0 || s > 0) ? 1u : 0u);
      commit(bar_o);
    }
    o_pending = true;
  }
  if (o_pending && !bad) {
    bad |= !mbar_wait(bar_o, (n_kt - 1) & 1);
    o_pending = bad;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    // drain: tensor-core work still in flight must finish before its TMEM is freed
    if (s_pending) mbar_wait(bar_s, kt & 1);
    if (o_pending) mbar_wait(bar_o, (kt - 1) & 1);
  }
  cp_async_wait<0>();
  fence_after();
  if (!bad) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* dst = p.o + ((start + t_row) * p.h + g * R + hd) * D;
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 32) {
      float ov[32];
      if (n_kt > 0) {
        tmem_ld32(t_lane + 128 + cc, ov);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = 0.f;
      }
      if (valid) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 pk;
          pk.x = pack_bf16(ov[j] * inv, ov[j + 1] * inv);
          pk.y = pack_bf16(ov[j + 2] * inv, ov[j + 3] * inv);
          pk.z = pack_bf16(ov[j + 4] * inv, ov[j + 5] * inv);
          pk.w = pack_bf16(ov[j + 6] * inv, ov[j + 7] * inv);
          *reinterpret_cast<uint4*>(dst + cc + j) = pk;
        }
      }
    }
    if (p.lse && valid) p.lse[(start + t_row) * p.h + g * R + hd] = l > 0.f ? (m + __log2f(l)) * kLn2 : kNegInf;
  }
  fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

// V [rows, hkv, D] -> V^T [hkv, D, pad] with pad = rows rounded up to 64.  Rows at or
// past `valid` (the rows the producer wrote; for compressed rows of packed sequences the
// sum of their counts) are written as zeros, so masked keys never multiply garbage.
__global__ void __launch_bounds__(256) transpose_kernel(const __nv_bfloat16* __restrict__ v,
                                                        __nv_bfloat16* __restrict__ vt, int64_t pad, int hkv,
                                                        int64_t valid, Seqs seqs, int kernel, int stride) {
  __shared__ __nv_bfloat16 tile[64][D + 8];
  if (valid < 0) valid = cmp_offset(seqs, seqs.n_seqs, kernel, stride);
  const int64_t r0 = (int64_t)blockIdx.x * 64;
  const int g = blockIdx.y;
  for (int c = threadIdx.x; c < 64 * (D / 8); c += 256) {
    const int r = c / (D / 8), ch = c % (D / 8);
    uint4 x = make_uint4(0, 0, 0, 0);
    if (r0 + r < valid) x = *reinterpret_cast<const uint4*>(v + ((r0 + r) * hkv + g) * D + ch * 8);
    *reinterpret_cast<uint4*>(&tile[r][ch * 8]) = x;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < D * 8; c += 256) {  // 128 d rows x 8 chunks of 8 keys
    const int d = c / 8, ch = c % 8;
    __align__(16) __nv_bfloat16 e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = tile[ch * 8 + j][d];
    *reinterpret_cast<uint4*>(vt + ((int64_t)g * D + d) * pad + r0 + ch * 8) = *reinterpret_cast<const uint4*>(e);
  }
}

}  // namespace tc

int64_t tc_vt_pad(int64_t rows) { return (rows + tc::KT - 1) / tc::KT * tc::KT; }

cudaError_t launch_transpose_v(const Seqs& s, const void* v, void* vt, int64_t rows, int hkv, bool compressed,
                               int kernel, int stride, cudaStream_t st) {
  const int64_t pad = tc_vt_pad(rows);
  if (pad == 0) return cudaSuccess;
  tc::transpose_kernel<<<dim3((unsigned)(pad / 64), hkv), 256, 0, st>>>(
      (const __nv_bfloat16*)v, (__nv_bfloat16*)vt, pad, hkv, compressed ? -1 : rows, s, kernel, stride);
  return cudaGetLastError();
}

cudaError_t launch_dense_attn_tc(int mode, const Seqs& s, const void* q, const void* k, const void* vt,
                                 int64_t kv_rows, int h, int hkv, int kernel, int stride, int window, float scale,
                                 void* o, float* lse, cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  tc::Params p{};
  p.q = (const __nv_bfloat16*)q;
  p.k = (const __nv_bfloat16*)k;
  p.vt = (const __nv_bfloat16*)vt;
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.R = h / hkv;
  p.kernel = kernel;
  p.stride = stride;
  p.window = window;
  p.kv_rows = kv_rows;
  p.kv_pad = tc_vt_pad(kv_rows);
  p.scale_log2 = scale * kLog2e;
  const int tpc = tc::ROWS / p.R;
  const dim3 grid((s.max_len + tpc - 1) / tpc, s.n_seqs, hkv);
  auto kern = mode == 0 ? tc::attn_kernel<0> : tc::attn_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, tc::SMEM_BYTES, st>>>(p);
  return cudaGetLastError();
}

cudaError_t read_device_status(int32_t* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_status, sizeof(int));
  if (e != cudaSuccess || !reset) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
}

}  // namespace nsa
