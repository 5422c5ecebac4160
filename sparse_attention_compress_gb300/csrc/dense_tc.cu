// Compressed and sliding-window branches on the 5th-generation tensor cores, and the
// block scores of the selection (fused into the compressed branch).
//
// [NSA-Triton] "DeepSeek NSA ... with Triton", sec. 1.1: the compressed branch attends
// to the mean-pooled keys/values, the sliding branch to the most recent tokens; both
// are dense attention over a contiguous key range per query.  [NOSA-Triton] mechanisms
// 2 and 3: the selection scores are the compressed attention probabilities, summed over
// the heads of a kv-group and mean-pooled over the compressed windows inside each
// 64-token block.
//
// GB300 design.  A CTA takes 128 (token, head) rows of one kv-group (8 tokens x 16 heads
// at group size 16): they share every K/V tile, so the contraction is an M = 128 GEMM.
// Warp roles (224 threads):
//   warp 4      TMA producer: Q once (a 3-D box of tokens x heads x d), then 64-key K
//               tiles and V^T tiles through 2-stage rings (128B-swizzled, K-major);
//   warp 5      S issuer (one lane): S(j) = Q K(j)^T into one of two TMEM S buffers,
//               issued while the softmax of tile j-1 runs;
//   warp 6      PV issuer: O += P(j) V(j) with P read from TMEM (a second issuing warp, on
//               another scheduler, since an issuing lane beside computing softmax warps
//               gets few issue slots);
//   warps 0..3  softmax, one row per thread (TMEM lane = row): mask, running max with
//               lazy rescale, base-2 exponentials, P (bf16) stored over its S buffer.
// Pass 2 (compressed branch with block scores): the issuer recomputes S over 64-key
// tiles aligned to the sequence's compressed index, so each tile holds 16 whole
// selection blocks; the softmax warps turn the scores into probabilities with the final
// normaliser, pool the three windows of each block, sum the group's heads with a
// reduce-scatter over lanes and write one fp32 score per (token, kv-head, block).
// Every mbarrier wait is bounded (about one second; a timeout sets the device status,
// makes the other roles leave their loops, drains the copies and MMAs in flight and
// frees the tensor memory).  Two CTAs share an SM (97 KB shared memory and 256 TMEM
// columns each).
#include "launch.h"
#include "sm100.cuh"

namespace nsa {
namespace tc {

constexpr int D = 128;
constexpr int ROWS = 128;  // query rows per CTA (= tcgen05 M)
constexpr int KT = 64;     // keys per tile
constexpr int NS = 2;      // K / V^T ring stages
constexpr int NTHREADS = 224;
// scores-only mode: no PV, so no PV issuer (warp 6)
constexpr int nthreads(int mode) { return mode == 2 ? NTHREADS - 32 : NTHREADS; }
constexpr int Q_BYTES = ROWS * D * 2;  // two 64-column halves of 16 KB
constexpr int K_BYTES = KT * D * 2;    // two halves of 8 KB
constexpr int V_BYTES = D * KT * 2;    // V^T tile: 128 d-rows of 64 keys
constexpr int SMEM_BYTES = Q_BYTES + NS * (K_BYTES + V_BYTES) + 1024;  // + 1 KB for alignment
constexpr int TMEM_COLS = 256;  // S buffers at columns 0 and 64 (P over their first 32), O at 128
// scores-only mode: no V ring and no O accumulator (three CTAs per SM)
constexpr int SMEM_BYTES_SCORES = Q_BYTES + NS * K_BYTES + 1024;
constexpr int TMEM_COLS_SCORES = 128;
constexpr uint32_t O_COL = 128;

// barrier slots
enum {
  B_Q = 0,
  B_KFULL = 1,
  B_KEMPTY = B_KFULL + NS,
  B_VFULL = B_KEMPTY + NS,
  B_VEMPTY = B_VFULL + NS,
  B_SFULL = B_VEMPTY + NS,  // [2] S(j) computed, indexed by j & 1
  B_SFREE = B_SFULL + 2,    // [2] pass 2: softmax has read S(j)
  B_PFULL = B_SFREE + 2,    // [2] softmax wrote P(j)
  B_ODONE = B_PFULL + 2,    // [2] PV(j) finished
  B_DRAIN = B_ODONE + 2,
  NBARS
};

// Reduce-scatter of 16 values over the R lanes of a group (R | 32, the lanes of a group
// contiguous): afterwards lane hd = lane % R holds in v[0 .. 16/R) the group sums of
// entries hd*(16/R) .. hd*(16/R) + 16/R - 1.
template <int R>
__device__ __forceinline__ void group_reduce_scatter(float (&v)[16], int lane) {
#pragma unroll
  for (int s = 0; (1 << s) < R; ++s) {
    const int off = R >> (s + 1), half = 8 >> s;
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}

// Maximum of a tile row, four independent chains.
__device__ __forceinline__ float row_max(const float (&v)[KT]) {
  float a = v[0], b = v[1], c = v[2], d = v[3];
#pragma unroll
  for (int j = 4; j < KT; j += 4) {
    a = fmaxf(a, v[j]);
    b = fmaxf(b, v[j + 1]);
    c = fmaxf(c, v[j + 2]);
    d = fmaxf(d, v[j + 3]);
  }
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

struct Params {
  __nv_bfloat16* o;
  float* lse;            // optional natural-log normaliser per (token, head)
  float* scores;         // MODE 0 with fused block scores, MODE 2: [tokens, hkv, nb_stride]
  const float* lse_in;   // MODE 2: normaliser given by the caller (pass 1 skipped), or null
  const __nv_bfloat16* k;  // MODE 0 / 2: key rows, for the copies of a tile that ends past them
  // MODE 0 / 2: key rows the buffer holds (-1: the packed compressed rows of all sequences;
  // 0, MODE 0 only: the buffer extends past every tile, no bounds checks)
  int64_t kv_total;
  const uint8_t* bmask;  // MODE 3: [batch, h, n_qb, n_qb] tile mask (query block, key block)
  int n_qb, causal;
  Seqs seqs;
  int h, hkv, R, kernel, stride, window, nb_stride;
  float scale_log2;
};

// Index of the last of items 0..last that went to ring stage st (-1 if none).
__device__ __forceinline__ int last_in_stage(int last, int st) {
  if (last < st) return -1;
  return last - (last - st) % NS;
}

// MODE 0: compressed branch (RS = group size when the block scores are fused, else 0);
// MODE 1: sliding window (RS = 0);
// MODE 2: block scores only (RS = group size): pass 1 keeps just the softmax statistics
//         (no V, no PV; skipped when the caller gives the normaliser), then pass 2;
// MODE 3: block-mask sparse attention, one head per CTA (128 tokens = two 64-token
//         query blocks): the key tiles are the 64-key blocks active for either query
//         block; each row masks the tiles its own block does not list.
template <int MODE, int RS>
__global__ void __launch_bounds__(nthreads(MODE), MODE == 2 ? 3 : 2)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_vt, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NBARS];
  __shared__ uint32_t tmem_holder;
  __shared__ int s_abort;
  const uint32_t base = (smem_u32(smem_raw) + 1023) & ~1023u;  // swizzle atoms need 1 KB alignment
  const uint32_t q_s = base, k_s = base + Q_BYTES, v_s = k_s + NS * K_BYTES;
  const uint32_t bar0 = smem_u32(&bars[0]);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // after a timeout anywhere on the device, later CTAs leave at once (the caller reads
  // the status word; the outputs of this launch are not valid)
  if (device_status_set()) return;
  const int R = RS > 0 ? RS : p.R;
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
  if (MODE == 0 || MODE == 2) {  // compressed keys
    n_c = num_cmp(L, p.kernel, p.stride);
    kv0 = cmp_offset(p.seqs, sq, p.kernel, p.stride);
    key_lo = 0;
    key_hi = num_causal_cmp(t_last, n_c, p.kernel, p.stride);
  } else {
    kv0 = start;
    key_lo = max(0, t0 - p.window + 1);
    key_hi = t_last + 1;
  }
  // MODE 3: per key block, bit 0 / bit 1 = active for the first / second query block
  uint8_t* tflag = smem_raw + (v_s - smem_u32(smem_raw)) + NS * V_BYTES;
  // pass 1: 64-key tiles in absolute key rows (64-aligned, so every V^T tile starts on a
  // 128-byte boundary); pass 2: tiles at kv0 + 64 i (16 whole selection blocks each)
  // (MODE 2 needs no V^T, so both of its passes use the sequence-aligned tiles)
  const int64_t a_lo = (kv0 + key_lo) / KT;
  const int n_kt2 = RS > 0 ? (key_hi + KT - 1) / KT : 0;
  int n_kt = MODE == 2 ? (p.lse_in ? 0 : n_kt2)
                       : (key_hi > key_lo ? (int)((kv0 + key_hi + KT - 1) / KT - a_lo) : 0);
  if (MODE == 3) {
    const int qb0 = t0 / KT, nbw = (p.n_qb + 3) / 4 * 4;
    const bool two = t0 + KT < L;
    const uint8_t* m0 = p.bmask + (((int64_t)sq * p.h + g) * p.n_qb + qb0) * p.n_qb;
    for (int kb = tid; kb < nbw; kb += nthreads(MODE)) {
      int f = 0;
      if (kb < p.n_qb) {
        if (m0[kb] && (!p.causal || kb <= qb0)) f |= 1;
        if (two && m0[p.n_qb + kb] && (!p.causal || kb <= qb0 + 1)) f |= 2;
      }
      tflag[kb] = (uint8_t)f;
    }
  }
  constexpr int kTmemCols = MODE == 2 ? TMEM_COLS_SCORES : TMEM_COLS;

  if (tid == 0) {
    mbar_init(bar(B_Q), 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SFREE + i), 128);
      mbar_init(bar(B_PFULL + i), 128);
      mbar_init(bar(B_ODONE + i), 1);
    }
    mbar_init(bar(B_DRAIN), MODE == 2 ? 1 : 2);  // the S and the PV issuer
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    fence_before();
  }
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_holder;
  int kb_cur = -1;  // MODE 3: this role's position in the active key blocks
  auto next_kb = [&]() {
    do ++kb_cur;
    while (tflag[kb_cur] == 0);
    return kb_cur;
  };
  if (MODE == 3) {  // every thread counts the active key blocks
    n_kt = 0;
    for (int w = 0; w < (p.n_qb + 3) / 4; ++w)
      n_kt += __popc(__vcmpne4(reinterpret_cast<const uint32_t*>(tflag)[w], 0u)) >> 3;
  }

  int last_k = -1, last_v = -1;  // producer: last K / V^T tile loads issued
  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(bar(B_Q), Q_BYTES);
      tma3d(q_s, &tm_q, 0, g * R, (int)(start + t0), bar(B_Q));
      tma3d(q_s + Q_BYTES / 2, &tm_q, 64, g * R, (int)(start + t0), bar(B_Q));
    }
    int64_t kv_total = p.kv_total;
    if ((MODE == 0 || MODE == 2) && kv_total < 0) {  // packed compressed rows of all sequences
      int64_t acc = 0;
      for (int i = lane; i < p.seqs.n_seqs; i += 32) acc += num_cmp(seq_len(p.seqs, i), p.kernel, p.stride);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      kv_total = acc;
    }
    for (int i = 0; i < n_kt + n_kt2; ++i) {
      const int st = i % NS;
      if (i >= NS && !warp_wait(bar(B_KEMPTY + st), ((i / NS) - 1) & 1, abort)) break;
      const int row = MODE == 3   ? (int)(kv0 + (int64_t)next_kb() * KT)
                      : MODE == 2 ? (int)(kv0 + (int64_t)(i < n_kt ? i : i - n_kt) * KT)
                                  : (i < n_kt ? (int)((a_lo + i) * KT) : (int)(kv0 + (int64_t)(i - n_kt) * KT));
      const uint32_t kb = bar(B_KFULL + st), ks = k_s + st * K_BYTES;
      if ((MODE == 2 || (MODE == 0 && kv_total != 0)) && row + KT > kv_total) {
        // a tile reaching past the caller's rows: bounds-checked copies (zeros past the
        // end) instead of TMA, then the async-proxy fence and a plain arrival
        for (int c = lane; c < KT * (D / 8); c += 32) {
          const int r = c / (D / 8), ch = c % (D / 8);
          const bool in = row + r < kv_total;
          const __nv_bfloat16* src = p.k + ((int64_t)(row + r) * p.hkv + g) * D + ch * 8;
          cp_async16(ks + (ch >> 3) * (K_BYTES / 2) + r * 128 + (((ch & 7) ^ (r & 7)) << 4),
                     in ? (const void*)src : (const void*)p.k, in ? 16 : 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(kb);
      } else if (lane == 0) {
        mbar_expect_tx(kb, K_BYTES);
        tma2d(ks, &tm_k, g * D, row, kb);
        tma2d(ks + K_BYTES / 2, &tm_k, g * D + 64, row, kb);
      }
      last_k = i;
      if (MODE != 2 && i < n_kt) {
        if (i >= NS && !warp_wait(bar(B_VEMPTY + st), ((i / NS) - 1) & 1, abort)) break;
        if (lane == 0) {
          const uint32_t vb = bar(B_VFULL + st);
          mbar_expect_tx(vb, V_BYTES);
          tma2d(v_s + st * V_BYTES, &tm_vt, row, g * D, vb);
        }
        last_v = i;
      }
      __syncwarp();
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    bool ok = warp_wait(bar(B_Q), 0, abort);
    if (MODE == 2) {
      // S buffer j & 1 is free once the softmax warps have read S(j - 2)
      for (int j = 0; ok && j < n_kt + n_kt2; ++j) {
        if (j >= 2) ok = warp_wait(bar(B_SFREE + (j & 1)), ((j - 2) >> 1) & 1, abort);
        if (ok) ok = warp_wait(bar(B_KFULL + j % NS), (j / NS) & 1, abort);
        if (!ok) break;
        if (lane == 0) {
          fence_after();
          const uint32_t ks = k_s + (j % NS) * K_BYTES;
#pragma unroll
          for (int s = 0; s < D / 16; ++s)
            mma_ss(tmem + (j & 1) * KT, sdesc(q_s + (s >> 2) * (Q_BYTES / 2) + (s & 3) * 32),
                   sdesc(ks + (s >> 2) * (K_BYTES / 2) + (s & 3) * 32), idesc(ROWS, KT), s > 0);
          commit(bar(B_SFULL + (j & 1)));
          commit(bar(B_KEMPTY + j % NS));
        }
        __syncwarp();
      }
    }
    // S(j) of the attention pass; PV is issued by warp 6
    for (int j = 0; MODE != 2 && ok && j < n_kt; ++j) {
      // S buffer j & 1 was last read by PV(j - 2)
      if (j >= 2) ok = warp_wait(bar(B_ODONE + (j & 1)), ((j - 2) >> 1) & 1, abort);
      if (ok) ok = warp_wait(bar(B_KFULL + j % NS), (j / NS) & 1, abort);
      if (!ok) break;
      if (lane == 0) {
        fence_after();
        const uint32_t ks = k_s + (j % NS) * K_BYTES;
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
          mma_ss(tmem + (j & 1) * KT, sdesc(q_s + (s >> 2) * (Q_BYTES / 2) + (s & 3) * 32),
                 sdesc(ks + (s >> 2) * (K_BYTES / 2) + (s & 3) * 32), idesc(ROWS, KT), s > 0);
        commit(bar(B_SFULL + (j & 1)));
        commit(bar(B_KEMPTY + j % NS));
      }
      __syncwarp();
    }
    for (int i = 0; MODE != 2 && ok && i < n_kt2; ++i) {
      const int j = n_kt + i, b = j & 1;
      if (i >= 2)
        ok = warp_wait(bar(B_SFREE + b), ((i - 2) >> 1) & 1, abort);
      else if (j >= 2)
        ok = warp_wait(bar(B_ODONE + b), ((j - 2) >> 1) & 1, abort);
      if (ok) ok = warp_wait(bar(B_KFULL + j % NS), (j / NS) & 1, abort);
      if (!ok) break;
      if (lane == 0) {
        fence_after();
        const uint32_t ks = k_s + (j % NS) * K_BYTES;
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
          mma_ss(tmem + b * KT, sdesc(q_s + (s >> 2) * (Q_BYTES / 2) + (s & 3) * 32),
                 sdesc(ks + (s >> 2) * (K_BYTES / 2) + (s & 3) * 32), idesc(ROWS, KT), s > 0);
        commit(bar(B_SFULL + b));
        commit(bar(B_KEMPTY + j % NS));
      }
      __syncwarp();
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------------ PV issuer
    // O += P(kt) V(kt) once the softmax warps wrote P(kt).  A second issuing warp, on
    // another scheduler than the S issuer: an issuing lane that shares its scheduler with
    // computing softmax warps gets few issue slots.
    bool ok = true;
    for (int kt = 0; MODE != 2 && ok && kt < n_kt; ++kt) {
      ok = warp_wait(bar(B_PFULL + (kt & 1)), (kt >> 1) & 1, abort);
      if (ok) ok = warp_wait(bar(B_VFULL + kt % NS), (kt / NS) & 1, abort);
      if (!ok) break;
      if (lane == 0) {
        fence_after();
        const uint32_t vs = v_s + (kt % NS) * V_BYTES;
#pragma unroll
        for (int s = 0; s < KT / 16; ++s)
          mma_ts(tmem + O_COL, tmem + (kt & 1) * KT + s * 8, sdesc(vs + s * 32), idesc(ROWS, D),
                 (kt > 0 || s > 0) ? 1u : 0u);
        commit(bar(B_ODONE + (kt & 1)));
        commit(bar(B_VEMPTY + kt % NS));
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int row = tid;
    const int tl = row / R, hd = row % R;
    const int t_row = t0 + tl;
    const bool valid = t_row < L;
    int b_lo = 0, b_hi = 0;  // attended keys [b_lo, b_hi), relative to kv0
    if (valid) {
      if (MODE == 0 || MODE == 2) {
        b_hi = num_causal_cmp(t_row, n_c, p.kernel, p.stride);
      } else {
        b_lo = max(0, t_row - p.window + 1);
        b_hi = t_row + 1;
      }
    }
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's 32 TMEM lanes
    float m = kNegInf, l = 0.f;
    bool ok = true;
    for (int kt = 0; MODE == 2 && kt < n_kt; ++kt) {
      // scores-only pass 1: running max and sum of the row, nothing else
      const int b = kt & 1;
      if (!(ok = warp_wait(bar(B_SFULL + b), (kt >> 1) & 1, abort))) break;
      fence_after();
      float sv[KT];
      tmem_ld64(t_lane + b * KT, sv);
      fence_before();
      mbar_arrive(bar(B_SFREE + b));
      const int j_hi = min(KT, max(0, b_hi - kt * KT));
      // max of the raw scores (scaling is monotonic), masked keys at -inf
      if (j_hi < KT) {
#pragma unroll
        for (int j = 0; j < KT; ++j) sv[j] = j < j_hi ? sv[j] : kNegInf;
      }
      float mx = row_max(sv) * p.scale_log2;
      if (mx > m + 8.f) {  // lazy rescale, as in the attention pass
        l *= ex2(m - mx);
        m = mx;
      }
      const float mu = m == kNegInf ? 0.f : m;
      float l4[4] = {0.f, 0.f, 0.f, 0.f};  // four chains of the row sum
#pragma unroll
      for (int j = 0; j < KT; ++j) l4[j & 3] += ex2(fmaf(sv[j], p.scale_log2, -mu));
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
    }
    for (int kt = 0; MODE != 2 && kt < n_kt; ++kt) {
      const int b = kt & 1;
      if (!(ok = warp_wait(bar(B_SFULL + b), (kt >> 1) & 1, abort))) break;
      fence_after();
      float sv[KT];
      tmem_ld64(t_lane + b * KT, sv);
      // key row a0 + j is key a0 + j - kv0 of the sequence: attended when in [b_lo, b_hi)
      int j_lo, j_hi;
      if (MODE == 3) {
        const int kb = next_kb();
        const bool on = valid && (tflag[kb] & (tl < KT ? 1 : 2));
        const int jh = on ? min(p.causal ? t_row - kb * KT + 1 : KT, L - kb * KT) : 0;
        j_lo = 0;
        j_hi = jh < 0 ? 0 : (jh > KT ? KT : jh);
      } else {
        const int64_t rel0 = (a_lo + kt) * KT - kv0;
        const int64_t jl = b_lo - rel0, jh = b_hi - rel0;
        j_lo = jl < 0 ? 0 : (jl > KT ? KT : (int)jl);
        j_hi = jh < 0 ? 0 : (jh > KT ? KT : (int)jh);
      }
      // max of the raw scores (scaling is monotonic); the mask only where the tile
      // reaches outside the row's keys
      if (j_lo > 0 || j_hi < KT) {
#pragma unroll
        for (int j = 0; j < KT; ++j) sv[j] = (j >= j_lo && j < j_hi) ? sv[j] : kNegInf;
      }
      const float mx = row_max(sv) * p.scale_log2;
      // lazy rescale: the running max moves only when a score exceeds it by 2^8
      const bool need = mx > m + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m - mx) : 1.f;  // need implies mx finite
        if (kt > 0) {
          // O must hold PV(kt-1) before it is rescaled
          if (!(ok = warp_wait(bar(B_ODONE + ((kt - 1) & 1)), ((kt - 1) >> 1) & 1, abort))) break;
          fence_after();
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            float ov[32];
            tmem_ld32(t_lane + O_COL + cc, ov);
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] *= alpha;
            tmem_st32(t_lane + O_COL + cc, reinterpret_cast<const uint32_t*>(ov));
          }
        }
        if (need) {
          l *= alpha;
          m = mx;
        }
      }
      const float mu = m == kNegInf ? 0.f : m;
      uint32_t pk[KT / 2];
      float l4[4] = {0.f, 0.f, 0.f, 0.f};  // four chains of the row sum
#pragma unroll
      for (int j = 0; j < KT; j += 2) {
        const float e0 = ex2(fmaf(sv[j], p.scale_log2, -mu)), e1 = ex2(fmaf(sv[j + 1], p.scale_log2, -mu));
        l4[(j >> 1) & 3] += e0 + e1;
        pk[j / 2] = pack_bf16(e0, e1);
      }
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      tmem_st32(t_lane + b * KT, pk);  // P over the first 32 columns of its S buffer
      fence_before();
      mbar_arrive(bar(B_PFULL + b));
    }
    if (MODE != 2 && ok && n_kt > 0) {
      ok = warp_wait(bar(B_ODONE + ((n_kt - 1) & 1)), ((n_kt - 1) >> 1) & 1, abort);
      fence_after();
    }
    if (MODE != 2 && ok) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = p.o + ((start + t_row) * p.h + g * R + hd) * D;
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        float ov[32];
        if (n_kt > 0) {
          tmem_ld32(t_lane + O_COL + cc, ov);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0.f;
        }
        if (valid) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 v;
            v.x = pack_bf16(ov[j] * inv, ov[j + 1] * inv);
            v.y = pack_bf16(ov[j + 2] * inv, ov[j + 3] * inv);
            v.z = pack_bf16(ov[j + 4] * inv, ov[j + 5] * inv);
            v.w = pack_bf16(ov[j + 6] * inv, ov[j + 7] * inv);
            *reinterpret_cast<uint4*>(dst + cc + j) = v;
          }
        }
      }
      if (p.lse && valid) p.lse[(start + t_row) * p.h + g * R + hd] = l > 0.f ? (m + __log2f(l)) * kLn2 : kNegInf;
    }
    if (RS > 0 && ok) {
      // ---------------------------------------------------------------- pass 2: block scores
      // base-2 normaliser of the scaled scores (0 for rows without keys)
      float lse2 = l > 0.f ? m + __log2f(l) : 0.f;
      if (MODE == 2 && p.lse_in && valid) {
        const float li = p.lse_in[(start + t_row) * p.h + g * R + hd];
        lse2 = li > kNegInf ? li * kLog2e : 0.f;
      }
      float* out = p.scores + ((start + t_row) * p.hkv + g) * p.nb_stride;
      constexpr int PER = RS > 0 ? 16 / RS : 1;  // blocks per lane after the head reduction
      for (int i = 0; i < n_kt2; ++i) {
        const int j = n_kt + i, b = j & 1;
        if (!(ok = warp_wait(bar(B_SFULL + b), (j >> 1) & 1, abort))) break;
        fence_after();
        float sv[KT];
        tmem_ld64(t_lane + b * KT, sv);
        fence_before();
        mbar_arrive(bar(B_SFREE + b));
        const int jh = min(KT, max(0, b_hi - i * KT));  // causal compressed keys of this tile
        float bs[16];
#pragma unroll
        for (int jb = 0; jb < 16; ++jb) {
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            const int jj = 4 * jb + c;
            acc += jj < jh ? ex2(fmaf(sv[jj], p.scale_log2, -lse2)) : 0.f;
          }
          bs[jb] = acc;
        }
        group_reduce_scatter<RS>(bs, lane);
        if (valid) {
#pragma unroll
          for (int u = 0; u < PER; ++u) {
            const int blk = i * 16 + hd * PER + u;
            if (blk < p.nb_stride) {
              const int c0 = 4 * blk;
              const int cnt = (c0 < n_c) + (c0 + 1 < n_c) + (c0 + 2 < n_c);
              out[blk] = bs[u] * (cnt == 3 ? (1.f / 3.f) : cnt == 2 ? 0.5f : cnt == 1 ? 1.f : 0.f);
            }
          }
        }
      }
      // blocks past the last tile hold no causal probability
      if (ok && valid)
        for (int blk = n_kt2 * 16 + hd; blk < p.nb_stride; blk += R) out[blk] = 0.f;
    }
  }

  __syncthreads();
  if (*abort) {
    // drain: copies and MMAs still in flight must land before the CTA leaves
    if (warp == 4) {
      mbar_drain(bar(B_Q), 0);
      for (int st = 0; st < NS; ++st) {
        const int ik = last_in_stage(last_k, st), iv = last_in_stage(last_v, st);
        if (ik >= 0) mbar_drain(bar(B_KFULL + st), (ik / NS) & 1);
        if (iv >= 0) mbar_drain(bar(B_VFULL + st), (iv / NS) & 1);
      }
    } else if (warp == 5 || warp == 6) {
      if (lane == 0) commit(bar(B_DRAIN));
      __syncwarp();
      mbar_drain(bar(B_DRAIN), 0);
    }
  } else if (warp == 4) {
    // every MMA completion that arrives on a ring barrier lands before the CTA leaves:
    // wait for the last release of each stage
    for (int st = 0; st < NS; ++st) {
      const int ik = last_in_stage(last_k, st), iv = last_in_stage(last_v, st);
      if (ik >= 0) mbar_drain(bar(B_KEMPTY + st), (ik / NS) & 1);
      if (iv >= 0) mbar_drain(bar(B_VEMPTY + st), (iv / NS) & 1);
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// V [rows, hkv, D] -> V^T [hkv, D, pad] with pad = rows rounded up to 64.  Rows at or
// past `valid` (the rows the producer wrote; for compressed rows of packed sequences the
// sum of their counts) are written as zeros, so masked keys never multiply garbage.
// The staging tile keeps row r's 16-byte chunk c at chunk c ^ (r / 8): the column reads
// of the transpose then hit eight different bank groups.
__global__ void __launch_bounds__(256) transpose_kernel(const __nv_bfloat16* __restrict__ v,
                                                        __nv_bfloat16* __restrict__ vt, int64_t pad, int hkv,
                                                        int64_t valid, Seqs seqs, int kernel, int stride) {
  __shared__ __align__(16) __nv_bfloat16 tile[64][D];
  if (valid < 0) valid = cmp_offset(seqs, seqs.n_seqs, kernel, stride);
  const int64_t r0 = (int64_t)blockIdx.x * 64;
  const int g = blockIdx.y;
  for (int c = threadIdx.x; c < 64 * (D / 8); c += 256) {
    const int r = c / (D / 8), ch = c % (D / 8);
    uint4 x = make_uint4(0, 0, 0, 0);
    if (r0 + r < valid) x = *reinterpret_cast<const uint4*>(v + ((r0 + r) * hkv + g) * D + ch * 8);
    *reinterpret_cast<uint4*>(&tile[r][(ch ^ (r >> 3)) * 8]) = x;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < D * 8; c += 256) {  // 128 d rows x 8 chunks of 8 keys
    const int d = c / 8, ch = c % 8;
    __align__(16) __nv_bfloat16 e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = tile[ch * 8 + j][(((d >> 3) ^ ch) << 3) | (d & 7)];
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

template <int MODE, int RS>
static cudaError_t run_tc(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const tc::Params& p,
                          dim3 grid, cudaStream_t st) {
  auto kern = tc::attn_kernel<MODE, RS>;
  constexpr int smem = MODE == 2 ? tc::SMEM_BYTES_SCORES : tc::SMEM_BYTES + (MODE == 3 ? 1024 : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, tc::nthreads(MODE), smem, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

cudaError_t launch_dense_attn_tc(int mode, const Seqs& s, const void* q, const void* k, const void* vt,
                                 int64_t kv_rows, int h, int hkv, int kernel, int stride, int window, float scale,
                                 void* o, float* lse, float* scores, int nb_stride, cudaStream_t st,
                                 int64_t kv_total) {
  if (s.tokens == 0) return cudaSuccess;
  const int R = h / hkv;
  const int tpc = tc::ROWS / R;
  // a map needs nonzero extents; with no key rows no tile is ever loaded
  const uint64_t rows = kv_rows > 0 ? (uint64_t)kv_rows : 1;
  const uint64_t pad = (uint64_t)tc_vt_pad((int64_t)rows);
  CUtensorMap mq, mk, mv;
  {
    const uint64_t dims[3] = {(uint64_t)tc::D, (uint64_t)h, (uint64_t)s.tokens};
    const uint64_t strides[2] = {(uint64_t)tc::D * 2, (uint64_t)h * tc::D * 2};
    const uint32_t box[3] = {64, (uint32_t)R, (uint32_t)tpc};
    if (!tc::make_map(&mq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)hkv * tc::D, rows};
    const uint64_t strides[1] = {(uint64_t)hkv * tc::D * 2};
    const uint32_t box[2] = {64, (uint32_t)tc::KT};
    if (!tc::make_map(&mk, k, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {pad, (uint64_t)hkv * tc::D};
    const uint64_t strides[1] = {pad * 2};
    const uint32_t box[2] = {64, (uint32_t)tc::D};
    if (!tc::make_map(&mv, vt, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  tc::Params p{};
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.scores = scores;
  p.k = (const __nv_bfloat16*)k;
  p.kv_total = mode == 0 ? kv_total : 0;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.R = R;
  p.kernel = kernel;
  p.stride = stride;
  p.window = window;
  p.nb_stride = nb_stride;
  p.scale_log2 = scale * kLog2e;
  const dim3 grid((s.max_len + tpc - 1) / tpc, s.n_seqs, hkv);
  if (mode == 1) return run_tc<1, 0>(mq, mk, mv, p, grid, st);
  if (!scores) return run_tc<0, 0>(mq, mk, mv, p, grid, st);
  switch (R) {
    case 1: return run_tc<0, 1>(mq, mk, mv, p, grid, st);
    case 2: return run_tc<0, 2>(mq, mk, mv, p, grid, st);
    case 4: return run_tc<0, 4>(mq, mk, mv, p, grid, st);
    case 8: return run_tc<0, 8>(mq, mk, mv, p, grid, st);
    case 16: return run_tc<0, 16>(mq, mk, mv, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_block_sparse_tc(const Seqs& s, const void* q, const void* k, const void* vt, int h,
                                   const uint8_t* mask, int causal, float scale, void* o, float* lse,
                                   cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  const uint64_t rows = (uint64_t)s.tokens;
  const uint64_t pad = (uint64_t)tc_vt_pad((int64_t)rows);
  CUtensorMap mq, mk, mv;
  {
    const uint64_t dims[3] = {(uint64_t)tc::D, (uint64_t)h, rows};
    const uint64_t strides[2] = {(uint64_t)tc::D * 2, (uint64_t)h * tc::D * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)tc::ROWS};
    if (!tc::make_map(&mq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)h * tc::D, rows};
    const uint64_t strides[1] = {(uint64_t)h * tc::D * 2};
    const uint32_t box[2] = {64, (uint32_t)tc::KT};
    if (!tc::make_map(&mk, k, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {pad, (uint64_t)h * tc::D};
    const uint64_t strides[1] = {pad * 2};
    const uint32_t box[2] = {64, (uint32_t)tc::D};
    if (!tc::make_map(&mv, vt, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  tc::Params p{};
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.bmask = mask;
  p.n_qb = (s.max_len + tc::KT - 1) / tc::KT;
  p.causal = causal;
  p.seqs = s;
  p.h = h;
  p.hkv = h;
  p.R = 1;
  p.scale_log2 = scale * kLog2e;
  const dim3 grid((s.max_len + tc::ROWS - 1) / tc::ROWS, s.n_seqs, h);
  return run_tc<3, 0>(mq, mk, mv, p, grid, st);
}

bool dense_tc_supported(int h, int hkv, int d) {
  const int R = hkv > 0 ? h / hkv : 0;
  return d == tc::D && R >= 1 && R * hkv == h && R <= tc::ROWS && (R & (R - 1)) == 0;
}

bool scores_tc_supported(int h, int hkv, int d, int kernel, int stride, int block_size) {
  const int R = hkv > 0 ? h / hkv : 0;
  return d == tc::D && kernel == 32 && stride == 16 && block_size == 64 && R * hkv == h &&
         (R == 1 || R == 2 || R == 4 || R == 8 || R == 16);
}

cudaError_t launch_scores_tc(const Seqs& s, const void* q, const void* k_cmp, int64_t kv_rows, int64_t kv_total,
                             int h, int hkv, float scale, const float* lse_in, float* scores, int nb_stride,
                             cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  const int R = h / hkv;
  const int tpc = tc::ROWS / R;
  const uint64_t rows = kv_rows > 0 ? (uint64_t)kv_rows : 1;
  CUtensorMap mq, mk;
  {
    const uint64_t dims[3] = {(uint64_t)tc::D, (uint64_t)h, (uint64_t)s.tokens};
    const uint64_t strides[2] = {(uint64_t)tc::D * 2, (uint64_t)h * tc::D * 2};
    const uint32_t box[3] = {64, (uint32_t)R, (uint32_t)tpc};
    if (!tc::make_map(&mq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)hkv * tc::D, rows};
    const uint64_t strides[1] = {(uint64_t)hkv * tc::D * 2};
    const uint32_t box[2] = {64, (uint32_t)tc::KT};
    if (!tc::make_map(&mk, k_cmp, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  tc::Params p{};
  p.scores = scores;
  p.lse_in = lse_in;
  p.k = (const __nv_bfloat16*)k_cmp;
  p.kv_total = kv_total;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.R = R;
  p.kernel = 32;
  p.stride = 16;
  p.nb_stride = nb_stride;
  p.scale_log2 = scale * kLog2e;
  const dim3 grid((s.max_len + tpc - 1) / tpc, s.n_seqs, hkv);
  switch (R) {  // the V map is never read in this mode
    case 1: return run_tc<2, 1>(mq, mk, mk, p, grid, st);
    case 2: return run_tc<2, 2>(mq, mk, mk, p, grid, st);
    case 4: return run_tc<2, 4>(mq, mk, mk, p, grid, st);
    case 8: return run_tc<2, 8>(mq, mk, mk, p, grid, st);
    case 16: return run_tc<2, 16>(mq, mk, mk, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

NSA_STATUS_ACCESSOR(dense_tc)

}  // namespace nsa
