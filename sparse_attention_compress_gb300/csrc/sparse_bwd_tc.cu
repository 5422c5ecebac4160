// dK and dV of selected-block attention (and of the compressed and sliding-window branches,
// the same kernel in their key spaces) on the fifth-generation tensor cores.
//
// The derivative is the one sparse_bwd.cu states ([TileLang-NSA] "TileLang operator
// development: Native Sparse Attention", sec. 2 for the forward; [NSA-Triton] "DeepSeek
// NSA ... with Triton", sec. 4 for training with it): per (token, head) row that reaches
// key e, p = exp(scale q.k_e - lse), ds = p (dO.v_e - D), dk[e] += scale ds q,
// dv[e] += p dO.
//
// GB300 design.  A work item is (sequence, kv-head, key block j, query chunk), as for
// sparse_bwd_dkv, and writes the same fp32 partials, so sparse_bwd_reduce sums them.
// The rows that reach block j are gathered 128 at a time (128 / r tokens of r heads):
//   S = Q K_j^T and dP = dO V_j^T      M = 128 rows, N = 64 keys, K = d   (TMEM)
//   P, dS from S, dP, lse, D            softmax warps, one row per thread
//   dV^T += dO^T P,  dK^T += Q^T dS     M = 128 (d), N = 64 keys, K = 128 rows (TMEM)
// The same shared-memory tile of Q (or dO) is the K-major A operand of the first
// product and the MN-major A operand of the second, so no transpose is made.  P and dS
// enter the second products as bf16 pairs (the rounded value and its remainder, so the
// operand carries about 16 bits), as in sparse_bwd_dkv.  Roles: warp 8 takes the tokens
// that reach j and gathers their Q and dO rows by TMA into a two-stage ring; warp 9
// issues S and dP (into one of two TMEM buffers, so the next tile's products run while
// the softmax warps work on this one), warps 10 and 11 the dV and the dK products (issuing
// warps on different schedulers: an issuing lane beside computing softmax warps gets few
// issue slots); warps 0-7, two per scheduler, form P and dS (each a half of every row's 64
// keys) and finally read dK^T and dV^T out of TMEM.  One CTA per SM (224 KB of shared
// memory).
#include <algorithm>

#include "sm100.cuh"
#include "sparse_bwd.cuh"
#include "topk.cuh"

namespace nsa {
namespace bwd {

namespace {

constexpr int kSoftWarps = 8;  // two per scheduler: warp w takes rows 32 (w % 4) .. and key half w / 4
constexpr int kSoft = kSoftWarps * 32;
constexpr int kProducer = kSoftWarps, kIssuer = kSoftWarps + 1;  // warp roles
constexpr int kThreads = kSoft + 64;
constexpr int kTileRows = 128;                   // gathered (token, head) rows per tile
constexpr int kKVBytes = kBS * kD * 2;           // K_j or V_j: two 64-column halves of 64 rows
constexpr int kHalfRows = kTileRows * 128;       // one 64-column half of a 128-row tile
constexpr int kQBytes = 2 * kHalfRows;           // Q (or dO) of one tile
constexpr int kStageBytes = 2 * kQBytes;         // Q and dO
constexpr int kPBytes = kTileRows * kBS * 2;     // P or dS (hi or lo) of one tile: 128 rows x 64 keys
constexpr int kSmemBytes = 2 * kKVBytes + 2 * kStageBytes + 4 * kPBytes + 1024;  // + base alignment
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S and dP of tile buffer b at 128 b and 128 b + 64; then dV^T and dK^T in
// two parts each, the products of the bf16-rounded P / dS and of their remainders (the
// epilogue adds the parts).  A part pair is contiguous, so one N = 128 product fills both:
// its B operand is the rounded and the remainder buffer (adjacent, kPBytes apart) as the
// two 64-column groups of one MN-major operand.
constexpr uint32_t kColDV = 256, kColDVlo = 320, kColDK = 384, kColDKlo = 448;
// P or dS values above these make the remainder products count (as in sparse_bwd_dkv)
constexpr float kLoP = 0.00390625f, kLoS = 0.0625f;

enum : int {
  B_FULL = 0,    // [2] a stage's Q, dO and token list landed
  B_EMPTY = 2,   // [2] the MMAs reading a stage are done
  B_KV = 4,      // K_j and V_j are in shared memory
  B_SFULL = 5,   // [2] S and dP of a tile buffer computed
  B_SFREE = 7,   // [2] the softmax warps have read a tile buffer
  B_PFULL = 9,   // P and dS of a tile are in shared memory
  B_PFREE = 10,  // the dV / dK products of that tile are done
  B_ADONE = 11,  // every product of the item is done
  B_DRAIN = 12,
  B_SDONE = 13,  // the S / dP issuer saw the list's last tile (the row-tile count is in s_nrows)
  B_COUNT = 14
};
// dkv_tc: the dV and the dK issuer (beside the S / dP issuer, kIssuer)
constexpr int kDvIssuer = kSoftWarps + 2, kDkIssuer = kSoftWarps + 3, kKVThreads = kThreads + 64;

// Shared-memory descriptor of an MN-major tile with 128-byte swizzling: rows of 64
// MN-elements (128 B) along K, 1024-byte atoms of 8 K-rows.  lbo: byte distance between
// groups of 64 MN-elements; sbo: between groups of 8 K-rows.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
// bf16 x bf16 -> fp32 with both operands MN-major
constexpr uint32_t idesc_mn(int M, int N) { return tc::idesc(M, N) | (1u << 15) | (1u << 16); }

// Item slot in the numbering of item_to_block (the order sparse_bwd_reduce reads).
__device__ __forceinline__ int slot_of(const BwdParams& p, int j, int c) {
  if (p.window) return j;
  if (p.cmp_kernel) {
    int s = 0;
    for (int jj = 0; jj < j; ++jj) s += p.n_chunks - first_query(p, jj) / kChunk;
    return s + c - first_query(p, j) / kChunk;
  }
  const int m = j / kGroup;
  int s = 0;
  for (int mm = 0; mm < m; ++mm) s += min(kGroup, p.nb - mm * kGroup) * (p.n_chunks - mm);
  return s + (j - m * kGroup) * (p.n_chunks - m) + (c - m);
}

// CTA x -> (sequence and kv-head bg, key block j, query chunk c).  Selected blocks: every
// block-0 item first (each token's list holds block 0, so these items are the longest),
// then per (sequence, kv-head) the chunks in order and, within a chunk, the blocks it
// reaches in order, so that the CTAs running together share their chunk's Q and dO in L2.
// Compressed keys: per (sequence, kv-head), chunk-major the same way.  Window: one item
// per block.
__device__ __forceinline__ void dispatch(const BwdParams& p, int x, int& bg, int& j, int& c) {
  const int n_bg = p.seqs.n_seqs * p.hkv;
  if (p.window) {
    bg = x / p.nb;
    j = x % p.nb;
    c = 0;
    return;
  }
  if (!p.cmp_kernel) {
    const int head = n_bg * p.n_chunks;
    if (x < head) {
      bg = x / p.n_chunks;
      j = 0;
      c = x % p.n_chunks;
      return;
    }
    x -= head;
    const int per = p.items_per_bg - p.n_chunks;
    bg = x / per;
    int rem = x % per;
    for (c = 0; c < p.n_chunks; ++c) {
      const int nbc = min(p.nb, (c + 1) * kGroup) - 1;  // blocks 1 .. reached by chunk c
      if (rem < nbc) {
        j = rem + 1;
        return;
      }
      rem -= nbc;
    }
    j = p.nb;  // not reached
    return;
  }
  bg = x / p.items_per_bg;
  int rem = x % p.items_per_bg;
  const int span = p.cmp_stride * kBS;  // tokens per compressed key block
  for (c = 0; c < p.n_chunks; ++c) {
    // blocks whose first reaching query lies in chunk c or before
    const int lim = (c + 1) * kChunk - p.cmp_kernel + 1;
    const int nbc = min(p.nb, lim > 0 ? (lim + span - 1) / span : 0);
    if (rem < nbc) {
      j = rem;
      return;
    }
    rem -= nbc;
  }
  j = p.nb;  // not reached
}

// Chunk-wise inverted lists of the selected blocks.  Block (chunk c, sequence and kv-head
// bg): the tokens t of the chunk whose list holds a block j with 64 j <= t (the entries
// that reach a key), grouped by j.  Eight warps own 256 consecutive tokens each; pass 1
// counts (warp, block) pairs, a prefix over the blocks and warps places each warp's run
// inside each block's bucket, and pass 2 writes the tokens in warp, token and list-entry
// order (ranks within a warp from __match_any_sync), so the lists, and the dK / dV sums
// over them, are the same on every run.  Shared memory: 8 x min(nb, (c + 1) * kGroup) ints.
__global__ void __launch_bounds__(256) invert_kernel(const BwdParams p) {
  extern __shared__ int s_cnt[];  // [8][nbr]
  __shared__ int s_tot[8];
  const int c = blockIdx.x, bg = blockIdx.y;
  const int b = bg / p.hkv, g = bg % p.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = seq_len(p.seqs, b);
  const int nbr = min(p.nb, (c + 1) * kGroup);  // blocks a query of chunk c can reach
  const size_t seg = (size_t)bg * p.n_chunks + c;
  int2* tab = p.inv_tab + seg * p.nb;
  for (int jj = nbr + tid; jj < p.nb; jj += 256) tab[jj] = make_int2(0, 0);
  const int t0 = c * kChunk, t1 = min(L, t0 + kChunk);
  for (int i = tid; i < 8 * nbr; i += 256) s_cnt[i] = 0;
  __syncthreads();
  const int64_t base = seq_start(p.seqs, b);
  const int wt0 = t0 + warp * (kChunk / 8), wt1 = min(t1, wt0 + kChunk / 8);
  auto entry = [&](int t, int e) -> int {  // block of list entry e of token t, or -1
    const int jj = __ldg(p.idx + ((base + t) * p.hkv + g) * p.S + e);
    return (jj >= 0 && jj < nbr && jj * kBS <= t) ? jj : -1;
  };
  for (int tb = wt0; tb < wt1; tb += 32) {
    const int t = tb + lane;
    if (t < wt1)
      for (int e = 0; e < p.S; ++e) {
        const int jj = entry(t, e);
        if (jj >= 0) atomicAdd(&s_cnt[warp * nbr + jj], 1);
      }
  }
  __syncthreads();
  // bucket offsets: blocks 4 tid .. 4 tid + 3 per thread (nbr <= 1024)
  int tot[4], sum = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int jj = 4 * tid + u;
    tot[u] = 0;
    if (jj < nbr)
      for (int w = 0; w < 8; ++w) tot[u] += s_cnt[w * nbr + jj];
    sum += tot[u];
  }
  int off = block_excl_scan<8>(sum, s_tot, lane, warp);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int jj = 4 * tid + u;
    if (jj < nbr) {
      tab[jj] = make_int2(off, tot[u]);
      int run = off;
      for (int w = 0; w < 8; ++w) {
        const int x = s_cnt[w * nbr + jj];
        s_cnt[w * nbr + jj] = run;
        run += x;
      }
    }
    off += tot[u];
  }
  __syncthreads();
  int32_t* list = p.inv_list + seg * kChunk * p.S;
  for (int tb = wt0; tb < wt1; tb += 32) {
    const int t = tb + lane;
    for (int e = 0; e < p.S; ++e) {
      const int jj = t < wt1 ? entry(t, e) : -1;
      const unsigned same = __match_any_sync(0xffffffffu, jj);
      const int rank = __popc(same & ((1u << lane) - 1u));
      if (jj >= 0) list[s_cnt[warp * nbr + jj] + rank] = t;
      __syncwarp();
      if (jj >= 0 && rank == 0) s_cnt[warp * nbr + jj] += __popc(same);
      __syncwarp();
    }
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint32_t (&v)[4]) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
               : "memory");
}

// P and dS of 32 keys of a gathered row (keys 64 j + 32 kh ..), as bf16 values and
// remainders into the four shared-memory tiles (the row's 16-byte chunks c8 = 4 kh + cc,
// 128-byte swizzled); MASK: keys outside [tl, tb] give 0.  Keeps the row's max P, |dS|.
struct PdsArgs {
  float fm, scale_log2, lse2, dsum;
  int tl, tb, kb0, row, kh;
  uint32_t p_hi, p_lo, s_hi, s_lo;
};
template <bool MASK>
__device__ __forceinline__ void form_pds(float (&sv)[32], float (&dpv)[32], const PdsArgs& a, float& pmax,
                                         float& smax) {
  // sv holds S on entry and P on return, dpv dP and then dS; the rounded parts are stored
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {  // keys 8 c8 .. 8 c8 + 7 (one 16-byte chunk), c8 = 4 kh + cc
    const int c8 = a.kh * 4 + cc;
    uint32_t ph[4], sh[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      float p0 = a.fm * ex2(fmaf(sv[cc * 8 + e], a.scale_log2, -a.lse2));
      float p1 = a.fm * ex2(fmaf(sv[cc * 8 + e + 1], a.scale_log2, -a.lse2));
      if (MASK) {
        const int k0 = a.kb0 + c8 * 8 + e;
        p0 = k0 <= a.tb && k0 >= a.tl ? p0 : 0.f;
        p1 = k0 + 1 <= a.tb && k0 + 1 >= a.tl ? p1 : 0.f;
      }
      const float d0 = p0 * (dpv[cc * 8 + e] - a.dsum), d1 = p1 * (dpv[cc * 8 + e + 1] - a.dsum);
      sv[cc * 8 + e] = p0;
      sv[cc * 8 + e + 1] = p1;
      dpv[cc * 8 + e] = d0;
      dpv[cc * 8 + e + 1] = d1;
      pmax = fmaxf(pmax, fmaxf(p0, p1));
      smax = fmaxf(smax, fmaxf(fabsf(d0), fabsf(d1)));
      ph[e / 2] = pack_bf16(p0, p1);
      sh[e / 2] = pack_bf16(d0, d1);
    }
    const uint32_t off = a.row * 128 + ((c8 ^ (a.row & 7)) << 4);
    st_shared_v4(a.p_hi + off, ph);
    st_shared_v4(a.s_hi + off, sh);
  }
}

// The bf16 remainders of the 32 values x into the remainder tile at base (the row's
// chunks c8 = 4 kh + cc), or zeros: a warp whose values all lie below the threshold
// drops its remainders (the remainder products then add nothing for its rows).
__device__ __forceinline__ void store_remainders(const float (&x)[32], uint32_t base, int row, int kh, bool need) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c8 = kh * 4 + cc;
    uint32_t r[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      if (need) {
        const uint32_t h = pack_bf16(x[cc * 8 + e], x[cc * 8 + e + 1]);
        const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h));
        r[e / 2] = pack_bf16(x[cc * 8 + e] - hf.x, x[cc * 8 + e + 1] - hf.y);
      } else {
        r[e / 2] = 0u;
      }
    }
    st_shared_v4(base + row * 128 + ((c8 ^ (row & 7)) << 4), r);
  }
}

template <int R>
__global__ void __launch_bounds__(kKVThreads, 1)
    dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_q3, const __grid_constant__ CUtensorMap tm_do3,
                  const BwdParams p) {
  constexpr int TPT = kTileRows / R;  // tokens per tile
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t s_bar[B_COUNT];
  __shared__ int s_meta[2][TPT + 2];  // per stage: (token << 7 | multiplicity) per slot, count, last
  __shared__ int s_need[kSoftWarps];  // per softmax warp, for the tile in the P buffer: remainder products needed
  __shared__ int s_nrows;             // tiles with rows (written by the S / dP issuer before SDONE)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bg, j, c;
  dispatch(p, blockIdx.x, bg, j, c);
  const int b = bg / p.hkv, g = bg % p.hkv;
  const int L = seq_len(p.seqs, b);
  const int Lk = key_len(p, L);
  const int m = p.window ? 0 : (p.cmp_kernel ? first_query(p, j) / kChunk : j / kGroup);
  if (j >= p.nb || j * kBS >= Lk || (c > m && c * kChunk >= L)) return;  // no partial is read for this item
  const int slot_item = slot_of(p, j, c);
  const int64_t base = seq_start(p.seqs, b);
  const int64_t kbase = key_base(p, b);
  const int t_begin = p.window ? j * kBS : max(first_query(p, j), c * kChunk);
  const int t_end = p.window ? min(j * kBS + kBS - 1 + p.window, L) : min((c + 1) * kChunk, L);

  const uint32_t sbase = (smem_u32(smem_raw) + 1023) & ~1023u;
  const uint32_t kt = sbase, vt = kt + kKVBytes;
  const uint32_t stage0 = vt + kKVBytes;
  const uint32_t p_hi = stage0 + 2 * kStageBytes, p_lo = p_hi + kPBytes, s_hi = p_lo + kPBytes, s_lo = s_hi + kPBytes;
  auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
  volatile int* abort = &s_abort;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar(B_FULL + i), 1);
      tc::mbar_init(bar(B_EMPTY + i), 2);  // the dV and the dK issuer
      tc::mbar_init(bar(B_SFULL + i), 1);
      tc::mbar_init(bar(B_SFREE + i), kSoft);
    }
    tc::mbar_init(bar(B_KV), kSoft);
    tc::mbar_init(bar(B_PFULL), kSoft);
    tc::mbar_init(bar(B_PFREE), 2);  // the dV and the dK issuer
    tc::mbar_init(bar(B_ADONE), 2);
    tc::mbar_init(bar(B_DRAIN), 3);  // the three issuing warps
    tc::mbar_init(bar(B_SDONE), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kIssuer) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    tc::fence_before();
  }
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = s_tmem;

  int n_tiles = 0;      // producer: tiles handed to the ring
  int last_full[2] = {-1, -1};  // producer: last tile with rows in each stage
  if (warp == kProducer) {
    // ------------------------------------------------------------------ token tiles + TMA
    // Every tile but an empty item's marker holds TPT slots; the item's last tile is
    // flagged.  Slots past the item's tokens repeat one of them with multiplicity 0.
    bool ok = true;
    auto begin_tile = [&]() -> bool {  // the stage of tile n_tiles is free (warp-uniform)
      if (n_tiles < 2) return true;
      return tc::warp_wait(bar(B_EMPTY + (n_tiles & 1)), ((n_tiles - 2) >> 1) & 1, abort);
    };
    auto end_tile = [&](int cnt, int last) {  // lane 0: the list's header, then the arrival
      const int s = n_tiles & 1;
      s_meta[s][TPT] = cnt;
      s_meta[s][TPT + 1] = last;
      tc::mbar_expect_tx(bar(B_FULL + s), cnt > 0 ? (uint32_t)kStageBytes : 0u);
    };
    if (!p.cmp_kernel && !p.window) {
      // selected blocks: the tokens of the chunk that list j, from the inverted lists (a
      // token listing j twice appears twice).  A tile's TPT tokens are gathered by TPT
      // lanes at once, each issuing its token's four copies (r rows per tensor half) and
      // writing its slot; lane 0 then adds the header and arrives.
      const size_t seg = (size_t)bg * p.n_chunks + c;
      const int2 bk = p.inv_tab[seg * p.nb + j];
      const int32_t* lst = p.inv_list + seg * kChunk * p.S + bk.x;
      for (int k0 = 0; ok && k0 < bk.y; k0 += TPT) {
        if (!(ok = begin_tile())) break;
        const int s = n_tiles & 1, n_tok = min(TPT, bk.y - k0);
        if (lane < TPT) {
          const bool in = lane < n_tok;
          const int t = __ldg(lst + k0 + (in ? lane : n_tok - 1));
          const uint32_t qs = stage0 + s * kStageBytes + lane * R * 128, ds = qs + kQBytes;
          const int y = (int)((base + t) * p.h + g * R);
          const uint32_t fb = bar(B_FULL + s);
          tc::tma2d(qs, &tm_q, 0, y, fb);
          tc::tma2d(qs + kHalfRows, &tm_q, 64, y, fb);
          tc::tma2d(ds, &tm_do, 0, y, fb);
          tc::tma2d(ds + kHalfRows, &tm_do, 64, y, fb);
          s_meta[s][lane] = (t << 7) | (in ? 1 : 0);
        }
        __syncwarp();  // (orders the lanes' slot writes before lane 0's arrival)
        if (lane == 0) end_tile(TPT, k0 + TPT >= bk.y ? 1 : 0);
        __syncwarp();
        last_full[s] = n_tiles;
        ++n_tiles;
      }
    } else {
      // compressed keys and window: the queries reaching j are the consecutive tokens
      // t_begin .. t_end - 1, each once (a query t reaches the block exactly when t lies in
      // that range), so a tile is one 3-D box of TPT tokens x r heads per tensor half
      // (four copies, few instructions on the scheduler this warp shares with softmax
      // warps); slots past t_end read rows of no query of the item and get multiplicity 0
      for (int tt = t_begin; ok && tt < t_end; tt += TPT) {
        if (!(ok = begin_tile())) break;
        const int s = n_tiles & 1, n_tok = min(TPT, t_end - tt);
        if (lane == 0) {
          for (int q = 0; q < TPT; ++q) s_meta[s][q] = ((q < n_tok ? tt + q : tt) << 7) | (q < n_tok ? 1 : 0);
          const uint32_t qs = stage0 + s * kStageBytes, ds = qs + kQBytes, fb = bar(B_FULL + s);
          const int z = (int)(base + tt);
          tc::tma3d(qs, &tm_q3, 0, g * R, z, fb);
          tc::tma3d(qs + kHalfRows, &tm_q3, 64, g * R, z, fb);
          tc::tma3d(ds, &tm_do3, 0, g * R, z, fb);
          tc::tma3d(ds + kHalfRows, &tm_do3, 64, g * R, z, fb);
          end_tile(TPT, tt + TPT >= t_end ? 1 : 0);
        }
        __syncwarp();
        last_full[s] = n_tiles;
        ++n_tiles;
      }
    }
    if (ok && n_tiles == 0 && begin_tile()) {  // no token of the chunk reaches j: a marker tile
      if (lane == 0) end_tile(0, 1);
      ++n_tiles;
    }
    __syncwarp();
  }

  int pn = 0;  // dV / dK issuer and softmax warps: tiles whose P and dS went through the P buffer
  bool adone = false;  // dV / dK issuer: the item's last commit was issued
  if (warp == kIssuer) {
    // ------------------------------------------------------------------ S / dP issuer
    // S and dP of each loaded tile with rows, once its TMEM buffer is free (the softmax
    // warps read the tile two before); at the list's last tile it publishes the number of
    // tiles with rows.  The dV / dK products come from a second issuing warp on another
    // scheduler: an issuing lane that shares its scheduler with computing softmax warps
    // gets few issue slots.
    bool ok = tc::warp_wait(bar(B_KV), 0, abort);
    int n_rows_tiles = 0;
    for (int next_s = 0; ok; ++next_s) {
      const int s = next_s & 1;
      if (!(ok = tc::warp_wait(bar(B_FULL + s), (next_s >> 1) & 1, abort))) break;
      int cnt = 0, last = 0;  // every lane observed the stage's arrival
      cnt = s_meta[s][TPT];
      last = s_meta[s][TPT + 1];
      if (cnt > 0) {
        if (next_s >= 2 && !(ok = tc::warp_wait(bar(B_SFREE + s), ((next_s - 2) >> 1) & 1, abort))) break;
        if (lane == 0) {
          tc::fence_after();
          const uint32_t qs = stage0 + s * kStageBytes, ds = qs + kQBytes;
          constexpr uint32_t id = tc::idesc(128, kBS);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) {
            const uint32_t ao = (k >> 2) * kHalfRows + (k & 3) * 32, bo = (k >> 2) * (kKVBytes / 2) + (k & 3) * 32;
            tc::mma_ss(tmem + s * 128, tc::sdesc(qs + ao), tc::sdesc(kt + bo), id, k > 0);
            tc::mma_ss(tmem + s * 128 + 64, tc::sdesc(ds + ao), tc::sdesc(vt + bo), id, k > 0);
          }
          tc::commit(bar(B_SFULL + s));
        }
        __syncwarp();
        ++n_rows_tiles;
      }
      if (last) {
        if (lane == 0) {
          s_nrows = n_rows_tiles;
          tc::mbar_arrive(bar(B_SDONE));  // (release: s_nrows is visible to its observers)
        }
        __syncwarp();
        break;
      }
    }
  }
  if (warp == kDvIssuer || warp == kDkIssuer) {
    // ------------------------------------------------------------------ dV and dK issuers
    // A polling loop (lane 0 probes, the warp follows): dV (warp 10) or dK (warp 11) of the
    // oldest tile whose P and dS are written, until the S / dP issuer's count of tiles with
    // rows is reached; each commits the P buffer's and the stage's release (two arrivals).
    // Waits are bounded: without progress for the unit's limit the item gives up.
    const bool is_dk = warp == kDkIssuer;
    bool ok = true;
    int n_rows_tiles = -1;  // unknown until SDONE
    bool lo_init = false;   // the remainder accumulators hold a first product
    unsigned long long t_idle = tc::globaltimer();
    const unsigned long long lim = tc::wait_limit();
    while (ok) {
      int act = 0;  // 1: dV / dK of tile pn; 2: the row-tile count arrived
      if (lane == 0) {
        if ((n_rows_tiles < 0 || pn < n_rows_tiles) && tc::mbar_test(bar(B_PFULL), pn & 1))
          act = 1;
        else if (n_rows_tiles < 0 && tc::mbar_test(bar(B_SDONE), 0))
          act = 2;
      }
      act = __shfl_sync(0xffffffffu, act, 0);
      if (act == 1) {
        const int u = pn;  // P tiles are the row tiles, in order
        if (lane == 0) {  // lane 0 observed the P buffer's arrival: it reads the warps' flags
          int lo = 3;
          if (lo_init) {
            lo = 0;
#pragma unroll
            for (int w = 0; w < kSoftWarps; ++w) lo |= s_need[w];
          }
          tc::fence_after();
          // dV^T += dO^T P from the P buffer, or dK^T += Q^T dS from the dS buffer; the first
          // tile runs both parts (it initialises the remainder columns), later tiles only
          // the parts their values need
          const uint32_t qs = stage0 + (u & 1) * kStageBytes, a_s = is_dk ? qs : qs + kQBytes;
          const uint32_t b_s = is_dk ? s_hi : p_hi, d_col = is_dk ? kColDK : kColDV;
          const uint32_t id = idesc_mn(128, (lo & (is_dk ? 2 : 1)) ? 2 * kBS : kBS);
#pragma unroll 1
          for (int k = 0; k < kTileRows / 16; ++k) {
            const uint32_t ro = k * 2048;
            const uint32_t acc = (u > 0 || k > 0) ? 1u : 0u;
            tc::mma_ss(tmem + d_col, sdesc_mn(a_s + ro, kHalfRows, 1024), sdesc_mn(b_s + ro, kPBytes, 1024), id, acc);
          }
          tc::commit(bar(B_PFREE));
          tc::commit(bar(B_EMPTY + (u & 1)));
        }
        __syncwarp();
        lo_init = true;
        ++pn;
        t_idle = tc::globaltimer();
      } else if (act == 2) {
        int n = 0;
        if (lane == 0) n = s_nrows;  // lane 0 observed SDONE
        n_rows_tiles = __shfl_sync(0xffffffffu, n, 0);
        t_idle = tc::globaltimer();
      } else {
        if (n_rows_tiles >= 0 && pn == n_rows_tiles) {  // every product is issued
          if (lane == 0) tc::commit(bar(B_ADONE));
          __syncwarp();
          adone = true;
          break;
        }
        if (*abort) {
          ok = false;
        } else if (tc::globaltimer() - t_idle >= lim) {
          *abort = 1;
          atomicExch(&g_device_status, (int)NSA_ERR_TIMEOUT);
          ok = false;
        }
        ok = __all_sync(0xffffffffu, ok);
        __nanosleep(32);  // leave the issue slots to the softmax warps on this scheduler
      }
    }
  }
  if (warp < kSoftWarps) {
    // ------------------------------------------------------------------ softmax warps
    // K_j and V_j, bounds-checked (rows past the sequence's keys read as zeros; no query
    // reaches them), in the K-major layout of the S and dP products; the async-proxy fence
    // makes these generic-proxy writes visible to the MMAs
    {
      const int64_t rs = (int64_t)p.hkv * kD;
      const __nv_bfloat16* kb = p.k + ((kbase + (int64_t)j * kBS) * p.hkv + g) * kD;
      const __nv_bfloat16* vb = p.v + ((kbase + (int64_t)j * kBS) * p.hkv + g) * kD;
      for (int e = tid; e < 2 * kBS * (kD / 8); e += kSoft) {
        const int which = e / (kBS * (kD / 8)), r = (e / (kD / 8)) % kBS, ch = e % (kD / 8);
        const bool in = j * kBS + r < Lk;
        const __nv_bfloat16* src = (which ? vb : kb) + r * rs + ch * 8;
        const uint32_t dst = (which ? vt : kt) + (ch >> 3) * (kKVBytes / 2) + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        cp_async16(dst, in ? (const void*)src : (const void*)p.k, in ? 16 : 0);
      }
      cp_async_commit();
      cp_async_wait<0>();
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      tc::mbar_arrive(bar(B_KV));
    }
    // TMEM lanes 32 (warp % 4) .. are this warp's rows; kh: its half of the 64 keys
    const int row = (warp & 3) * 32 + lane, kh = warp >> 2, slot = row / R, hd = row % R;
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int s = i & 1;
      if (!(ok = tc::warp_wait(bar(B_FULL + s), (i >> 1) & 1, abort))) break;
      const int cnt = s_meta[s][TPT], last = s_meta[s][TPT + 1];
      if (cnt == 0) break;  // the marker that ends the list
      const int info = s_meta[s][slot];
      const int t = info >> 7, mult = info & 127;
      float lse2 = __builtin_inff(), dsum = 0.f;
      if (mult > 0) {
        const int64_t rg = (base + t) * p.h + (int64_t)g * R + hd;
        lse2 = lse_to_log2(p.lse[rg]);
        dsum = p.dsum[rg];
      }
      const int tb = key_bound(p, t, Lk), tl = key_lo(p, t);
      if (!(ok = tc::warp_wait(bar(B_SFULL + s), (i >> 1) & 1, abort))) break;
      tc::fence_after();
      float sv[32], dpv[32];
      tc::tmem_ld32_nowait(t_lane + s * 128 + kh * 32, sv);
      tc::tmem_ld32_nowait(t_lane + s * 128 + 64 + kh * 32, dpv);
      tc::tmem_wait_ld();
      tc::fence_before();
      tc::mbar_arrive(bar(B_SFREE + s));
      // the P buffer is free once the previous tile's dV / dK products are done
      if (pn > 0 && !(ok = tc::warp_wait(bar(B_PFREE), (pn - 1) & 1, abort))) break;
      float pmax = 0.f, smax = 0.f;
      // every key of the warp's 32 inside every row's range (the usual case: blocks before
      // the row's own): no per-key mask
      const int kw = j * kBS + kh * 32;
      const PdsArgs pa{(float)mult, p.scale_log2, lse2, dsum, tl, tb, j * kBS, row, kh, p_hi, p_lo, s_hi, s_lo};
      if (__all_sync(0xffffffffu, kw >= tl && kw + 31 <= tb))
        form_pds<false>(sv, dpv, pa, pmax, smax);
      else
        form_pds<true>(sv, dpv, pa, pmax, smax);
      {  // which remainder products this warp's rows need (read by the issuers after PFULL)
        const unsigned bp = __ballot_sync(0xffffffffu, pmax > kLoP), bs = __ballot_sync(0xffffffffu, smax > kLoS);
        if (lane == 0) s_need[warp] = (bp ? 1 : 0) | (bs ? 2 : 0);
        store_remainders(sv, p_lo, row, kh, bp != 0);
        store_remainders(dpv, s_lo, row, kh, bs != 0);
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      tc::mbar_arrive(bar(B_PFULL));
      ++pn;
      if (last) break;
    }
    // ------------------------------------------------------------------ epilogue
    // TMEM lane = d: row d of dK^T and dV^T holds the 64 keys' values of column d; this
    // thread writes keys 32 kh .. 32 kh + 31
    float* out = p.part + ((size_t)bg * p.items_per_bg + slot_item) * 2 * kBS * kD;
    if (ok && pn > 0) ok = tc::warp_wait(bar(B_ADONE), 0, abort);
    if (ok) {
      tc::fence_after();
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        {
          const int cc = kh * 32;
          float v[32];
          if (pn > 0) {
            float w[32];
            tc::tmem_ld32_nowait(t_lane + (which ? kColDV : kColDK) + cc, v);
            tc::tmem_ld32_nowait(t_lane + (which ? kColDVlo : kColDKlo) + cc, w);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] += w[e];
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.f;
          }
          float* o = out + (size_t)which * kBS * kD + (size_t)cc * kD + row;
#pragma unroll
          for (int e = 0; e < 32; ++e) o[(size_t)e * kD] = v[e];
        }
      }
    }
  }

  __syncthreads();
  if (*abort) {
    // copies and tensor-core work still in flight land before the CTA leaves
    if (warp == kProducer) {
      for (int s = 0; s < 2; ++s) {
        const int i = n_tiles - 1 - ((n_tiles - 1 - s) & 1);  // last tile handed to stage s
        if (i >= 0 && (i & 1) == s) tc::warp_drain(bar(B_FULL + s), (i >> 1) & 1);
      }
    } else if (warp == kIssuer || warp == kDvIssuer || warp == kDkIssuer) {
      if (lane == 0) tc::commit(bar(B_DRAIN));
      __syncwarp();
      tc::warp_drain(bar(B_DRAIN), 0);
    }
  } else if (warp == kProducer) {
    // the dV / dK issuer's last release of each stage lands before the CTA leaves
    for (int s = 0; s < 2; ++s)
      if (last_full[s] >= 0) tc::warp_drain(bar(B_EMPTY + s), (last_full[s] >> 1) & 1);
  } else if (warp == kDvIssuer || warp == kDkIssuer) {
    if (pn > 0) tc::warp_drain(bar(B_PFREE), (pn - 1) & 1);
    if (adone) tc::warp_drain(bar(B_ADONE), 0);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kIssuer)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ---------------------------------------------------------------------------- dQ, dense key spaces
// dQ of the compressed and sliding-window branches (group sizes 8 and 16).  There a query
// reaches a contiguous key range, and the 128 / r tokens of a 128-row tile reach nearly
// the same one, so the tile walks 128-key tiles of that range (masked per row at its
// edges, as the tensor-core forward does):
//   S = Q K^T, dP = dO V^T        M = 128 rows, N = 128 keys, K = d
//   dS = P (dP - D), P = exp(scale S - lse) from the forward's lse (no running max)
//   dQ += dS K                    M = 128 rows, N = 128 (d), K = 128 keys; dS is the TMEM A
//                                 operand (bf16 value and remainder), the K tile the
//                                 MN-major B operand (the same tile as S's K-major B)
// 128-key tiles, since a tcgen05 product occupies the tensor pipe for about as long at
// N = 64 as at N = 128 (measured: 74 against 70 cycles per M = 128, K = 16 product).
// TMEM holds two S buffers (dS is written over its tile's S, once every thread has its
// S values in registers), one dP buffer and the dQ accumulator: 4 x 128 columns.
// The kernel also stores D = dO . o per row, which the dK / dV kernel reads.  Roles as
// in dkv_tc_kernel: warp 8 loads Q and dO once and streams K tiles through a three-stage
// and V tiles through a two-stage ring (V is free once dP is done), warps 9 and 11 issue
// S and dP (of the next tile while the softmax warps work on this one), warp 10 the dQ
// products, warps 0-7 (rows 32 (w % 4) .., keys 64 (w / 4) .. of every tile) form dS and
// finally store dQ.
namespace dqk {
constexpr int KT = 128;                // keys per tile
constexpr int NK = 3, NV = 2;          // K and V ring stages
constexpr int TILE = KT * kD * 2;      // a K or V tile: two 64-column halves of 16 KB
constexpr int QB = kTileRows * kD * 2;  // Q or dO of the 128 rows: two halves of 16 KB
constexpr int SMEM = 2 * QB + (NK + NV) * TILE + 1024;
constexpr uint32_t COL_DP = 256, COL_DQ = 384;  // S / dS buffers at 0 and 128
enum : int {
  QB_Q = 0,                    // Q and dO landed
  QB_KFULL = 1,                // [NK]
  QB_KEMPTY = QB_KFULL + NK,   // [NK] dQ of the tile done
  QB_VFULL = QB_KEMPTY + NK,   // [NV]
  QB_VEMPTY = QB_VFULL + NV,   // [NV] dP of the tile done
  QB_SFULL = QB_VEMPTY + NV,   // [2] S and dP of a tile computed (S buffer = tile % 2)
  QB_DPFREE = QB_SFULL + 2,    // the softmax warps hold dP of the current tile
  QB_DSFULL = QB_DPFREE + 1,   // [2] dS written over its tile's S
  QB_DQDONE = QB_DSFULL + 2,   // [2] dQ += dS K of the buffer's tile done
  QB_ADONE = QB_DQDONE + 2,    // every product of the CTA done
  QB_DRAIN,
  QB_COUNT
};
}  // namespace dqk

// dS of 64 keys of a row from S and dP (P from the forward's base-2 normaliser lse2):
// dv holds dP on entry and dS on return, hi the bf16-rounded pairs; MASK: keys outside
// [tl, tb] give 0.  Returns max |dS|.
template <bool MASK>
__device__ __forceinline__ float form_ds(const float (&sv)[64], float (&dv)[64], int k0, int tl, int tb,
                                         float scale_log2, float lse2, float dsum, uint32_t (&hi)[32]) {
  float smax = 0.f;
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    float p0 = ex2(fmaf(sv[e], scale_log2, -lse2)), p1 = ex2(fmaf(sv[e + 1], scale_log2, -lse2));
    if (MASK) {
      const int k = k0 + e;
      p0 = k >= tl && k <= tb ? p0 : 0.f;
      p1 = k + 1 >= tl && k + 1 <= tb ? p1 : 0.f;
    }
    const float d0 = p0 * (dv[e] - dsum), d1 = p1 * (dv[e + 1] - dsum);
    dv[e] = d0;
    dv[e + 1] = d1;
    smax = fmaxf(smax, fmaxf(fabsf(d0), fabsf(d1)));
    hi[e / 2] = pack_bf16(d0, d1);
  }
  return smax;
}

// The bf16 remainders x - bf16(x) of value pairs whose rounded parts are hi, or zeros:
// a warp whose values all lie below the split threshold drops its remainders (the
// remainder products then add nothing for its rows, as when no warp needs them).
template <int N>
__device__ __forceinline__ void remainders(const float (&x)[2 * N], const uint32_t (&hi)[N], bool need,
                                           uint32_t (&lo)[N]) {
#pragma unroll
  for (int w = 0; w < N; ++w) {
    if (need) {
      const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi[w]));
      lo[w] = pack_bf16(x[2 * w] - h.x, x[2 * w + 1] - h.y);
    } else {
      lo[w] = 0u;
    }
  }
}

// dq_tc: issuing warps of the dQ and the dP products beside the S issuer (kIssuer)
constexpr int kQIssuer = kSoftWarps + 2, kPIssuer = kSoftWarps + 3, kQThreads = kThreads + 64;

template <int R>
__global__ void __launch_bounds__(kQThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const BwdParams p) {
  using namespace dqk;
  constexpr int TPC = kTileRows / R;  // tokens per CTA
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t s_bar[QB_COUNT];
  __shared__ int s_need[2][kSoftWarps];  // per S buffer and softmax warp: remainder products needed
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tc::device_status_set()) return;  // after a timeout elsewhere, later CTAs leave at once
  const int sq = blockIdx.y, g = blockIdx.z;
  const int L = seq_len(p.seqs, sq);
  const int tile = (L + TPC - 1) / TPC - 1 - (int)blockIdx.x;  // longest key ranges first
  if (tile < 0) return;
  const int t0 = tile * TPC, t_last = min(t0 + TPC, L) - 1;
  const int64_t start = seq_start(p.seqs, sq);
  const int Lk = key_len(p, L);
  const int64_t kv0 = key_base(p, sq);  // key row of the sequence's first key
  const int k_lo = key_lo(p, t0), k_hi = key_bound(p, t_last, Lk) + 1;
  const int64_t a_lo = (kv0 + k_lo) / KT;  // key tiles at absolute 128-row offsets
  const int n_kt = k_hi > k_lo ? (int)((kv0 + k_hi + KT - 1) / KT - a_lo) : 0;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023) & ~1023u;
  const uint32_t q_s = sbase, do_s = q_s + QB, k_ring = do_s + QB, v_ring = k_ring + NK * TILE;
  auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
  volatile int* abort = &s_abort;
  if (tid == 0) {
    tc::mbar_init(bar(QB_Q), 1);
    for (int i = 0; i < NK; ++i) {
      tc::mbar_init(bar(QB_KFULL + i), 1);
      tc::mbar_init(bar(QB_KEMPTY + i), 1);
    }
    for (int i = 0; i < NV; ++i) {
      tc::mbar_init(bar(QB_VFULL + i), 1);
      tc::mbar_init(bar(QB_VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar(QB_SFULL + i), 2);  // the S and the dP issuer
      tc::mbar_init(bar(QB_DSFULL + i), kSoft);
      tc::mbar_init(bar(QB_DQDONE + i), 1);
    }
    tc::mbar_init(bar(QB_DPFREE), kSoft);
    tc::mbar_init(bar(QB_ADONE), 1);
    tc::mbar_init(bar(QB_DRAIN), 3);  // the three issuing warps
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == kIssuer) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    tc::fence_before();
  }
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = s_tmem;

  int last_k = -1, last_v = -1;  // producer: last K / V tile handed to its ring
  if (warp == kProducer) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && n_kt > 0) {
      tc::mbar_expect_tx(bar(QB_Q), 2 * QB);
      tc::tma3d(q_s, &tm_q, 0, g * R, (int)(start + t0), bar(QB_Q));
      tc::tma3d(q_s + QB / 2, &tm_q, 64, g * R, (int)(start + t0), bar(QB_Q));
      tc::tma3d(do_s, &tm_do, 0, g * R, (int)(start + t0), bar(QB_Q));
      tc::tma3d(do_s + QB / 2, &tm_do, 64, g * R, (int)(start + t0), bar(QB_Q));
    }
    // key rows the buffers hold: the tokens (window), or the packed compressed rows of all
    // sequences, counted here; a tile that reaches past them is copied with bounds checks
    int64_t kv_total = p.seqs.tokens;
    if (p.cmp_kernel) {
      int64_t acc = 0;
      for (int i = lane; i < p.seqs.n_seqs; i += 32) acc += num_cmp(seq_len(p.seqs, i), p.cmp_kernel, p.cmp_stride);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      kv_total = acc;
    }
    // one K or V tile into the stage at dst (warp-uniform)
    auto load = [&](const CUtensorMap* map, const __nv_bfloat16* src, uint32_t dst, uint32_t fb, int64_t row) {
      if (p.cmp_kernel && row + KT > kv_total) {
        for (int c = lane; c < KT * (kD / 8); c += 32) {
          const int r = c / (kD / 8), ch = c % (kD / 8);
          const bool in = row + r < kv_total;
          const int64_t off = ((row + r) * p.hkv + g) * kD + ch * 8;
          cp_async16(dst + (ch >> 3) * (TILE / 2) + r * 128 + (((ch & 7) ^ (r & 7)) << 4),
                     in ? (const void*)(src + off) : (const void*)p.k, in ? 16 : 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(fb);
      } else if (lane == 0) {
        tc::mbar_expect_tx(fb, TILE);
        tc::tma2d(dst, map, g * kD, (int)row, fb);
        tc::tma2d(dst + TILE / 2, map, g * kD + 64, (int)row, fb);
      }
      __syncwarp();
    };
    for (int i = 0; i < n_kt; ++i) {
      const int64_t row = (a_lo + i) * KT;
      const int sk = i % NK, sv = i % NV;
      if (i >= NK && !tc::warp_wait(bar(QB_KEMPTY + sk), ((i / NK) - 1) & 1, abort)) break;
      load(&tm_k, p.k, k_ring + sk * TILE, bar(QB_KFULL + sk), row);
      last_k = i;
      if (i >= NV && !tc::warp_wait(bar(QB_VEMPTY + sv), ((i / NV) - 1) & 1, abort)) break;
      load(&tm_v, p.v, v_ring + sv * TILE, bar(QB_VFULL + sv), row);
      last_v = i;
    }
  }

  if ((warp == kIssuer || warp == kPIssuer) && n_kt > 0) {
    // ------------------------------------------------------------------ S and dP issuers
    // Warp 9 issues S of tile u + 1 into buffer (u + 1) % 2 once dQ of tile u - 1, which
    // read the dS over that buffer, is done; warp 11 issues dP(u + 1) once the softmax
    // warps hold dP(u).  Each commits the tile's SFULL (two arrivals).
    constexpr uint32_t id_s = tc::idesc(128, KT);
    auto issue_s = [&](int j) -> bool {  // warp-uniform
      const int sk = j % NK;
      if (!tc::warp_wait(bar(QB_KFULL + sk), (j / NK) & 1, abort)) return false;
      if (lane == 0) {
        tc::fence_after();
        const uint32_t ks = k_ring + sk * TILE;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t ao = (k >> 2) * (QB / 2) + (k & 3) * 32, bo = (k >> 2) * (TILE / 2) + (k & 3) * 32;
          tc::mma_ss(tmem + (j & 1) * 128, tc::sdesc(q_s + ao), tc::sdesc(ks + bo), id_s, k > 0);
        }
        tc::commit(bar(QB_SFULL + (j & 1)));
      }
      __syncwarp();
      return true;
    };
    auto issue_dp = [&](int j) -> bool {
      const int sv = j % NV;
      if (j >= 1 && !tc::warp_wait(bar(QB_DPFREE), (j - 1) & 1, abort)) return false;
      if (!tc::warp_wait(bar(QB_VFULL + sv), (j / NV) & 1, abort)) return false;
      if (lane == 0) {
        tc::fence_after();
        const uint32_t vs = v_ring + sv * TILE;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t ao = (k >> 2) * (QB / 2) + (k & 3) * 32, bo = (k >> 2) * (TILE / 2) + (k & 3) * 32;
          tc::mma_ss(tmem + COL_DP, tc::sdesc(do_s + ao), tc::sdesc(vs + bo), id_s, k > 0);
        }
        tc::commit(bar(QB_SFULL + (j & 1)));
        tc::commit(bar(QB_VEMPTY + sv));
      }
      __syncwarp();
      return true;
    };
    bool ok = tc::warp_wait(bar(QB_Q), 0, abort);
    if (warp == kIssuer) {  // S
      if (ok) ok = issue_s(0);
      for (int u = 0; ok && u + 1 < n_kt; ++u) {
        if (u >= 1 && !(ok = tc::warp_wait(bar(QB_DQDONE + ((u - 1) & 1)), ((u - 1) >> 1) & 1, abort))) break;
        ok = issue_s(u + 1);
      }
    } else {  // dP
      for (int u = 0; ok && u < n_kt; ++u) ok = issue_dp(u);
    }
  }
  if (warp == kQIssuer && n_kt > 0) {
    // ------------------------------------------------------------------ dQ issuer
    // dQ += dS K of tile u once its dS is written.  A second issuing warp, on another
    // scheduler: an issuing lane that shares its scheduler with two computing softmax
    // warps gets few issue slots (measured with eight FMA-bound warps beside it: 158 - 178
    // cycles per product against 68 - 71 alone), so S / dP and dQ issue in parallel.
    bool ok = true;
    for (int u = 0; ok && u < n_kt; ++u) {
      const int b = u & 1, sk = u % NK;
      if (!(ok = tc::warp_wait(bar(QB_DSFULL + b), (u >> 1) & 1, abort))) break;
      if (lane == 0) {  // lane 0 observed the dS arrival: it reads the warps' flags
        int lo = 0;
#pragma unroll
        for (int w = 0; w < kSoftWarps; ++w) lo |= s_need[b][w];
        tc::fence_after();
        const uint32_t ks = k_ring + sk * TILE;
        constexpr uint32_t id = tc::idesc(128, kD) | (1u << 16);  // B (the K tile) MN-major
#pragma unroll
        for (int s = 0; s < KT / 16; ++s) {
          // dS of keys 16 s .. 16 s + 15: the bf16 values of key half s / 4 over its 64 S
          // columns, the rounded parts first and the remainders 32 columns on
          const uint32_t a = tmem + b * 128 + (s >> 2) * 64 + (s & 3) * 8;
          const uint64_t bk = sdesc_mn(ks + s * 2048, TILE / 2, 1024);
          tc::mma_ts(tmem + COL_DQ, a, bk, id, (u > 0 || s > 0) ? 1u : 0u);
          if (lo) tc::mma_ts(tmem + COL_DQ, a + 32, bk, id, 1u);
        }
        tc::commit(bar(QB_DQDONE + b));
        tc::commit(bar(QB_KEMPTY + sk));
        if (u == n_kt - 1) tc::commit(bar(QB_ADONE));
      }
      __syncwarp();
    }
  }
  if (warp < kSoftWarps) {
    // ------------------------------------------------------------------ softmax warps
    // TMEM lanes 32 (warp % 4) .. are this warp's rows; kh: its half of every tile's keys
    __shared__ float s_dd[2][kTileRows];  // D = dO . o, the two halves of d
    const int row = (warp & 3) * 32 + lane, kh = warp >> 2, slot = row / R, hd = row % R;
    const int t = t0 + slot;
    const bool valid = t <= t_last;
    const int64_t rg = (start + t) * p.h + (int64_t)g * R + hd;
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    {
      float acc = 0.f;
      if (valid) {
        const uint4* a = reinterpret_cast<const uint4*>(p.dout + rg * kD + kh * 64);
        const uint4* b = reinterpret_cast<const uint4*>(p.o + rg * kD + kh * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = __ldg(a + c), y = __ldg(b + c);
          acc += dot_bf16x2(x.x, y.x) + dot_bf16x2(x.y, y.y) + dot_bf16x2(x.z, y.z) + dot_bf16x2(x.w, y.w);
        }
      }
      s_dd[kh][row] = acc;
    }
    asm volatile("bar.sync 1, %0;\n" ::"n"(kSoft) : "memory");
    const float dsum = s_dd[0][row] + s_dd[1][row];
    if (valid && kh == 0) p.dsum[rg] = dsum;
    const float lse2 = valid ? lse_to_log2(p.lse[rg]) : __builtin_inff();
    const int tl = key_lo(p, t), tb = valid ? key_bound(p, t, Lk) : -1;
    bool ok = true;
    for (int u = 0; u < n_kt; ++u) {
      const int b = u & 1;
      if (!(ok = tc::warp_wait(bar(QB_SFULL + b), (u >> 1) & 1, abort))) break;
      tc::fence_after();
      float sv[64], dpv[64];
      const uint32_t sc = t_lane + b * 128 + kh * 64;  // this thread's S (then dS) columns
      tc::tmem_ld32_nowait(sc, sv);
      tc::tmem_ld32_nowait(sc + 32, sv + 32);
      tc::tmem_ld32_nowait(t_lane + COL_DP + kh * 64, dpv);
      tc::tmem_ld32_nowait(t_lane + COL_DP + kh * 64 + 32, dpv + 32);
      tc::tmem_wait_ld();
      tc::fence_before();
      tc::mbar_arrive(bar(QB_DPFREE));
      const int k0 = (int)((a_lo + u) * KT - kv0) + kh * 64;  // key of sv[0] within the sequence
      uint32_t hi[32], lo[32];
      // every key of the warp's 64 inside every row's range: no per-key mask (fewer
      // instructions on the schedulers the MMA warp shares)
      const float smax = __all_sync(0xffffffffu, k0 >= tl && k0 + 63 <= tb)
                             ? form_ds<false>(sv, dpv, k0, tl, tb, p.scale_log2, lse2, dsum, hi)
                             : form_ds<true>(sv, dpv, k0, tl, tb, p.scale_log2, lse2, dsum, hi);
      {
        const unsigned bs = __ballot_sync(0xffffffffu, smax > kLoS);
        if (lane == 0) s_need[b][warp] = bs ? 1 : 0;
        remainders<32>(dpv, hi, bs != 0, lo);
      }
      // dS over this thread's own S columns (already read): the MMA warp reuses the
      // buffer only after the dQ product of this tile
      tc::tmem_st32(sc, hi);  // (waits for its stores)
      tc::tmem_st32(sc + 32, lo);
      tc::fence_before();
      tc::mbar_arrive(bar(QB_DSFULL + b));
    }
    // ------------------------------------------------------------------ epilogue
    // every product is done; then the last arrivals on both dQ barriers land (their
    // earlier phases were observed by the MMA warp)
    if (ok && n_kt > 0) ok = tc::warp_wait(bar(QB_ADONE), 0, abort);
    if (ok && n_kt > 0) ok = tc::warp_wait(bar(QB_DQDONE + ((n_kt - 1) & 1)), ((n_kt - 1) >> 1) & 1, abort);
    if (ok && n_kt > 1) ok = tc::warp_wait(bar(QB_DQDONE + ((n_kt - 2) & 1)), ((n_kt - 2) >> 1) & 1, abort);
    if (ok) {
      float v[64];
      if (n_kt > 0) {
        tc::fence_after();
        tc::tmem_ld32_nowait(t_lane + COL_DQ + kh * 64, v);
        tc::tmem_ld32_nowait(t_lane + COL_DQ + kh * 64 + 32, v + 32);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) v[e] = 0.f;
      }
      if (valid) {
        uint4* o = reinterpret_cast<uint4*>(p.dq + rg * kD + kh * 64);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float* x = v + 8 * c;
          o[c] = make_uint4(pack_bf16(x[0] * p.scale, x[1] * p.scale), pack_bf16(x[2] * p.scale, x[3] * p.scale),
                            pack_bf16(x[4] * p.scale, x[5] * p.scale), pack_bf16(x[6] * p.scale, x[7] * p.scale));
        }
      }
    }
  }

  __syncthreads();
  if (*abort) {
    // copies and tensor-core work still in flight land before the CTA leaves
    if (warp == kProducer) {
      if (n_kt > 0) tc::warp_drain(bar(QB_Q), 0);
      for (int st = 0; st < NK; ++st) {
        const int i = last_k - ((last_k - st) % NK + NK) % NK;  // last K tile handed to stage st
        if (i >= 0) tc::warp_drain(bar(QB_KFULL + st), (i / NK) & 1);
      }
      for (int st = 0; st < NV; ++st) {
        const int i = last_v - ((last_v - st) % NV + NV) % NV;
        if (i >= 0) tc::warp_drain(bar(QB_VFULL + st), (i / NV) & 1);
      }
    } else if (warp == kIssuer || warp == kQIssuer || warp == kPIssuer) {
      if (lane == 0) tc::commit(bar(QB_DRAIN));
      __syncwarp();
      tc::warp_drain(bar(QB_DRAIN), 0);
    }
  } else if (warp == kProducer) {
    // the MMA warps' last release of each stage lands before the CTA leaves
    for (int st = 0; st < NK; ++st) {
      const int i = last_k - ((last_k - st) % NK + NK) % NK;
      if (i >= 0) tc::warp_drain(bar(QB_KEMPTY + st), (i / NK) & 1);
    }
    for (int st = 0; st < NV; ++st) {
      const int i = last_v - ((last_v - st) % NV + NV) % NV;
      if (i >= 0) tc::warp_drain(bar(QB_VEMPTY + st), (i / NV) & 1);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kIssuer)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

}  // namespace

cudaError_t launch_invert(const BwdParams& p, cudaStream_t st) {
  const int n_bg = p.seqs.n_seqs * p.hkv;
  if (n_bg == 0 || p.n_chunks == 0) return cudaSuccess;
  const int smem = 8 * std::min(p.nb, p.n_chunks * kGroup) * 4;
  cudaError_t e = cudaFuncSetAttribute(invert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  invert_kernel<<<dim3(p.n_chunks, n_bg), 256, smem, st>>>(p);
  return cudaGetLastError();
}

// The inverted lists take up to 1024 key blocks per chunk (4 per thread of invert_kernel).
bool dkv_tc_supported(const BwdParams& p) { return dkv_tc_shape(p.h / p.hkv, p.cmp_kernel || p.window, p.nb); }

// q_rows: rows of q and dout ([tokens, h, d]), the extent of their tensor maps.
cudaError_t launch_dkv_tc(const BwdParams& p, int64_t items, int64_t q_rows, cudaStream_t st) {
  if (items <= 0) return cudaSuccess;
  const int r = p.h / p.hkv;
  CUtensorMap mq, mdo, mq3, mdo3;
  const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)q_rows};
  const uint64_t strides[1] = {(uint64_t)kD * 2};
  const uint32_t box[2] = {64, (uint32_t)r};
  if (!tc::make_map(&mq, p.q, 2, dims, strides, box) || !tc::make_map(&mdo, p.dout, 2, dims, strides, box))
    return cudaErrorInvalidValue;
  // the same tensors as (d, h, tokens) with boxes of 128 / r consecutive tokens x r heads
  const uint64_t dims3[3] = {(uint64_t)kD, (uint64_t)p.h, (uint64_t)(q_rows / p.h)};
  const uint64_t strides3[2] = {(uint64_t)kD * 2, (uint64_t)p.h * kD * 2};
  const uint32_t box3[3] = {64, (uint32_t)r, (uint32_t)(kTileRows / r)};
  if (!tc::make_map(&mq3, p.q, 3, dims3, strides3, box3) || !tc::make_map(&mdo3, p.dout, 3, dims3, strides3, box3))
    return cudaErrorInvalidValue;
  auto kern = r == 16 ? dkv_tc_kernel<16> : dkv_tc_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)items, kKVThreads, kSmemBytes, st>>>(mq, mdo, mq3, mdo3, p);
  return cudaGetLastError();
}

bool dq_tc_supported(const BwdParams& p) {
  const int r = p.h / p.hkv;
  return (r == 8 || r == 16) && (p.cmp_kernel > 0 || p.window > 0);
}

// kv_rows: rows of k and v ([kv_rows, hkv, d]; for the compressed keys a bound on the
// packed rows, past which the kernel reads nothing).
cudaError_t launch_dq_tc(const BwdParams& p, int64_t kv_rows, cudaStream_t st) {
  const Seqs& s = p.seqs;
  if (s.tokens == 0) return cudaSuccess;
  const int r = p.h / p.hkv, tpc = kTileRows / r;
  CUtensorMap mq, mdo, mk, mv;
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)p.h, (uint64_t)s.tokens};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)p.h * kD * 2};
    const uint32_t box[3] = {64, (uint32_t)r, (uint32_t)tpc};
    if (!tc::make_map(&mq, p.q, 3, dims, strides, box) || !tc::make_map(&mdo, p.dout, 3, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)p.hkv * kD, (uint64_t)std::max<int64_t>(kv_rows, 1)};
    const uint64_t strides[1] = {(uint64_t)p.hkv * kD * 2};
    const uint32_t box[2] = {64, (uint32_t)dqk::KT};
    if (!tc::make_map(&mk, p.k, 2, dims, strides, box) || !tc::make_map(&mv, p.v, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  auto kern = r == 16 ? dq_tc_kernel<16> : dq_tc_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dqk::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((s.max_len + tpc - 1) / tpc), (unsigned)s.n_seqs, (unsigned)p.hkv);
  kern<<<grid, kQThreads, dqk::SMEM, st>>>(mq, mdo, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace bwd

NSA_STATUS_ACCESSOR(sparse_bwd_tc)

}  // namespace nsa
