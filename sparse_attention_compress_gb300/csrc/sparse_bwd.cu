// Backward of selected-block attention (prefill): dQ, dK, dV for an upstream dO.
//
// The forward is [TileLang-NSA] "TileLang operator development: Native Sparse
// Attention", sec. 2 (a listed block starting at index*block_size is attended when it
// starts at or before the query; keys past the query are masked); the pages train with
// it ([NSA-Triton] "DeepSeek NSA ... with Triton", sec. 4) but print no backward, so
// this is the derivative of that forward.  Per (token, head) row with list keys e:
//   p_e = exp(scale q.k_e - lse),  dp_e = dO.v_e,  D = dO.o,  ds_e = p_e (dp_e - D),
//   dq = scale sum_e ds_e k_e,  dk[e] += scale ds_e q,  dv[e] += p_e dO.
//
// GB300 design, three launches:
//   1. sparse_bwd_dq: one CTA per (token, kv-head), the forward's structure (four warps
//      own the four 16-key slices of every listed block and stream them through private
//      cp.async rings), recomputing p from the forward's lse (no online softmax), with a
//      second product dO.V^T and dq accumulated in registers; it also stores D = dO.o.
//   2. sparse_bwd_dkv: the transpose problem.  A work item is (sequence, kv-head, key
//      block j, chunk of 2048 query positions); its CTA finds, in token order, the
//      tokens of the chunk whose list holds j (with multiplicity), keeps K_j and V_j in
//      shared memory and streams those tokens' Q and dO rows (all r heads of the group:
//      the N = 16 of one mma tile) through a CTA-wide cp.async ring.  Warp w owns keys
//      16w..16w+15 of the block: it holds their K and V rows as mma A fragments for
//      the whole item, forms S^T = K_w Q_t^T and dP^T = V_w dO_t^T with the keys as the
//      M dimension (so P^T and dS^T come out as the A operands of dV and dK with no
//      transpose) and accumulates its dK and dV rows in registers.  Each item writes
//      fp32 partials.
//   3. sparse_bwd_reduce: per (sequence, kv-head, block) the partials are summed in
//      chunk order (deterministic: no floating-point atomics anywhere) and stored.
// For group sizes 8 and 16 (run_bwd below) the tensor-core kernels of sparse_bwd_tc.cu
// take over: dK / dV always (dkv_tc_kernel, with invert_kernel first building the
// selected blocks' token lists), and dQ with D in the compressed and window key spaces
// (dq_tc_kernel); sparse_bwd_dq keeps the selected blocks' dQ, and the mma.sync dK / dV
// the other group sizes.
#include <algorithm>

#include "sparse_bwd.cuh"

namespace nsa {

namespace {

using namespace bwd;

// ---------------------------------------------------------------------------- dQ
template <int NSTAGE>
__global__ void __launch_bounds__(128, 2) sparse_bwd_dq(const BwdParams p) {
  constexpr int D = kD, BS = kBS;
  constexpr int SLICE_BYTES = 16 * D * 2;
  constexpr int STAGE_BYTES = 2 * SLICE_BYTES;
  constexpr int CH = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_list[4][64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slice = warp;
  const int g = blockIdx.y;
  const int r = p.r;
  const int64_t qrow = blockIdx.x;
  const int sq = seq_of_token(p.seqs, qrow);
  const int t = (int)(qrow - seq_start(p.seqs, sq));
  const int64_t kv_base = key_base(p, sq);
  const int tb = key_bound(p, t, key_len(p, seq_len(p.seqs, sq)));  // last reachable key
  const int tl = key_lo(p, t);                                       // first reachable key
  const int hbase = g * r;
  const int rlo = lane >> 2, rhi = rlo + 8;
  const bool w0 = rlo < r, w1 = rhi < r;
  const int64_t row0 = qrow * p.h + hbase;

  uint32_t qa[D / 16][4], da[D / 16][4];
  load_a_frags<D>(qa, w0 ? p.q + (row0 + rlo) * D : nullptr, w1 ? p.q + (row0 + rhi) * D : nullptr, lane);
  load_a_frags<D>(da, w0 ? p.dout + (row0 + rlo) * D : nullptr, w1 ? p.dout + (row0 + rhi) * D : nullptr, lane);
  float d0 = 0.f, d1 = 0.f;
  {
    uint32_t oa[D / 16][4];
    load_a_frags<D>(oa, w0 ? p.o + (row0 + rlo) * D : nullptr, w1 ? p.o + (row0 + rhi) * D : nullptr, lane);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      d0 += dot_bf16x2(da[kk][0], oa[kk][0]) + dot_bf16x2(da[kk][2], oa[kk][2]);
      d1 += dot_bf16x2(da[kk][1], oa[kk][1]) + dot_bf16x2(da[kk][3], oa[kk][3]);
    }
    d0 = quad_sum(d0);
    d1 = quad_sum(d1);
  }
  const float L0 = w0 ? lse_to_log2(p.lse[row0 + rlo]) : __builtin_inff();
  const float L1 = w1 ? lse_to_log2(p.lse[row0 + rhi]) : __builtin_inff();
  if (warp == 0 && (lane & 3) == 0) {
    if (w0) p.dsum[row0 + rlo] = d0;
    if (w1) p.dsum[row0 + rhi] = d1;
  }

  // this warp's list: listed blocks whose slice starts at or before the bound (every
  // such block for the compressed branch)
  int cnt = 0;
  if (p.window) {  // blocks whose slice overlaps [tl, tb]
    const int j0 = tl / BS, j1 = tb / BS;
    for (int jj = j0 + lane; jj <= j1; jj += 32) {
      const int k0 = jj * BS + slice * 16;
      const bool ok = k0 <= tb && k0 + 15 >= tl;
      const unsigned m = __ballot_sync(__activemask(), ok);
      if (ok) s_list[warp][cnt + __popc(m & ((1u << lane) - 1u))] = jj;
      cnt += __popc(m);
    }
    cnt = __shfl_sync(0xffffffffu, cnt, 0);
  } else if (p.cmp_kernel) {
    cnt = tb >= slice * 16 ? (tb - slice * 16) / BS + 1 : 0;
    for (int e = lane; e < cnt; e += 32) s_list[warp][e] = e;
  } else {
    const int32_t* il = p.idx + (qrow * p.hkv + g) * p.S;
    for (int base = 0; base < p.S; base += 32) {
      const int e = base + lane;
      int blk = -1;
      bool ok = false;
      if (e < p.S) {
        blk = il[e];
        ok = blk >= 0 && (int64_t)blk * BS + slice * 16 <= tb;
      }
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (ok) s_list[warp][cnt + __popc(m & ((1u << lane) - 1u))] = blk;
      cnt += __popc(m);
    }
  }
  __syncwarp();

  const __nv_bfloat16* kb = p.k + (kv_base * p.hkv + g) * D;
  const __nv_bfloat16* vb = p.v + (kv_base * p.hkv + g) * D;
  const int64_t rs = (int64_t)p.hkv * D;
  const uint32_t wbase = smem_u32(smem) + warp * NSTAGE * STAGE_BYTES;
  const int* list = s_list[warp];
  auto issue = [&](int i) {
    const int64_t key0 = (int64_t)list[i] * BS + slice * 16;
    const uint32_t sb = wbase + (i % NSTAGE) * STAGE_BYTES;
    const bool full = key0 + 15 <= tb;
#pragma unroll
    for (int c = lane; c < 16 * CH; c += 32) {
      const int row = c / CH, ch = c % CH;
      const bool ok = full || key0 + row <= tb;
      const int64_t off = (key0 + row) * rs + ch * 8;
      cp_async16(tile_addr<D>(sb, row, ch), ok ? kb + off : (const void*)p.k, ok ? 16 : 0);
      cp_async16(tile_addr<D>(sb + SLICE_BYTES, row, ch), ok ? vb + off : (const void*)p.k, ok ? 16 : 0);
    }
  };

  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
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
    float s[2][4] = {}, s2[2][4] = {}, dp[2][4] = {}, dp2[2][4] = {};
    qk_16keys_2acc<D>(s, s2, qa, sb, 0, lane);
    qk_16keys_2acc<D>(dp, dp2, da, sb + SLICE_BYTES, 0, lane);
    const int64_t key0 = (int64_t)list[i] * BS + slice * 16;
    float ds[2][4], big = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t key = key0 + nt * 8 + (lane & 3) * 2 + (j & 1);
        const float pe = key <= tb && key >= tl
                             ? ex2((s[nt][j] + s2[nt][j]) * p.scale_log2 - (j < 2 ? L0 : L1)) : 0.f;
        ds[nt][j] = pe * ((dp[nt][j] + dp2[nt][j]) - (j < 2 ? d0 : d1));
        big = fmaxf(big, fabsf(ds[nt][j]));
      }
    uint32_t dsa[4], dsl[4];
    split_bf16x2(ds[0][0], ds[0][1], dsa[0], dsl[0]);
    split_bf16x2(ds[0][2], ds[0][3], dsa[1], dsl[1]);
    split_bf16x2(ds[1][0], ds[1][1], dsa[2], dsl[2]);
    split_bf16x2(ds[1][2], ds[1][3], dsa[3], dsl[3]);
    pv_16keys<D>(acc, dsa, sb, 0, lane);  // dq += dS . K
    if (__any_sync(0xffffffffu, big > kSplitAbove)) pv_16keys<D>(acc, dsl, sb, 0, lane);
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();  // every ring is drained: the fold below reuses the shared memory

  constexpr int OS = D + 8;
  float* sm = reinterpret_cast<float*>(smem);  // [3][16][OS]
  if (warp > 0) {
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(&sm[((warp - 1) * 16 + rlo) * OS + col]) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(&sm[((warp - 1) * 16 + rhi) * OS + col]) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + (lane & 3) * 2;
    float a0 = acc[nt][0], a1 = acc[nt][1], a2 = acc[nt][2], a3 = acc[nt][3];
#pragma unroll
    for (int w = 0; w < 3; ++w) {
      const float2 x = *reinterpret_cast<const float2*>(&sm[(w * 16 + rlo) * OS + col]);
      const float2 y = *reinterpret_cast<const float2*>(&sm[(w * 16 + rhi) * OS + col]);
      a0 += x.x;
      a1 += x.y;
      a2 += y.x;
      a3 += y.y;
    }
    if (w0) *reinterpret_cast<uint32_t*>(p.dq + (row0 + rlo) * D + col) = pack_bf16(a0 * p.scale, a1 * p.scale);
    if (w1) *reinterpret_cast<uint32_t*>(p.dq + (row0 + rhi) * D + col) = pack_bf16(a2 * p.scale, a3 * p.scale);
  }
}

// ---------------------------------------------------------------------------- dK, dV
// Shared memory of sparse_bwd_dkv: K_j and V_j tiles, the token ring (Q rows, dO rows,
// log2-lse and D of 16 head rows per stage) and the item's token list.
template <int NSTAGE>
constexpr int dkv_smem_bytes() {
  return 2 * kTileBytes + NSTAGE * (2 * kRowsBytes + 2 * 16 * 4) + kChunk * 4;
}

template <int NSTAGE>
__global__ void __launch_bounds__(128, 2) sparse_bwd_dkv(const BwdParams p) {
  constexpr int D = kD, BS = kBS, CH = D / 8;
  constexpr int STAGE = 2 * kRowsBytes + 2 * 16 * 4;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_wcount[4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_bg = p.seqs.n_seqs * p.hkv;
  const int bg = blockIdx.x % n_bg;
  const int item = blockIdx.x / n_bg;
  const int b = bg / p.hkv, g = bg % p.hkv;
  int j, c, m;
  item_to_block(p, item, j, c, m);
  const int L = seq_len(p.seqs, b);
  const int Lk = key_len(p, L);
  if (j * BS >= Lk || (c > m && c * kChunk >= L)) return;  // no partial is read for this item
  const int64_t base = seq_start(p.seqs, b);
  const int64_t kbase = key_base(p, b);
  const int t_begin = p.window ? j * BS : max(first_query(p, j), c * kChunk);
  const int t_end = p.window ? min(j * BS + BS - 1 + p.window, L) : min((c + 1) * kChunk, L);

  const uint32_t kt = smem_u32(smem), vt = kt + kTileBytes;
  const uint32_t ring = vt + kTileBytes;
  int* s_tok = reinterpret_cast<int*>(smem + 2 * kTileBytes + NSTAGE * STAGE);

  // K_j and V_j (rows past the sequence read as zeros; no query reaches them)
  {
    const int64_t rs = (int64_t)p.hkv * D;
    const __nv_bfloat16* kb = p.k + ((kbase + (int64_t)j * BS) * p.hkv + g) * D;
    const __nv_bfloat16* vb = p.v + ((kbase + (int64_t)j * BS) * p.hkv + g) * D;
    for (int i = threadIdx.x; i < BS * CH; i += 128) {
      const int row = i / CH, ch = i % CH;
      const bool ok = j * BS + row < Lk;
      cp_async16(tile_addr<D>(kt, row, ch), ok ? kb + row * rs + ch * 8 : (const void*)p.k, ok ? 16 : 0);
      cp_async16(tile_addr<D>(vt, row, ch), ok ? vb + row * rs + ch * 8 : (const void*)p.k, ok ? 16 : 0);
    }
    cp_async_commit();
  }

  // tokens of the chunk whose list holds j, in token order, with multiplicity
  int n = 0;
  for (int t0 = t_begin; t0 < t_end; t0 += 128) {
    const int t = t0 + threadIdx.x;
    int mult = 0;
    if (t < t_end) {
      if (p.window) {
        mult = key_lo(p, t) <= j * BS + BS - 1;  // t >= j*BS here
      } else if (p.cmp_kernel) {
        mult = key_bound(p, t, Lk) >= j * BS;
      } else {
        const int32_t* il = p.idx + ((base + t) * p.hkv + g) * p.S;
        for (int e = 0; e < p.S; ++e) mult += il[e] == j;
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, mult > 0);
    if (lane == 0) s_wcount[warp] = __popc(bal);
    __syncthreads();
    int off = n;
    for (int w = 0; w < warp; ++w) off += s_wcount[w];
    if (mult > 0) s_tok[off + __popc(bal & ((1u << lane) - 1u))] = (t << 7) | mult;
    n += s_wcount[0] + s_wcount[1] + s_wcount[2] + s_wcount[3];
    __syncthreads();
  }

  const int r = p.r;
  const int hbase = g * r;
  auto issue = [&](int i) {
    const int t = s_tok[i] >> 7;
    const int64_t row0 = (base + t) * p.h + hbase;
    const uint32_t sb = ring + (i % NSTAGE) * STAGE;
#pragma unroll
    for (int e = threadIdx.x; e < 2 * 16 * CH; e += 128) {
      const int which = e / (16 * CH), rr = (e / CH) % 16, ch = e % CH;
      const bool ok = rr < r;
      const __nv_bfloat16* src = (which ? p.dout : p.q) + (row0 + rr) * D + ch * 8;
      cp_async16(tile_addr<D>(sb + which * kRowsBytes, rr, ch), ok ? (const void*)src : (const void*)p.q,
                 ok ? 16 : 0);
    }
    if (threadIdx.x < 32) {
      const int rr = threadIdx.x & 15;
      const bool ok = rr < r;
      const float* src = (threadIdx.x < 16 ? p.lse : p.dsum) + row0 + rr;
      cp_async4(sb + 2 * kRowsBytes + threadIdx.x * 4, ok ? (const void*)src : (const void*)p.lse, ok ? 4 : 0);
    }
  };

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < NSTAGE - 1; ++i) {
    if (i < n) issue(i);
    cp_async_commit();
  }
  cp_async_wait<NSTAGE - 1>();  // K_j and V_j (the oldest group) have landed
  __syncthreads();
  // A fragments of this warp's 16 keys of K_j and V_j, held for the whole item: the
  // products are S^T = K_w Q_t^T and dP^T = V_w dO_t^T (16 keys x 16 heads), whose C
  // fragments are already the A fragments of P^T and dS^T for dV and dK.
  uint32_t ka[D / 16][4], va[D / 16][4];
  {
    const int arow = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), acol = lane >> 4;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      ldsm_x4(ka[kk], tile_addr<D>(kt, arow, 2 * kk + acol));
      ldsm_x4(va[kk], tile_addr<D>(vt, arow, 2 * kk + acol));
    }
  }
  const int brow = (lane & 7) + ((lane >> 4) << 3), bcol = (lane >> 3) & 1;
  const int hc = (lane & 3) * 2;  // head columns hc, hc+1 (and hc+8, hc+9)
  const int krow_lo = j * BS + warp * 16 + (lane >> 2), krow_hi = krow_lo + 8;
  for (int i = 0; i < n; ++i) {
    if (i + NSTAGE - 1 < n) issue(i + NSTAGE - 1);
    cp_async_commit();
    cp_async_wait<NSTAGE - 1>();
    __syncthreads();
    const int t = s_tok[i] >> 7;
    const int tb = key_bound(p, t, Lk), tl = key_lo(p, t);
    const float mult = (float)(s_tok[i] & 127);
    const uint32_t qt = ring + (i % NSTAGE) * STAGE, dt = qt + kRowsBytes;
    const float* lrow = reinterpret_cast<const float*>(smem + 2 * kTileBytes + (i % NSTAGE) * STAGE + 2 * kRowsBytes);
    const float* drow = lrow + 16;
    float st[2][4] = {}, dpt[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t bq[4], bd[4];
      ldsm_x4(bq, tile_addr<D>(qt, brow, 2 * kk + bcol));
      ldsm_x4(bd, tile_addr<D>(dt, brow, 2 * kk + bcol));
      mma_bf16(st[0], ka[kk], bq[0], bq[1]);
      mma_bf16(st[1], ka[kk], bq[2], bq[3]);
      mma_bf16(dpt[0], va[kk], bd[0], bd[1]);
      mma_bf16(dpt[1], va[kk], bd[2], bd[3]);
    }
    float pr[2][4], ds[2][4], big = 0.f, pbig = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int head = nt * 8 + hc + (q & 1);
        const int key = q < 2 ? krow_lo : krow_hi;
        const float pe =
            key <= tb && key >= tl ? ex2(st[nt][q] * p.scale_log2 - lse_to_log2(lrow[head])) : 0.f;
        pr[nt][q] = pe * mult;
        ds[nt][q] = pe * mult * (dpt[nt][q] - drow[head]);
        big = fmaxf(big, fabsf(ds[nt][q]));
        pbig = fmaxf(pbig, pr[nt][q]);
      }
    uint32_t ph[4], pl[4], sh[4], sl[4];
    split_bf16x2(pr[0][0], pr[0][1], ph[0], pl[0]);
    split_bf16x2(pr[0][2], pr[0][3], ph[1], pl[1]);
    split_bf16x2(pr[1][0], pr[1][1], ph[2], pl[2]);
    split_bf16x2(pr[1][2], pr[1][3], ph[3], pl[3]);
    split_bf16x2(ds[0][0], ds[0][1], sh[0], sl[0]);
    split_bf16x2(ds[0][2], ds[0][3], sh[1], sl[1]);
    split_bf16x2(ds[1][0], ds[1][1], sh[2], sl[2]);
    split_bf16x2(ds[1][2], ds[1][3], sh[3], sl[3]);
    pv_16keys<D>(dv, ph, dt, 0, lane);  // dV_w += P^T . dO_t
    pv_16keys<D>(dk, sh, qt, 0, lane);  // dK_w += dS^T . Q_t
    if (__any_sync(0xffffffffu, pbig > kSplitPAbove)) pv_16keys<D>(dv, pl, dt, 0, lane);
    if (__any_sync(0xffffffffu, big > kSplitAbove)) pv_16keys<D>(dk, sl, qt, 0, lane);
    __syncthreads();  // the stage is refilled at the next iteration
  }
  cp_async_wait<0>();

  const int rlo = lane >> 2;
  float* out = p.part + ((size_t)bg * p.items_per_bg + item) * 2 * BS * D;
  const int k0 = warp * 16 + rlo, k1 = k0 + 8;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + (lane & 3) * 2;
    *reinterpret_cast<float2*>(out + k0 * D + col) = make_float2(dk[nt][0], dk[nt][1]);
    *reinterpret_cast<float2*>(out + k1 * D + col) = make_float2(dk[nt][2], dk[nt][3]);
    *reinterpret_cast<float2*>(out + BS * D + k0 * D + col) = make_float2(dv[nt][0], dv[nt][1]);
    *reinterpret_cast<float2*>(out + BS * D + k1 * D + col) = make_float2(dv[nt][2], dv[nt][3]);
  }
}

// Sum of the partials of one (sequence, kv-head, key block) in chunk order.
__global__ void __launch_bounds__(256) sparse_bwd_reduce(const BwdParams p) {
  constexpr int D = kD, BS = kBS;
  const int bg = blockIdx.x / p.nb, j = blockIdx.x % p.nb;
  const int b = bg / p.hkv, g = bg % p.hkv;
  const int L = seq_len(p.seqs, b);
  const int Lk = key_len(p, L);
  if (j * BS >= Lk) return;
  int m, first = 0;
  if (p.window) {
    m = 0;
    first = j;
  } else if (p.cmp_kernel) {
    for (int jj = 0; jj < j; ++jj) first += p.n_chunks - first_query(p, jj) / kChunk;
    m = first_query(p, j) / kChunk;
  } else {
    m = j / kGroup;
    for (int mm = 0; mm < m; ++mm) first += min(kGroup, p.nb - mm * kGroup) * (p.n_chunks - mm);
    first += (j - m * kGroup) * (p.n_chunks - m);
  }
  int n_items = 1;
  while (!p.window && m + n_items < p.n_chunks && (m + n_items) * kChunk < L) ++n_items;
  const float4* src = reinterpret_cast<const float4*>(p.part + ((size_t)bg * p.items_per_bg + first) * 2 * BS * D);
  constexpr int N4 = 2 * BS * D / 4;
  const int64_t base = key_base(p, b);
  for (int e = threadIdx.x; e < N4; e += 256) {
    float4 a = src[e];
    for (int it = 1; it < n_items; ++it) {
      const float4 x = src[(size_t)it * N4 + e];
      a.x += x.x;
      a.y += x.y;
      a.z += x.z;
      a.w += x.w;
    }
    const int which = e / (BS * D / 4), key = (e / (D / 4)) % BS, col = (e % (D / 4)) * 4;
    if (j * BS + key >= Lk) continue;
    const float f = which ? 1.f : p.scale;
    __nv_bfloat16* dst = (which ? p.dv : p.dk) + ((base + (int64_t)j * BS + key) * p.hkv + g) * D + col;
    uint2 w;
    w.x = pack_bf16(a.x * f, a.y * f);
    w.y = pack_bf16(a.z * f, a.w * f);
    *reinterpret_cast<uint2*>(dst) = w;
  }
}

struct BwdLayout {
  int n_chunks, nb, items_per_bg;
  size_t dsum, part, inv_list, inv_tab, total;
};

// cmp_kernel > 0: the compressed branch (keys are the n_c(L) compressed rows).  S > 0:
// selected blocks with lists of S entries (room for the inverted lists).
BwdLayout bwd_layout(const Seqs& s, int h, int hkv, int cmp_kernel = 0, int cmp_stride = 0, int window = 0,
                     int S = 0) {
  BwdLayout l{};
  const int Lmax = s.max_len;
  l.n_chunks = (Lmax + kChunk - 1) / kChunk;
  if (window) {  // one item per key block
    l.nb = (Lmax + kBS - 1) / kBS;
    l.items_per_bg = l.nb;
  } else if (cmp_kernel) {
    const int nk = Lmax >= cmp_kernel ? (Lmax - cmp_kernel) / cmp_stride + 1 : 0;
    l.nb = (nk + kBS - 1) / kBS;
    for (int j = 0; j < l.nb; ++j) l.items_per_bg += l.n_chunks - (cmp_stride * kBS * j + cmp_kernel - 1) / kChunk;
  } else {
    l.nb = (Lmax + kBS - 1) / kBS;
    for (int m = 0; m < l.n_chunks; ++m) l.items_per_bg += std::min(kGroup, l.nb - m * kGroup) * (l.n_chunks - m);
  }
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  l.dsum = 0;
  l.part = a256((size_t)s.tokens * h * 4);
  l.inv_list = a256(l.part + (size_t)s.n_seqs * hkv * l.items_per_bg * 2 * kBS * kD * 4);
  const bool inv = !cmp_kernel && !window && S > 0 && dkv_tc_shape(h / hkv, false, l.nb);
  const size_t lists = inv ? (size_t)s.n_seqs * hkv * l.n_chunks : 0;
  l.inv_tab = a256(l.inv_list + lists * kChunk * S * 4);
  l.total = a256(l.inv_tab + lists * l.nb * 8);
  return l;
}

cudaError_t run_bwd(const BwdParams& p0, const BwdLayout& l, void* workspace, cudaStream_t st) {
  BwdParams p = p0;
  p.dsum = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + l.dsum);
  p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + l.part);
  p.inv_list = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + l.inv_list);
  p.inv_tab = reinterpret_cast<int2*>(static_cast<uint8_t*>(workspace) + l.inv_tab);
  p.r = p.h / p.hkv;
  p.scale_log2 = p.scale * kLog2e;
  p.n_chunks = l.n_chunks;
  p.nb = l.nb;
  p.items_per_bg = l.items_per_bg;
  const Seqs& s = p.seqs;
  constexpr int NS_Q = 2, NS_KV = 3;
  constexpr int dq_bytes = 4 * NS_Q * 2 * 16 * kD * 2;
  static_assert(dq_bytes >= 3 * 16 * (kD + 8) * 4, "dq fold needs the ring's shared memory");
  cudaError_t e;
  if (dq_tc_supported(p)) {  // compressed keys and window, group sizes 8 and 16: the tensor-core kernel
    const int64_t kv_rows = !p.cmp_kernel ? s.tokens
                            : s.cu        ? s.tokens / p.cmp_stride + s.n_seqs
                                          : (int64_t)s.n_seqs * (s.T >= p.cmp_kernel ? (s.T - p.cmp_kernel) / p.cmp_stride + 1 : 0);
    if ((e = launch_dq_tc(p, kv_rows, st)) != cudaSuccess) return e;
  } else {
    e = cudaFuncSetAttribute(sparse_bwd_dq<NS_Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq_bytes);
    if (e != cudaSuccess) return e;
    sparse_bwd_dq<NS_Q><<<dim3((unsigned)s.tokens, p.hkv), 128, dq_bytes, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int64_t items = (int64_t)s.n_seqs * p.hkv * l.items_per_bg;
  if (items > 0) {
    if (dkv_tc_supported(p)) {  // group sizes 8 and 16: the tensor-core kernel
      if (!p.cmp_kernel && !p.window && (e = launch_invert(p, st)) != cudaSuccess) return e;
      if ((e = launch_dkv_tc(p, items, s.tokens * p.h, st)) != cudaSuccess) return e;
    } else {
      constexpr int kv_bytes = dkv_smem_bytes<NS_KV>();
      e = cudaFuncSetAttribute(sparse_bwd_dkv<NS_KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kv_bytes);
      if (e != cudaSuccess) return e;
      sparse_bwd_dkv<NS_KV><<<(unsigned)items, 128, kv_bytes, st>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    sparse_bwd_reduce<<<(unsigned)((int64_t)s.n_seqs * p.hkv * l.nb), 256, 0, st>>>(p);
  }
  return cudaGetLastError();
}

// Backward of the mean pooling: token row t of sequence b receives, from each window c
// of that sequence with c*stride <= t < c*stride + kernel, the window's gradient / kernel.
// One thread per (token, kv-head, 8 columns).
__global__ void __launch_bounds__(256) compress_bwd_kernel(const __nv_bfloat16* __restrict__ dkc,
                                                           __nv_bfloat16* __restrict__ dk, Seqs s, int hkv, int d,
                                                           int kernel, int stride) {
  const int cpr = d / 8;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= s.tokens * hkv * cpr) return;
  const int ch = (int)(i % cpr);
  const int64_t rg = i / cpr;
  const int g = (int)(rg % hkv);
  const int64_t tok = rg / hkv;
  const int sq = seq_of_token(s, tok);
  const int t = (int)(tok - seq_start(s, sq));
  const int n_c = num_cmp(seq_len(s, sq), kernel, stride);
  const int64_t c0 = cmp_offset(s, sq, kernel, stride);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int c_hi = min(t / stride, n_c - 1);
  for (int c = max(0, (t - kernel) / stride); c <= c_hi; ++c) {
    if (c * stride > t || t >= c * stride + kernel) continue;
    const uint4 w = *reinterpret_cast<const uint4*>(dkc + ((c0 + c) * hkv + g) * d + ch * 8);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      acc[2 * e] += f.x;
      acc[2 * e + 1] += f.y;
    }
  }
  const float inv = 1.f / (float)kernel;
  uint4 o;
  o.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  o.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  o.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  o.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(dk + (tok * hkv + g) * d + ch * 8) = o;
}

// Backward of the gate combine: with g_i = sigmoid(a_i) and o = sum_i g_i o_i, the branch
// gradients are g_i dO and the logit gradients g_i (1 - g_i) (dO . o_i).  One warp per
// (token, head) row, 8 columns per lane and step; HBM bound.
__global__ void __launch_bounds__(256) gate_bwd_kernel(const __nv_bfloat16* __restrict__ dout,
                                                       const __nv_bfloat16* __restrict__ o_cmp,
                                                       const __nv_bfloat16* __restrict__ o_slc,
                                                       const __nv_bfloat16* __restrict__ o_swa,
                                                       const float* __restrict__ logits, __nv_bfloat16* d_cmp,
                                                       __nv_bfloat16* d_slc, __nv_bfloat16* d_swa, float* d_logits,
                                                       int64_t rows, int d) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float g[3], dot[3] = {0.f, 0.f, 0.f};
#pragma unroll
  for (int b = 0; b < 3; ++b) g[b] = 1.f / (1.f + expf(-logits[row * 3 + b]));
  const __nv_bfloat16* src[3] = {o_cmp, o_slc, o_swa};
  __nv_bfloat16* dst[3] = {d_cmp, d_slc, d_swa};
  for (int c = lane * 8; c < d; c += 256) {
    const uint4 w = *reinterpret_cast<const uint4*>(dout + row * d + c);
    const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&w);
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(w2[e]);
      x[2 * e] = f.x;
      x[2 * e + 1] = f.y;
    }
#pragma unroll
    for (int b = 0; b < 3; ++b) {
      const uint4 u = *reinterpret_cast<const uint4*>(src[b] + row * d + c);
      const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(u2[e]);
        dot[b] += x[2 * e] * f.x + x[2 * e + 1] * f.y;
      }
      uint4 o;
      o.x = pack_bf16(g[b] * x[0], g[b] * x[1]);
      o.y = pack_bf16(g[b] * x[2], g[b] * x[3]);
      o.z = pack_bf16(g[b] * x[4], g[b] * x[5]);
      o.w = pack_bf16(g[b] * x[6], g[b] * x[7]);
      *reinterpret_cast<uint4*>(dst[b] + row * d + c) = o;
    }
  }
#pragma unroll
  for (int b = 0; b < 3; ++b)
    for (int off = 16; off; off >>= 1) dot[b] += __shfl_xor_sync(0xffffffffu, dot[b], off);
  if (lane < 3) {
    const float gb = lane == 0 ? g[0] : lane == 1 ? g[1] : g[2];
    const float db = lane == 0 ? dot[0] : lane == 1 ? dot[1] : dot[2];
    d_logits[row * 3 + lane] = gb * (1.f - gb) * db;
  }
}

}  // namespace

// out = a + b + c elementwise (bf16 in and out, fp32 sum); n a multiple of 8.
__global__ void __launch_bounds__(256) add3_kernel(const uint4* __restrict__ a, const uint4* __restrict__ b,
                                                   const uint4* __restrict__ c, uint4* __restrict__ out, int64_t n8) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint4 x = a[i], y = b[i], z = c[i];
  const __nv_bfloat162* xs = reinterpret_cast<const __nv_bfloat162*>(&x);
  const __nv_bfloat162* ys = reinterpret_cast<const __nv_bfloat162*>(&y);
  const __nv_bfloat162* zs = reinterpret_cast<const __nv_bfloat162*>(&z);
  uint32_t r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 u = __bfloat1622float2(xs[e]), v = __bfloat1622float2(ys[e]), w = __bfloat1622float2(zs[e]);
    r[e] = pack_bf16(u.x + v.x + w.x, u.y + v.y + w.y);
  }
  out[i] = make_uint4(r[0], r[1], r[2], r[3]);
}

cudaError_t launch_add3(const void* a, const void* b, const void* c, void* out, int64_t n, cudaStream_t st) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  add3_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>((const uint4*)a, (const uint4*)b, (const uint4*)c,
                                                             (uint4*)out, n8);
  return cudaGetLastError();
}

cudaError_t launch_gate_bwd(int64_t rows, int d, const void* dout, const void* o_cmp, const void* o_slc,
                            const void* o_swa, const float* logits, void* d_cmp, void* d_slc, void* d_swa,
                            float* d_logits, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  gate_bwd_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(
      (const __nv_bfloat16*)dout, (const __nv_bfloat16*)o_cmp, (const __nv_bfloat16*)o_slc,
      (const __nv_bfloat16*)o_swa, logits, (__nv_bfloat16*)d_cmp, (__nv_bfloat16*)d_slc, (__nv_bfloat16*)d_swa,
      d_logits, rows, d);
  return cudaGetLastError();
}

size_t sparse_bwd_workspace_bytes(const Seqs& s, int h, int hkv, int S) {
  if (s.tokens == 0 || s.max_len == 0) return 0;
  return bwd_layout(s, h, hkv, 0, 0, 0, S).total;
}

size_t cmp_attn_bwd_workspace_bytes(const Seqs& s, int h, int hkv, int kernel, int stride) {
  if (s.tokens == 0 || s.max_len == 0) return 0;
  return bwd_layout(s, h, hkv, kernel, stride).total;
}

static BwdParams bwd_params(const Seqs& s, const void* q, const void* k, const void* v, int h, int hkv, float scale,
                            const void* o, const float* lse, const void* dout, void* dq, void* dk, void* dv) {
  BwdParams p{};
  p.q = (const __nv_bfloat16*)q;
  p.k = (const __nv_bfloat16*)k;
  p.v = (const __nv_bfloat16*)v;
  p.o = (const __nv_bfloat16*)o;
  p.dout = (const __nv_bfloat16*)dout;
  p.lse = lse;
  p.dq = (__nv_bfloat16*)dq;
  p.dk = (__nv_bfloat16*)dk;
  p.dv = (__nv_bfloat16*)dv;
  p.seqs = s;
  p.h = h;
  p.hkv = hkv;
  p.scale = scale;
  return p;
}

cudaError_t launch_sparse_bwd(const Seqs& s, const void* q, const void* k, const void* v, const int32_t* idx, int S,
                              int h, int hkv, float scale, const void* o, const float* lse, const void* dout,
                              void* dq, void* dk, void* dv, void* workspace, cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  BwdParams p = bwd_params(s, q, k, v, h, hkv, scale, o, lse, dout, dq, dk, dv);
  p.idx = idx;
  p.S = S;
  return run_bwd(p, bwd_layout(s, h, hkv, 0, 0, 0, S), workspace, st);
}

cudaError_t launch_cmp_attn_bwd(const Seqs& s, const void* q, const void* k_cmp, const void* v_cmp, int h, int hkv,
                                int kernel, int stride, float scale, const void* o, const float* lse,
                                const void* dout, void* dq, void* dk_cmp, void* dv_cmp, void* workspace,
                                cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  BwdParams p = bwd_params(s, q, k_cmp, v_cmp, h, hkv, scale, o, lse, dout, dq, dk_cmp, dv_cmp);
  p.cmp_kernel = kernel;
  p.cmp_stride = stride;
  return run_bwd(p, bwd_layout(s, h, hkv, kernel, stride), workspace, st);
}

size_t swa_bwd_workspace_bytes(const Seqs& s, int h, int hkv, int window) {
  if (s.tokens == 0 || s.max_len == 0) return 0;
  return bwd_layout(s, h, hkv, 0, 0, window).total;
}

cudaError_t launch_swa_bwd(const Seqs& s, const void* q, const void* k, const void* v, int h, int hkv, int window,
                           float scale, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* workspace, cudaStream_t st) {
  if (s.tokens == 0) return cudaSuccess;
  BwdParams p = bwd_params(s, q, k, v, h, hkv, scale, o, lse, dout, dq, dk, dv);
  p.window = window;
  return run_bwd(p, bwd_layout(s, h, hkv, 0, 0, window), workspace, st);
}

cudaError_t launch_compress_bwd(const Seqs& s, const void* dk_cmp, int hkv, int d, int kernel, int stride, void* dk,
                                cudaStream_t st) {
  const int64_t n = s.tokens * hkv * (d / 8);
  if (n == 0) return cudaSuccess;
  compress_bwd_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>((const __nv_bfloat16*)dk_cmp, (__nv_bfloat16*)dk,
                                                                    s, hkv, d, kernel, stride);
  return cudaGetLastError();
}

}  // namespace nsa
