"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against a library routine that computes the same
definition (avg_pool1d, scaled_dot_product_attention, topk), a hand-computed
value, or an invariant that determines the result uniquely.  None of them
re-types the oracle's own formula.  CPU only.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc
from sparse_attention_compress_gb300 import inputs as gen

F64 = torch.float64


def _t(a):
    """numpy (bf16 bits or fp32) -> torch float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = gen.bf16_bits_to_f32(a)
    return torch.from_numpy(np.asarray(a, np.float64))


def _rand(shape, seed, dtype="bf16"):
    return gen.normal(np.random.Generator(np.random.PCG64(seed)), shape, dtype)


def _sdpa_probs(q, k, mask):
    """Attention probabilities through the library SDPA, using V = identity.
    q [T,h,d], k [Tk,h,d] (already expanded per head), mask [T,Tk] bool."""
    T, h, d = q.shape
    Tk = k.shape[0]
    eye = torch.eye(Tk, dtype=F64).expand(h, Tk, Tk)
    return F.scaled_dot_product_attention(q.permute(1, 0, 2), k.permute(1, 0, 2), eye,
                                          attn_mask=mask).permute(1, 0, 2)  # [T,h,Tk]


def _sdpa(q, k, v, mask):
    """SDPA float64 with GQA expansion; q [T,h,d], k/v [Tk,hkv,d], mask [T,Tk] bool."""
    h, hkv = q.shape[1], k.shape[1]
    r = h // hkv
    ke = k.repeat_interleave(r, dim=1)
    ve = v.repeat_interleave(r, dim=1)
    return F.scaled_dot_product_attention(q.permute(1, 0, 2), ke.permute(1, 0, 2), ve.permute(1, 0, 2),
                                          attn_mask=mask).permute(1, 0, 2)


# --------------------------------------------------------------------------- S1
def test_num_cmp_hand_values():
    # full windows of 32 at stride 16 (hand-counted)
    expect = {0: 0, 1: 0, 31: 0, 32: 1, 33: 1, 47: 1, 48: 2, 63: 2, 64: 3, 4100: 255, 32768: 2047,
              65536: 4095}
    for L, n in expect.items():
        assert orc.num_cmp(L) == n, L


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_compress_equals_avg_pool1d(dtype):
    lengths = [1, 31, 32, 47, 48, 100, 257]
    cu = gen.varlen_cu_seqlens(lengths)
    hkv, d = 2, 8
    k = _rand((cu[-1], hkv, d), 11, dtype)
    exact, rounded = orc.compress(k, cu)
    kt = _t(k)
    off = orc.cmp_offsets(cu)
    for i, L in enumerate(lengths):
        n_c = off[i + 1] - off[i]
        if L < 32:
            assert n_c == 0
            continue
        x = kt[cu[i]:cu[i + 1]].reshape(L, hkv * d).T.unsqueeze(1)  # [hkv*d, 1, L]
        ref = F.avg_pool1d(x, 32, 16).squeeze(1).T.reshape(-1, hkv, d)
        assert ref.shape[0] == n_c
        got = torch.from_numpy(exact[off[i]:off[i + 1]])
        assert torch.allclose(got, ref, rtol=0, atol=1e-14)
    # the stored value is the nearest representable value of the storage dtype
    if dtype == "f32":
        assert np.array_equal(rounded, exact.astype(np.float32))
    else:
        r = rounded.astype(np.int64)
        val = gen.bf16_bits_to_f32(rounded).astype(np.float64)
        up = gen.bf16_bits_to_f32(((r & 0x7FFF) + 1 | (r & 0x8000)).astype(np.uint16)).astype(np.float64)
        dn = gen.bf16_bits_to_f32(np.where((r & 0x7FFF) > 0, r - 1, r).astype(np.uint16)).astype(np.float64)
        err = np.abs(val - exact)
        assert np.all(err <= np.abs(up - exact))
        assert np.all(err <= np.abs(dn - exact))
        tie = (err == np.abs(up - exact)) | (err == np.abs(dn - exact))
        tie &= err > 0
        assert np.all((r[tie] & 1) == 0)  # ties go to the even pattern


def test_compress_constant_and_window_independence():
    cu = gen.varlen_cu_seqlens([64, 80])
    k = np.full((144, 1, 4), 3.25, np.float32)
    k[64:] = -1.5  # the second sequence must not leak into the first one's windows
    exact, _ = orc.compress(k, cu)
    assert np.all(exact[:3] == 3.25) and np.all(exact[3:] == -1.5)


# --------------------------------------------------------------------------- S2
def test_cmp_probs_kernel1_is_dense_causal_attention():
    """With kernel = stride = 1 each compressed key is one token and the window rule
    reduces to plain causal masking: the group probabilities must be the summed
    causal attention probabilities of the group's heads."""
    T, h, hkv, d = 40, 4, 2, 16
    cu = gen.dense_cu_seqlens(1, T)
    q = _rand((T, h, d), 1)
    k = _rand((T, hkv, d), 2)
    _, kc = orc.compress(k, cu, kernel=1, stride=1)
    assert np.array_equal(kc, k)
    pg = orc.cmp_probs(q, kc, cu, kernel=1, stride=1)
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    probs = _sdpa_probs(_t(q), _t(k).repeat_interleave(2, dim=1), mask)  # [T,h,T]
    ref = probs.reshape(T, hkv, 2, T).sum(2)
    assert torch.allclose(torch.from_numpy(pg), ref, atol=1e-13, rtol=0)


def test_cmp_probs_window_causality_via_sdpa_mask():
    lengths = [200, 77]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d = 4, 1, 32
    q = _rand((cu[-1], h, d), 3)
    k = _rand((cu[-1], hkv, d), 4)
    _, kc = orc.compress(k, cu)
    pg = orc.cmp_probs(q, kc, cu)
    off = orc.cmp_offsets(cu)
    for i, L in enumerate(lengths):
        n_c = off[i + 1] - off[i]
        t = torch.arange(L)[:, None]
        c = torch.arange(n_c)[None, :]
        mask = (16 * c + 31) <= t
        live = mask.any(1)
        qs = _t(q[cu[i]:cu[i + 1]])[live]
        ks = _t(kc[off[i]:off[i + 1]]).repeat_interleave(h, dim=1)
        ref = _sdpa_probs(qs, ks, mask[live]).sum(1)
        got = torch.from_numpy(pg[cu[i]:cu[i + 1], 0, :n_c])
        assert torch.allclose(got[live], ref, atol=1e-13, rtol=0)
        assert torch.all(got[~live] == 0)
        # every row with a causal compressed key sums to the group size
        assert torch.allclose(got[live].sum(1), torch.full((int(live.sum()),), float(h), dtype=F64))


# --------------------------------------------------------------------------- S3
@pytest.mark.parametrize("L,expect", [
    (31, [0.0]), (32, [0.0]), (47, [0.0]), (48, [0.5]), (63, [0.5]), (64, [1.0]),
    (128, [1.0, 5.0]), (112, [1.0, 4.5]),
])
def test_pool_ramp_hand_values(L, expect):
    # P_g[c] = c: block j averages c = 4j, 4j+1, 4j+2 where those windows exist
    n_c = orc.num_cmp(L)
    n_b = -(-L // 64)
    got = orc.pool_row(np.arange(max(n_c, 1), dtype=np.float64), n_c, n_b)
    assert got.tolist() == expect


def test_pool_ramp_long_tail():
    L = 4100
    n_c, n_b = orc.num_cmp(L), -(-L // 64)
    got = orc.pool_row(np.arange(n_c, dtype=np.float64), n_c, n_b)
    assert n_c == 255 and n_b == 65
    assert got[:64].tolist() == [4.0 * j + 1 for j in range(64)]
    assert got[64] == 0.0


@pytest.mark.parametrize("n_c", [3, 4, 5, 6, 7, 64, 255, 2047])
def test_pool_equals_avg_pool1d_ceil(n_c):
    rng = np.random.default_rng(n_c)
    pg = rng.random(n_c)
    n_b = (16 * (n_c - 1) + 32 + 63) // 64 + 1  # room for trailing empty blocks
    got = orc.pool_row(pg, n_c, n_b)
    ref = F.avg_pool1d(torch.from_numpy(pg).view(1, 1, -1), 3, 4, ceil_mode=True).flatten().numpy()
    m = len(ref)
    assert np.allclose(got[:m], ref, atol=1e-15, rtol=0)
    assert np.all(got[m:] == 0)


def test_cmp_scores_pool_equals_sdpa_then_avg_pool():
    """S2+S3 in one call on ragged varlen sequences with GQA groups, a non-default scale,
    a padded block stride and a row subset: the library SDPA's probabilities under the
    window-end mask, summed over each group's heads, then avg_pool1d(3, 4, ceil_mode)
    over the window axis; blocks past the pooled ones, rows without a causal window and
    the stride padding are 0."""
    lengths = [1, 31, 64, 65, 130, 257, 300]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d, scale = 8, 2, 32, 0.3
    r = h // hkv
    q = _rand((cu[-1], h, d), 11)
    k = _rand((cu[-1], hkv, d), 12)
    _, kc = orc.compress(k, cu)
    off = orc.cmp_offsets(cu)
    nb_stride = -(-max(lengths) // 64) + 3
    got = orc.cmp_scores_pool(q, kc, cu, scale=scale, nb_stride=nb_stride)
    assert got.shape == (cu[-1], hkv, nb_stride)
    for i, L in enumerate(lengths):
        rows = slice(cu[i], cu[i + 1])
        n_c = off[i + 1] - off[i]
        ref = torch.zeros(L, hkv, nb_stride, dtype=F64)
        if n_c > 0:
            assert n_c >= 3  # avg_pool1d needs a full first window; the lengths above ensure it
            t = torch.arange(L)[:, None]
            mask = (16 * torch.arange(n_c)[None, :] + 31) <= t
            live = mask.any(1)
            qs = _t(q[rows])[live].permute(1, 0, 2)
            ks = _t(kc[off[i]:off[i + 1]]).repeat_interleave(r, dim=1).permute(1, 0, 2)
            eye = torch.eye(n_c, dtype=F64).expand(h, n_c, n_c)
            probs = F.scaled_dot_product_attention(qs, ks, eye, attn_mask=mask[live], scale=scale)
            pg = probs.permute(1, 0, 2).reshape(-1, hkv, r, n_c).sum(2)  # [live rows, hkv, n_c]
            pooled = F.avg_pool1d(pg.reshape(-1, 1, n_c), 3, 4, ceil_mode=True).reshape(pg.shape[0], hkv, -1)
            m = pooled.shape[-1]
            assert m <= -(-L // 64)
            ref[live, :, :m] = pooled
        assert torch.allclose(torch.from_numpy(got[rows]), ref, atol=1e-13, rtol=0), L
    sub = [0, 1, 40, cu[3] - 1, cu[5] + 200, cu[-1] - 1]
    part = orc.cmp_scores_pool(q, kc, cu, scale=scale, nb_stride=nb_stride, rows=sub)
    assert np.array_equal(part, got[sub])


# --------------------------------------------------------------------------- S4
def _check_topk_row(sc, t, bs, n_init, n_local, k, row):
    own = t // bs
    ncand = own + 1
    take = min(k, ncand)
    chosen = row[:take]
    assert np.all(row[take:] == -1)
    assert np.all(np.diff(chosen) > 0), "ascending and distinct"
    assert chosen.min() >= 0 and chosen.max() <= own, "causal"
    forced = {j for j in range(ncand) if j < n_init or j > own - n_local}
    cs = set(chosen.tolist())
    if len(forced) <= k:
        assert forced <= cs
    # dominance: anything chosen and not forced beats anything not chosen
    for a in cs - forced:
        for b in set(range(ncand)) - cs:
            assert b not in forced
            assert sc[a] > sc[b] or (sc[a] == sc[b] and a < b)


@pytest.mark.parametrize("seed", range(6))
def test_topk_invariants(seed):
    rng = np.random.default_rng(seed)
    bs = 64
    L = int(rng.integers(1, 3000))
    n_init, n_local, k = int(rng.integers(0, 3)), int(rng.integers(0, 3)), int(rng.integers(1, 20))
    cu = gen.dense_cu_seqlens(1, L)
    nb = -(-L // bs)
    # few distinct levels -> many exact ties
    sc = rng.integers(0, 4, size=(L, 1, nb)).astype(np.float64) / 4
    idx = orc.topk(sc, cu, bs, n_init, n_local, k)
    for t in range(0, L, max(1, L // 97)):
        _check_topk_row(sc[t, 0], t, bs, n_init, n_local, k, idx[t, 0])


def test_topk_equals_torch_topk_without_forcing():
    rng = np.random.default_rng(7)
    L, bs, k = 2048, 64, 9
    sc = rng.permutation(L * 32).reshape(L, 1, 32).astype(np.float64)  # all distinct
    idx = orc.topk(sc, gen.dense_cu_seqlens(1, L), bs, 0, 0, k)
    for t in (0, 63, 64, 600, 2047):
        own = t // bs
        ref = torch.topk(torch.from_numpy(sc[t, 0, :own + 1]), min(k, own + 1)).indices.sort().values
        assert idx[t, 0, :len(ref)].tolist() == ref.tolist()


# --------------------------------------------------------------------------- S5
def _all_causal_idx(cu, hkv, bs):
    T = int(np.max(np.diff(cu)))
    nb = -(-T // bs)
    rows = []
    for i in range(len(cu) - 1):
        for t in range(cu[i + 1] - cu[i]):
            rows.append([j if j <= t // bs else -1 for j in range(nb)])
    return np.repeat(np.asarray(rows, np.int32)[:, None, :], hkv, axis=1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sparse_all_blocks_equals_dense_causal(dtype):
    lengths = [150, 64, 33]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d, bs = 4, 2, 16, 32
    q, k, v = (_rand((cu[-1], hh, d), s, dtype) for s, hh in ((5, h), (6, hkv), (7, hkv)))
    idx = _all_causal_idx(cu, hkv, bs)
    o, lse = orc.sparse_attn(q, k, v, idx, cu, bs)
    for i, L in enumerate(lengths):
        sl = slice(cu[i], cu[i + 1])
        mask = torch.ones(L, L, dtype=torch.bool).tril()
        ref = _sdpa(_t(q[sl]), _t(k[sl]), _t(v[sl]), mask)
        assert torch.allclose(torch.from_numpy(o[sl]), ref, atol=1e-12, rtol=0)
        s = torch.einsum("thd,shd->ths", _t(q[sl]), _t(k[sl]).repeat_interleave(2, 1)) * d ** -0.5
        ref_lse = torch.logsumexp(s.masked_fill(~mask[:, None, :], -torch.inf), -1)
        assert torch.allclose(torch.from_numpy(lse[sl]), ref_lse, atol=1e-12, rtol=0)


def test_sparse_own_block_is_local_attention():
    T, h, hkv, d, bs = 130, 2, 1, 8, 32
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v = _rand((T, h, d), 8), _rand((T, hkv, d), 9), _rand((T, hkv, d), 10)
    idx = (np.arange(T) // bs).astype(np.int32).reshape(T, 1, 1)
    o, _ = orc.sparse_attn(q, k, v, idx, cu, bs)
    t = torch.arange(T)
    mask = (t[:, None] >= t[None, :]) & (t[:, None] // bs == t[None, :] // bs)
    assert torch.allclose(torch.from_numpy(o), _sdpa(_t(q), _t(k), _t(v), mask), atol=1e-12, rtol=0)


def test_sparse_order_padding_noncausal_and_duplicates():
    T, h, hkv, d, bs = 256, 2, 1, 8, 32
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v = _rand((T, h, d), 12), _rand((T, hkv, d), 13), _rand((T, hkv, d), 14)
    t = np.arange(T)
    own = t // bs
    base = np.stack([np.zeros(T), own], 1).astype(np.int32)       # {0, own}
    shuf = np.stack([own, np.full(T, -1), np.full(T, 7), np.zeros(T)], 1).astype(np.int32)
    o1, _ = orc.sparse_attn(q, k, v, base[:, None, :], cu, bs)
    o2, _ = orc.sparse_attn(q, k, v, shuf[:, None, :], cu, bs)
    # block 7 starts at 224: it is non-causal (skipped) for t < 224 only
    early = t < 224
    assert np.allclose(o1[early], o2[early], atol=1e-13, rtol=0)
    # a block listed twice counts twice: same as attention with its keys duplicated
    tq = 100
    dup = np.array([[[0, 0, 3]]], np.int32)  # block 0 twice, own block 3 once
    o3, _ = orc.sparse_attn(q, k, v, np.repeat(dup, T, 0), cu, bs, rows=[tq])
    keys = list(range(0, 32)) * 2 + list(range(96, 101))
    kk, vv = _t(k)[keys], _t(v)[keys]
    ref = _sdpa(_t(q[tq:tq + 1]), kk, vv, torch.ones(1, len(keys), dtype=torch.bool))
    assert torch.allclose(torch.from_numpy(o3), ref, atol=1e-12, rtol=0)


def test_sparse_empty_list_gives_zero():
    T, h, d = 40, 2, 8
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v = _rand((T, h, d), 15), _rand((T, 1, d), 16), _rand((T, 1, d), 17)
    idx = np.full((T, 1, 2), -1, np.int32)
    o, lse = orc.sparse_attn(q, k, v, idx, cu, 32)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


# --------------------------------------------------------------------------- S7, S8, S9
def test_cmp_attn_kernel1_equals_dense_causal():
    T, h, hkv, d = 70, 4, 2, 16
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v = _rand((T, h, d), 18), _rand((T, hkv, d), 19), _rand((T, hkv, d), 20)
    o, _ = orc.cmp_attn(q, k, v, cu, kernel=1, stride=1)
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    assert torch.allclose(torch.from_numpy(o), _sdpa(_t(q), _t(k), _t(v), mask), atol=1e-12, rtol=0)


def test_cmp_attn_window_mask_via_sdpa():
    T, h, hkv, d = 300, 4, 2, 16
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v = _rand((T, h, d), 21), _rand((T, hkv, d), 22), _rand((T, hkv, d), 23)
    _, kc = orc.compress(k, cu)
    _, vc = orc.compress(v, cu)
    o, _ = orc.cmp_attn(q, kc, vc, cu)
    n_c = kc.shape[0]
    mask = (16 * torch.arange(n_c)[None, :] + 31) <= torch.arange(T)[:, None]
    live = mask.any(1)
    ref = _sdpa(_t(q)[live], _t(kc), _t(vc), mask[live])
    assert torch.allclose(torch.from_numpy(o)[live], ref, atol=1e-12, rtol=0)
    assert np.all(o[~live.numpy()] == 0)


@pytest.mark.parametrize("window", [1, 17, 64, 1000])
def test_swa_equals_banded_sdpa(window):
    T, h, hkv, d = 150, 4, 2, 16
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v = _rand((T, h, d), 24), _rand((T, hkv, d), 25), _rand((T, hkv, d), 26)
    o, _ = orc.swa(q, k, v, cu, window=window)
    t = torch.arange(T)
    mask = (t[:, None] >= t[None, :]) & (t[:, None] - t[None, :] < window)
    assert torch.allclose(torch.from_numpy(o), _sdpa(_t(q), _t(k), _t(v), mask), atol=1e-12, rtol=0)


def test_gate_combine_saturation_and_half():
    rng = np.random.default_rng(3)
    a, b, c = (rng.standard_normal((5, 2, 4)) for _ in range(3))
    sat = np.zeros((5, 2, 3), np.float32)
    sat[..., 0], sat[..., 1], sat[..., 2] = 60.0, -60.0, -60.0
    assert np.allclose(orc.gate_combine(a, b, c, sat), a, atol=1e-20, rtol=1e-15)
    half = np.zeros((5, 2, 3), np.float32)  # sigmoid(0) = 1/2
    assert np.allclose(orc.gate_combine(a, b, c, half), (a + b + c) / 2, atol=0, rtol=1e-15)


# --------------------------------------------------------------------------- S6 and the layer
def test_decode_equals_prefill_last_row():
    B, L, h, hkv, d = 3, 700, 4, 2, 16
    seqlens = np.array([700, 513, 64], np.int32)
    q = _rand((B, h, d), 27)
    kcache, vcache = _rand((B, L, hkv, d), 28), _rand((B, L, hkv, d), 29)
    ncs = orc.num_cmp(L)
    kc_cache = np.zeros((B, ncs, hkv, d), np.uint16)
    for b in range(B):
        _, kc = orc.compress(kcache[b, :seqlens[b]], [0, seqlens[b]])
        kc_cache[b, :len(kc)] = kc
    idx, o = orc.decode(q, kcache, vcache, kc_cache, seqlens, k=5)
    for b in range(B):
        Lb = int(seqlens[b])
        cu = np.array([0, Lb], np.int32)
        qf = np.zeros((Lb, h, d), np.uint16)
        qf[-1] = q[b]
        kb, vb = kcache[b, :Lb], vcache[b, :Lb]
        _, kc = orc.compress(kb, cu)
        sc = orc.cmp_scores_pool(qf, kc, cu, rows=[Lb - 1])
        ib = orc.topk(sc, cu, k=5, rows=[Lb - 1])
        assert np.array_equal(ib[0], idx[b])
        ob, _ = orc.sparse_attn(qf, kb, vb, np.repeat(ib, Lb, 0), cu, rows=[Lb - 1])
        assert np.allclose(ob[0], o[b], atol=1e-13, rtol=0)


def test_decode_all_blocks_is_dense_last_row():
    B, L, h, hkv, d = 2, 300, 4, 2, 16
    q = _rand((B, h, d), 30)
    kcache, vcache = _rand((B, L, hkv, d), 31), _rand((B, L, hkv, d), 32)
    kc_cache = np.zeros((B, orc.num_cmp(L), hkv, d), np.uint16)
    for b in range(B):
        kc_cache[b] = orc.compress(kcache[b], [0, L])[1]
    _, o = orc.decode(q, kcache, vcache, kc_cache, np.full(B, L, np.int32), k=64)
    for b in range(B):
        ref = _sdpa(_t(q[b:b + 1]), _t(kcache[b]), _t(vcache[b]), torch.ones(1, L, dtype=torch.bool))
        assert torch.allclose(torch.from_numpy(o[b:b + 1]), ref, atol=1e-12, rtol=0)


def test_layer_is_composition_of_branches():
    T, h, hkv, d = 400, 4, 2, 16
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v = _rand((T, h, d), 33), _rand((T, hkv, d), 34), _rand((T, hkv, d), 35)
    gates = np.random.default_rng(1).standard_normal((T, h, 3)).astype(np.float32)
    rows = [0, 31, 63, 64, 200, 399]
    out = orc.layer(q, k, v, gates, cu, S=4, window=100, rows=rows, branches=True)
    _, kc = orc.compress(k, cu)
    _, vc = orc.compress(v, cu)
    oc, _ = orc.cmp_attn(q, kc, vc, cu, rows=rows)
    sc = orc.cmp_scores_pool(q, kc, cu, rows=rows)
    idx = orc.topk(sc, cu, k=4, rows=rows)
    assert np.array_equal(idx, out["idx"])
    full_idx = np.full((T, hkv, 4), -1, np.int32)
    full_idx[rows] = idx
    os_, _ = orc.sparse_attn(q, k, v, full_idx, cu, rows=rows)
    ow, _ = orc.swa(q, k, v, cu, window=100, rows=rows)
    assert np.allclose(out["o_cmp"], oc, atol=1e-14, rtol=0)
    assert np.allclose(out["o_slc"], os_, atol=1e-14, rtol=0)
    assert np.allclose(out["o_swa"], ow, atol=1e-14, rtol=0)
    ref = orc.gate_combine(oc, os_, ow, gates[rows])
    assert np.allclose(out["o"], ref, atol=1e-14, rtol=0)


# --------------------------------------------------------------------------- input generator
def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]  # exact ties
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gen.f32_to_bf16_bits(x), ref)


def test_random_indices_structure():
    w = gen.prefill(B=2, T=1000)
    t = np.tile(np.arange(1000), 2)
    own = t // 64
    idx = w.idx[:, 0, :]
    for r in range(0, 2000, 37):
        row = idx[r]
        valid = row[row >= 0]
        assert np.all(np.diff(valid) > 0)
        assert valid.max() == own[r] and valid.min() == 0
        assert len(valid) == min(16, own[r] + 1)
        assert np.all(row[len(valid):] == -1)


# --------------------------------------------------------------------------- block-mask variant
def _token_mask(block_mask_bh, T, block, causal):
    """Expand one (batch, head) block mask to the token level by a Kronecker product."""
    m = np.kron(block_mask_bh, np.ones((block, block), np.uint8))[:T, :T].astype(bool)
    if causal:
        m &= np.tril(np.ones((T, T), bool))
    return torch.from_numpy(m)


@pytest.mark.parametrize("causal", [True, False])
def test_block_sparse_equals_masked_sdpa(causal):
    """Random 64x64 tile masks on ragged lengths: the oracle's key lists equal SDPA with
    the token-level mask built by expanding the tiles."""
    B, T, h, d, block = 2, 150, 3, 16, 64
    q, k, v = (_rand((B * T, h, d), s) for s in (61, 62, 63))
    mask = gen.block_mask(np.random.Generator(np.random.PCG64(64)), B, h, T, 0.5, causal, block)
    o, lse = orc.block_sparse_attn(q, k, v, mask, causal=causal, block=block)
    for b in range(B):
        sl = slice(b * T, (b + 1) * T)
        tm = torch.stack([_token_mask(mask[b, hh], T, block, causal) for hh in range(h)])  # [h, T, T]
        qt, kt, vt = (_t(a[sl]).permute(1, 0, 2) for a in (q, k, v))
        ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=tm).permute(1, 0, 2)
        assert torch.allclose(torch.from_numpy(o[sl]), ref, atol=1e-12, rtol=0)
        s = torch.einsum("htd,hsd->hts", qt, kt) * d ** -0.5
        ref_lse = torch.logsumexp(s.masked_fill(~tm, -torch.inf), -1).T
        assert torch.allclose(torch.from_numpy(lse[sl]), ref_lse, atol=1e-12, rtol=0)


def test_block_sparse_full_mask_is_dense_causal_and_empty_row_is_zero():
    B, T, h, d, block = 1, 130, 2, 8, 64
    q, k, v = (_rand((T, h, d), s) for s in (65, 66, 67))
    nb = -(-T // block)
    full = np.ones((B, h, nb, nb), np.uint8)
    o, _ = orc.block_sparse_attn(q, k, v, full, causal=True, block=block)
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    assert torch.allclose(torch.from_numpy(o), _sdpa(_t(q), _t(k), _t(v), mask), atol=1e-12, rtol=0)
    # non-causal: query block 1 of head 0 attends nothing -> zero output, lse -inf
    m = full.copy()
    m[0, 0, 1, :] = 0
    o2, lse2 = orc.block_sparse_attn(q, k, v, m, causal=False, block=block)
    assert np.all(o2[64:128, 0] == 0) and np.all(np.isneginf(lse2[64:128, 0]))
    assert np.all(np.isfinite(lse2[:64, 0])) and np.all(np.isfinite(lse2[:, 1]))


# --------------------------------------------------------------------------- S5 backward
def _bwd_lists(cu, hkv, bs, S, seed, dup=True):
    """Per (token, kv-head) lists: own block, random blocks (some non-causal), a -1 and,
    on every other token, a repeated entry."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(len(cu) - 1):
        L = int(cu[i + 1] - cu[i])
        nb = -(-L // bs)
        for t in range(L):
            per_g = []
            for _ in range(hkv):
                e = [t // bs] + list(rng.integers(0, nb, S - 2)) + [-1]
                if dup and t % 2:
                    e[-1] = e[1]
                per_g.append(e)
            rows.append(per_g)
    return np.asarray(rows, np.int32)


def _autograd_selected(q, k, v, do, idx, cu, bs, scale):
    """Selected attention written densely in float64 torch ops (logit + log multiplicity
    of each key in the token's expanded list), differentiated by autograd."""
    Q, K, V = (_t(a).requires_grad_(True) for a in (q, k, v))
    dO = _t(do)
    h, hkv = Q.shape[1], K.shape[1]
    r = h // hkv
    loss = 0.0
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        L = b - a
        mult = np.zeros((L, hkv, L))
        for t in range(L):
            for g in range(hkv):
                for j in idx[a + t, g]:
                    if j < 0 or j * bs > t:
                        continue
                    for tau in range(j * bs, min((j + 1) * bs, t + 1, L)):
                        mult[t, g, tau] += 1
        logm = torch.from_numpy(np.where(mult > 0, np.log(np.maximum(mult, 1)), -np.inf))
        logm = logm.repeat_interleave(r, dim=1)                          # [L, h, L]
        s = torch.einsum("thd,shd->ths", Q[a:b], K[a:b].repeat_interleave(r, 1)) * scale + logm
        p = torch.softmax(s, dim=-1)
        o = torch.einsum("ths,shd->thd", p, V[a:b].repeat_interleave(r, 1))
        loss = loss + (o * dO[a:b]).sum()
    loss.backward()
    return Q.grad, K.grad, V.grad


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sparse_bwd_equals_autograd(dtype):
    lengths = [150, 97]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d, bs, S = 4, 2, 16, 32, 5
    q, do = _rand((cu[-1], h, d), 31, dtype), _rand((cu[-1], h, d), 32, dtype)
    k, v = _rand((cu[-1], hkv, d), 33, dtype), _rand((cu[-1], hkv, d), 34, dtype)
    idx = _bwd_lists(cu, hkv, bs, S, 35)
    dq, dk, dv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs)
    gq, gk, gv = _autograd_selected(q, k, v, do, idx, cu, bs, d ** -0.5)
    for ours, ref in ((dq, gq), (dk, gk), (dv, gv)):
        assert torch.allclose(torch.from_numpy(ours), ref, atol=1e-12, rtol=1e-10)


def test_sparse_bwd_finite_differences():
    """Directional derivatives of sum(dO * o) through the (separately pinned) forward."""
    T, h, hkv, d, bs, S = 70, 2, 1, 8, 16, 3
    cu = gen.dense_cu_seqlens(1, T)
    q, k, v, do = (_rand((T, hh, d), s, "f32") for s, hh in ((41, h), (42, hkv), (43, hkv), (44, h)))
    idx = _bwd_lists(cu, hkv, bs, S, 45, dup=False)
    dq, dk, dv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs)
    rng = np.random.default_rng(46)
    eps = 1e-2

    def loss(qq, kk, vv):
        o, _ = orc.sparse_attn(qq, kk, vv, idx, cu, bs)
        return float((o * do.astype(np.float64)).sum())

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        args = [q, k, v]
        delta = rng.standard_normal(args[which].shape)
        plus, minus = list(args), list(args)
        plus[which] = (args[which] + eps * delta).astype(np.float32)
        minus[which] = (args[which] - eps * delta).astype(np.float32)
        step = plus[which].astype(np.float64) - minus[which].astype(np.float64)
        fd = loss(*plus) - loss(*minus)
        an = float((grad * step).sum())
        assert abs(fd - an) <= 1e-4 * max(1.0, abs(an)), (which, fd, an)


def test_sparse_bwd_invariants_and_sampling():
    """Per sequence and kv-head: the dK rows sum to zero (each row's ds sums to zero)
    and the dV rows sum to the dO of every row that has keys.  Requested subsets of
    rows equal the same rows of the full result."""
    lengths = [300, 129]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d, bs, S = 4, 2, 32, 32, 5
    q, do = _rand((cu[-1], h, d), 51), _rand((cu[-1], h, d), 52)
    k, v = _rand((cu[-1], hkv, d), 53), _rand((cu[-1], hkv, d), 54)
    idx = _bwd_lists(cu, hkv, bs, S, 55)
    dq, dk, dv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs)
    dof = gen.bf16_bits_to_f32(do).astype(np.float64)
    for i in range(len(lengths)):
        sl = slice(cu[i], cu[i + 1])
        for g in range(hkv):
            assert np.abs(dk[sl, g].sum(0)).max() < 1e-10
            want = dof[sl, 2 * g:2 * g + 2].sum((0, 1))  # every row lists its own block
            assert np.allclose(dv[sl, g].sum(0), want, atol=1e-10, rtol=0)
    qr = [0, 5, 149, 150, 428]
    kr = [1, 31, 32, 200, 299, 300, 301, 428]
    sq, sk, sv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs, q_rows=qr, kv_rows=kr)
    assert np.allclose(sq, dq[qr], atol=1e-13, rtol=0)
    assert np.allclose(sk, dk[kr], atol=1e-13, rtol=0) and np.allclose(sv, dv[kr], atol=1e-13, rtol=0)


def test_sparse_bwd_stored_output_reading():
    """D taken from a given forward output: with the exact output (fp32 here) it agrees
    with the exact D = sum_e p_e dp_e; a different output changes the result."""
    lengths = [130, 77]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d, bs, S = 4, 1, 16, 32, 4
    q, do = _rand((cu[-1], h, d), 61, "f32"), _rand((cu[-1], h, d), 62, "f32")
    k, v = _rand((cu[-1], hkv, d), 63, "f32"), _rand((cu[-1], hkv, d), 64, "f32")
    idx = _bwd_lists(cu, hkv, bs, S, 65, dup=False)
    o, _ = orc.sparse_attn(q, k, v, idx, cu, bs)
    exact = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs)
    stored = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs, o=o.astype(np.float32))
    for a, b in zip(exact, stored):
        assert np.allclose(a, b, atol=1e-6, rtol=1e-5)
    off = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs, o=np.zeros_like(q))
    assert not np.allclose(off[0], exact[0], atol=1e-3)


# --------------------------------------------------------------------------- NOSA stage 2
def test_cis_block_scores_equal_two_avg_pools():
    """Windows: avg_pool1d(32, 16) of each sequence's CIS; blocks: avg_pool1d(3, 4,
    ceil_mode) of the windows (the S3 rule), zero where a block holds no window."""
    lengths = [10, 31, 32, 47, 100, 700, 1001]
    cu = gen.varlen_cu_seqlens(lengths)
    cis = gen.cis_scores(np.random.default_rng(71), int(cu[-1]), 2)
    got = orc.cis_block_scores(cis, cu)
    nb = got.shape[2]
    for i, L in enumerate(lengths):
        for g in range(2):
            x = torch.from_numpy(cis[cu[i]:cu[i + 1], g].astype(np.float64)).view(1, 1, -1)
            ref = np.zeros(nb)
            if L >= 32:
                win = F.avg_pool1d(x, 32, 16)
                r = F.avg_pool1d(win, 3, 4, ceil_mode=True).flatten().numpy()
                ref[:len(r)] = r
            assert np.allclose(got[i, g], ref, atol=1e-14, rtol=0), (L, g)


def test_cis_block_scores_ramp_hand_values():
    """cis[t] = t: window c averages 16c .. 16c+31 = 16c + 15.5; a full block j averages
    windows 4j, 4j+1, 4j+2, i.e. 64j + 31.5."""
    L = 256
    cis = np.arange(L, dtype=np.float64)[:, None]
    got = orc.cis_block_scores(cis, gen.dense_cu_seqlens(1, L))[0, 0]
    assert np.allclose(got, [31.5, 95.5, 159.5, 223.5], atol=1e-12)


def _brute_two_stage(sc, cs, t, bs, n_init, n_local, qk, k):
    own = t // bs
    forced = lambda j: j < n_init or j > own - n_local  # noqa: E731
    key1 = lambda j: (-(np.inf if forced(j) else sc[j]), j)  # noqa: E731
    first = sorted(range(own + 1), key=key1)[:qk]
    key2 = lambda j: (-(np.inf if forced(j) else cs[j]), j)  # noqa: E731
    pick = sorted(sorted(first, key=key2)[:k])
    return pick + [-1] * (k - len(pick))


@pytest.mark.parametrize("qk,k", [(8, 4), (16, 16), (6, 3), (40, 16)])
def test_topk_two_stage_brute_force_and_reductions(qk, k):
    rng = np.random.default_rng(qk * 100 + k)
    lengths = [700, 2000, 64, 1]
    cu = gen.varlen_cu_seqlens(lengths)
    nb = 32
    sc = np.round(rng.random((int(cu[-1]), 2, nb)) * 8) / 8          # many exact ties
    cs = np.round(rng.random((len(lengths), 2, nb)) * 8) / 8
    got = orc.topk_two_stage(sc, cs, cu, qk, k)
    for i in range(len(lengths)):
        for t in range(lengths[i]):
            for g in range(2):
                want = _brute_two_stage(sc[cu[i] + t, g], cs[i, g], t, 64, 1, 2, qk, k)
                assert got[cu[i] + t, g].tolist() == want
    # qk_select = k: stage 2 keeps stage 1's choice
    assert np.array_equal(orc.topk_two_stage(sc, cs, cu, k, k), orc.topk(sc, cu, 64, 1, 2, k))
    # stage 1 keeps every causal block: the choice is S4 on the CIS scores of the sequence
    per_row = np.concatenate([np.repeat(cs[i][None], lengths[i], 0) for i in range(len(lengths))])
    assert np.array_equal(orc.topk_two_stage(sc, cs, cu, nb, k), orc.topk(per_row, cu, 64, 1, 2, k))


def _cis_case(dtype, seed):
    lengths = [150, 64, 33]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d, bs = 4, 2, 16, 32
    q, k, v = (_rand((cu[-1], hh, d), seed + i, dtype) for i, hh in enumerate((h, hkv, hkv)))
    idx = _bwd_lists(cu, hkv, bs, 4, seed + 5)
    cis = gen.cis_scores(np.random.default_rng(seed + 6), int(cu[-1]), hkv)
    return lengths, cu, q, k, v, idx, cis, bs


def test_sparse_cis_unit_weights_and_pages_construction():
    """cis = 1 gives the plain selected attention; otherwise the output equals the pages'
    recipe: attention of v * cis divided by attention of ones * cis."""
    lengths, cu, q, k, v, idx, cis, bs = _cis_case("f32", 80)
    o1, l1 = orc.sparse_attn_cis(q, k, v, np.ones_like(cis), idx, cu, bs)
    o0, l0 = orc.sparse_attn(q, k, v, idx, cu, bs)
    assert np.allclose(o1, o0, atol=1e-13) and np.allclose(l1, l0, atol=1e-13)
    o, _ = orc.sparse_attn_cis(q, k, v, cis, idx, cu, bs)
    vs = (v * cis[:, :, None]).astype(np.float32)
    ones = np.repeat(cis[:, :, None], v.shape[2], 2).astype(np.float32)
    num, _ = orc.sparse_attn(q, k, vs, idx, cu, bs)
    den, _ = orc.sparse_attn(q, k, ones, idx, cu, bs)
    assert np.allclose(o, num / den, atol=1e-6, rtol=1e-6)


def test_sparse_cis_equals_sdpa_with_log_weight_bias():
    """Weights p * cis = softmax(s + log cis): SDPA with a float mask (log cis on the listed
    keys, times their multiplicity; -inf elsewhere)."""
    lengths, cu, q, k, v, idx, cis, bs = _cis_case("bf16", 90)
    o, lse = orc.sparse_attn_cis(q, k, v, cis, idx, cu, bs)
    h, hkv, d = q.shape[1], k.shape[1], q.shape[2]
    for i, L in enumerate(lengths):
        a = int(cu[i])
        for g in range(hkv):
            mult = np.zeros((L, L))
            for t in range(L):
                for j in idx[a + t, g]:
                    if j < 0 or j * bs > t:
                        continue
                    for tau in range(j * bs, min((j + 1) * bs, t + 1)):
                        mult[t, tau] += 1
            bias = np.where(mult > 0, np.log(np.maximum(mult, 1)) + np.log(cis[a:a + L, g].astype(np.float64))[None, :],
                            -np.inf)
            heads = slice(g * (h // hkv), (g + 1) * (h // hkv))
            qq = _t(q[a:a + L, heads]).permute(1, 0, 2)
            kk = _t(k[a:a + L, g:g + 1]).permute(1, 0, 2).expand(h // hkv, L, d)
            vv = _t(v[a:a + L, g:g + 1]).permute(1, 0, 2).expand(h // hkv, L, d)
            ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=torch.from_numpy(bias)).permute(1, 0, 2)
            assert torch.allclose(torch.from_numpy(o[a:a + L, heads]), ref, atol=1e-12, rtol=0)
            s = torch.einsum("hld,hmd->hlm", qq, kk) * d ** -0.5 + torch.from_numpy(bias)
            assert torch.allclose(torch.from_numpy(lse[a:a + L, heads]).T, torch.logsumexp(s, -1), atol=1e-12)


def test_sparse_cis_zero_weights_give_zero():
    lengths, cu, q, k, v, idx, cis, bs = _cis_case("f32", 100)
    o, lse = orc.sparse_attn_cis(q, k, v, np.zeros_like(cis), idx, cu, bs)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


# --------------------------------------------------------------------------- S7 and S1 backward
def _cmp_case(dtype, seed, lengths=(150, 97, 20), h=4, hkv=2, d=16):
    cu = gen.varlen_cu_seqlens(list(lengths))
    q, do = _rand((cu[-1], h, d), seed, dtype), _rand((cu[-1], h, d), seed + 1, dtype)
    n_cmp = int(orc.cmp_offsets(cu)[-1])
    kc, vc = _rand((n_cmp, hkv, d), seed + 2, dtype), _rand((n_cmp, hkv, d), seed + 3, dtype)
    return list(lengths), cu, q, do, kc, vc


def _autograd_cmp(q, kc, vc, do, cu, scale):
    Q, K, V = (_t(a).requires_grad_(True) for a in (q, kc, vc))
    dO = _t(do)
    h, hkv = Q.shape[1], K.shape[1]
    r = h // hkv
    off = orc.cmp_offsets(cu)
    loss = 0.0
    for i in range(len(cu) - 1):
        a, L = int(cu[i]), int(cu[i + 1] - cu[i])
        n_c = orc.num_cmp(L)
        if n_c == 0:
            continue
        kk = K[off[i]:off[i] + n_c].repeat_interleave(r, 1)
        vv = V[off[i]:off[i] + n_c].repeat_interleave(r, 1)
        t = torch.arange(31, L)                      # rows with at least one causal window
        ok = (torch.arange(n_c)[None, :] * 16 + 31) <= t[:, None]
        s = torch.einsum("thd,chd->thc", Q[a + 31:a + L], kk) * scale
        s = s.masked_fill(~ok[:, None, :], -torch.inf)
        o = torch.einsum("thc,chd->thd", torch.softmax(s, -1), vv)
        loss = loss + (o * dO[a + 31:a + L]).sum()
    loss.backward()
    return Q.grad, K.grad, V.grad


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cmp_attn_bwd_equals_autograd(dtype):
    lengths, cu, q, do, kc, vc = _cmp_case(dtype, 121)
    dq, dkc, dvc = orc.cmp_attn_bwd(q, kc, vc, do, cu)
    gq, gk, gv = _autograd_cmp(q, kc, vc, do, cu, 16 ** -0.5)
    for ours, ref in ((dq, gq), (dkc, gk), (dvc, gv)):
        assert torch.allclose(torch.from_numpy(ours), ref, atol=1e-12, rtol=1e-10)


def test_cmp_attn_bwd_finite_differences_invariants_and_rows():
    lengths, cu, q, do, kc, vc = _cmp_case("f32", 131, lengths=(120, 64))
    dq, dkc, dvc = orc.cmp_attn_bwd(q, kc, vc, do, cu)
    rng = np.random.default_rng(132)
    eps = 1e-2

    def loss(qq, kk, vv):
        o, _ = orc.cmp_attn(qq, kk, vv, cu)
        return float((o * do.astype(np.float64)).sum())

    for which, grad in ((0, dq), (1, dkc), (2, dvc)):
        args = [q, kc, vc]
        delta = rng.standard_normal(args[which].shape)
        plus, minus = list(args), list(args)
        plus[which] = (args[which] + eps * delta).astype(np.float32)
        minus[which] = (args[which] - eps * delta).astype(np.float32)
        step = plus[which].astype(np.float64) - minus[which].astype(np.float64)
        fd = loss(*plus) - loss(*minus)
        an = float((grad * step).sum())
        assert abs(fd - an) <= 1e-4 * max(1.0, abs(an)), (which, fd, an)
    off = orc.cmp_offsets(cu)
    for i, L in enumerate(lengths):
        sl = slice(off[i], off[i + 1])
        for g in range(2):
            assert np.abs(dkc[sl, g].sum(0)).max() < 1e-10
            rows = slice(cu[i] + 31, cu[i + 1])          # rows with at least one causal window
            assert np.allclose(dvc[sl, g].sum(0), do[rows, 2 * g:2 * g + 2].astype(np.float64).sum((0, 1)),
                               atol=1e-10, rtol=0)
    qr, kr = [0, 30, 31, 100, 183], [0, 3, 5, 8]
    sq, sk, sv = orc.cmp_attn_bwd(q, kc, vc, do, cu, q_rows=qr, kv_rows=kr)
    assert np.allclose(sq, dq[qr], atol=1e-13) and np.allclose(sk, dkc[kr], atol=1e-13)
    assert np.allclose(sv, dvc[kr], atol=1e-13)


def test_compress_bwd_is_the_adjoint_of_compress():
    """<compress(x), y> = <x, compress_bwd(y)> for every x, y (exact means), and it equals
    autograd of avg_pool1d(32, 16) per sequence."""
    lengths = [10, 31, 32, 47, 100, 333]
    cu = gen.varlen_cu_seqlens(lengths)
    x = _rand((cu[-1], 2, 8), 141, "f32")
    xe, _ = orc.compress(x, cu)
    y = np.random.default_rng(142).standard_normal(xe.shape)
    gx = orc.compress_bwd(y, cu)
    assert abs(float((xe * y).sum()) - float((x.astype(np.float64) * gx).sum())) < 1e-9
    off = orc.cmp_offsets(cu)
    for i, L in enumerate(lengths):
        X = torch.from_numpy(x[cu[i]:cu[i + 1]].astype(np.float64)).permute(1, 2, 0).requires_grad_(True)
        if L < 32:
            assert np.all(gx[cu[i]:cu[i + 1]] == 0)
            continue
        P = F.avg_pool1d(X.reshape(1, -1, L), 32, 16).reshape(2, 8, -1)
        (P * torch.from_numpy(y[off[i]:off[i + 1]]).permute(1, 2, 0)).sum().backward()
        assert torch.allclose(X.grad.permute(2, 0, 1), torch.from_numpy(gx[cu[i]:cu[i + 1]]), atol=1e-14)


# --------------------------------------------------------------------------- S8 and S9 backward
@pytest.mark.parametrize("window", [1, 17, 64, 1000])
def test_swa_bwd_equals_autograd(window):
    lengths = [150, 97, 20]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d = 4, 2, 16
    q, do = _rand((cu[-1], h, d), 151, "bf16"), _rand((cu[-1], h, d), 152, "bf16")
    k, v = _rand((cu[-1], hkv, d), 153, "bf16"), _rand((cu[-1], hkv, d), 154, "bf16")
    dq, dk, dv = orc.swa_bwd(q, k, v, do, cu, window)
    Q, K, V = (_t(a).requires_grad_(True) for a in (q, k, v))
    loss = 0.0
    for i, L in enumerate(lengths):
        a = int(cu[i])
        t = torch.arange(L)
        mask = (t[:, None] >= t[None, :]) & (t[:, None] - t[None, :] < window)
        loss = loss + (_sdpa(Q[a:a + L], K[a:a + L], V[a:a + L], mask) * _t(do[a:a + L])).sum()
    loss.backward()
    for ours, ref in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
        assert torch.allclose(torch.from_numpy(ours), ref, atol=1e-12, rtol=1e-10)
    # row subsets and the stored-output reading with the exact output
    o, _ = orc.swa(q, k, v, cu, window)
    sq, sk, sv = orc.swa_bwd(q, k, v, do, cu, window, q_rows=[0, 5, 200], kv_rows=[1, 149, 260])
    assert np.allclose(sq, dq[[0, 5, 200]], atol=1e-13) and np.allclose(sk, dk[[1, 149, 260]], atol=1e-13)
    assert np.allclose(sv, dv[[1, 149, 260]], atol=1e-13)


def test_gate_bwd_equals_autograd():
    rng = np.random.default_rng(161)
    n, h, d = 37, 4, 8
    br = [rng.standard_normal((n, h, d)) for _ in range(3)]
    gates = (rng.standard_normal((n, h, 3)) * 3).astype(np.float32)
    do = rng.standard_normal((n, h, d))
    got = orc.gate_bwd(*br, gates, do)
    B = [torch.from_numpy(b).requires_grad_(True) for b in br]
    A = torch.from_numpy(gates.astype(np.float64)).requires_grad_(True)
    o = sum(torch.sigmoid(A[..., i:i + 1]) * B[i] for i in range(3))
    (o * torch.from_numpy(do)).sum().backward()
    for i in range(3):
        assert torch.allclose(torch.from_numpy(got[i]), B[i].grad, atol=1e-14)
    assert torch.allclose(torch.from_numpy(got[3]), A.grad, atol=1e-13)


# --------------------------------------------------------------------------- layer backward
def test_layer_bwd_equals_autograd_of_the_layer():
    """The whole layer written in float64 torch ops (avg_pool1d compression, window-masked
    compressed attention, the selected attention on fixed lists, the banded window, the
    sigmoid gates), differentiated by autograd, against the oracle's composition of branch
    backwards (fp32 inputs: the stored compressed keys and branch gradients round to fp32)."""
    lengths = [130, 97]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d, bs, S, win = 4, 2, 16, 64, 3, 40
    q, do = _rand((cu[-1], h, d), 171, "f32"), _rand((cu[-1], h, d), 172, "f32")
    k, v = _rand((cu[-1], hkv, d), 173, "f32"), _rand((cu[-1], hkv, d), 174, "f32")
    gates = np.random.default_rng(175).standard_normal((int(cu[-1]), h, 3)).astype(np.float32)
    idx = gen.random_block_indices(np.random.default_rng(176), cu, hkv, S, bs, force_first=True)
    dq, dk, dv, dg = orc.layer_bwd(q, k, v, gates, idx, do, cu, 32, 16, bs, win)
    Q, K, V, A = (_t(a).requires_grad_(True) for a in (q, k, v, gates))
    r, scale = h // hkv, d ** -0.5
    loss = 0.0
    for i, L in enumerate(lengths):
        a = int(cu[i])
        qq, kk, vv, aa = Q[a:a + L], K[a:a + L], V[a:a + L], A[a:a + L]
        t = torch.arange(L)
        # compressed branch
        kc = F.avg_pool1d(kk.permute(1, 2, 0), 32, 16).permute(2, 0, 1)  # [n_c, hkv, d]
        vc = F.avg_pool1d(vv.permute(1, 2, 0), 32, 16).permute(2, 0, 1)
        n_c = kc.shape[0]
        ok = (torch.arange(n_c)[None, :] * 16 + 31) <= t[:, None]
        s = torch.einsum("thd,chd->thc", qq, kc.repeat_interleave(r, 1)) * scale
        s = s.masked_fill(~ok[:, None, :], -torch.inf)
        p = torch.softmax(s[31:], -1)
        o_cmp = torch.cat([torch.zeros(31, h, d, dtype=F64),
                           torch.einsum("thc,chd->thd", p, vc.repeat_interleave(r, 1))])
        # selected branch on the fixed lists
        mult = np.zeros((L, hkv, L))
        for tt in range(L):
            for g in range(hkv):
                for j in idx[a + tt, g]:
                    if j < 0 or j * bs > tt:
                        continue
                    for tau in range(j * bs, min((j + 1) * bs, tt + 1)):
                        mult[tt, g, tau] += 1
        logm = torch.from_numpy(np.where(mult > 0, np.log(np.maximum(mult, 1)), -np.inf)).repeat_interleave(r, 1)
        s2 = torch.einsum("thd,shd->ths", qq, kk.repeat_interleave(r, 1)) * scale + logm
        o_slc = torch.einsum("ths,shd->thd", torch.softmax(s2, -1), vv.repeat_interleave(r, 1))
        # sliding window
        band = (t[:, None] >= t[None, :]) & (t[:, None] - t[None, :] < win)
        o_swa = _sdpa(qq, kk, vv, band)
        g = torch.sigmoid(aa)
        o = g[..., 0:1] * o_cmp + g[..., 1:2] * o_slc + g[..., 2:3] * o_swa
        loss = loss + (o * _t(do[a:a + L])).sum()
    loss.backward()
    for ours, ref, what in ((dq, Q.grad, "dq"), (dk, K.grad, "dk"), (dv, V.grad, "dv"), (dg, A.grad, "dgate")):
        assert torch.allclose(torch.from_numpy(ours), ref, atol=2e-6, rtol=1e-5), what


def test_decode_cis_reductions():
    """cis = 1 and qk_select = k reduce the NOSA decode step to the plain decode step; with
    qk_select covering every causal block the choice is S4 on the CIS block scores."""
    w = gen.decode(B=3, L=1500, seqlens=[1500, 700, 90], topk=8, H=8, HKV=2)
    ncs = orc.num_cmp(1500)
    kc = np.zeros((3, ncs, 2, 128), np.uint16)
    for b in range(3):
        kc[b] = orc.compress(w.k_cache[b], [0, 1500])[1]
    ones = np.ones((3, 1500, 2), np.float32)
    i0, o0 = orc.decode(w.q, w.k_cache, w.v_cache, kc, w.seqlens, k=8)
    i1, o1, _ = orc.decode_cis(w.q, w.k_cache, w.v_cache, kc, ones, w.seqlens, 8, k=8)
    assert np.array_equal(i0, i1) and np.allclose(o0, o1, atol=1e-12)
    cis = gen.cis_scores(np.random.default_rng(181), 3 * 1500, 2).reshape(3, 1500, 2)
    i2, _, _ = orc.decode_cis(w.q, w.k_cache, w.v_cache, kc, cis, w.seqlens, 64, k=8)
    for b, L in enumerate([1500, 700, 90]):
        cs = orc.cis_block_scores(cis[b, :L], np.array([0, L], np.int32), nb_stride=24)
        want = orc.topk(cs[0][None], np.array([0, L], np.int32), 64, 1, 2, 8, rows=[L - 1])[0]
        assert np.array_equal(i2[b], want)
