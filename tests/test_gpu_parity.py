"""GPU parity: every kernel through the C ABI against the CPU oracle on the same
seeded inputs.  Indices bit-exact (top-k on identical scores) or within the tie band
(fused selection); outputs within |gpu - oracle| <= 1e-2 + 1e-2|oracle|.
"""
import numpy as np
import pytest
import torch

import sparse_attention_compress_gb300 as nsa
from oracle import oracle as orc
from sparse_attention_compress_gb300 import inputs as gen
from tests.parity import as_f64, assert_close, dev, host, pinned, selection_mismatches

pytestmark = pytest.mark.gpu


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _t_of_rows(cu):
    cu = np.asarray(cu)
    return np.concatenate([np.arange(cu[i + 1] - cu[i]) for i in range(len(cu) - 1)])


# --------------------------------------------------------------------------- S1
@pytest.mark.parametrize("dtype,hkv,d,kernel,stride", [
    ("bf16", 2, 128, 32, 16), ("bf16", 4, 128, 32, 16), ("bf16", 1, 64, 16, 16), ("bf16", 2, 128, 64, 16),
    ("f32", 1, 64, 32, 16)])
def test_compress(dtype, hkv, d, kernel, stride):
    lengths = [1, 31, 32, 100, 1000, 4097]
    cu = gen.varlen_cu_seqlens(lengths)
    k = gen.normal(_rng(1), (cu[-1], hkv, d), dtype)
    exact, rounded = orc.compress(k, cu, kernel, stride)
    out = nsa.nsa_compress_k(dev(k), kernel, stride, cu_seqlens=dev(cu), max_seqlen=max(lengths))
    torch.cuda.synchronize()
    g = host(out)
    assert g.shape == rounded.shape
    # the mean of bf16 inputs in fp32 rounds to the same bf16 as the exact mean except
    # at a rounding tie boundary: allow one unit in the last place there
    assert_close(out, exact, atol=1e-6, rtol=2 ** -7, what="compress")
    if dtype == "bf16":
        same = np.mean(g == rounded)
        assert same > 0.999, same


def test_compress_dense_batch_layout():
    B, T, hkv, d = 3, 1000, 2, 128
    k = gen.normal(_rng(2), (B * T, hkv, d), "bf16")
    _, rounded = orc.compress(k, gen.dense_cu_seqlens(B, T))
    out = nsa.nsa_compress_k(dev(k).view(B, T, hkv, d))
    torch.cuda.synchronize()
    assert np.mean(host(out) == rounded) > 0.999


# --------------------------------------------------------------------------- S2+S3
@pytest.mark.parametrize("H,hkv,d", [(16, 2, 128), (16, 1, 128), (8, 2, 64), (4, 4, 128), (8, 4, 128)])
def test_cmp_scores_pool(H, hkv, d):
    lengths = [40, 700, 3001, 64]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(3)
    q = gen.normal(rng, (cu[-1], H, d), "bf16")
    k = gen.normal(rng, (cu[-1], hkv, d), "bf16")
    _, kc = orc.compress(k, cu)
    nb = -(-max(lengths) // 64) + 3
    ref = orc.cmp_scores_pool(q, kc, cu, nb_stride=nb)
    out = nsa.nsa_cmp_scores_pool(dev(q), dev(kc), hkv, cu_seqlens=dev(cu), max_seqlen=max(lengths), nb_stride=nb)
    torch.cuda.synchronize()
    g = host(out).astype(np.float64)
    assert np.all(g[ref == 0] == 0)
    np.testing.assert_allclose(g, ref, rtol=1e-4, atol=1e-9)


@pytest.mark.parametrize("B,T,H,hkv", [(2, 1000, 16, 1), (3, 4100, 32, 4), (1, 31, 16, 2)])
def test_cmp_scores_pool_dense(B, T, H, hkv):
    """Dense layout: the compressed-key buffer holds exactly B * n_c(T) rows, so the last
    64-key tile of the last sequence reaches past it (read with bounds checks)."""
    d = 128
    cu = gen.dense_cu_seqlens(B, T)
    rng = _rng(31)
    q = gen.normal(rng, (B * T, H, d), "bf16")
    k = gen.normal(rng, (B * T, hkv, d), "bf16")
    _, kc = orc.compress(k, cu)
    ref = orc.cmp_scores_pool(q, kc, cu)
    kcd = dev(kc).view(B, -1, hkv, d) if kc.shape[0] else None
    out = nsa.nsa_cmp_scores_pool(dev(q).view(B, T, H, d), kcd, hkv)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    g = host(out).astype(np.float64).reshape(ref.shape)
    assert np.all(g[ref == 0] == 0)
    np.testing.assert_allclose(g, ref, rtol=1e-4, atol=1e-9)


def test_cmp_scores_pool_with_given_normaliser():
    lengths = [1200, 333]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(4)
    H, hkv, d = 16, 1, 128
    q, k, v = (gen.normal(rng, (cu[-1], hh, d), "bf16") for hh in (H, hkv, hkv))
    _, kc = orc.compress(k, cu)
    _, vc = orc.compress(v, cu)
    dcu = dev(cu)
    lse = torch.empty((cu[-1], H), dtype=torch.float32, device="cuda")
    nsa.nsa_cmp_attn_fwd(dev(q), dev(kc), dev(vc), hkv, cu_seqlens=dcu, max_seqlen=1200, lse=lse)
    a = nsa.nsa_cmp_scores_pool(dev(q), dev(kc), hkv, cu_seqlens=dcu, max_seqlen=1200, lse_in=lse)
    b = nsa.nsa_cmp_scores_pool(dev(q), dev(kc), hkv, cu_seqlens=dcu, max_seqlen=1200)
    torch.cuda.synchronize()
    ref = orc.cmp_scores_pool(q, kc, cu)
    np.testing.assert_allclose(host(a), ref, rtol=1e-4, atol=1e-9)
    np.testing.assert_allclose(host(b), ref, rtol=1e-4, atol=1e-9)


# --------------------------------------------------------------------------- S4
@pytest.mark.parametrize("nb_stride,k,n_init,n_local,levels", [
    (40, 16, 1, 2, 0), (40, 16, 1, 2, 3), (129, 7, 0, 0, 5), (512, 64, 1, 2, 0), (1024, 16, 2, 1, 4),
    (2048, 64, 1, 2, 0), (3, 1, 1, 2, 0), (64, 64, 0, 0, 2), (1024, 16, 1, 2, 0), (2048, 32, 1, 2, 0),
    (256, 32, 0, 0, 50), (1024, 16, 1, 2, 1000)])
def test_topk_bit_exact(nb_stride, k, n_init, n_local, levels):
    bs = 64
    max_len = nb_stride * bs
    lengths = [max_len, max(1, max_len // 3), 77]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(5 + k)
    sc = rng.random((cu[-1], 2, nb_stride), dtype=np.float32)
    if levels:
        sc = np.floor(sc * levels).astype(np.float32) / levels  # exact ties
    ref = orc.topk(sc, cu, bs, n_init, n_local, k)
    out = nsa.nsa_topk_select(dev(sc), k, bs, n_init, n_local, cu_seqlens=dev(cu), max_seqlen=max_len)
    torch.cuda.synchronize()
    assert np.array_equal(host(out), ref)


# --------------------------------------------------------------------------- S5
def test_sparse_fwd_tiny_fp32():
    w = gen.tiny()
    ref, lse_ref = orc.sparse_attn(w.q, w.k, w.v, w.idx, w.cu_seqlens, w.block_size)
    lse = torch.empty((w.tokens, w.h), dtype=torch.float32, device="cuda")
    out = nsa.nsa_sparse_fwd(dev(w.q).view(1, 256, 4, 64), dev(w.k), dev(w.v), dev(w.idx), w.block_size, lse=lse)
    torch.cuda.synchronize()
    err = assert_close(out.reshape(w.tokens, w.h, w.d), ref, what="tiny fp32")
    assert err < 1e-5
    assert_close(lse, lse_ref, atol=1e-5, rtol=1e-5, what="tiny lse")


@pytest.mark.parametrize("H,hkv,d,bs,S", [(16, 1, 128, 64, 16), (16, 2, 128, 64, 8), (8, 1, 64, 32, 6),
                                          (32, 1, 128, 64, 5), (4, 2, 128, 16, 9), (12, 1, 128, 64, 16)])
def test_sparse_fwd_bf16_varlen(H, hkv, d, bs, S):
    lengths = [1, 63, 64, 65, 900, 2000]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(6)
    q, k, v = (gen.normal(rng, (cu[-1], hh, d), "bf16") for hh in (H, hkv, hkv))
    idx = gen.random_block_indices(rng, cu, hkv, S, bs, force_first=True)
    ref, lse_ref = orc.sparse_attn(q, k, v, idx, cu, bs)
    lse = torch.empty((cu[-1], H), dtype=torch.float32, device="cuda")
    out = nsa.nsa_sparse_fwd(dev(q), dev(k), dev(v), dev(idx), bs, cu_seqlens=dev(cu), max_seqlen=max(lengths),
                             lse=lse)
    torch.cuda.synchronize()
    assert_close(out, ref, what="sparse bf16")
    assert_close(lse, lse_ref, atol=1e-3, rtol=1e-3, what="sparse lse")


def test_sparse_fwd_edge_lists():
    """-1 padding, non-causal entries, duplicates and empty lists."""
    T, H, hkv, d, bs = 300, 16, 1, 128, 64
    cu = gen.dense_cu_seqlens(1, T)
    rng = _rng(7)
    q, k, v = (gen.normal(rng, (T, hh, d), "bf16") for hh in (H, hkv, hkv))
    t = np.arange(T)
    idx = np.stack([t // bs, np.full(T, -1), np.full(T, 3), np.zeros(T), np.zeros(T)], 1).astype(np.int32)
    idx[:10] = -1  # empty lists -> zero output
    idx = idx[:, None, :]
    ref, _ = orc.sparse_attn(q, k, v, idx, cu, bs)
    out = nsa.nsa_sparse_fwd(dev(q), dev(k), dev(v), dev(idx), bs)
    torch.cuda.synchronize()
    assert_close(out, ref, what="edge lists")
    assert np.all(as_f64(host(out))[:10] == 0)


def test_sparse_fwd_prefill_full_size_sampled():
    """B=8, T=16384, H=16, Hkv=1, d=128, block 64, S=16 (the benchmark launch);
    oracle on sampled rows, including first/last tokens of every sequence."""
    w = gen.prefill()
    out = nsa.nsa_sparse_fwd(dev(w.q).view(8, 16384, 16, 128), dev(w.k), dev(w.v), dev(w.idx), 64)
    torch.cuda.synchronize()
    rng = _rng(8)
    rows = np.unique(np.concatenate([rng.integers(0, w.tokens, 400), np.arange(8) * 16384,
                                     np.arange(1, 9) * 16384 - 1, [63, 64, 65, 16383 + 64]]))
    ref, _ = orc.sparse_attn(w.q, w.k, w.v, w.idx, w.cu_seqlens, 64, rows=rows)
    g = out.reshape(w.tokens, 16, 128)[torch.from_numpy(rows).cuda()]
    assert_close(g, ref, what="prefill sampled")


# --------------------------------------------------------------------------- S5 backward
# The backward takes the forward's stored output o (bf16) and lse; D = dO . o comes from
# that o.  Both sides get the oracle's own forward (o rounded to bf16, lse in fp32), so
# the comparison covers the backward alone.
def _oracle_fwd_inputs(q, k, v, idx, cu, rows=None, bs=64):
    o64, lse64 = orc.sparse_attn(q, k, v, idx, cu, bs, rows=rows)
    return gen.f32_to_bf16_bits(o64.astype(np.float32)), lse64.astype(np.float32)


def _sparse_bwd_gpu(q, k, v, idx, o, lse, do, cu, max_len, bs=64):
    gq, gk, gv = nsa.nsa_sparse_bwd(dev(q), dev(k), dev(v), dev(idx), dev(o), dev(lse), dev(do), bs,
                                    cu_seqlens=dev(cu), max_seqlen=max_len)
    torch.cuda.synchronize()
    return gq, gk, gv


@pytest.mark.parametrize("H,hkv,S", [(16, 1, 4), (8, 2, 8), (4, 4, 3), (16, 2, 6)])
def test_sparse_bwd_varlen(H, hkv, S):
    """Ragged lengths: single-token sequences, block edges, and sequences spanning two and
    three 2048-query chunks (several dK/dV partials per block)."""
    lengths = [1, 63, 64, 65, 700, 2100, 4200]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(21)
    q, do = gen.normal(rng, (cu[-1], H, 128), "bf16"), gen.normal(rng, (cu[-1], H, 128), "bf16")
    k, v = gen.normal(rng, (cu[-1], hkv, 128), "bf16"), gen.normal(rng, (cu[-1], hkv, 128), "bf16")
    idx = gen.random_block_indices(rng, cu, hkv, S, 64, force_first=True)
    o, lse = _oracle_fwd_inputs(q, k, v, idx, cu)
    gq, gk, gv = _sparse_bwd_gpu(q, k, v, idx, o, lse, do, cu, max(lengths))
    assert nsa.nsa_device_status() == 0
    rq, rk, rv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, 64, o=o)
    assert_close(gq, rq, what="dq")
    assert_close(gk, rk, what="dk")
    assert_close(gv, rv, what="dv")


def test_sparse_bwd_edge_lists_and_determinism():
    """-1 padding, non-causal entries, duplicates (count twice) and empty lists (no
    gradient); two runs give identical bits."""
    T, H, hkv, bs = 300, 16, 1, 64
    cu = gen.dense_cu_seqlens(1, T)
    rng = _rng(22)
    q, do = gen.normal(rng, (T, H, 128), "bf16"), gen.normal(rng, (T, H, 128), "bf16")
    k, v = gen.normal(rng, (T, hkv, 128), "bf16"), gen.normal(rng, (T, hkv, 128), "bf16")
    t = np.arange(T)
    idx = np.stack([t // bs, np.full(T, -1), np.full(T, 3), np.zeros(T), np.zeros(T)], 1).astype(np.int32)
    idx[:10] = -1
    idx = idx[:, None, :]
    o, lse = _oracle_fwd_inputs(q, k, v, idx, cu)
    gq, gk, gv = _sparse_bwd_gpu(q, k, v, idx, o, lse, do, cu, T)
    rq, rk, rv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, bs, o=o)
    assert_close(gq, rq, what="dq edge")
    assert_close(gk, rk, what="dk edge")
    assert_close(gv, rv, what="dv edge")
    assert np.all(as_f64(host(gq))[:10] == 0)
    g2 = _sparse_bwd_gpu(q, k, v, idx, o, lse, do, cu, T)
    for a, b in zip((gq, gk, gv), g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_sparse_bwd_full_size_sampled():
    """B=8, T=16384, H=16, Hkv=1, d=128, block 64, S=16 (the benchmark launch, fed by the
    GPU forward): dq on sampled query rows, dk and dv on sampled key rows of blocks 1, 100
    and 255.  The oracle takes D from its own forward output on every token it visits."""
    w = gen.prefill()
    do = gen.normal(_rng(23), (w.tokens, 16, 128), "bf16")
    q, k, v, di = dev(w.q), dev(w.k), dev(w.v), dev(w.idx)
    lse = torch.empty((w.tokens, 16), dtype=torch.float32, device="cuda")
    o = nsa.nsa_sparse_fwd(q.view(8, 16384, 16, 128), k, v, di, 64, lse=lse).view(w.tokens, 16, 128)
    gq, gk, gv = nsa.nsa_sparse_bwd(q.view(8, 16384, 16, 128), k, v, di, o, lse, dev(do), 64)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    rng = _rng(24)
    qr = np.unique(np.concatenate([rng.integers(0, w.tokens, 48), [0, 16383, 16384, 131071]]))
    kr = np.array([3 * 16384 + 64, 3 * 16384 + 127, 5 * 16384 + 6400 + 17, 7 * 16384 + 16320, 7 * 16384 + 16383])
    # tokens whose lists reach the sampled key rows (same sequence, block listed, key causal)
    tok = np.arange(w.tokens)
    seq, t = tok // 16384, tok % 16384
    hit = np.zeros(w.tokens, bool)
    for r_ in kr:
        s_, j_ = r_ // 16384, (r_ % 16384) // 64
        hit |= (seq == s_) & (t >= r_ % 16384) & (w.idx[:, 0, :] == j_).any(1)
    need = np.unique(np.concatenate([qr, tok[hit]]))
    o_ref = np.zeros((w.tokens, 16, 128), np.uint16)
    o_ref[need] = _oracle_fwd_inputs(w.q, w.k, w.v, w.idx, w.cu_seqlens, rows=need)[0]
    rq, _, _ = orc.sparse_attn_bwd(w.q, w.k, w.v, w.idx, do, w.cu_seqlens, 64, q_rows=qr, want_dkv=False, o=o_ref)
    _, rk, rv = orc.sparse_attn_bwd(w.q, w.k, w.v, w.idx, do, w.cu_seqlens, 64, kv_rows=kr, want_dq=False,
                                    o=o_ref)
    assert_close(gq.reshape(w.tokens, 16, 128)[torch.from_numpy(qr).cuda()], rq, what="dq sampled")
    assert_close(gk[torch.from_numpy(kr).cuda()], rk, what="dk sampled")
    assert_close(gv[torch.from_numpy(kr).cuda()], rv, what="dv sampled")


# --------------------------------------------------------------------------- S7 and S1 backward
@pytest.mark.parametrize("H,hkv", [(16, 1), (16, 2), (16, 4), (8, 8), (64, 4)])
def test_cmp_attn_bwd_varlen(H, hkv):
    """Ragged lengths (no window, one window, several key blocks and query chunks); both
    sides take the oracle's forward (o rounded to bf16, lse)."""
    lengths = [10, 31, 32, 47, 500, 2100, 4500]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(41)
    q, do = gen.normal(rng, (cu[-1], H, 128), "bf16"), gen.normal(rng, (cu[-1], H, 128), "bf16")
    k, v = gen.normal(rng, (cu[-1], hkv, 128), "bf16"), gen.normal(rng, (cu[-1], hkv, 128), "bf16")
    _, kc = orc.compress(k, cu)
    _, vc = orc.compress(v, cu)
    o64, lse64 = orc.cmp_attn(q, kc, vc, cu)
    o = gen.f32_to_bf16_bits(o64.astype(np.float32))
    lse = lse64.astype(np.float32)
    gq, gk, gv = nsa.nsa_cmp_attn_bwd(dev(q), dev(kc), dev(vc), dev(o), dev(lse), dev(do), hkv, cu_seqlens=dev(cu),
                                      max_seqlen=max(lengths))
    gk_tok = nsa.nsa_compress_bwd(gk, int(cu[-1]), cu_seqlens=dev(cu), max_seqlen=max(lengths))
    torch.cuda.synchronize()
    rq, rk, rv = orc.cmp_attn_bwd(q, kc, vc, do, cu, o=o)
    assert_close(gq, rq, what="cmp dq")
    assert_close(gk, rk, what="cmp dk")
    assert_close(gv, rv, what="cmp dv")
    # the pooling backward on the GPU's own window gradient
    assert_close(gk_tok, orc.compress_bwd(as_f64(host(gk)), cu), atol=1e-3, rtol=1e-2, what="compress bwd")


def test_cmp_attn_bwd_layer_size_sampled():
    """T=65536, H=64, Hkv=4 (4095 compressed keys): GPU forward then backward; dq on sampled
    rows, d k_cmp / d v_cmp on late compressed rows (the oracle visits every token that
    reaches them), and determinism."""
    w = gen.layer()
    cu, T = w.cu_seqlens, w.tokens
    do = gen.normal(_rng(42), (T, 64, 128), "bf16")
    dq_, dk_, dv_ = dev(w.q), dev(w.k), dev(w.v)
    kc = nsa.nsa_compress_k(dk_)
    vc = nsa.nsa_compress_k(dv_)
    lse = torch.empty((T, 64), dtype=torch.float32, device="cuda")
    o = nsa.nsa_cmp_attn_fwd(dq_, kc, vc, 4, lse=lse)
    gq, gk, gv = nsa.nsa_cmp_attn_bwd(dq_, kc, vc, o, lse, dev(do), 4)
    g2 = nsa.nsa_cmp_attn_bwd(dq_, kc, vc, o, lse, dev(do), 4)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    for a, b in zip((gq, gk, gv), g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    kch, vch = host(kc), host(vc)
    qr = np.array([0, 31, 32, 1000, 33333, 65535])
    kr = np.array([4088, 4094])
    need = np.unique(np.concatenate([qr, np.arange(16 * 4088 + 31, T)]))
    o_ref = np.zeros((T, 64, 128), np.uint16)
    o64, _ = orc.cmp_attn(w.q, kch, vch, cu, rows=need)
    o_ref[need] = gen.f32_to_bf16_bits(o64.astype(np.float32))
    rq, _, _ = orc.cmp_attn_bwd(w.q, kch, vch, do, cu, q_rows=qr, want_dkv=False, o=o_ref)
    _, rk, rv = orc.cmp_attn_bwd(w.q, kch, vch, do, cu, kv_rows=kr, want_dq=False, o=o_ref)
    assert_close(gq[torch.from_numpy(qr).cuda()], rq, what="cmp dq sampled")
    assert_close(gk[torch.from_numpy(kr).cuda()], rk, what="cmp dk sampled")
    assert_close(gv[torch.from_numpy(kr).cuda()], rv, what="cmp dv sampled")


# --------------------------------------------------------------------------- S8 and S9 backward
@pytest.mark.parametrize("window,H,hkv", [(512, 16, 1), (1, 16, 2), (64, 8, 8), (1984, 16, 4), (100, 64, 4)])
def test_swa_bwd_varlen(window, H, hkv):
    lengths = [1, 63, 64, 65, 700, 2100]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(51)
    q, do = gen.normal(rng, (cu[-1], H, 128), "bf16"), gen.normal(rng, (cu[-1], H, 128), "bf16")
    k, v = gen.normal(rng, (cu[-1], hkv, 128), "bf16"), gen.normal(rng, (cu[-1], hkv, 128), "bf16")
    o64, lse64 = orc.swa(q, k, v, cu, window)
    o = gen.f32_to_bf16_bits(o64.astype(np.float32))
    gq, gk, gv = nsa.nsa_swa_bwd(dev(q), dev(k), dev(v), dev(o), dev(lse64.astype(np.float32)), dev(do), window,
                                 cu_seqlens=dev(cu), max_seqlen=max(lengths))
    torch.cuda.synchronize()
    rq, rk, rv = orc.swa_bwd(q, k, v, do, cu, window, o=o)
    assert_close(gq, rq, what="swa dq")
    assert_close(gk, rk, what="swa dk")
    assert_close(gv, rv, what="swa dv")


def test_swa_bwd_layer_size_sampled():
    """T=65536, H=64, Hkv=4, window 512: GPU forward then backward; sampled rows.  The GPU
    backward takes D from the GPU forward's o, the oracle from its own; key rows near the
    start collect large-p terms from rows with few keys, where those two D differ most, so
    the sampled key rows lie past the first window (rows with few keys are covered above,
    where both sides share one forward output)."""
    w = gen.layer()
    T = w.tokens
    do = gen.normal(_rng(52), (T, 64, 128), "bf16")
    q, k, v = dev(w.q), dev(w.k), dev(w.v)
    lse = torch.empty((T, 64), dtype=torch.float32, device="cuda")
    o = nsa.nsa_swa_fwd(q, k, v, 512, lse=lse)
    gq, gk, gv = nsa.nsa_swa_bwd(q, k, v, o, lse, dev(do), 512)
    torch.cuda.synchronize()
    qr = np.array([0, 1, 511, 512, 40000, 65535])
    kr = np.array([1000, 1023, 1024, 30000, 65535])
    need = np.unique(np.concatenate([qr] + [np.arange(r_, min(r_ + 512, T)) for r_ in kr]))
    o_ref = np.zeros((T, 64, 128), np.uint16)
    o64, _ = orc.swa(w.q, w.k, w.v, w.cu_seqlens, 512, rows=need)
    o_ref[need] = gen.f32_to_bf16_bits(o64.astype(np.float32))
    rq, _, _ = orc.swa_bwd(w.q, w.k, w.v, do, w.cu_seqlens, 512, q_rows=qr, want_dkv=False, o=o_ref)
    _, rk, rv = orc.swa_bwd(w.q, w.k, w.v, do, w.cu_seqlens, 512, kv_rows=kr, want_dq=False, o=o_ref)
    assert_close(gq[torch.from_numpy(qr).cuda()], rq, what="swa dq sampled")
    assert_close(gk[torch.from_numpy(kr).cuda()], rk, what="swa dk sampled")
    assert_close(gv[torch.from_numpy(kr).cuda()], rv, what="swa dv sampled")


def test_gate_combine_bwd():
    rng = _rng(53)
    n, h, d = 777, 16, 128
    br = [gen.normal(rng, (n, h, d), "bf16") for _ in range(3)]
    do = gen.normal(rng, (n, h, d), "bf16")
    logits = (rng.standard_normal((n, h, 3)) * 2).astype(np.float32)
    got = nsa.nsa_gate_combine_bwd(dev(do), *(dev(b) for b in br), dev(logits))
    torch.cuda.synchronize()
    ref = orc.gate_bwd(*(as_f64(b) for b in br), logits, as_f64(do))
    for i in range(3):
        assert_close(got[i], ref[i], what=f"gate branch {i}")
    assert_close(got[3], ref[3], atol=1e-4, rtol=1e-4, what="gate logits")


# --------------------------------------------------------------------------- layer training pair
def _layer_train_case(lengths, H, hkv):
    w = gen.layer(H=H, HKV=hkv, lengths=lengths)
    cu = w.cu_seqlens
    do = gen.normal(_rng(61), (w.tokens, H, 128), "bf16")
    return w, cu, do


def test_layer_fwd_train_matches_layer_fwd_and_oracle():
    """The training forward gives the same output as nsa_layer_fwd (same kernels) and
    keeps branch outputs and normalisers that match the oracle's branches."""
    lengths = [700, 1500, 40]
    w, cu, _ = _layer_train_case(lengths, 16, 2)
    dcu, L = dev(cu), max(lengths)
    n_cmp = int(orc.cmp_offsets(cu)[-1])
    saved = nsa.nsa_layer_saved_buffers(w.tokens, n_cmp, 16, 2, 128, 16, "cuda")
    q, k, v, gl = dev(w.q), dev(w.k), dev(w.v), dev(w.gates)
    o_tr = nsa.nsa_layer_fwd_train(q, k, v, gl, saved, cu_seqlens=dcu, max_seqlen=L)
    o = torch.empty_like(o_tr)
    idx = torch.empty((w.tokens, 2, 16), dtype=torch.int32, device="cuda")
    nsa.nsa_layer_fwd(q, k, v, gl, cu_seqlens=dcu, max_seqlen=L, out=o, idx_out=idx)
    torch.cuda.synchronize()
    assert torch.equal(o_tr.view(torch.int16), o.view(torch.int16))
    assert torch.equal(saved["idx"], idx)
    _, kc = orc.compress(w.k, cu)
    assert np.array_equal(host(saved["k_cmp"]), kc)
    gi = host(saved["idx"])
    ref_c, lc = orc.cmp_attn(w.q, host(saved["k_cmp"]), host(saved["v_cmp"]), cu)
    ref_s, ls = orc.sparse_attn(w.q, w.k, w.v, gi, cu, 64)
    ref_w, lw = orc.swa(w.q, w.k, w.v, cu, 512)
    for got, ref, what in (("o_cmp", ref_c, "cmp"), ("o_slc", ref_s, "slc"), ("o_swa", ref_w, "swa")):
        assert_close(saved[got], ref, what=f"saved {what}")
    for got, ref in (("lse_cmp", lc), ("lse_slc", ls), ("lse_swa", lw)):
        g = host(saved[got])
        fin = np.isfinite(ref)
        assert np.array_equal(np.isfinite(g), fin), got
        assert np.allclose(g[fin], ref[fin], atol=1e-3, rtol=1e-3), got


@pytest.mark.parametrize("lengths,H,hkv", [([700, 1500, 40], 16, 2), ([2100], 16, 1), ([300, 64], 8, 8)])
def test_layer_bwd(lengths, H, hkv):
    """nsa_layer_bwd on buffers the oracle's forward filled (branch outputs rounded to bf16,
    normalisers, block lists) against the oracle's composition of branch backwards."""
    w, cu, do = _layer_train_case(lengths, H, hkv)
    dcu, L = dev(cu), max(lengths)
    ref = orc.layer(w.q, w.k, w.v, w.gates, cu, branches=True)
    idx = ref["idx"]
    _, kc = orc.compress(w.k, cu)
    _, vc = orc.compress(w.v, cu)
    oc, lc = orc.cmp_attn(w.q, kc, vc, cu)
    os_, ls = orc.sparse_attn(w.q, w.k, w.v, idx, cu, 64)
    ow, lw = orc.swa(w.q, w.k, w.v, cu, 512)
    rb = [gen.f32_to_bf16_bits(x.astype(np.float32)) for x in (oc, os_, ow)]
    saved = {"k_cmp": dev(kc), "v_cmp": dev(vc), "o_cmp": dev(rb[0]), "o_slc": dev(rb[1]), "o_swa": dev(rb[2]),
             "lse_cmp": dev(lc.astype(np.float32)), "lse_slc": dev(ls.astype(np.float32)),
             "lse_swa": dev(lw.astype(np.float32)), "idx": dev(idx)}
    gq, gk, gv, gg = nsa.nsa_layer_bwd(dev(w.q), dev(w.k), dev(w.v), dev(w.gates), saved, dev(do), cu_seqlens=dcu,
                                       max_seqlen=L)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    rq, rk, rv, rg = orc.layer_bwd(w.q, w.k, w.v, w.gates, idx, do, cu, branches=rb)
    assert_close(gq, rq, what="layer dq")
    assert_close(gk, rk, what="layer dk")
    assert_close(gv, rv, what="layer dv")
    assert_close(gg, rg, atol=1e-3, rtol=1e-3, what="layer d gates")


# --------------------------------------------------------------------------- NOSA stage 2
def test_cis_block_scores():
    lengths = [10, 31, 32, 47, 100, 700, 5000]
    cu = gen.varlen_cu_seqlens(lengths)
    cis = gen.cis_scores(_rng(31), int(cu[-1]), 2)
    nb = -(-max(lengths) // 64)
    got = nsa.nsa_cis_block_scores(dev(cis), cu_seqlens=dev(cu), max_seqlen=max(lengths), nb_stride=nb)
    torch.cuda.synchronize()
    ref = orc.cis_block_scores(cis, cu, nb_stride=nb)
    assert np.allclose(host(got), ref, atol=2e-6, rtol=0)


@pytest.mark.parametrize("qk,k,nb", [(32, 16, 64), (64, 64, 260), (16, 16, 40), (48, 13, 1024), (3, 1, 8)])
def test_topk_two_stage_bit_exact(qk, k, nb):
    """Same fp32 inputs on both sides: the chosen lists must match exactly (many ties)."""
    rng = _rng(32 + qk)
    L = nb * 64
    lengths = [L, min(L, 700), 65]
    cu = gen.varlen_cu_seqlens(lengths)
    sc = (np.round(rng.random((int(cu[-1]), 2, nb)) * 16) / 16).astype(np.float32)
    cs = (np.round(rng.random((len(lengths), 2, nb)) * 16) / 16).astype(np.float32)
    got = nsa.nsa_topk_two_stage(dev(sc), dev(cs), qk, k, cu_seqlens=dev(cu), max_seqlen=L)
    torch.cuda.synchronize()
    ref = orc.topk_two_stage(sc, cs, cu, qk, k)
    assert np.array_equal(host(got), ref)


@pytest.mark.parametrize("H,hkv,d", [(16, 1, 128), (16, 4, 128), (8, 8, 128), (16, 2, 64), (32, 1, 128)])
def test_sparse_cis_fwd(H, hkv, d):
    lengths = [1, 63, 64, 65, 900, 2000]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(33)
    q, k, v = (gen.normal(rng, (cu[-1], hh, d), "bf16") for hh in (H, hkv, hkv))
    idx = gen.random_block_indices(rng, cu, hkv, 16, 64, force_first=True)
    cis = gen.cis_scores(rng, int(cu[-1]), hkv)
    cis[:40] = 0.0  # the first sequences' early keys carry no weight: some rows sum to zero
    ref, lse_ref = orc.sparse_attn_cis(q, k, v, cis, idx, cu, 64)
    lse = torch.empty((cu[-1], H), dtype=torch.float32, device="cuda")
    out = nsa.nsa_sparse_cis_fwd(dev(q), dev(k), dev(v), dev(cis), dev(idx), 64, cu_seqlens=dev(cu),
                                 max_seqlen=max(lengths), lse=lse)
    torch.cuda.synchronize()
    assert_close(out, ref, what="cis-weighted attention")
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(host(lse)), fin)
    assert_close(host(lse)[fin], lse_ref[fin], atol=1e-3, rtol=1e-3, what="cis lse")


def test_nosa_pipeline():
    """compress -> block scores -> block CIS -> two-stage selection -> CIS-weighted attention,
    each stage checked against the oracle on the GPU's own inputs to that stage."""
    w = gen.selection(n_seqs=3, lo=1500, hi=4000)
    cu, L = w.cu_seqlens, w.max_len
    dcu = dev(cu)
    cis = gen.cis_scores(_rng(34), w.tokens, w.hkv)
    kc = nsa.nsa_compress_k(dev(w.k), cu_seqlens=dcu, max_seqlen=L)
    nb = ((-(-L // 64)) + 3) // 4 * 4
    sc = nsa.nsa_cmp_scores_pool(dev(w.q), kc, w.hkv, cu_seqlens=dcu, max_seqlen=L, nb_stride=nb)
    cs = nsa.nsa_cis_block_scores(dev(cis), cu_seqlens=dcu, max_seqlen=L, nb_stride=nb)
    idx = nsa.nsa_topk_two_stage(sc, cs, 32, 16, cu_seqlens=dcu, max_seqlen=L)
    out = nsa.nsa_sparse_cis_fwd(dev(w.q), dev(w.k), dev(w.v), dev(cis), idx, 64, cu_seqlens=dcu, max_seqlen=L)
    torch.cuda.synchronize()
    assert np.allclose(host(cs), orc.cis_block_scores(cis, cu, nb_stride=nb), atol=2e-6, rtol=0)
    assert np.array_equal(host(idx), orc.topk_two_stage(host(sc), host(cs), cu, 32, 16))
    rows = np.unique(np.concatenate([_rng(35).integers(0, w.tokens, 300), cu[:-1], cu[1:] - 1]))
    ref, _ = orc.sparse_attn_cis(w.q, w.k, w.v, cis, host(idx), cu, 64, rows=rows)
    assert_close(out[torch.from_numpy(rows).cuda()], ref, what="nosa pipeline")


# --------------------------------------------------------------------------- S7, S8, S9
# d 128 with a power-of-two group runs on the tcgen05 kernel (group 128: one token per
# CTA); group 48 and d 64 run on mma.sync
@pytest.mark.parametrize("H,hkv,d", [(16, 1, 128), (32, 2, 128), (8, 1, 64), (16, 4, 128), (64, 1, 128),
                                     (48, 1, 128), (128, 1, 128)])
def test_cmp_attn(H, hkv, d):
    lengths = [10, 31, 32, 47, 500, 1777]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(9)
    q, k, v = (gen.normal(rng, (cu[-1], hh, d), "bf16") for hh in (H, hkv, hkv))
    _, kc = orc.compress(k, cu)
    _, vc = orc.compress(v, cu)
    ref, lse_ref = orc.cmp_attn(q, kc, vc, cu)
    lse = torch.empty((cu[-1], H), dtype=torch.float32, device="cuda")
    out = nsa.nsa_cmp_attn_fwd(dev(q), dev(kc), dev(vc), hkv, cu_seqlens=dev(cu), max_seqlen=max(lengths), lse=lse)
    torch.cuda.synchronize()
    assert_close(out, ref, what="cmp attn")
    l = host(lse)
    assert np.array_equal(np.isneginf(l), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(l[fin], lse_ref[fin], atol=1e-3, rtol=1e-4)


@pytest.mark.parametrize("window,H,hkv", [(512, 16, 1), (1, 16, 2), (100, 8, 1), (5000, 16, 1), (64, 64, 4),
                                          (300, 32, 1), (77, 48, 1)])
def test_swa(window, H, hkv):
    lengths = [3, 600, 2100]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = _rng(10)
    d = 128
    q, k, v = (gen.normal(rng, (cu[-1], hh, d), "bf16") for hh in (H, hkv, hkv))
    ref, _ = orc.swa(q, k, v, cu, window=window)
    out = nsa.nsa_swa_fwd(dev(q), dev(k), dev(v), window, cu_seqlens=dev(cu), max_seqlen=max(lengths))
    torch.cuda.synchronize()
    assert_close(out, ref, what="swa")


def test_gate_combine():
    rng = _rng(11)
    n, h, d = 1000, 16, 128
    a, b, c = (gen.normal(rng, (n, h, d), "bf16") for _ in range(3))
    gates = rng.standard_normal((n, h, 3), dtype=np.float32)
    gates[:5] = [[40.0, -40.0, -40.0]]
    ref = orc.gate_combine(as_f64(a), as_f64(b), as_f64(c), gates)
    out = nsa.nsa_gate_combine(dev(a), dev(b), dev(c), dev(gates))
    torch.cuda.synchronize()
    assert_close(out, ref, what="gate")


# --------------------------------------------------------------------------- S6
def _decode_case(B, L, seqlens, k, seed, H=16, HKV=2):
    w = gen.decode(B=B, L=L, seqlens=seqlens, topk=k, H=H, HKV=HKV)
    ncs = orc.num_cmp(L)
    kc_cache = np.zeros((B, ncs, w.hkv, w.d), np.uint16)
    for b in range(B):
        kc_cache[b] = orc.compress(w.k_cache[b], [0, L])[1]
    return w, kc_cache


@pytest.mark.parametrize("B,L,seqlens,k", [(4, 4096, [4096, 2500, 70, 1], 64), (3, 2048, [2048, 2047, 1000], 16),
                                           (2, 300, [300, 33], 64)])
def test_decode(B, L, seqlens, k):
    w, kc_cache = _decode_case(B, L, seqlens, k, 0)
    ref_idx, _, ref_sc = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, want_scores=True)
    idx = torch.empty((B, w.hkv, k), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode(dev(w.q), dev(w.k_cache), dev(w.v_cache), dev(kc_cache), dev(w.seqlens), k=k,
                                idx_out=idx)
    torch.cuda.synchronize()
    gi = host(idx)
    n_mis, outside = selection_mismatches(gi, ref_idx, ref_sc, np.asarray(w.seqlens) - 1)
    assert outside == 0, (n_mis, outside)
    # attention over the GPU's own choice
    _, ref_o = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, idx_in=gi)
    assert_close(out, ref_o, what="decode")


@pytest.mark.parametrize("B,L,seqlens,k,H,HKV", [
    (3, 3000, [3000, 1500, 40], 64, 16, 1),     # group 16
    (2, 2000, [2000, 999], 7, 4, 4),            # group 1, small k
    (5, 1500, [1500, 31, 64, 65, 1200], 1, 8, 2),  # group 4, k = 1, rows without compressed keys
    (40, 1024, None, 32, 16, 2)])               # 80 rows: more work items than resident CTAs
def test_decode_group_sizes(B, L, seqlens, k, H, HKV):
    w, kc_cache = _decode_case(B, L, seqlens, k, 0, H=H, HKV=HKV)
    ref_idx, _, ref_sc = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, want_scores=True)
    idx = torch.empty((B, HKV, k), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode(dev(w.q), dev(w.k_cache), dev(w.v_cache), dev(kc_cache), dev(w.seqlens), k=k,
                                idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    gi = host(idx)
    n_mis, outside = selection_mismatches(gi, ref_idx, ref_sc, np.asarray(w.seqlens) - 1)
    assert outside == 0, (n_mis, outside)
    _, ref_o = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, idx_in=gi)
    assert_close(out, ref_o, what="decode groups")


@pytest.mark.parametrize("L,k", [(20000, 64), (4000, 16)])
def test_decode_exact_ties(L, k):
    """A cache of identical keys: every compressed key scores alike, so every block that is
    not forced has the same pooled score (three windows each) on both sides, bit for bit.
    The choice must then be the lowest blocks, exactly: with 310 tied candidates the CTA
    top-k settles every bit and takes ties by block order; with 60 it ranks the bin."""
    B, H, HKV = 2, 16, 2
    rng = _rng(77)
    q = gen.normal(rng, (B, H, 128), "bf16")
    kcache = np.full((B, L, HKV, 128), gen.f32_to_bf16_bits(np.float32(0.25)), np.uint16)
    vcache = gen.normal(rng, (B, L, HKV, 128), "bf16")
    seqlens = np.array([L, L - 37], np.int32)
    ncs = orc.num_cmp(L)
    kc_cache = np.zeros((B, ncs, HKV, 128), np.uint16)
    for b in range(B):
        kc_cache[b] = orc.compress(kcache[b], [0, L])[1]
    ref_idx, _ = orc.decode(q, kcache, vcache, kc_cache, seqlens, k=k)
    idx = torch.empty((B, HKV, k), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode(dev(q), dev(kcache), dev(vcache), dev(kc_cache), dev(seqlens), k=k, idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    assert np.array_equal(host(idx), ref_idx)
    _, ref_o = orc.decode(q, kcache, vcache, kc_cache, seqlens, k=k, idx_in=host(idx))
    assert_close(out, ref_o, what="decode ties")


def test_decode_full_size():
    """B=32, context 32768, H=16, Hkv=2, d=128, top-k 64: all rows."""
    w = gen.decode()
    kc = nsa.nsa_compress_k(dev(w.k_cache))  # [B*n_c, Hkv, d]
    kc_cache = kc.view(32, orc.num_cmp(32768), 2, 128)
    idx = torch.empty((32, 2, 64), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode(dev(w.q), dev(w.k_cache), dev(w.v_cache), kc_cache, dev(w.seqlens), k=64,
                                idx_out=idx)
    torch.cuda.synchronize()
    kch = host(kc_cache)
    ref_idx, _, ref_sc = orc.decode(w.q, w.k_cache, w.v_cache, kch, w.seqlens, k=64, want_scores=True)
    gi = host(idx)
    n_mis, outside = selection_mismatches(gi, ref_idx, ref_sc, np.asarray(w.seqlens) - 1)
    assert outside == 0, (n_mis, outside)
    _, ref_o = orc.decode(w.q, w.k_cache, w.v_cache, kch, w.seqlens, k=64, idx_in=gi)
    assert_close(out, ref_o, what="decode full")


@pytest.mark.parametrize("B,L,seqlens,k,H,HKV", [(4, 4096, [4096, 2500, 70, 1], 64, 16, 2),
                                                  (5, 1500, [1500, 31, 64, 65, 1200], 1, 8, 2),
                                                  (3, 3000, [3000, 1500, 40], 64, 16, 1)])
def test_decode_offloaded_cache(B, L, seqlens, k, H, HKV):
    """K/V cache in page-locked host memory, compressed keys on the device: the chosen
    blocks are read over the CPU-GPU link.  Same kernels, so the outputs equal those of
    the device-resident cache bit for bit, and they match the oracle."""
    w, kc_cache = _decode_case(B, L, seqlens, k, 0, H=H, HKV=HKV)
    hk, hv = pinned(w.k_cache), pinned(w.v_cache)
    assert hk.device.type == "cpu" and hk.is_pinned()
    q, kc, sl = dev(w.q), dev(kc_cache), dev(w.seqlens)
    idx_h = torch.empty((B, HKV, k), dtype=torch.int32, device="cuda")
    out_h = nsa.nsa_sparse_decode(q, hk, hv, kc, sl, k=k, idx_out=idx_h)
    idx_d = torch.empty_like(idx_h)
    out_d = nsa.nsa_sparse_decode(q, dev(w.k_cache), dev(w.v_cache), kc, sl, k=k, idx_out=idx_d)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    assert torch.equal(idx_h, idx_d)
    assert torch.equal(out_h.view(torch.int16), out_d.view(torch.int16))
    gi = host(idx_h)
    ref_idx, _, ref_sc = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, want_scores=True)
    n_mis, outside = selection_mismatches(gi, ref_idx, ref_sc, np.asarray(w.seqlens) - 1)
    assert outside == 0, (n_mis, outside)
    _, ref_o = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, idx_in=gi)
    assert_close(out_h, ref_o, what="decode offloaded")


def _stage1_near_tie_rows(sc, seqlens, qk, n_init=1, n_local=2, tau=1e-6):
    """Rows whose stage-1 cut (the qk-th kept block) has a near tie in the oracle's scores."""
    B, hkv, nb = sc.shape
    near = np.zeros((B, hkv), bool)
    for b in range(B):
        own = (int(seqlens[b]) - 1) // 64
        for g in range(hkv):
            free = [j for j in range(own + 1) if not (j < n_init or j > own - n_local)]
            nf = own + 1 - len(free)
            keep = qk - nf
            if 0 < keep < len(free):
                s_ = np.sort(sc[b, g, free])[::-1]
                near[b, g] = s_[keep - 1] - s_[keep] < tau * 16
    return near


@pytest.mark.parametrize("B,L,seqlens,k,qk,H,HKV", [(4, 4096, [4096, 2500, 700, 1], 16, 32, 16, 2),
                                                    (3, 3000, [3000, 1500, 40], 64, 64, 16, 1),
                                                    (5, 1500, [1500, 31, 64, 65, 1200], 4, 12, 8, 2)])
def test_decode_cis(B, L, seqlens, k, qk, H, HKV):
    """NOSA decode: two-stage selection and CIS-weighted attention."""
    w, kc_cache = _decode_case(B, L, seqlens, k, 0, H=H, HKV=HKV)
    cis = gen.cis_scores(_rng(71), B * L, HKV).reshape(B, L, HKV)
    nb = -(-L // 64)
    cb = nsa.nsa_cis_block_scores(dev(cis.reshape(B * L, HKV)), batch=B, seqlen=L, nb_stride=nb)
    idx = torch.empty((B, HKV, k), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode_cis(dev(w.q), dev(w.k_cache), dev(w.v_cache), dev(kc_cache), dev(cis),
                                    dev(w.seqlens), cb, qk, k=k, idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    gi = host(idx)
    ref_idx, _, sc = orc.decode_cis(w.q, w.k_cache, w.v_cache, kc_cache, cis, w.seqlens, qk, k=k)
    near = _stage1_near_tie_rows(sc, w.seqlens, qk)
    diff = np.any(gi != ref_idx, axis=2)
    assert not np.any(diff & ~near), np.argwhere(diff & ~near)
    _, ref_o, _ = orc.decode_cis(w.q, w.k_cache, w.v_cache, kc_cache, cis, w.seqlens, qk, k=k, idx_in=gi)
    assert_close(out, ref_o, what="decode cis")


def test_decode_cis_weights_only_keeps_the_plain_selection():
    """Without block CIS scores the choice is the plain decode's, bit for bit; the output is
    the CIS-weighted attention over it."""
    w, kc_cache = _decode_case(3, 2048, [2048, 2047, 1000], 16, 0)
    cis = gen.cis_scores(_rng(72), 3 * 2048, 2).reshape(3, 2048, 2)
    cis[1, :100] = 0.0
    i0 = torch.empty((3, 2, 16), dtype=torch.int32, device="cuda")
    i1 = torch.empty_like(i0)
    nsa.nsa_sparse_decode(dev(w.q), dev(w.k_cache), dev(w.v_cache), dev(kc_cache), dev(w.seqlens), k=16, idx_out=i0)
    out = nsa.nsa_sparse_decode_cis(dev(w.q), dev(w.k_cache), dev(w.v_cache), dev(kc_cache), dev(cis),
                                    dev(w.seqlens), k=16, idx_out=i1)
    torch.cuda.synchronize()
    assert torch.equal(i0, i1)
    _, ref_o, _ = orc.decode_cis(w.q, w.k_cache, w.v_cache, kc_cache, cis, w.seqlens, 16, k=16, idx_in=host(i1))
    assert_close(out, ref_o, what="decode cis weights only")


def test_decode_offloaded_full_size_sampled():
    """B=32, context 32768, H=16, Hkv=2, d=128, top-k 64 with the 1 GB K/V cache in
    page-locked host memory; the oracle checks eight sampled sequences."""
    w = gen.decode()
    kc_cache = nsa.nsa_compress_k(dev(w.k_cache)).view(32, orc.num_cmp(32768), 2, 128)
    hk, hv = pinned(w.k_cache), pinned(w.v_cache)
    idx = torch.empty((32, 2, 64), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode(dev(w.q), hk, hv, kc_cache, dev(w.seqlens), k=64, idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    rows = np.random.default_rng(5).choice(32, 8, replace=False)
    kch, gi, go = host(kc_cache)[rows], host(idx)[rows], host(out)[rows]
    sl = np.asarray(w.seqlens)[rows]
    ref_idx, _, ref_sc = orc.decode(w.q[rows], w.k_cache[rows], w.v_cache[rows], kch, sl, k=64, want_scores=True)
    n_mis, outside = selection_mismatches(gi, ref_idx, ref_sc, sl - 1)
    assert outside == 0, (n_mis, outside)
    _, ref_o = orc.decode(w.q[rows], w.k_cache[rows], w.v_cache[rows], kch, sl, k=64, idx_in=gi)
    assert_close(go, ref_o, what="decode offloaded full")


def test_decode_rejects_pageable_cache():
    """A pageable host cache has no device address: the call fails before any launch."""
    w, kc_cache = _decode_case(2, 300, [300, 33], 16, 0)
    kp = torch.from_numpy(np.ascontiguousarray(w.k_cache).view(np.int16)).view(torch.bfloat16)
    assert not kp.is_pinned()
    with pytest.raises(RuntimeError, match="page-locked"):
        nsa.nsa_sparse_decode(dev(w.q), kp, dev(w.v_cache), dev(kc_cache), dev(w.seqlens), k=16)


# --------------------------------------------------------------------------- fused selection and the layer
def test_selection_varlen_end_to_end():
    """compress -> scores -> top-k at reduced size of the varlen selection workload."""
    w = gen.selection(n_seqs=3, lo=1000, hi=3000)
    dcu = dev(w.cu_seqlens)
    kc = nsa.nsa_compress_k(dev(w.k), cu_seqlens=dcu, max_seqlen=w.max_len)
    sc = nsa.nsa_cmp_scores_pool(dev(w.q), kc, w.hkv, cu_seqlens=dcu, max_seqlen=w.max_len)
    idx = nsa.nsa_topk_select(sc, 16, cu_seqlens=dcu, max_seqlen=w.max_len)
    torch.cuda.synchronize()
    kch = host(kc)
    ref_sc = orc.cmp_scores_pool(w.q, kch, w.cu_seqlens)
    ref_idx = orc.topk(ref_sc, w.cu_seqlens, k=16)
    n_mis, outside = selection_mismatches(host(idx), ref_idx, ref_sc, _t_of_rows(w.cu_seqlens))
    assert outside == 0
    assert n_mis <= max(3, ref_idx.shape[0] * ref_idx.shape[1] // 200), n_mis
    # top-k on the GPU's own scores is bit-exact with the oracle's top-k of those scores
    assert np.array_equal(host(idx), orc.topk(host(sc), w.cu_seqlens, k=16))


@pytest.mark.parametrize("T,H,hkv", [(1500, 32, 2), (700, 16, 1), (1100, 16, 2), (900, 8, 2), (333, 4, 4)])
def test_layer_small(T, H, hkv):
    w = gen.layer(T=T, H=H, HKV=hkv)
    idx = torch.empty((T, hkv, 16), dtype=torch.int32, device="cuda")
    out = nsa.nsa_layer_fwd(dev(w.q), dev(w.k), dev(w.v), dev(w.gates), idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    gi = host(idx)
    ref = orc.layer(w.q, w.k, w.v, w.gates, w.cu_seqlens, idx_in=gi)
    _, kc = orc.compress(w.k, w.cu_seqlens)
    ref_sc = orc.cmp_scores_pool(w.q, kc, w.cu_seqlens)
    n_mis, outside = selection_mismatches(gi, ref["idx"], ref_sc, _t_of_rows(w.cu_seqlens))
    assert outside == 0, (n_mis, outside)
    assert_close(out, ref["o"], what="layer")


def test_select_fused_call():
    """nsa_select (S2-S4 in one call) equals scores + top-k by separate calls, bit for
    bit, and matches the oracle's selection up to near ties."""
    w = gen.selection(n_seqs=3, lo=900, hi=2500)
    dcu = dev(w.cu_seqlens)
    kc = nsa.nsa_compress_k(dev(w.k), cu_seqlens=dcu, max_seqlen=w.max_len)
    one = nsa.nsa_select(dev(w.q), kc, w.hkv, k=16, cu_seqlens=dcu, max_seqlen=w.max_len)
    sc = nsa.nsa_cmp_scores_pool(dev(w.q), kc, w.hkv, cu_seqlens=dcu, max_seqlen=w.max_len)
    two = nsa.nsa_topk_select(sc, 16, cu_seqlens=dcu, max_seqlen=w.max_len)
    torch.cuda.synchronize()
    assert np.array_equal(host(one), host(two))
    ref_sc = orc.cmp_scores_pool(w.q, host(kc), w.cu_seqlens)
    ref_idx = orc.topk(ref_sc, w.cu_seqlens, k=16)
    _, outside = selection_mismatches(host(one), ref_idx, ref_sc, _t_of_rows(w.cu_seqlens))
    assert outside == 0


def test_selection_full_size_sampled():
    """The varlen selection workload at its stated size (4 packed sequences of 7733,
    14932, 24577 and 8673 tokens, H 16, H_kv 2, d 128, top-16 with 1 initial and 2 local
    blocks), through the same calls the benchmark times: compression checked on every
    compressed key; block scores and block lists against the oracle on sampled rows (the
    first and last row of every sequence, rows around the first compression window and
    the first selection blocks, and random rows); the top-k of the GPU's own scores
    bit-exact with the oracle's top-k of those scores on every row; the one-call
    selection identical to the separate calls."""
    w = gen.selection()
    cu = w.cu_seqlens
    assert list(np.diff(cu)) == [7733, 14932, 24577, 8673]
    dcu = dev(cu)
    kc = nsa.nsa_compress_k(dev(w.k), cu_seqlens=dcu, max_seqlen=w.max_len)
    sc = nsa.nsa_cmp_scores_pool(dev(w.q), kc, w.hkv, cu_seqlens=dcu, max_seqlen=w.max_len)
    idx = nsa.nsa_topk_select(sc, 16, cu_seqlens=dcu, max_seqlen=w.max_len)
    one = nsa.nsa_select(dev(w.q), kc, w.hkv, k=16, cu_seqlens=dcu, max_seqlen=w.max_len)
    torch.cuda.synchronize()
    kch = host(kc)
    exact, rounded = orc.compress(w.k, cu)
    assert_close(kc, exact, atol=1e-6, rtol=2 ** -7, what="selection compress")
    assert np.mean(kch == rounded) > 0.999
    nb = sc.shape[-1]
    assert nb == -(-w.max_len // 64)
    starts, ends = cu[:-1], cu[1:] - 1
    special = np.concatenate([starts, ends] + [starts + t for t in (30, 31, 32, 47, 63, 64, 127, 128, 1023)])
    rows = np.unique(np.concatenate([_rng(13).integers(0, w.tokens, 400), special]))
    ref_sc = orc.cmp_scores_pool(w.q, kch, cu, rows=rows, nb_stride=nb)
    g_sc = host(sc)[rows].astype(np.float64)
    assert np.all(g_sc[ref_sc == 0] == 0)
    np.testing.assert_allclose(g_sc, ref_sc, rtol=1e-4, atol=1e-9)
    gi = host(idx)
    ref_idx = orc.topk(ref_sc, cu, k=16, rows=rows)
    n_mis, outside = selection_mismatches(gi[rows], ref_idx, ref_sc, _t_of_rows(cu)[rows])
    assert outside == 0, (n_mis, outside)
    assert n_mis <= max(3, len(rows) * w.hkv // 200), n_mis
    assert np.array_equal(gi, orc.topk(host(sc), cu, k=16))
    assert np.array_equal(host(one), gi)


def test_layer_varlen():
    """Packed sequences of ragged lengths (shorter than one compression window, one
    selection block, one sliding window, and longer): every tile of the tensor-core
    branches may mix keys of two sequences, which the masks must exclude."""
    lengths = [700, 65, 1300, 31, 200, 513]
    w = gen.layer(H=32, HKV=2, lengths=lengths)
    dcu = dev(w.cu_seqlens)
    idx = torch.empty((w.tokens, 2, 16), dtype=torch.int32, device="cuda")
    out = nsa.nsa_layer_fwd(dev(w.q), dev(w.k), dev(w.v), dev(w.gates), cu_seqlens=dcu, max_seqlen=max(lengths),
                            idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    gi = host(idx)
    ref = orc.layer(w.q, w.k, w.v, w.gates, w.cu_seqlens, idx_in=gi)
    _, kc = orc.compress(w.k, w.cu_seqlens)
    ref_sc = orc.cmp_scores_pool(w.q, kc, w.cu_seqlens)
    n_mis, outside = selection_mismatches(gi, ref["idx"], ref_sc, _t_of_rows(w.cu_seqlens))
    assert outside == 0, (n_mis, outside)
    assert_close(out, ref["o"], what="layer varlen")


def test_layer_full_size_sampled():
    """B=1, T=65536, H=64, Hkv=4, d=128: the three-branch layer, oracle on sampled rows."""
    w = gen.layer()
    idx = torch.empty((w.tokens, 4, 16), dtype=torch.int32, device="cuda")
    out = nsa.nsa_layer_fwd(dev(w.q), dev(w.k), dev(w.v), dev(w.gates), idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    gi = host(idx)
    rows = np.unique(np.concatenate([_rng(12).integers(0, w.tokens, 24), [0, 31, 32, 511, 512, 65535]]))
    ref = orc.layer(w.q, w.k, w.v, w.gates, w.cu_seqlens, idx_in=gi, rows=rows)
    assert_close(out[torch.from_numpy(rows).cuda()], ref["o"], what="layer full")
    _, kc = orc.compress(w.k, w.cu_seqlens)
    ref_sc = orc.cmp_scores_pool(w.q, kc, w.cu_seqlens, rows=rows)
    n_mis, outside = selection_mismatches(gi[rows], ref["idx"], ref_sc, rows)
    assert outside == 0, (n_mis, outside)


# --------------------------------------------------------------------------- block-mask variant
@pytest.mark.parametrize("B,T,H,causal,density", [(2, 1024, 4, True, 0.5), (2, 1024, 4, False, 0.5),
                                                  (1, 960, 2, False, 0.3), (3, 384, 2, True, 1.0)])
def test_block_sparse(B, T, H, causal, density):
    w = gen.block_sparse(B=B, T=T, H=H, density=density, causal=causal, salt=T)
    mask = w.idx
    if not causal:  # a query block with no active tile: zero output, lse -inf
        mask = mask.copy()
        mask[0, 0, 1, :] = 0
    lse = torch.empty((B * T, H), dtype=torch.float32, device="cuda")
    out = nsa.nsa_block_sparse_fwd(dev(w.q).view(B, T, H, 128), dev(w.k).view(B, T, H, 128),
                                   dev(w.v).view(B, T, H, 128), dev(mask), causal=causal, lse=lse)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    ref, ref_lse = orc.block_sparse_attn(w.q, w.k, w.v, mask, causal=causal)
    assert_close(out.reshape(B * T, H, 128), ref, what="block sparse")
    l = host(lse)
    assert np.array_equal(np.isneginf(l), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(l[fin], ref_lse[fin], atol=1e-3, rtol=1e-4)


def test_block_sparse_full_size_sampled():
    """B=8, T=16384, H=16, d=128, 50% of the 64x64 tiles (the pages' block-sparse table
    shape), causal; oracle on sampled rows."""
    w = gen.block_sparse()
    out = nsa.nsa_block_sparse_fwd(dev(w.q).view(8, 16384, 16, 128), dev(w.k).view(8, 16384, 16, 128),
                                   dev(w.v).view(8, 16384, 16, 128), dev(w.idx), causal=True)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([_rng(32).integers(0, w.tokens, 48), [0, 63, 64, 127, 128, 16383,
                                                                         7 * 16384 + 16383]]))
    ref, _ = orc.block_sparse_attn(w.q, w.k, w.v, w.idx, causal=True, rows=rows)
    g = out.reshape(w.tokens, 16, 128)[torch.from_numpy(rows).cuda()]
    assert_close(g, ref, what="block sparse full")


# --------------------------------------------------------------------------- sizes at the edges
def test_zero_token_calls():
    """A batch without tokens is valid input: every forward entry point returns without
    launching and leaves its (empty) outputs alone."""
    q = torch.empty((0, 16, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    cu = dev(np.zeros(2, np.int32))
    assert nsa.nsa_compress_k(kv, cu_seqlens=cu, max_seqlen=0).shape[0] == 0
    assert nsa.nsa_sparse_fwd(q, kv, kv, torch.empty((0, 1, 16), dtype=torch.int32, device="cuda"), 64,
                              cu_seqlens=cu, max_seqlen=0).shape == (0, 16, 128)
    assert nsa.nsa_swa_fwd(q, kv, kv, 512, cu_seqlens=cu, max_seqlen=0).shape == (0, 16, 128)
    assert nsa.nsa_cmp_attn_fwd(q, kv, kv, 1, cu_seqlens=cu, max_seqlen=0).shape == (0, 16, 128)
    sc = torch.empty((0, 1, 4), dtype=torch.float32, device="cuda")
    assert nsa.nsa_topk_select(sc, 16, cu_seqlens=cu, max_seqlen=0).shape == (0, 1, 16)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0


def test_sparse_fwd_longest_list():
    """S = 64, the longest block list the entry point takes: with every causal block of a
    4096-token sequence listed, selected attention is dense causal attention."""
    T, H, d, S = 4096, 16, 128, 64
    cu = gen.dense_cu_seqlens(1, T)
    rng = _rng(14)
    q, k, v = (gen.normal(rng, (T, hh, d), "bf16") for hh in (H, 1, 1))
    t = np.arange(T)
    idx = np.where(np.arange(S)[None, :] <= (t // 64)[:, None], np.arange(S)[None, :], -1).astype(np.int32)[:, None, :]
    out = nsa.nsa_sparse_fwd(dev(q), dev(k), dev(v), dev(idx), 64)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([_rng(15).integers(0, T, 200), [0, 1, 63, 64, 4095]]))
    ref, _ = orc.sparse_attn(q, k, v, idx, cu, 64, rows=rows)
    assert_close(out[torch.from_numpy(rows).cuda()], ref, what="S = 64")


def test_decode_longest_context():
    """A decode step at the longest context it takes (65536 tokens, 4095 compressed keys,
    1024 selection blocks), top-64, with a ragged second sequence."""
    B, L, k = 2, 65536, 64
    w, kc_cache = _decode_case(B, L, [65536, 40000], k, 0)
    ref_idx, _, ref_sc = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, want_scores=True)
    idx = torch.empty((B, w.hkv, k), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode(dev(w.q), dev(w.k_cache), dev(w.v_cache), dev(kc_cache), dev(w.seqlens), k=k,
                                idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    gi = host(idx)
    n_mis, outside = selection_mismatches(gi, ref_idx, ref_sc, np.asarray(w.seqlens) - 1)
    assert outside == 0, (n_mis, outside)
    _, ref_o = orc.decode(w.q, w.k_cache, w.v_cache, kc_cache, w.seqlens, k=k, idx_in=gi)
    assert_close(out, ref_o, what="decode at 65536")
