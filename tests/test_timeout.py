"""Bounded waits that run out, on purpose, without breaking any kernel.

The kernels that wait (the tensor-core branches and the TMA-fed selected attention of the
layer, the decode step's wait for a row's block list, the tensor-core dK / dV and dQ of
the backward) bound every first-level wait.  Here
that limit is set to 1 ns through the C ABI (nsa_set_wait_limit_ns), far below any wait's
normal length; nothing else changes: no copy is withheld, no barrier left unarrived.  The
waits give up, the kernels set the device status word to NSA_ERR_TIMEOUT, drain the copies
and tensor-core work they have in flight and return, so the stream synchronises and the
context stays usable.  With the limit and the word reset, the next call is checked against
the oracle.
"""
import numpy as np
import pytest
import torch

import sparse_attention_compress_gb300 as nsa
from oracle import oracle as orc
from sparse_attention_compress_gb300 import inputs as gen
from tests.parity import assert_close, dev, host

pytestmark = pytest.mark.gpu

NSA_ERR_TIMEOUT = 4


def _flush_l2():
    """Write a buffer larger than the L2 (129 MB): the first copies of the next kernel then
    come from DRAM, slower than a wait's first probe, so a 1 ns limit runs out."""
    buf = torch.empty(96 * 2 ** 20, dtype=torch.float32, device="cuda")
    buf.fill_(1.0)
    torch.cuda.synchronize()
    del buf


@pytest.fixture
def clean_status():
    assert nsa.nsa_device_status(reset=True) == 0
    yield
    nsa.nsa_set_wait_limit_ns(0)
    nsa.nsa_device_status(reset=True)


def _decode_inputs():
    B, L, seqlens, k = 8, 4096, [4096, 4000, 3000, 2500, 1000, 700, 70, 1], 16
    w = gen.decode(B=B, L=L, seqlens=seqlens, topk=k)
    kc = nsa.nsa_compress_k(dev(w.k_cache)).view(B, orc.num_cmp(L), w.hkv, w.d)
    return w, kc, k


def test_decode_wait_runs_out_then_recovers(clean_status):
    w, kc, k = _decode_inputs()
    q, kcache, vcache, sl = dev(w.q), dev(w.k_cache), dev(w.v_cache), dev(w.seqlens)
    torch.cuda.synchronize()
    _flush_l2()
    nsa.nsa_set_wait_limit_ns(1)
    nsa.nsa_sparse_decode(q, kcache, vcache, kc, sl, k=k)
    torch.cuda.synchronize()  # the kernel returned: no hang, no fault
    assert nsa.nsa_device_status(reset=True) == NSA_ERR_TIMEOUT
    nsa.nsa_set_wait_limit_ns(0)
    idx = torch.empty((w.batch, w.hkv, k), dtype=torch.int32, device="cuda")
    out = nsa.nsa_sparse_decode(q, kcache, vcache, kc, sl, k=k, idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    _, ref_o = orc.decode(w.q, w.k_cache, w.v_cache, host(kc), w.seqlens, k=k, idx_in=host(idx))
    assert_close(out, ref_o, what="decode after a timeout")


def test_selected_attention_wait_runs_out_then_recovers(clean_status):
    lengths = [2000, 900, 65]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = np.random.Generator(np.random.PCG64(41))
    q, k, v = (gen.normal(rng, (cu[-1], hh, 128), "bf16") for hh in (16, 1, 1))
    idx = gen.random_block_indices(rng, cu, 1, 16, 64, force_first=True)
    dq, dk, dv, di, dcu = dev(q), dev(k), dev(v), dev(idx), dev(cu)
    torch.cuda.synchronize()
    _flush_l2()
    nsa.nsa_set_wait_limit_ns(1)
    nsa.nsa_sparse_fwd(dq, dk, dv, di, 64, cu_seqlens=dcu, max_seqlen=max(lengths))
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(reset=True) == NSA_ERR_TIMEOUT
    nsa.nsa_set_wait_limit_ns(0)
    out = nsa.nsa_sparse_fwd(dq, dk, dv, di, 64, cu_seqlens=dcu, max_seqlen=max(lengths))
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    ref, _ = orc.sparse_attn(q, k, v, idx, cu, 64)
    assert_close(out, ref, what="selected attention after a timeout")


def test_layer_wait_runs_out_then_recovers(clean_status):
    T, H, hkv = 1100, 16, 2
    w = gen.layer(T=T, H=H, HKV=hkv)
    q, k, v, g = dev(w.q), dev(w.k), dev(w.v), dev(w.gates)
    torch.cuda.synchronize()
    _flush_l2()
    nsa.nsa_set_wait_limit_ns(1)
    nsa.nsa_layer_fwd(q, k, v, g)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(reset=True) == NSA_ERR_TIMEOUT
    nsa.nsa_set_wait_limit_ns(0)
    idx = torch.empty((T, hkv, 16), dtype=torch.int32, device="cuda")
    out = nsa.nsa_layer_fwd(q, k, v, g, idx_out=idx)
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    ref = orc.layer(w.q, w.k, w.v, w.gates, w.cu_seqlens, idx_in=host(idx))
    assert_close(out, ref["o"], what="layer after a timeout")


def test_sparse_bwd_wait_runs_out_then_recovers(clean_status):
    """The tensor-core dK / dV kernel (group size 16): its producer, MMA and softmax roles
    give up, drain the gathers and products in flight and free the TMEM."""
    lengths = [2100, 700, 65]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = np.random.Generator(np.random.PCG64(43))
    q, do = (gen.normal(rng, (cu[-1], 16, 128), "bf16") for _ in range(2))
    k, v = (gen.normal(rng, (cu[-1], 1, 128), "bf16") for _ in range(2))
    idx = gen.random_block_indices(rng, cu, 1, 8, 64, force_first=True)
    o64, lse64 = orc.sparse_attn(q, k, v, idx, cu, 64)
    o, lse = gen.f32_to_bf16_bits(o64.astype(np.float32)), lse64.astype(np.float32)
    args = [dev(x) for x in (q, k, v, idx, o, lse, do)]
    dcu = dev(cu)
    torch.cuda.synchronize()
    _flush_l2()
    nsa.nsa_set_wait_limit_ns(1)
    nsa.nsa_sparse_bwd(*args, 64, cu_seqlens=dcu, max_seqlen=max(lengths))
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(reset=True) == NSA_ERR_TIMEOUT
    nsa.nsa_set_wait_limit_ns(0)
    gq, gk, gv = nsa.nsa_sparse_bwd(*args, 64, cu_seqlens=dcu, max_seqlen=max(lengths))
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    rq, rk, rv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, 64, o=o)
    assert_close(gq, rq, what="dq after a timeout")
    assert_close(gk, rk, what="dk after a timeout")
    assert_close(gv, rv, what="dv after a timeout")


def test_cmp_bwd_wait_runs_out_then_recovers(clean_status):
    """The compressed branch's tensor-core dQ (its S, dP and dQ issuing warps) and dK / dV
    kernels (group size 16): every role gives up, drains the copies and products in flight
    and frees the TMEM; the next call with the default limit is correct."""
    lengths = [2100, 700, 65]
    cu = gen.varlen_cu_seqlens(lengths)
    rng = np.random.Generator(np.random.PCG64(44))
    q, do = (gen.normal(rng, (cu[-1], 16, 128), "bf16") for _ in range(2))
    k, v = (gen.normal(rng, (cu[-1], 1, 128), "bf16") for _ in range(2))
    _, kc = orc.compress(k, cu)
    _, vc = orc.compress(v, cu)
    o64, lse64 = orc.cmp_attn(q, kc, vc, cu)
    o, lse = gen.f32_to_bf16_bits(o64.astype(np.float32)), lse64.astype(np.float32)
    args = [dev(x) for x in (q, kc, vc, o, lse, do)]
    dcu = dev(cu)
    torch.cuda.synchronize()
    _flush_l2()
    nsa.nsa_set_wait_limit_ns(1)
    nsa.nsa_cmp_attn_bwd(*args, 1, cu_seqlens=dcu, max_seqlen=max(lengths))
    torch.cuda.synchronize()
    assert nsa.nsa_device_status(reset=True) == NSA_ERR_TIMEOUT
    nsa.nsa_set_wait_limit_ns(0)
    gq, gk, gv = nsa.nsa_cmp_attn_bwd(*args, 1, cu_seqlens=dcu, max_seqlen=max(lengths))
    torch.cuda.synchronize()
    assert nsa.nsa_device_status() == 0
    rq, rk, rv = orc.cmp_attn_bwd(q, kc, vc, do, cu, o=o)
    assert_close(gq, rq, what="cmp dq after a timeout")
    assert_close(gk, rk, what="cmp dk after a timeout")
    assert_close(gv, rv, what="cmp dv after a timeout")
