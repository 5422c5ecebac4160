"""The allocation-free decode entry point (nsa_sparse_decode_noalloc) against the
regular one (nsa_sparse_decode with a caller-provided workspace).

Callers such as allocator or memory-pool callbacks, runtimes that reserve all device
memory up front, or plug-ins given only their input and output buffers cannot allocate
scratch when a decode step runs; the allocation-free call serves them from a fixed
device array owned by the library.  It must give the same block choice and output as
the regular call, also when called twice in a row with different inputs (the shared
array keeps the previous call's contents).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_compress_gb300 as nsa
from sparse_attention_compress_gb300 import _lib
from sparse_attention_compress_gb300 import inputs as gen
from tests.parity import assert_close, dev, host


def _case(B, L, seqlens, seed):
    w = gen.decode(B=B, L=L, seqlens=seqlens, topk=64)
    rng = np.random.Generator(np.random.PCG64(seed))
    q = gen.normal(rng, w.q.shape, "bf16")  # a different query per case
    kc = dev(w.k_cache)
    kcmp = nsa.nsa_compress_k(kc).view(B, nsa.num_cmp(L), w.hkv, w.d)
    return dev(q), kc, dev(w.v_cache), kcmp, dev(w.seqlens), w


@pytest.mark.gpu
def test_noalloc_decode_matches_regular_decode_twice():
    cases = [(8, 8192, [8192, 8000, 5000, 4097, 100, 64, 33, 1], 1),
             (4, 4096, [4096, 1, 2500, 700], 2)]
    for B, L, seqlens, seed in cases:
        q, kc, vc, kcmp, sl, w = _case(B, L, seqlens, seed)
        ref_idx = torch.empty((B, w.hkv, 64), dtype=torch.int32, device="cuda")
        ref = nsa.nsa_sparse_decode(q, kc, vc, kcmp, sl, k=64, idx_out=ref_idx)
        idx = torch.full((B, w.hkv, 64), -7, dtype=torch.int32, device="cuda")
        out = torch.full_like(q, float("nan"))
        nsa.nsa_sparse_decode_noalloc(q, kc, vc, kcmp, sl, k=64, idx_out=idx, out=out)
        torch.cuda.synchronize()
        assert np.array_equal(host(idx), host(ref_idx))
        assert_close(out, _f64(ref), what="noalloc decode")


@pytest.mark.gpu
def test_noalloc_decode_keeps_its_block_lists_in_the_shared_array():
    """Without idx_out the block lists live in the shared array too.  A larger step first
    leaves its lists (and everything else) there; a smaller step after it, with other
    inputs, must still give the regular call's output."""
    big = _case(8, 8192, [8192, 8000, 5000, 4097, 100, 64, 33, 1], 3)
    small = _case(4, 4096, [4096, 1, 2500, 700], 4)
    for q, kc, vc, kcmp, sl, w in (big, small):
        ref = nsa.nsa_sparse_decode(q, kc, vc, kcmp, sl, k=64)
        out = torch.full_like(q, float("nan"))
        nsa.nsa_sparse_decode_noalloc(q, kc, vc, kcmp, sl, k=64, out=out)
        torch.cuda.synchronize()
        assert_close(out, _f64(ref), what="noalloc decode without idx_out")


def _f64(t):
    return host(t.float()).astype(np.float64)


def test_noalloc_rejects_steps_beyond_the_fixed_scratch():
    lib = nsa.load()
    cap = int(lib.nsa_sparse_decode_noalloc_max_bytes())
    assert cap == 16 << 20
    # 1024 sequences of 32768 tokens need far more scratch than the fixed array holds
    need = nsa.nsa_sparse_decode_workspace_size(1024, 32768, 16, 2, 128, k=64)
    assert need > cap
    fake = ctypes.c_void_p(0x10000)
    rc = lib.nsa_sparse_decode_noalloc(1024, fake, 32768, 16, 2, 128, fake, fake, fake, fake, 32, 16, 64, 1, 2, 64,
                                       0.0, None, fake, None)
    assert rc == 2
    msg = lib.nsa_last_error()
    assert b"scratch" in msg and str(cap).encode() in msg
