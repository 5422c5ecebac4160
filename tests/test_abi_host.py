"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
entry point its header declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

import sparse_attention_compress_gb300 as nsa
from sparse_attention_compress_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nsa.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^NSA_API\s+[\w\s\*]+?\b(nsa_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = nsa.load()
    names = _declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib._SIGS), "binding and header disagree"


def test_version_and_empty_error():
    lib = nsa.load()
    assert lib.nsa_version().startswith(b"nsa-gb300")


def _shape(**kw):
    s = _lib.NsaShape()
    s.batch, s.seqlen, s.h, s.h_kv, s.d, s.dtype = 1, 128, 16, 1, 128, _lib.NSA_BF16
    for k, v in kw.items():
        setattr(s, k, v)
    return s


P = ctypes.c_void_p
FAKE = P(0x10000)  # aligned, never dereferenced: every call below fails validation first
MIS = P(0x10008)


@pytest.mark.parametrize("kw,expect", [
    ({"h": 0}, 1), ({"h": 15, "h_kv": 2}, 1), ({"dtype": 7}, 1), ({"batch": -1}, 1), ({"d": 96}, 2),
])
def test_sparse_fwd_rejects_bad_shapes(kw, expect):
    lib = nsa.load()
    s = _shape(**kw)
    rc = lib.nsa_sparse_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, 16, 64, 0.0, FAKE, None, None)
    assert rc == expect
    assert lib.nsa_last_error()


def test_null_and_misaligned_pointers():
    lib = nsa.load()
    s = _shape()
    assert lib.nsa_sparse_fwd(ctypes.byref(s), None, FAKE, FAKE, FAKE, 16, 64, 0.0, FAKE, None, None) == 1
    assert b"null" in lib.nsa_last_error()
    assert lib.nsa_sparse_fwd(ctypes.byref(s), MIS, FAKE, FAKE, FAKE, 16, 64, 0.0, FAKE, None, None) == 1
    assert b"aligned" in lib.nsa_last_error()
    assert lib.nsa_sparse_fwd(None, FAKE, FAKE, FAKE, FAKE, 16, 64, 0.0, FAKE, None, None) == 1


def test_unsupported_parameters():
    lib = nsa.load()
    s = _shape(h=16, h_kv=2)
    assert lib.nsa_cmp_scores_pool(ctypes.byref(s), FAKE, FAKE, 32, 8, 64, 0.0, None, FAKE, 2, None) == 2
    assert lib.nsa_cmp_scores_pool(ctypes.byref(s), FAKE, FAKE, 32, 16, 64, 0.0, None, FAKE, 1, None) == 1
    assert lib.nsa_topk_select(ctypes.byref(s), FAKE, 2, 64, 1, 2, 65, FAKE, None) == 2
    assert lib.nsa_topk_select(ctypes.byref(s), FAKE, 4096, 64, 1, 2, 16, FAKE, None) == 2
    assert lib.nsa_compress_k(ctypes.byref(s), FAKE, FAKE, 40, 16, None) == 2
    assert lib.nsa_sparse_decode(2, FAKE, 1024, 16, 2, 64, FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 1, 2, 64, 0.0,
                                 None, FAKE, FAKE, 1 << 30, None) == 2
    assert lib.nsa_swa_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, 0, 0.0, FAKE, None, None, 0, None) == 1


def test_decode_workspace_checks():
    lib = nsa.load()
    need = nsa.nsa_sparse_decode_workspace_size(32, 32768, 16, 2, 128, k=64)
    assert need > 0
    rc = lib.nsa_sparse_decode(32, FAKE, 32768, 16, 2, 128, FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 1, 2, 64, 0.0,
                               None, FAKE, FAKE, need - 1, None)
    assert rc == 1 and b"workspace" in lib.nsa_last_error()
    rc = lib.nsa_sparse_decode(32, FAKE, 32768, 16, 2, 128, FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 1, 2, 64, 0.0,
                               None, FAKE, P(0x10010), need, None)
    assert rc == 1 and b"256-byte" in lib.nsa_last_error()


def test_empty_inputs_are_no_ops():
    lib = nsa.load()
    s = _shape(batch=0)
    assert lib.nsa_sparse_fwd(ctypes.byref(s), None, None, None, None, 16, 64, 0.0, None, None, None) == 0
    assert lib.nsa_gate_combine(0, 16, 128, None, None, None, None, None, None) == 0


def test_layer_workspace_size_scales_with_tokens():
    s1 = _lib.make_shape(65536, 64, 4, 128, _lib.NSA_BF16, batch=1, seqlen=65536)
    s2 = _lib.make_shape(32768, 64, 4, 128, _lib.NSA_BF16, batch=1, seqlen=32768)
    a, b = nsa.nsa_layer_fwd_workspace_size(s1), nsa.nsa_layer_fwd_workspace_size(s2)
    assert a > 1.9 * b > 0


def _items_per_seq_head(T, chunk=2048, block=64):
    """Brute-force count of dK/dV work items: one per (key block j, query chunk c) with
    the chunk reaching at or past the block's first key."""
    nb, nch = -(-T // block), -(-T // chunk)
    return sum(1 for j in range(nb) for c in range(nch) if (c + 1) * chunk > j * block)


@pytest.mark.parametrize("B,T,h,hkv", [(8, 16384, 16, 1), (2, 4500, 8, 2), (1, 64, 16, 16), (3, 1, 4, 1)])
def test_sparse_bwd_workspace_size(B, T, h, hkv):
    s = _shape(batch=B, seqlen=T, h=h, h_kv=hkv)
    got = nsa.nsa_sparse_bwd_workspace_size(s, 16)
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    dsum = a256(B * T * h * 4)
    part = a256(dsum + B * hkv * _items_per_seq_head(T) * 2 * 64 * 128 * 4)
    # group sizes 8 and 16 (the tensor-core dK/dV kernel): chunk-wise inverted lists, 2048 * S
    # token slots and an (offset, count) pair per key block for each (sequence, kv-head, chunk)
    lists = B * hkv * -(-T // 2048) if h // hkv in (8, 16) else 0
    nb = -(-T // 64)
    want = a256(a256(part + lists * 2048 * 16 * 4) + lists * nb * 8)
    assert got == want


def test_sparse_bwd_rejects_unsupported():
    lib = nsa.load()
    args = lambda s, S=16, bs=64, lse=FAKE, ws=FAKE, wsb=1 << 40: (  # noqa: E731
        ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, S, bs, 0.0, FAKE, lse, FAKE, FAKE, FAKE, FAKE, ws, wsb, None)
    assert lib.nsa_sparse_bwd(*args(_shape(d=64))) == 2
    assert lib.nsa_sparse_bwd(*args(_shape(dtype=_lib.NSA_F32))) == 2
    assert lib.nsa_sparse_bwd(*args(_shape(), bs=32)) == 2
    assert lib.nsa_sparse_bwd(*args(_shape(), S=65)) == 2
    assert lib.nsa_sparse_bwd(*args(_shape(h=32, h_kv=1))) == 2
    assert lib.nsa_sparse_bwd(*args(_shape(), lse=None)) == 1
    assert lib.nsa_sparse_bwd(*args(_shape(), ws=MIS)) == 1
    assert lib.nsa_sparse_bwd(*args(_shape(), wsb=16)) == 1
    assert b"workspace" in lib.nsa_last_error()
    assert lib.nsa_sparse_bwd(*args(_shape(batch=0))) == 0


@pytest.mark.parametrize("B,T,h,hkv", [(1, 65536, 64, 4), (2, 4500, 16, 1), (3, 31, 8, 2), (1, 2048 + 31, 16, 16)])
def test_cmp_attn_bwd_workspace_size(B, T, h, hkv):
    """Work items: (compressed key block j, 2048-query chunk c) with the chunk reaching the
    first query that sees block j (query 1024 j + 31 for windows of 32 at step 16)."""
    s = _shape(batch=B, seqlen=T, h=h, h_kv=hkv)
    n_c = (T - 32) // 16 + 1 if T >= 32 else 0
    nb, nch = -(-n_c // 64), -(-T // 2048)
    items = sum(1 for j in range(nb) for c in range(nch) if (c + 1) * 2048 > 1024 * j + 31)
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    want = a256(a256(B * T * h * 4) + B * hkv * items * 2 * 64 * 128 * 4)
    assert nsa.nsa_cmp_attn_bwd_workspace_size(s, 32, 16) == want


def test_cmp_attn_bwd_rejects_unsupported():
    lib = nsa.load()
    args = lambda s, ws=FAKE, wsb=1 << 40: (ctypes.byref(s), FAKE, FAKE, FAKE, 32, 16, 0.0, FAKE, FAKE, FAKE,  # noqa: E731
                                            FAKE, FAKE, FAKE, ws, wsb, None)
    assert lib.nsa_cmp_attn_bwd(*args(_shape(d=64))) == 2
    assert lib.nsa_cmp_attn_bwd(*args(_shape(seqlen=70000))) == 2
    assert lib.nsa_cmp_attn_bwd(*args(_shape(), wsb=8)) == 1
    assert lib.nsa_compress_bwd(ctypes.byref(_shape(d=12)), FAKE, 32, 16, FAKE, None) == 2


def test_new_entry_points_reject_bad_arguments():
    """Validation before any launch for the NOSA, backward and layer-training calls."""
    lib = nsa.load()
    s = _shape()
    # NOSA stage 2
    assert lib.nsa_cis_block_scores(ctypes.byref(s), FAKE, 32, 16, 64, 1, FAKE, None) == 1  # nb_stride too small
    assert lib.nsa_topk_two_stage(ctypes.byref(s), FAKE, 2, FAKE, 64, 1, 2, 8, 16, FAKE, None) == 2  # k > qk
    assert lib.nsa_topk_two_stage(ctypes.byref(s), FAKE, 2, FAKE, 64, 1, 2, 65, 16, FAKE, None) == 2  # qk > 64
    assert lib.nsa_sparse_cis_fwd(ctypes.byref(_shape(dtype=_lib.NSA_F32)), FAKE, FAKE, FAKE, FAKE, FAKE, 16, 64,
                                  0.0, FAKE, None, None) == 2
    assert lib.nsa_sparse_cis_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, 16, 32, 0.0, FAKE, None, None) == 2
    assert lib.nsa_sparse_cis_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, None, FAKE, 16, 64, 0.0, FAKE, None, None) == 1
    # NOSA decode: null CIS cache, qk outside [k, 64]
    dec = lambda cis, cb, qk: lib.nsa_sparse_decode_cis(  # noqa: E731
        2, FAKE, 4096, 16, 2, 128, FAKE, FAKE, FAKE, FAKE, cis, cb, 64, qk, 32, 16, 64, 1, 2, 16, 0.0, None, FAKE,
        FAKE, 1 << 30, None)
    assert dec(None, None, 0) == 1
    assert dec(FAKE, FAKE, 8) == 2
    assert dec(FAKE, FAKE, 65) == 2
    # sliding-window and gate backward
    sw = lambda window, ws=FAKE, wsb=1 << 40: lib.nsa_swa_bwd(  # noqa: E731
        ctypes.byref(s), FAKE, FAKE, FAKE, window, 0.0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, wsb, None)
    assert sw(1985) == 2 and sw(0) == 2
    assert sw(512, wsb=8) == 1
    assert lib.nsa_gate_combine_bwd(10, 4, 12, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 2
    assert lib.nsa_gate_combine_bwd(10, 4, 128, FAKE, FAKE, FAKE, FAKE, MIS, FAKE, FAKE, FAKE, FAKE, None) == 1
    # layer training pair
    assert lib.nsa_layer_fwd_train(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 16, 1, 2, 512, 0.0, FAKE,
                                   None, FAKE, 1 << 40, None) == 1
    assert lib.nsa_layer_bwd(ctypes.byref(_shape(d=64)), FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 16, 512, 0.0, None,
                             FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 2
    assert lib.nsa_layer_bwd(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 16, 4000, 0.0, None,
                             FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 2
    assert lib.nsa_layer_bwd(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 16, 512, 0.0, None,
                             FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 1  # saved is NULL


@pytest.mark.parametrize("T,h,hkv,window", [(65536, 64, 4, 512), (1000, 16, 2, 1984)])
def test_layer_bwd_workspace_size(T, h, hkv, window):
    """Branch gradients, per-branch dq/dk/dv and compressed-key gradients, plus the largest
    branch-backward scratch (used in turn)."""
    lib = nsa.load()
    s = _shape(seqlen=T, h=h, h_kv=hkv)
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    qsz, ksz = T * h * 128 * 2, T * hkv * 128 * 2
    ncr = (T - 32) // 16 + 1
    off = 0
    for sz in (3 * qsz, 3 * qsz, 3 * ksz, 3 * ksz, ncr * hkv * 256, ncr * hkv * 256):
        off = a256(off + sz)
    scratch = max(lib.nsa_sparse_bwd_workspace_size(ctypes.byref(s), 16, 64),
                  lib.nsa_cmp_attn_bwd_workspace_size(ctypes.byref(s), 32, 16),
                  lib.nsa_swa_bwd_workspace_size(ctypes.byref(s), window))
    got = lib.nsa_layer_bwd_workspace_size(ctypes.byref(s), 32, 16, 64, 16, window)
    assert got == a256(off + scratch)


def test_select_block_mask_cmp_layer_reject_bad_arguments():
    """The entry points without a dedicated host check above: each rejects an
    unsupported or malformed argument with its status and a message, before any launch."""
    lib = nsa.load()
    s = _shape()  # B 1, T 128, h 16, h_kv 1, d 128, bf16
    ref = ctypes.byref

    def select(shape=s, kernel=32, k=16, n_init=1, ws=P(0x10000), ws_bytes=1 << 20):
        return lib.nsa_select(ref(shape), FAKE, FAKE, kernel, 16, 64, 0.0, n_init, 2, k, FAKE, ws, ws_bytes, None)

    assert select(kernel=16) == 2
    assert select(k=65) == 2
    assert select(n_init=-1) == 1
    assert select(shape=_shape(d=96)) == 2
    assert select(shape=_shape(dtype=_lib.NSA_F32)) == 2
    assert select(ws=P(0x10100 + 16)) == 1 and b"aligned" in lib.nsa_last_error()
    assert select(ws_bytes=512) == 1 and b"workspace" in lib.nsa_last_error()
    assert select(ws=None) == 1

    def block_mask(shape, block_size=64, mask=FAKE, ws_bytes=1 << 30):
        return lib.nsa_block_sparse_fwd(ref(shape), FAKE, FAKE, FAKE, mask, block_size, 1, 0.0, FAKE, None, FAKE,
                                        ws_bytes, None)

    mh = dict(h=2, h_kv=2)
    assert block_mask(_shape()) == 2  # needs h_kv == h
    assert block_mask(_shape(d=64, **mh)) == 2
    assert block_mask(_shape(seqlen=100, **mh)) == 2
    assert block_mask(_shape(**mh), block_size=32) == 2
    assert block_mask(_shape(**mh), mask=None) == 1
    assert block_mask(_shape(**mh), ws_bytes=256) == 1 and b"workspace" in lib.nsa_last_error()

    def cmp_fwd(shape=s, kernel=32, lse=None, ws=FAKE, ws_bytes=1 << 30):
        return lib.nsa_cmp_attn_fwd(ref(shape), FAKE, FAKE, FAKE, kernel, 16, 0.0, FAKE, lse, ws, ws_bytes, None)

    assert cmp_fwd(shape=_shape(dtype=_lib.NSA_F32)) == 2
    assert cmp_fwd(shape=_shape(h=12, h_kv=4)) == 2  # group of 3 heads
    assert cmp_fwd(kernel=0) == 1
    assert cmp_fwd(lse=P(0x10002)) == 1 and b"misaligned" in lib.nsa_last_error()
    # d 128 with a power-of-two group runs on the tensor cores and needs the V^T workspace
    assert cmp_fwd(ws=None) == 1 and b"workspace" in lib.nsa_last_error()
    assert cmp_fwd(ws_bytes=256) == 1 and b"workspace" in lib.nsa_last_error()
    assert lib.nsa_swa_fwd(ref(s), FAKE, FAKE, FAKE, 512, 0.0, FAKE, None, None, 0, None) == 1
    assert b"workspace" in lib.nsa_last_error()


    def layer(shape=s, kernel=32, S=16, window=512, ws_bytes=1 << 30):
        return lib.nsa_layer_fwd(ref(shape), FAKE, FAKE, FAKE, FAKE, kernel, 16, 64, S, 1, 2, window, 0.0, FAKE,
                                 None, FAKE, ws_bytes, None)

    assert layer(kernel=16) == 2
    assert layer(S=65) == 2
    assert layer(window=0) == 1
    assert layer(shape=_shape(h=32, h_kv=1)) == 2  # group of 32 heads: selection limit
    need = lib.nsa_layer_fwd_workspace_size(ref(s), 32, 16, 64, 16)
    assert need > 0 and need % 256 == 0
    assert layer(ws_bytes=need - 1) == 1 and b"workspace" in lib.nsa_last_error()


@pytest.mark.parametrize("B,T,h,hkv,d,tc", [(1, 128, 16, 1, 128, True), (2, 1000, 16, 2, 128, True),
                                            (3, 100, 64, 1, 128, True), (2, 100, 48, 1, 128, False),
                                            (2, 100, 16, 1, 64, False)])
def test_branch_workspace_sizes(B, T, h, hkv, d, tc):
    """The compressed and sliding branches ask for V transposed (bf16, rows padded to 64 per
    kv-head) exactly when they run on the tensor cores (d 128, power-of-two group)."""
    lib = nsa.load()
    s = _shape(batch=B, seqlen=T, h=h, h_kv=hkv, d=d)
    pad = lambda rows: -(-rows // 64) * 64
    up = lambda x: -(-x // 256) * 256
    n_c = max(0, (T - 32) // 16 + 1)
    want_cmp = up(pad(B * n_c) * hkv * d * 2) if tc else 0
    want_swa = up(pad(B * T) * hkv * d * 2) if tc else 0
    assert lib.nsa_cmp_attn_fwd_workspace_size(ctypes.byref(s), 32, 16) == want_cmp
    assert lib.nsa_swa_fwd_workspace_size(ctypes.byref(s)) == want_swa

@pytest.mark.parametrize("B,T,hkv", [(1, 128, 1), (2, 1000, 2), (3, 64, 4)])
def test_select_and_block_mask_workspace_sizes(B, T, hkv):
    lib = nsa.load()
    s = _shape(batch=B, seqlen=T, h=16, h_kv=hkv)
    nb = -(-T // 64)
    want = B * T * hkv * nb * 4
    assert lib.nsa_select_workspace_size(ctypes.byref(s), 64) == -(-want // 256) * 256
    assert lib.nsa_select_workspace_size(ctypes.byref(s), 0) == 0
    m = _shape(batch=B, seqlen=T, h=hkv, h_kv=hkv)
    ws = lib.nsa_block_sparse_workspace_size(ctypes.byref(m))
    assert ws % 256 == 0 and ws >= hkv * 128 * B * T * 2  # V transposed per head, bf16
    assert lib.nsa_block_sparse_workspace_size(ctypes.byref(_shape(h=0))) == 0


def test_decode_noalloc_refuses_steps_beyond_its_scratch():
    """A supported step whose scratch exceeds the fixed array is refused with the sizes,
    before any CUDA call; sizes the decode step does not support get the regular entry
    point's message, not the scratch one."""
    lib = nsa.load()
    cap = lib.nsa_sparse_decode_noalloc_max_bytes()
    assert cap > 0
    big = (1024, 32768, 16, 2, 128, 32, 16, 64, 64)  # batch, max_len, h, h_kv, d, kernel, stride, block, k
    assert lib.nsa_sparse_decode_workspace_size(*big) > cap
    B, L, h, hkv, d, kern, st, bs, k = big
    rc = lib.nsa_sparse_decode_noalloc(B, FAKE, L, h, hkv, d, FAKE, FAKE, FAKE, FAKE, kern, st, bs, 1, 2, k, 0.0,
                                       None, FAKE, None)
    assert rc == 2
    msg = lib.nsa_last_error()
    assert b"scratch" in msg and str(cap).encode() in msg
    # unsupported sizes whose scratch would also exceed the array: the size check speaks
    for args, word in [((256, 131072, 64, 4, 128, 32, 16, 64, 64), b"max_len"),
                       ((1024, 32768, 16, 2, 128, 32, 16, 64, 65), b"k must"),
                       ((1024, 32768, 16, 2, 64, 32, 16, 64, 64), b"d must"),
                       ((1024, 32768, 16, 2, 128, 64, 16, 64, 64), b"kernel 32")]:
        B, L, h, hkv, d, kern, st, bs, k = args
        rc = lib.nsa_sparse_decode_noalloc(B, FAKE, L, h, hkv, d, FAKE, FAKE, FAKE, FAKE, kern, st, bs, 1, 2, k,
                                           0.0, None, FAKE, None)
        msg = lib.nsa_last_error()
        assert rc == 2 and word in msg and b"scratch" not in msg, (args, msg)
    rc = lib.nsa_sparse_decode_noalloc(2, FAKE, 1024, 0, 1, 128, FAKE, FAKE, FAKE, FAKE, 32, 16, 64, 1, 2, 16, 0.0,
                                       None, FAKE, None)
    assert rc == 1
