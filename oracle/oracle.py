"""ctypes binding of the plain CPU oracle (``nsa_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline / reference arm are the only users.  The CUDA library
never loads it and it never loads the CUDA library.

Arrays are numpy: bf16 tensors travel as ``uint16`` bit patterns, fp32 as
``float32``; every floating-point result comes back as ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nsa_oracle.c")
_SO = os.path.join(_HERE, "libnsa_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fp contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_SO)
        _lib.nsa_oracle_num_cmp.restype = ctypes.c_int
        _lib.nsa_oracle_threads.restype = ctypes.c_int
    return _lib


def _p(a):
    return ctypes.c_void_p(0 if a is None else a.ctypes.data)


def _dt(a) -> int:
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float32:
        return 0
    raise TypeError(f"oracle inputs must be bf16 bits (uint16) or float32, got {a.dtype}")


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _rows(rows, total):
    if rows is None:
        return None, total
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, len(r)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def threads() -> int:
    return _load().nsa_oracle_threads()


def num_cmp(L: int, kernel: int = 32, stride: int = 16) -> int:
    return _load().nsa_oracle_num_cmp(int(L), int(kernel), int(stride))


def cmp_offsets(cu, kernel=32, stride=16):
    cu = np.asarray(cu)
    n = [num_cmp(int(cu[i + 1] - cu[i]), kernel, stride) for i in range(len(cu) - 1)]
    return np.concatenate([[0], np.cumsum(n)]).astype(np.int64)


def compress(k, cu, kernel=32, stride=16):
    """S1: returns (exact fp64 means, means rounded to k's dtype), both [n_cmp, hkv, d]."""
    k = np.ascontiguousarray(k)
    cu = _i32(cu)
    _, hkv, d = k.shape
    n = int(cmp_offsets(cu, kernel, stride)[-1])
    exact = np.zeros((n, hkv, d), np.float64)
    rounded = np.zeros((n, hkv, d), k.dtype)
    _check(_load().nsa_oracle_compress(_p(k), _dt(k), _p(cu), len(cu) - 1, hkv, d, kernel, stride,
                                       _p(exact), _p(rounded)), "compress")
    return exact, rounded


def cmp_probs(q, kc, cu, kernel=32, stride=16, scale=None, rows=None, nc_stride=None):
    """S2: group-summed probabilities P_g [rows, hkv, nc_stride]."""
    q, kc, cu = np.ascontiguousarray(q), np.ascontiguousarray(kc), _i32(cu)
    tot, h, d = q.shape
    hkv = kc.shape[1]
    scale = d ** -0.5 if scale is None else scale
    if nc_stride is None:
        nc_stride = max(1, max(num_cmp(int(cu[i + 1] - cu[i]), kernel, stride) for i in range(len(cu) - 1)))
    rows, n = _rows(rows, tot)
    out = np.zeros((n, hkv, nc_stride), np.float64)
    _check(_load().nsa_oracle_cmp_probs(_p(q), _p(kc), _dt(q), _p(cu), len(cu) - 1, h, hkv, d, kernel,
                                        stride, ctypes.c_double(scale), _p(rows), ctypes.c_int64(n),
                                        _p(out), nc_stride), "cmp_probs")
    return out


def pool_row(pg, n_c, n_b, block_size=64, kernel=32, stride=16):
    """S3 on one row of group probabilities."""
    pg = np.ascontiguousarray(np.asarray(pg, np.float64))
    out = np.zeros(n_b, np.float64)
    _check(_load().nsa_oracle_pool_row(_p(pg), int(n_c), int(n_b), block_size, kernel, stride, _p(out)),
           "pool_row")
    return out


def cmp_scores_pool(q, kc, cu, kernel=32, stride=16, block_size=64, scale=None, rows=None,
                    nb_stride=None):
    """S2+S3: pooled block scores [rows, hkv, nb_stride]."""
    q, kc, cu = np.ascontiguousarray(q), np.ascontiguousarray(kc), _i32(cu)
    tot, h, d = q.shape
    hkv = kc.shape[1]
    scale = d ** -0.5 if scale is None else scale
    if nb_stride is None:
        nb_stride = max(1, -(-int(np.max(np.diff(cu))) // block_size))
    rows, n = _rows(rows, tot)
    out = np.zeros((n, hkv, nb_stride), np.float64)
    _check(_load().nsa_oracle_cmp_scores_pool(_p(q), _p(kc), _dt(q), _p(cu), len(cu) - 1, h, hkv, d,
                                              kernel, stride, block_size, ctypes.c_double(scale),
                                              _p(rows), ctypes.c_int64(n), _p(out), nb_stride),
           "cmp_scores_pool")
    return out


def topk(scores, cu, block_size=64, n_init=1, n_local=2, k=16, rows=None):
    """S4: block indices [rows, hkv, k] from scores [rows, hkv, nb_stride] (float64 or float32)."""
    scores = np.ascontiguousarray(np.asarray(scores, np.float64))
    cu = _i32(cu)
    n_rows, hkv, nb_stride = scores.shape
    rows, n = _rows(rows, int(cu[-1]))
    if n != n_rows:
        raise ValueError("scores must have one row per requested token")
    out = np.zeros((n, hkv, k), np.int32)
    _check(_load().nsa_oracle_topk(_p(scores), nb_stride, _p(cu), len(cu) - 1, hkv, block_size, n_init,
                                   n_local, k, _p(rows), ctypes.c_int64(n), _p(out)), "topk")
    return out


def sparse_attn(q, k, v, idx, cu, block_size=64, scale=None, rows=None):
    """S5: selected-block attention; returns (o [rows,h,d], lse [rows,h]) in fp64."""
    q, k, v, idx, cu = (np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v),
                        _i32(idx), _i32(cu))
    tot, h, d = q.shape
    hkv = k.shape[1]
    S = idx.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    rows, n = _rows(rows, tot)
    o = np.zeros((n, h, d), np.float64)
    lse = np.zeros((n, h), np.float64)
    _check(_load().nsa_oracle_sparse_attn(_p(q), _p(k), _p(v), _dt(q), _p(cu), len(cu) - 1, h, hkv, d,
                                          _p(idx), S, block_size, ctypes.c_double(scale), _p(rows),
                                          ctypes.c_int64(n), _p(o), _p(lse)), "sparse_attn")
    return o, lse


def sparse_attn_bwd(q, k, v, idx, do, cu, block_size=64, scale=None, q_rows=None, kv_rows=None, want_dq=True,
                    want_dkv=True, o=None):
    """Backward of S5 for upstream gradient do [tokens, h, d] (same dtype as q).
    Returns (dq [q_rows, h, d], dk [kv_rows, hkv, d], dv [kv_rows, hkv, d]) in fp64; a
    part not wanted is None.  q_rows / kv_rows select token rows (all when None).
    o (optional, like q): the stored forward output; D = dO . o is then taken from it
    instead of the exact sum over the row's keys."""
    q, k, v, do, idx, cu = (np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v),
                            np.ascontiguousarray(do), _i32(idx), _i32(cu))
    if do.dtype != q.dtype or do.shape != q.shape:
        raise ValueError("do must match q in dtype and shape")
    if o is not None:
        o = np.ascontiguousarray(o)
        if o.dtype != q.dtype or o.shape != q.shape:
            raise ValueError("o must match q in dtype and shape")
    tot, h, d = q.shape
    hkv = k.shape[1]
    S = idx.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    qr, nq = _rows(q_rows, tot)
    kr, nkv = _rows(kv_rows, tot)
    if not want_dq:
        nq = -1
    if not want_dkv:
        nkv = -1
    dq = np.zeros((max(nq, 0), h, d), np.float64)
    dk = np.zeros((max(nkv, 0), hkv, d), np.float64)
    dv = np.zeros((max(nkv, 0), hkv, d), np.float64)
    _check(_load().nsa_oracle_sparse_attn_bwd(_p(q), _p(k), _p(v), _p(do), _p(o), _dt(q), _p(cu), len(cu) - 1, h, hkv,
                                              d, _p(idx), S, block_size, ctypes.c_double(scale), _p(qr),
                                              ctypes.c_int64(nq), _p(dq), _p(kr), ctypes.c_int64(nkv), _p(dk),
                                              _p(dv)), "sparse_attn_bwd")
    return (dq if want_dq else None), (dk if want_dkv else None), (dv if want_dkv else None)


def cis_block_scores(cis, cu, kernel=32, stride=16, block_size=64, nb_stride=None):
    """NOSA stage 2: CIS [tokens, hkv] pooled over the compressor's windows, then to
    blocks as in S3; returns [n_seqs, hkv, nb_stride] fp64."""
    cis = np.ascontiguousarray(np.asarray(cis, np.float64))
    cu = _i32(cu)
    hkv = cis.shape[1]
    if nb_stride is None:
        nb_stride = max(1, -(-int(np.max(np.diff(cu))) // block_size))
    out = np.zeros((len(cu) - 1, hkv, nb_stride), np.float64)
    _check(_load().nsa_oracle_cis_block_scores(_p(cis), _p(cu), len(cu) - 1, hkv, kernel, stride, block_size,
                                               nb_stride, _p(out)), "cis_block_scores")
    return out


def topk_two_stage(scores, cis_scores, cu, qk_select, k, block_size=64, n_init=1, n_local=2, rows=None):
    """NOSA two-stage selection: S4 with k = qk_select on the attention block scores, then
    the best k of those by pooled CIS score (forced blocks kept).  [rows, hkv, k] int32."""
    scores = np.ascontiguousarray(np.asarray(scores, np.float64))
    cis_scores = np.ascontiguousarray(np.asarray(cis_scores, np.float64))
    cu = _i32(cu)
    n, hkv, nb_stride = scores.shape
    if cis_scores.shape != (len(cu) - 1, hkv, nb_stride):
        raise ValueError("cis_scores must be [n_seqs, hkv, nb_stride]")
    rows, nr = _rows(rows, int(cu[-1]))
    if nr != n:
        raise ValueError("scores must have one row per requested token")
    out = np.zeros((n, hkv, k), np.int32)
    _check(_load().nsa_oracle_topk_two_stage(_p(scores), nb_stride, _p(cis_scores), _p(cu), len(cu) - 1, hkv,
                                             block_size, n_init, n_local, qk_select, k, _p(rows),
                                             ctypes.c_int64(n), _p(out)), "topk_two_stage")
    return out


def sparse_attn_cis(q, k, v, cis, idx, cu, block_size=64, scale=None, rows=None):
    """NOSA sparse_forward: selected attention with weights p_e * cis_e (normalised);
    returns (o [rows,h,d], lse [rows,h]) fp64."""
    q, k, v, idx, cu = (np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v), _i32(idx),
                        _i32(cu))
    cis = np.ascontiguousarray(np.asarray(cis, np.float64))
    tot, h, d = q.shape
    hkv = k.shape[1]
    if cis.shape != (tot, hkv):
        raise ValueError("cis must be [tokens, hkv]")
    S = idx.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    rows, n = _rows(rows, tot)
    o = np.zeros((n, h, d), np.float64)
    lse = np.zeros((n, h), np.float64)
    _check(_load().nsa_oracle_sparse_attn_cis(_p(q), _p(k), _p(v), _dt(q), _p(cis), _p(cu), len(cu) - 1, h, hkv, d,
                                              _p(idx), S, block_size, ctypes.c_double(scale), _p(rows),
                                              ctypes.c_int64(n), _p(o), _p(lse)), "sparse_attn_cis")
    return o, lse


def swa(q, k, v, cu, window=512, scale=None, rows=None):
    """S8: sliding-window attention; returns (o, lse)."""
    q, k, v, cu = np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v), _i32(cu)
    tot, h, d = q.shape
    hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    rows, n = _rows(rows, tot)
    o = np.zeros((n, h, d), np.float64)
    lse = np.zeros((n, h), np.float64)
    _check(_load().nsa_oracle_swa(_p(q), _p(k), _p(v), _dt(q), _p(cu), len(cu) - 1, h, hkv, d, window,
                                  ctypes.c_double(scale), _p(rows), ctypes.c_int64(n), _p(o), _p(lse)),
           "swa")
    return o, lse


def block_sparse_attn(q, k, v, mask, causal=True, block=64, scale=None, rows=None):
    """Block-mask sparse attention; q [B*T, h, d], k/v [B*T, hkv, d], mask uint8
    [B, h, nb, nb]; returns (o, lse) for the requested token rows."""
    q, k, v = np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v)
    mask = np.ascontiguousarray(np.asarray(mask, dtype=np.uint8))
    B, h, nb, _ = mask.shape
    tot, _, d = q.shape
    T = tot // B
    hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    rows, n = _rows(rows, tot)
    o = np.zeros((n, h, d), np.float64)
    lse = np.zeros((n, h), np.float64)
    _check(_load().nsa_oracle_block_sparse_attn(_p(q), _p(k), _p(v), _dt(q), B, T, h, hkv, d, _p(mask), block,
                                                int(bool(causal)), ctypes.c_double(scale), _p(rows),
                                                ctypes.c_int64(n), _p(o), _p(lse)),
           "block_sparse_attn")
    return o, lse


def cmp_attn(q, kc, vc, cu, kernel=32, stride=16, scale=None, rows=None):
    """S7: compressed-attention branch over stored compressed keys/values; (o, lse)."""
    q, kc, vc, cu = (np.ascontiguousarray(q), np.ascontiguousarray(kc), np.ascontiguousarray(vc),
                     _i32(cu))
    tot, h, d = q.shape
    hkv = kc.shape[1]
    scale = d ** -0.5 if scale is None else scale
    rows, n = _rows(rows, tot)
    o = np.zeros((n, h, d), np.float64)
    lse = np.zeros((n, h), np.float64)
    _check(_load().nsa_oracle_cmp_attn(_p(q), _p(kc), _p(vc), _dt(q), _p(cu), len(cu) - 1, h, hkv, d,
                                       kernel, stride, ctypes.c_double(scale), _p(rows),
                                       ctypes.c_int64(n), _p(o), _p(lse)), "cmp_attn")
    return o, lse


def cmp_attn_bwd(q, kc, vc, do, cu, kernel=32, stride=16, scale=None, q_rows=None, kv_rows=None, want_dq=True,
                 want_dkv=True, o=None):
    """Backward of S7 for upstream gradient do: (dq [q_rows, h, d], dkc, dvc [kv_rows, hkv, d]) fp64
    (kv_rows index the packed compressed rows).  o: optional stored forward output for D."""
    q, kc, vc, do, cu = (np.ascontiguousarray(q), np.ascontiguousarray(kc), np.ascontiguousarray(vc),
                         np.ascontiguousarray(do), _i32(cu))
    if do.dtype != q.dtype or do.shape != q.shape:
        raise ValueError("do must match q in dtype and shape")
    if o is not None:
        o = np.ascontiguousarray(o)
        if o.dtype != q.dtype or o.shape != q.shape:
            raise ValueError("o must match q in dtype and shape")
    tot, h, d = q.shape
    hkv = kc.shape[1]
    scale = d ** -0.5 if scale is None else scale
    qr, nq = _rows(q_rows, tot)
    kr, nkv = _rows(kv_rows, kc.shape[0])
    nq = nq if want_dq else -1
    nkv = nkv if want_dkv else -1
    dq = np.zeros((max(nq, 0), h, d), np.float64)
    dk = np.zeros((max(nkv, 0), hkv, d), np.float64)
    dv = np.zeros((max(nkv, 0), hkv, d), np.float64)
    _check(_load().nsa_oracle_cmp_attn_bwd(_p(q), _p(kc), _p(vc), _p(do), _p(o), _dt(q), _p(cu), len(cu) - 1, h,
                                           hkv, d, kernel, stride, ctypes.c_double(scale), _p(qr),
                                           ctypes.c_int64(nq), _p(dq), _p(kr), ctypes.c_int64(nkv), _p(dk), _p(dv)),
           "cmp_attn_bwd")
    return (dq if want_dq else None), (dk if want_dkv else None), (dv if want_dkv else None)


def compress_bwd(dkc, cu, kernel=32, stride=16):
    """Backward of S1: token-row gradient [tokens, hkv, d] fp64 from the window gradient."""
    dkc = np.ascontiguousarray(np.asarray(dkc, np.float64))
    cu = _i32(cu)
    _, hkv, d = dkc.shape
    out = np.zeros((int(cu[-1]), hkv, d), np.float64)
    _check(_load().nsa_oracle_compress_bwd(_p(dkc), _p(cu), len(cu) - 1, hkv, d, kernel, stride, _p(out)),
           "compress_bwd")
    return out


def gate_combine(o_cmp, o_slc, o_swa, gates):
    """S9: sigmoid-gated sum of the three branch outputs."""
    o_cmp, o_slc, o_swa = (np.ascontiguousarray(np.asarray(a, np.float64)) for a in (o_cmp, o_slc, o_swa))
    gates = np.ascontiguousarray(np.asarray(gates, np.float32))
    n, h, d = o_cmp.shape
    out = np.zeros_like(o_cmp)
    _check(_load().nsa_oracle_gate_combine(_p(o_cmp), _p(o_slc), _p(o_swa), _p(gates), ctypes.c_int64(n),
                                           h, d, _p(out)), "gate_combine")
    return out


def swa_bwd(q, k, v, do, cu, window=512, scale=None, q_rows=None, kv_rows=None, want_dq=True, want_dkv=True,
            o=None):
    """Backward of S8: (dq [q_rows, h, d], dk, dv [kv_rows, hkv, d]) fp64; o optional (D = dO . o)."""
    q, k, v, do, cu = (np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v),
                       np.ascontiguousarray(do), _i32(cu))
    if do.dtype != q.dtype or do.shape != q.shape:
        raise ValueError("do must match q in dtype and shape")
    if o is not None:
        o = np.ascontiguousarray(o)
        if o.dtype != q.dtype or o.shape != q.shape:
            raise ValueError("o must match q in dtype and shape")
    tot, h, d = q.shape
    hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    qr, nq = _rows(q_rows, tot)
    kr, nkv = _rows(kv_rows, tot)
    nq = nq if want_dq else -1
    nkv = nkv if want_dkv else -1
    dq = np.zeros((max(nq, 0), h, d), np.float64)
    dk = np.zeros((max(nkv, 0), hkv, d), np.float64)
    dv = np.zeros((max(nkv, 0), hkv, d), np.float64)
    _check(_load().nsa_oracle_swa_bwd(_p(q), _p(k), _p(v), _p(do), _p(o), _dt(q), _p(cu), len(cu) - 1, h, hkv, d,
                                      window, ctypes.c_double(scale), _p(qr), ctypes.c_int64(nq), _p(dq), _p(kr),
                                      ctypes.c_int64(nkv), _p(dk), _p(dv)), "swa_bwd")
    return (dq if want_dq else None), (dk if want_dkv else None), (dv if want_dkv else None)


def gate_bwd(o_cmp, o_slc, o_swa, gates, do):
    """Backward of S9: (d o_cmp, d o_slc, d o_swa [n, h, d], d gate logits [n, h, 3]) fp64."""
    o_cmp, o_slc, o_swa, do = (np.ascontiguousarray(np.asarray(a, np.float64)) for a in (o_cmp, o_slc, o_swa, do))
    gates = np.ascontiguousarray(np.asarray(gates, np.float32))
    n, h, d = o_cmp.shape
    outs = [np.zeros_like(o_cmp) for _ in range(3)]
    dg = np.zeros((n, h, 3), np.float64)
    _check(_load().nsa_oracle_gate_bwd(_p(o_cmp), _p(o_slc), _p(o_swa), _p(gates), _p(do), ctypes.c_int64(n), h, d,
                                       _p(outs[0]), _p(outs[1]), _p(outs[2]), _p(dg)), "gate_bwd")
    return outs[0], outs[1], outs[2], dg


def _to_dtype(x, like):
    """fp64 values rounded to the dtype of `like` (bf16 bits or fp32)."""
    x32 = np.asarray(x, np.float64).astype(np.float32)
    if np.asarray(like).dtype == np.uint16:
        u = x32.view(np.uint32).astype(np.uint64)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return x32


def layer_bwd(q, k, v, gates, idx, do, cu, kernel=32, stride=16, block_size=64, window=512, scale=None,
              branches=None):
    """Backward of the three-branch layer for fixed block lists idx (the selection is not
    differentiated): returns (dq, dk, dv [fp64], d gates [n, h, 3]).  The composition of the
    branch backwards: the gate backward, then each branch's backward on its gradient, which
    the layer holds in the input dtype (rounded here alike), the pooling backward of the
    compressed keys and values, and the sum over branches.  branches: optional stored
    (o_cmp, o_slc, o_swa) in q's dtype (for D and the gate); else the exact outputs."""
    cu = _i32(cu)
    _, kc = compress(k, cu, kernel, stride)
    _, vc = compress(v, cu, kernel, stride)
    if branches is None:
        o_cmp, _ = cmp_attn(q, kc, vc, cu, kernel, stride, scale)
        o_slc, _ = sparse_attn(q, k, v, idx, cu, block_size, scale)
        o_swa, _ = swa(q, k, v, cu, window, scale)
        stored = None
    else:
        stored = [np.ascontiguousarray(b) for b in branches]
        o_cmp, o_slc, o_swa = (_to_f64(b) for b in stored)
    d_cmp, d_slc, d_swa, dg = gate_bwd(o_cmp, o_slc, o_swa, gates, _to_f64(do))
    d_cmp, d_slc, d_swa = (_to_dtype(x, q) for x in (d_cmp, d_slc, d_swa))
    st = stored or [None, None, None]
    dq_c, dkc, dvc = cmp_attn_bwd(q, kc, vc, d_cmp, cu, kernel, stride, scale, o=st[0])
    dq_s, dk_s, dv_s = sparse_attn_bwd(q, k, v, idx, d_slc, cu, block_size, scale, o=st[1])
    dq_w, dk_w, dv_w = swa_bwd(q, k, v, d_swa, cu, window, scale, o=st[2])
    dk_c = compress_bwd(dkc, cu, kernel, stride)
    dv_c = compress_bwd(dvc, cu, kernel, stride)
    return dq_c + dq_s + dq_w, dk_c + dk_s + dk_w, dv_c + dv_s + dv_w, dg


def _to_f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def decode(q, k_cache, v_cache, kc_cache, seqlens, kernel=32, stride=16, block_size=64, n_init=1,
           n_local=2, k=64, scale=None, idx_in=None, want_scores=False):
    """S6: one decode step; returns (idx [B,hkv,k], o [B,h,d] fp64[, scores [B,hkv,nb]])."""
    q, k_cache, v_cache, kc_cache = (np.ascontiguousarray(a) for a in (q, k_cache, v_cache, kc_cache))
    seqlens = _i32(seqlens)
    B, h, d = q.shape
    max_len, hkv = k_cache.shape[1], k_cache.shape[2]
    scale = d ** -0.5 if scale is None else scale
    nb = -(-max_len // block_size)
    idx = np.zeros((B, hkv, k), np.int32)
    o = np.zeros((B, h, d), np.float64)
    sc = np.zeros((B, hkv, nb), np.float64) if want_scores else None
    ii = None if idx_in is None else _i32(idx_in)
    _check(_load().nsa_oracle_decode(_p(q), _p(k_cache), _p(v_cache), _p(kc_cache), _dt(q), B,
                                     _p(seqlens), max_len, h, hkv, d, kernel, stride, block_size, n_init,
                                     n_local, k, ctypes.c_double(scale), _p(ii), _p(idx), _p(o), _p(sc),
                                     nb), "decode")
    return (idx, o, sc) if want_scores else (idx, o)


def decode_cis(q, k_cache, v_cache, kc_cache, cis_cache, seqlens, qk_select, k=64, block_size=64, n_init=1,
               n_local=2, scale=None, idx_in=None):
    """NOSA decode step: the decode scores (S2, S3) of the newest query, the two-stage
    selection (top qk_select by attention score, then top k by the CIS block score of the
    sequence) and the CIS-weighted attention over the chosen blocks.  cis_cache [B, max_len,
    hkv] (fp32); returns (idx [B, hkv, k], o [B, h, d] fp64, stage-1 scores [B, hkv, nb])."""
    q = np.ascontiguousarray(q)
    seqlens = _i32(seqlens)
    B, h, d = q.shape
    hkv = k_cache.shape[2]
    idx1, _, sc = decode(q, k_cache, v_cache, kc_cache, seqlens, block_size=block_size, n_init=n_init,
                         n_local=n_local, k=k, scale=scale, want_scores=True)
    nb = sc.shape[2]
    idx = np.zeros((B, hkv, k), np.int32)
    o = np.zeros((B, h, d), np.float64)
    for b in range(B):
        L = int(seqlens[b])
        cu = np.array([0, L], np.int32)
        cs = cis_block_scores(cis_cache[b, :L], cu, block_size=block_size, nb_stride=nb)
        rows = [L - 1]
        if idx_in is None:
            sc_rows = np.zeros((1, hkv, nb))
            sc_rows[0] = sc[b]
            idx[b] = topk_two_stage(sc_rows, cs, cu, qk_select, k, block_size, n_init, n_local, rows=rows)[0]
        else:
            idx[b] = np.asarray(idx_in)[b]
        full_idx = np.zeros((L, hkv, k), np.int32)
        full_idx[L - 1] = idx[b]
        ob, _ = sparse_attn_cis(q[b][None].repeat(L, 0), k_cache[b, :L], v_cache[b, :L], cis_cache[b, :L],
                                full_idx, cu, block_size, scale, rows=rows)
        o[b] = ob[0]
    return idx, o, sc


def layer(q, k, v, gates, cu, kernel=32, stride=16, block_size=64, S=16, n_init=1, n_local=2,
          window=512, scale=None, idx_in=None, rows=None, branches=False):
    """Three-branch layer; returns dict with idx, o (and o_cmp/o_slc/o_swa if branches)."""
    q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
    gates = np.ascontiguousarray(np.asarray(gates, np.float32))
    cu = _i32(cu)
    tot, h, d = q.shape
    hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    rows, n = _rows(rows, tot)
    idx = np.zeros((n, hkv, S), np.int32)
    o = np.zeros((n, h, d), np.float64)
    oc = np.zeros((n, h, d), np.float64) if branches else None
    os_ = np.zeros((n, h, d), np.float64) if branches else None
    ow = np.zeros((n, h, d), np.float64) if branches else None
    ii = None if idx_in is None else _i32(idx_in)
    _check(_load().nsa_oracle_layer(_p(q), _p(k), _p(v), _p(gates), _dt(q), _p(cu), len(cu) - 1, h, hkv,
                                    d, kernel, stride, block_size, S, n_init, n_local, window,
                                    ctypes.c_double(scale), _p(ii), _p(rows), ctypes.c_int64(n), _p(idx),
                                    _p(o), _p(oc), _p(os_), _p(ow)), "layer")
    out = {"idx": idx, "o": o}
    if branches:
        out.update(o_cmp=oc, o_slc=os_, o_swa=ow)
    return out
