"""ctypes binding of libnsa.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see include/nsa.h)
and does nothing but shape bookkeeping, output allocation through PyTorch and the
call itself; all arithmetic of the path runs in the CUDA kernels.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# NSA_LIBRARY may point at another build of the same library (e.g. with other tuning flags)
LIB_PATH = os.environ.get("NSA_LIBRARY") or os.path.join(_PKG, "libnsa.so")

NSA_F32, NSA_BF16 = 0, 1
_c_int, _c_i64, _c_p, _c_f, _c_sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t


class NsaShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seqlen", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p),
                ("n_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int64), ("h", ctypes.c_int32),
                ("h_kv", ctypes.c_int32), ("d", ctypes.c_int32), ("dtype", ctypes.c_int)]


class NsaLayerSaved(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("k_cmp", "v_cmp", "o_cmp", "o_slc", "o_swa", "lse_cmp", "lse_slc",
                                                "lse_swa", "idx")]


_SIGS = {
    "nsa_version": ([], ctypes.c_char_p),
    "nsa_last_error": ([], ctypes.c_char_p),
    "nsa_device_status": ([_c_p, _c_int], _c_int),
    "nsa_set_wait_limit_ns": ([ctypes.c_uint64], _c_int),
    "nsa_compress_k": ([_c_p, _c_p, _c_p, _c_int, _c_int, _c_p], _c_int),
    "nsa_cmp_scores_pool": ([_c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_f, _c_p, _c_p, _c_int, _c_p], _c_int),
    "nsa_topk_select": ([_c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p], _c_int),
    "nsa_cis_block_scores": ([_c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p], _c_int),
    "nsa_topk_two_stage": ([_c_p, _c_p, _c_int, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p], _c_int),
    "nsa_sparse_cis_fwd": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p], _c_int),
    "nsa_select_workspace_size": ([_c_p, _c_int], _c_sz),
    "nsa_block_sparse_workspace_size": ([_c_p], _c_sz),
    "nsa_block_sparse_fwd": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p, _c_sz, _c_p],
                             _c_int),
    "nsa_select": ([_c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_f, _c_int, _c_int, _c_int, _c_p, _c_p, _c_sz,
                    _c_p], _c_int),
    "nsa_sparse_fwd": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p], _c_int),
    "nsa_sparse_bwd_workspace_size": ([_c_p, _c_int, _c_int], _c_sz),
    "nsa_cmp_attn_bwd_workspace_size": ([_c_p, _c_int, _c_int], _c_sz),
    "nsa_cmp_attn_bwd": ([_c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                          _c_sz, _c_p], _c_int),
    "nsa_compress_bwd": ([_c_p, _c_p, _c_int, _c_int, _c_p, _c_p], _c_int),
    "nsa_swa_bwd_workspace_size": ([_c_p, _c_int], _c_sz),
    "nsa_swa_bwd": ([_c_p, _c_p, _c_p, _c_p, _c_int, _c_f, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p],
                    _c_int),
    "nsa_gate_combine_bwd": ([_c_i64, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p],
                             _c_int),
    "nsa_sparse_bwd": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                        _c_sz, _c_p], _c_int),
    "nsa_cmp_attn_fwd_workspace_size": ([_c_p, _c_int, _c_int], _c_sz),
    "nsa_cmp_attn_fwd": ([_c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p, _c_sz, _c_p], _c_int),
    "nsa_swa_fwd_workspace_size": ([_c_p], _c_sz),
    "nsa_swa_fwd": ([_c_p, _c_p, _c_p, _c_p, _c_int, _c_f, _c_p, _c_p, _c_p, _c_sz, _c_p], _c_int),
    "nsa_gate_combine": ([_c_i64, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p], _c_int),
    "nsa_sparse_decode_workspace_size": ([_c_int] * 9, _c_sz),
    "nsa_sparse_decode": ([_c_int, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int,
                           _c_int, _c_int, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p, _c_sz, _c_p], _c_int),
    "nsa_sparse_decode_cis": ([_c_int, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                               _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p,
                               _c_sz, _c_p], _c_int),
    "nsa_sparse_decode_noalloc_max_bytes": ([], _c_sz),
    "nsa_sparse_decode_noalloc": ([_c_int, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_int,
                                   _c_int, _c_int, _c_int, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p], _c_int),
    "nsa_layer_fwd_workspace_size": ([_c_p, _c_int, _c_int, _c_int, _c_int], _c_sz),
    "nsa_layer_fwd_train": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                             _c_f, _c_p, _c_p, _c_p, _c_sz, _c_p], _c_int),
    "nsa_layer_bwd_workspace_size": ([_c_p, _c_int, _c_int, _c_int, _c_int, _c_int], _c_sz),
    "nsa_layer_bwd": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f, _c_p, _c_p, _c_p,
                       _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p], _c_int),
    "nsa_layer_fwd": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f,
                       _c_p, _c_p, _c_p, _c_sz, _c_p], _c_int),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libnsa.so (built by __graft_entry__.build() / build.py); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


class NsaError(RuntimeError):
    pass


def _check(rc: int, fn: str) -> None:
    if rc != 0:
        msg = load().nsa_last_error().decode()
        raise NsaError(f"{fn} failed (status {rc}): {msg}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NSA_BF16
    if t.dtype == torch.float32:
        return NSA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_shape(tokens: int, h: int, h_kv: int, d: int, dtype: int, *, cu_seqlens=None, max_seqlen=None,
               batch=None, seqlen=None) -> NsaShape:
    """Dense layout (batch, seqlen) or packed varlen (cu_seqlens device int32, max_seqlen)."""
    s = NsaShape()
    s.h, s.h_kv, s.d, s.dtype = h, h_kv, d, dtype
    if cu_seqlens is not None:
        if max_seqlen is None:
            raise ValueError("varlen needs max_seqlen")
        s.cu_seqlens = cu_seqlens.data_ptr()
        s.n_seqs = cu_seqlens.numel() - 1
        s.total_tokens = tokens
        s.seqlen = int(max_seqlen)
    else:
        if batch is None:
            batch, seqlen = 1, tokens
        s.batch, s.seqlen = int(batch), int(seqlen)
        if batch * seqlen != tokens:
            raise ValueError("batch * seqlen must equal the token count")
        s.cu_seqlens = None
        s.total_tokens = tokens
    return s


def _flat(t: torch.Tensor):
    """[B, T, H, d] -> ([B*T, H, d], B, T); [N, H, d] -> (t, None, None)."""
    if t.dim() == 4:
        B, T = t.shape[0], t.shape[1]
        return t.reshape(B * T, t.shape[2], t.shape[3]), B, T
    if t.dim() == 3:
        return t, None, None
    raise ValueError("expected [B, T, H, d] or [tokens, H, d]")


def _shape_for(q, h_kv, cu_seqlens, max_seqlen):
    qf, B, T = _flat(q)
    if cu_seqlens is None and B is None:
        B, T = 1, qf.shape[0]
    return qf, make_shape(qf.shape[0], qf.shape[1], h_kv, qf.shape[2], _dtype(qf), cu_seqlens=cu_seqlens,
                          max_seqlen=max_seqlen, batch=B, seqlen=T)


def num_cmp(L: int, kernel: int = 32, stride: int = 16) -> int:
    return (L - kernel) // stride + 1 if L >= kernel else 0


# ----------------------------------------------------------------------------- entry points
def nsa_compress_k(k, kernel=32, stride=16, *, cu_seqlens=None, max_seqlen=None, n_cmp=None, out=None,
                   stream=None):
    """S1.  k [B,T,Hkv,d] or packed [tokens,Hkv,d] -> packed compressed rows [n_cmp, Hkv, d]."""
    kf, shp = _shape_for(k, k.shape[-2], cu_seqlens, max_seqlen)
    if out is None:
        if n_cmp is None:
            if cu_seqlens is not None:
                lens = (cu_seqlens[1:] - cu_seqlens[:-1]).tolist()
                n_cmp = sum(num_cmp(int(L), kernel, stride) for L in lens)
            else:
                n_cmp = shp.batch * num_cmp(shp.seqlen, kernel, stride)
        out = torch.empty((n_cmp, kf.shape[1], kf.shape[2]), dtype=kf.dtype, device=kf.device)
    _check(load().nsa_compress_k(ctypes.byref(shp), _ptr(kf), _ptr(out), kernel, stride, _stream(stream)),
           "nsa_compress_k")
    return out


def nsa_cmp_scores_pool(q, k_cmp, h_kv, kernel=32, stride=16, block_size=64, scale=0.0, *, lse_in=None,
                        cu_seqlens=None, max_seqlen=None, nb_stride=None, out=None, stream=None):
    """S2+S3.  Returns block scores [tokens, Hkv, nb_stride] fp32."""
    qf, shp = _shape_for(q, h_kv, cu_seqlens, max_seqlen)
    if nb_stride is None:
        nb_stride = -(-shp.seqlen // block_size)
    if out is None:
        out = torch.empty((qf.shape[0], h_kv, nb_stride), dtype=torch.float32, device=qf.device)
    _check(load().nsa_cmp_scores_pool(ctypes.byref(shp), _ptr(qf), _ptr(k_cmp), kernel, stride, block_size,
                                      float(scale), _ptr(lse_in), _ptr(out), nb_stride, _stream(stream)),
           "nsa_cmp_scores_pool")
    return out


def nsa_block_sparse_workspace_size(shape: NsaShape) -> int:
    return int(load().nsa_block_sparse_workspace_size(ctypes.byref(shape)))


def nsa_select_workspace_size(shape: NsaShape, block_size=64) -> int:
    return int(load().nsa_select_workspace_size(ctypes.byref(shape), block_size))


def nsa_block_sparse_fwd(q, k, v, block_mask, causal=True, block_size=64, scale=0.0, *, workspace=None, out=None,
                         lse=None, stream=None):
    """Block-mask sparse attention; q/k/v [B, T, H, d] bf16, block_mask uint8 [B, H, T/64, T/64]."""
    qf, shp = _shape_for(q, k.shape[-2], None, None)
    if workspace is None:
        ws = int(load().nsa_block_sparse_workspace_size(ctypes.byref(shp)))
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=qf.device)
    if out is None:
        out = torch.empty_like(qf)
    _check(load().nsa_block_sparse_fwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), _ptr(block_mask), block_size,
                                       int(bool(causal)), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                       workspace.numel(), _stream(stream)), "nsa_block_sparse_fwd")
    return out


def nsa_select(q, k_cmp, h_kv, k=16, kernel=32, stride=16, block_size=64, n_init=1, n_local=2, scale=0.0, *,
               cu_seqlens=None, max_seqlen=None, workspace=None, out=None, stream=None):
    """S2-S4 in one call: block indices [tokens, Hkv, k] int32 from q and the compressed keys."""
    qf, shp = _shape_for(q, h_kv, cu_seqlens, max_seqlen)
    if workspace is None:
        ws = int(load().nsa_select_workspace_size(ctypes.byref(shp), block_size))
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=qf.device)
    if out is None:
        out = torch.empty((qf.shape[0], h_kv, k), dtype=torch.int32, device=qf.device)
    _check(load().nsa_select(ctypes.byref(shp), _ptr(qf), _ptr(k_cmp), kernel, stride, block_size, float(scale),
                             n_init, n_local, k, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)),
           "nsa_select")
    return out


def nsa_topk_select(block_scores, k, block_size=64, n_init=1, n_local=2, *, cu_seqlens=None, max_seqlen=None,
                    batch=None, seqlen=None, out=None, stream=None):
    """S4.  block_scores [tokens, Hkv, nb_stride] fp32 -> indices [tokens, Hkv, k] int32."""
    tokens, h_kv, nb_stride = block_scores.shape
    if cu_seqlens is None and batch is None:
        batch, seqlen = 1, tokens
    shp = make_shape(tokens, h_kv, h_kv, 1, NSA_F32, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen, batch=batch,
                     seqlen=seqlen)
    if out is None:
        out = torch.empty((tokens, h_kv, k), dtype=torch.int32, device=block_scores.device)
    _check(load().nsa_topk_select(ctypes.byref(shp), _ptr(block_scores), nb_stride, block_size, n_init, n_local, k,
                                  _ptr(out), _stream(stream)), "nsa_topk_select")
    return out


def nsa_cis_block_scores(cis, kernel=32, stride=16, block_size=64, *, cu_seqlens=None, max_seqlen=None, batch=None,
                         seqlen=None, nb_stride=None, out=None, stream=None):
    """NOSA stage 2.  cis [tokens, Hkv] fp32 -> block CIS scores [n_seqs, Hkv, nb_stride] fp32."""
    tokens, h_kv = cis.shape
    if cu_seqlens is None and batch is None:
        batch, seqlen = 1, tokens
    shp = make_shape(tokens, h_kv, h_kv, 1, NSA_F32, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen, batch=batch,
                     seqlen=seqlen)
    n_seqs = shp.n_seqs if cu_seqlens is not None else shp.batch
    if nb_stride is None:
        nb_stride = max(1, -(-shp.seqlen // block_size))
    if out is None:
        out = torch.empty((n_seqs, h_kv, nb_stride), dtype=torch.float32, device=cis.device)
    _check(load().nsa_cis_block_scores(ctypes.byref(shp), _ptr(cis), kernel, stride, block_size, nb_stride,
                                       _ptr(out), _stream(stream)), "nsa_cis_block_scores")
    return out


def nsa_topk_two_stage(block_scores, cis_block_scores, qk_select, k, block_size=64, n_init=1, n_local=2, *,
                       cu_seqlens=None, max_seqlen=None, batch=None, seqlen=None, out=None, stream=None):
    """NOSA two-stage selection: block_scores [tokens, Hkv, nb_stride], cis_block_scores
    [n_seqs, Hkv, nb_stride] -> indices [tokens, Hkv, k] int32."""
    tokens, h_kv, nb_stride = block_scores.shape
    if cu_seqlens is None and batch is None:
        batch, seqlen = 1, tokens
    shp = make_shape(tokens, h_kv, h_kv, 1, NSA_F32, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen, batch=batch,
                     seqlen=seqlen)
    if out is None:
        out = torch.empty((tokens, h_kv, k), dtype=torch.int32, device=block_scores.device)
    _check(load().nsa_topk_two_stage(ctypes.byref(shp), _ptr(block_scores), nb_stride, _ptr(cis_block_scores),
                                     block_size, n_init, n_local, qk_select, k, _ptr(out), _stream(stream)),
           "nsa_topk_two_stage")
    return out


def nsa_sparse_cis_fwd(q, k, v, cis, block_indices, block_size=64, scale=0.0, *, cu_seqlens=None, max_seqlen=None,
                       out=None, lse=None, stream=None):
    """NOSA sparse_forward: selected attention with weights p * cis (normalised); cis [tokens, Hkv] fp32."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    S = block_indices.shape[-1]
    if out is None:
        out = torch.empty_like(qf)
    _check(load().nsa_sparse_cis_fwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), _ptr(cis), _ptr(block_indices),
                                     S, block_size, float(scale), _ptr(out), _ptr(lse), _stream(stream)),
           "nsa_sparse_cis_fwd")
    return out.view(q.shape) if q.dim() == 4 else out


def nsa_sparse_fwd(q, k, v, block_indices, block_size=64, scale=0.0, *, cu_seqlens=None, max_seqlen=None,
                   out=None, lse=None, stream=None):
    """S5.  q [B,T,H,d] / [tokens,H,d]; k, v with Hkv heads; block_indices [..., Hkv, S] int32."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    S = block_indices.shape[-1]
    if out is None:
        out = torch.empty_like(qf)
    _check(load().nsa_sparse_fwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), _ptr(block_indices), S, block_size,
                                 float(scale), _ptr(out), _ptr(lse), _stream(stream)), "nsa_sparse_fwd")
    return out.view(q.shape) if q.dim() == 4 else out


def nsa_sparse_bwd_workspace_size(shape: NsaShape, S: int, block_size: int = 64) -> int:
    return int(load().nsa_sparse_bwd_workspace_size(ctypes.byref(shape), S, block_size))


def nsa_sparse_bwd(q, k, v, block_indices, o, lse, d_o, block_size=64, scale=0.0, *, cu_seqlens=None,
                   max_seqlen=None, workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Backward of S5: returns (dq, dk, dv) shaped like q, k, v.  o and lse come from
    nsa_sparse_fwd on the same inputs; d_o is the upstream gradient (like q)."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    S = block_indices.shape[-1]
    if workspace is None:
        ws = nsa_sparse_bwd_workspace_size(shp, S, block_size)
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(load().nsa_sparse_bwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), _ptr(block_indices), S, block_size,
                                 float(scale), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(workspace), workspace.numel(), _stream(stream)), "nsa_sparse_bwd")
    return dq, dk, dv


def nsa_cmp_attn_bwd_workspace_size(shape: NsaShape, kernel: int = 32, stride: int = 16) -> int:
    return int(load().nsa_cmp_attn_bwd_workspace_size(ctypes.byref(shape), kernel, stride))


def nsa_cmp_attn_bwd(q, k_cmp, v_cmp, o, lse, d_o, h_kv, kernel=32, stride=16, scale=0.0, *, cu_seqlens=None,
                     max_seqlen=None, workspace=None, dq=None, dk_cmp=None, dv_cmp=None, stream=None):
    """Backward of S7: (dq like q, dk_cmp and dv_cmp like k_cmp) from the forward's o, lse."""
    qf, shp = _shape_for(q, h_kv, cu_seqlens, max_seqlen)
    if workspace is None:
        ws = nsa_cmp_attn_bwd_workspace_size(shp, kernel, stride)
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk_cmp = torch.empty_like(k_cmp) if dk_cmp is None else dk_cmp
    dv_cmp = torch.empty_like(v_cmp) if dv_cmp is None else dv_cmp
    _check(load().nsa_cmp_attn_bwd(ctypes.byref(shp), _ptr(qf), _ptr(k_cmp), _ptr(v_cmp), kernel, stride,
                                   float(scale), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk_cmp), _ptr(dv_cmp),
                                   _ptr(workspace), workspace.numel(), _stream(stream)), "nsa_cmp_attn_bwd")
    return dq, dk_cmp, dv_cmp


def nsa_compress_bwd(dk_cmp, tokens, kernel=32, stride=16, *, cu_seqlens=None, max_seqlen=None, batch=None,
                     seqlen=None, out=None, stream=None):
    """Backward of S1: token-row gradient [tokens, Hkv, d] from the window gradient dk_cmp."""
    _, h_kv, d = dk_cmp.shape
    if cu_seqlens is None and batch is None:
        batch, seqlen = 1, tokens
    shp = make_shape(tokens, h_kv, h_kv, d, NSA_BF16, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen, batch=batch,
                     seqlen=seqlen)
    if out is None:
        out = torch.empty((tokens, h_kv, d), dtype=dk_cmp.dtype, device=dk_cmp.device)
    _check(load().nsa_compress_bwd(ctypes.byref(shp), _ptr(dk_cmp), kernel, stride, _ptr(out), _stream(stream)),
           "nsa_compress_bwd")
    return out


def nsa_swa_bwd_workspace_size(shape: NsaShape, window: int = 512) -> int:
    return int(load().nsa_swa_bwd_workspace_size(ctypes.byref(shape), window))


def nsa_swa_bwd(q, k, v, o, lse, d_o, window=512, scale=0.0, *, cu_seqlens=None, max_seqlen=None, workspace=None,
                dq=None, dk=None, dv=None, stream=None):
    """Backward of S8: (dq, dk, dv) shaped like q, k, v from the forward's o and lse."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    if workspace is None:
        ws = nsa_swa_bwd_workspace_size(shp, window)
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(load().nsa_swa_bwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), window, float(scale), _ptr(o),
                              _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                              workspace.numel(), _stream(stream)), "nsa_swa_bwd")
    return dq, dk, dv


def nsa_gate_combine_bwd(d_o, o_cmp, o_slc, o_swa, gate_logits, *, stream=None):
    """Backward of S9: (d o_cmp, d o_slc, d o_swa, d gate_logits)."""
    tokens, h, d = d_o.shape
    outs = [torch.empty_like(d_o) for _ in range(3)]
    dg = torch.empty_like(gate_logits)
    _check(load().nsa_gate_combine_bwd(tokens, h, d, _ptr(d_o), _ptr(o_cmp), _ptr(o_slc), _ptr(o_swa),
                                       _ptr(gate_logits), _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(dg),
                                       _stream(stream)), "nsa_gate_combine_bwd")
    return outs[0], outs[1], outs[2], dg


def _workspace(nbytes, device, workspace=None):
    """Caller's workspace, or a fresh one of nbytes (None when nothing is needed)."""
    if workspace is not None or nbytes == 0:
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def nsa_cmp_attn_fwd(q, k_cmp, v_cmp, h_kv, kernel=32, stride=16, scale=0.0, *, cu_seqlens=None,
                     max_seqlen=None, out=None, lse=None, workspace=None, stream=None):
    """S7.  Compressed branch over packed compressed keys / values."""
    qf, shp = _shape_for(q, h_kv, cu_seqlens, max_seqlen)
    if out is None:
        out = torch.empty_like(qf)
    ws = _workspace(int(load().nsa_cmp_attn_fwd_workspace_size(ctypes.byref(shp), kernel, stride)), qf.device,
                    workspace)
    _check(load().nsa_cmp_attn_fwd(ctypes.byref(shp), _ptr(qf), _ptr(k_cmp), _ptr(v_cmp), kernel, stride,
                                   float(scale), _ptr(out), _ptr(lse), _ptr(ws), 0 if ws is None else ws.numel(),
                                   _stream(stream)), "nsa_cmp_attn_fwd")
    return out


def nsa_swa_fwd(q, k, v, window=512, scale=0.0, *, cu_seqlens=None, max_seqlen=None, out=None, lse=None,
                workspace=None, stream=None):
    """S8.  Sliding-window branch."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    if out is None:
        out = torch.empty_like(qf)
    ws = _workspace(int(load().nsa_swa_fwd_workspace_size(ctypes.byref(shp))), qf.device, workspace)
    _check(load().nsa_swa_fwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), window, float(scale), _ptr(out),
                              _ptr(lse), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)), "nsa_swa_fwd")
    return out


def nsa_gate_combine(o_cmp, o_slc, o_swa, gate_logits, *, out=None, stream=None):
    """S9.  out = sigmoid(g0) o_cmp + sigmoid(g1) o_slc + sigmoid(g2) o_swa."""
    tokens, h, d = o_cmp.shape
    if out is None:
        out = torch.empty_like(o_cmp)
    _check(load().nsa_gate_combine(tokens, h, d, _ptr(o_cmp), _ptr(o_slc), _ptr(o_swa), _ptr(gate_logits),
                                   _ptr(out), _stream(stream)), "nsa_gate_combine")
    return out


def nsa_sparse_decode_workspace_size(batch, max_len, h, h_kv, d, kernel=32, stride=16, block_size=64, k=64):
    return int(load().nsa_sparse_decode_workspace_size(batch, max_len, h, h_kv, d, kernel, stride, block_size, k))


def nsa_sparse_decode(q, k_cache, v_cache, k_cmp_cache, seqlens, k=64, kernel=32, stride=16, block_size=64,
                      n_init=1, n_local=2, scale=0.0, *, workspace=None, idx_out=None, out=None, stream=None):
    """S6.  q [B,H,d]; caches [B,L,Hkv,d]; k_cmp_cache [B,n_c(L),Hkv,d]; seqlens device int32 [B]."""
    B, h, d = q.shape
    max_len, h_kv = k_cache.shape[1], k_cache.shape[2]
    if workspace is None:
        ws = nsa_sparse_decode_workspace_size(B, max_len, h, h_kv, d, kernel, stride, block_size, k)
        workspace = torch.empty(ws, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _check(load().nsa_sparse_decode(B, _ptr(seqlens), max_len, h, h_kv, d, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_cmp_cache), kernel, stride, block_size, n_init, n_local, k, float(scale),
                                    _ptr(idx_out), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)),
           "nsa_sparse_decode")
    return out


def nsa_sparse_decode_cis(q, k_cache, v_cache, k_cmp_cache, cis_cache, seqlens, cis_block_scores=None, qk_select=0,
                          k=64, kernel=32, stride=16, block_size=64, n_init=1, n_local=2, scale=0.0, *,
                          workspace=None, idx_out=None, out=None, stream=None):
    """NOSA decode step: CIS-weighted attention, two-stage selection when cis_block_scores
    [B, Hkv, nb_stride] is given.  cis_cache [B, max_len, Hkv] fp32."""
    B, h, d = q.shape
    max_len, h_kv = k_cache.shape[1], k_cache.shape[2]
    if workspace is None:
        ws = nsa_sparse_decode_workspace_size(B, max_len, h, h_kv, d, kernel, stride, block_size, k)
        workspace = torch.empty(ws, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    nb_stride = 0 if cis_block_scores is None else cis_block_scores.shape[-1]
    _check(load().nsa_sparse_decode_cis(B, _ptr(seqlens), max_len, h, h_kv, d, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(k_cmp_cache), _ptr(cis_cache), _ptr(cis_block_scores), nb_stride,
                                        qk_select, kernel, stride, block_size, n_init, n_local, k, float(scale),
                                        _ptr(idx_out), _ptr(out), _ptr(workspace), workspace.numel(),
                                        _stream(stream)), "nsa_sparse_decode_cis")
    return out


def nsa_sparse_decode_noalloc(q, k_cache, v_cache, k_cmp_cache, seqlens, k=64, kernel=32, stride=16,
                              block_size=64, n_init=1, n_local=2, scale=0.0, *, idx_out=None, out=None, stream=None):
    """S6 without a workspace: the scratch is the library's fixed device array (see nsa.h)."""
    B, h, d = q.shape
    max_len, h_kv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty_like(q)
    _check(load().nsa_sparse_decode_noalloc(B, _ptr(seqlens), max_len, h, h_kv, d, _ptr(q), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(k_cmp_cache), kernel, stride, block_size, n_init,
                                            n_local, k, float(scale), _ptr(idx_out), _ptr(out), _stream(stream)),
           "nsa_sparse_decode_noalloc")
    return out


def nsa_device_status(reset: bool = False) -> int:
    """Device status word (0 or NSA_ERR_TIMEOUT = 4); synchronises the device."""
    st = ctypes.c_int32(0)
    _check(load().nsa_device_status(ctypes.byref(st), int(bool(reset))), "nsa_device_status")
    return int(st.value)


def nsa_set_wait_limit_ns(ns: int = 0) -> None:
    """Limit of the kernels' first-level bounded waits in ns (0: the default second)."""
    _check(load().nsa_set_wait_limit_ns(int(ns)), "nsa_set_wait_limit_ns")


def nsa_layer_fwd_workspace_size(shape: NsaShape, kernel=32, stride=16, block_size=64, S=16) -> int:
    return int(load().nsa_layer_fwd_workspace_size(ctypes.byref(shape), kernel, stride, block_size, S))


def nsa_layer_fwd(q, k, v, gate_logits, kernel=32, stride=16, block_size=64, S=16, n_init=1, n_local=2,
                  window=512, scale=0.0, *, cu_seqlens=None, max_seqlen=None, workspace=None, idx_out=None,
                  out=None, stream=None):
    """Full three-branch layer forward."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    if workspace is None:
        ws = nsa_layer_fwd_workspace_size(shp, kernel, stride, block_size, S)
        workspace = torch.empty(ws, dtype=torch.uint8, device=qf.device)
    if out is None:
        out = torch.empty_like(qf)
    _check(load().nsa_layer_fwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), _ptr(gate_logits), kernel, stride,
                                block_size, S, n_init, n_local, window, float(scale), _ptr(out), _ptr(idx_out),
                                _ptr(workspace), workspace.numel(), _stream(stream)), "nsa_layer_fwd")
    return out


def nsa_layer_saved_buffers(tokens, n_cmp, h, h_kv, d, S, device):
    """Allocate the tensors a training forward keeps for the backward (a dict of tensors)."""
    bf = torch.bfloat16
    return {"k_cmp": torch.empty((n_cmp, h_kv, d), dtype=bf, device=device),
            "v_cmp": torch.empty((n_cmp, h_kv, d), dtype=bf, device=device),
            "o_cmp": torch.empty((tokens, h, d), dtype=bf, device=device),
            "o_slc": torch.empty((tokens, h, d), dtype=bf, device=device),
            "o_swa": torch.empty((tokens, h, d), dtype=bf, device=device),
            "lse_cmp": torch.empty((tokens, h), dtype=torch.float32, device=device),
            "lse_slc": torch.empty((tokens, h), dtype=torch.float32, device=device),
            "lse_swa": torch.empty((tokens, h), dtype=torch.float32, device=device),
            "idx": torch.empty((tokens, h_kv, S), dtype=torch.int32, device=device)}


def _saved_struct(saved):
    st = NsaLayerSaved()
    for name, _ in NsaLayerSaved._fields_:
        setattr(st, name, saved[name].data_ptr())
    return st


def nsa_layer_fwd_train(q, k, v, gate_logits, saved, kernel=32, stride=16, block_size=64, S=16, n_init=1,
                        n_local=2, window=512, scale=0.0, *, cu_seqlens=None, max_seqlen=None, workspace=None,
                        out=None, stream=None):
    """Layer forward that also fills `saved` (nsa_layer_saved_buffers) for nsa_layer_bwd."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    if workspace is None:
        ws = int(load().nsa_layer_fwd_workspace_size(ctypes.byref(shp), kernel, stride, block_size, S))
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(qf) if out is None else out
    st = _saved_struct(saved)
    _check(load().nsa_layer_fwd_train(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), _ptr(gate_logits), kernel,
                                      stride, block_size, S, n_init, n_local, window, float(scale), _ptr(out),
                                      ctypes.byref(st), _ptr(workspace), workspace.numel(), _stream(stream)),
           "nsa_layer_fwd_train")
    return out


def nsa_layer_bwd(q, k, v, gate_logits, saved, d_o, kernel=32, stride=16, block_size=64, S=16, window=512,
                  scale=0.0, *, cu_seqlens=None, max_seqlen=None, workspace=None, stream=None):
    """Layer backward: returns (dq, dk, dv, d_gate_logits)."""
    qf, shp = _shape_for(q, k.shape[-2], cu_seqlens, max_seqlen)
    if workspace is None:
        ws = int(load().nsa_layer_bwd_workspace_size(ctypes.byref(shp), kernel, stride, block_size, S, window))
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty_like(gate_logits)
    st = _saved_struct(saved)
    _check(load().nsa_layer_bwd(ctypes.byref(shp), _ptr(qf), _ptr(k), _ptr(v), _ptr(gate_logits), kernel, stride,
                                block_size, S, window, float(scale), ctypes.byref(st), _ptr(d_o), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(dg), _ptr(workspace), workspace.numel(), _stream(stream)),
           "nsa_layer_bwd")
    return dq, dk, dv, dg
