"""Helpers shared by the GPU parity tests: host<->device marshalling and comparisons.

The tolerance for floating-point outputs is the one the pages use for their kernel
check (TileLang NSA correctness test: assert_close with atol = rtol = 1e-2):
|gpu - oracle| <= 1e-2 + 1e-2 * |oracle| elementwise.
"""
import numpy as np
import torch

from sparse_attention_compress_gb300 import inputs as gen

ATOL = 1e-2
RTOL = 1e-2


def dev(a, device="cuda"):
    """numpy array (bf16 bits as uint16, fp32, int32) -> device tensor."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def pinned(a):
    """numpy array -> page-locked host tensor (bf16 bits as uint16 -> bfloat16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).pin_memory().view(torch.bfloat16)
    return torch.from_numpy(a).pin_memory()


def host(t):
    """device tensor -> numpy (bf16 -> uint16 bits, others as is)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = gen.bf16_bits_to_f32(a)
    return a.astype(np.float64)


def assert_close(gpu, ref, atol=ATOL, rtol=RTOL, what=""):
    g = as_f64(host(gpu) if isinstance(gpu, torch.Tensor) else gpu)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - r)
    bad = err > atol + rtol * np.abs(r)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(r))), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu {g[i]!r} oracle {r[i]!r}; max abs err {err.max():.3g}")
    return float(err.max())


def selection_mismatches(gpu_idx, ref_idx, ref_scores, t_of_row, block_size=64, n_init=1, n_local=2,
                         rel_band=2e-5):
    """Compare block lists row by row.  Returns (n_exact_mismatch_rows, n_outside_band).

    A row may differ from the oracle only by swapping blocks whose oracle scores lie
    within the tie band of the row's selection threshold: an fp64 oracle and fp32 GPU
    scores cannot agree at every rounding boundary.  rel_band is relative to the
    threshold score (fp32 scores carry ~1e-6 relative error; the band leaves 20x).
    """
    g = np.asarray(gpu_idx)
    r = np.asarray(ref_idx)
    rows = np.where(np.any(g != r, axis=-1))
    n_mis = len(rows[0])
    outside = 0
    for ri in zip(*rows):
        gs = set(int(x) for x in g[ri] if x >= 0)
        rs = set(int(x) for x in r[ri] if x >= 0)
        sc = ref_scores[ri]
        t = int(t_of_row[ri[0]])
        own = t // block_size
        forced = {j for j in range(own + 1) if j < n_init or j > own - n_local}
        if len(gs) != len(rs) or not forced <= gs:
            outside += 1
            continue
        chosen = [sc[j] for j in rs - forced]
        if not chosen:
            outside += 1
            continue
        thr = min(chosen)
        band = rel_band * abs(thr) + 1e-12
        for j in gs ^ rs:
            if abs(sc[j] - thr) > band:
                outside += 1
                break
    return n_mis, outside
