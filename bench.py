#!/usr/bin/env python
"""Benchmark of the native-sparse-attention hot path on GB300.

Headline: selected-attention prefill forward (B=8, T=16384, H=16, Hkv=1, d=128, bf16,
block 64, S=16 random causal blocks incl. block 0 and the own block) in TFLOP/s of
algorithmic work (4*d per attended (query head, key) pair).  One step = one
nsa_sparse_fwd over the whole batch.  Also measured in the same run (N=1): the decode
step (B=32, context 32768, top-k 64; KV GB/s), the varlen selection stage
(compress -> block scores -> top-k; tokens/s) and the full three-branch layer at
65536 tokens (TFLOP/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica (weak scaling, no collective on the data
path); rank 0 prints one JSON line.  --impl reference times the CPU oracle instead, on a
bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_compress_gb300 import inputs as gen  # noqa: E402
from sparse_attention_compress_gb300.dist import max_over_ranks  # noqa: E402

METRIC = "NSA selected-attn fwd TFLOP/s (prefill), KV GB/s (decode) vs GB300 roofline"
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the TMA-fed
# prefill kernel sparse_fwd_tma<2> (with the L2 prefetch of later tokens' query rows),
# captured by ncu at B=2 (153.22 MB read + 99.70 MB written), times 4 for the B=8 launch:
# every query token reads its own Q row and writes its own O row, and the K/V read grows
# with the batch in the same way.  To be set to None once the kernel changes again.
PREFILL_NCU_TRAFFIC = 4 * (153.22e6 + 99.70e6)
L2_BYTES = 129 * 2 ** 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- algorithmic work
def selected_pairs(idx: np.ndarray, cu: np.ndarray, block_size: int) -> np.ndarray:
    """Attended keys per (token, kv-head) row of a block list (causal masking inside blocks)."""
    t = np.concatenate([np.arange(cu[i + 1] - cu[i]) for i in range(len(cu) - 1)])
    i = idx.astype(np.int64)
    n = np.clip(t[:, None, None] - i * block_size + 1, 0, block_size)
    n = np.where(i >= 0, n, 0)
    return n.sum(axis=-1)  # [tokens, hkv]


def prefill_flops(w) -> float:
    r = w.h // w.hkv
    return float(selected_pairs(w.idx, w.cu_seqlens, w.block_size).sum()) * r * 4 * w.d


# ----------------------------------------------------------------------------- clocks
class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc = index, None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- timing
def timed(torch, fn, steps, warmup, flush=None, barrier=None):
    """Warm up, then time exactly `steps` calls of fn with CUDA events on the current stream.
    The L2 flush (if any) runs between the event pairs.  Returns per-step ms."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        if flush is not None:
            flush()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return [a.elapsed_time(b) for a, b in ev]


def dev(torch, a, device):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def pinned(torch, a):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.pin_memory()


# ----------------------------------------------------------------------------- oracle (CPU) runs
def oracle_prefill_sample(w, n_rows: int, seed: int = 0):
    """Time the CPU oracle on n_rows sampled query tokens; returns (TFLOP/s, seconds, flops, threads)."""
    from oracle import oracle as orc
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.tokens, size=n_rows, replace=False))
    t = rows % w.seqlen
    i = w.idx[rows].astype(np.int64)
    n = np.where(i >= 0, np.clip(t[:, None, None] - i * w.block_size + 1, 0, w.block_size), 0)
    flops = float(n.sum()) * (w.h // w.hkv) * 4 * w.d
    t0 = time.perf_counter()
    orc.sparse_attn(w.q, w.k, w.v, w.idx, w.cu_seqlens, w.block_size, rows=rows)
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, flops, orc.threads()


def run_reference(args):
    """CPU oracle arm: each step is the oracle on a bounded sample of the prefill workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as orc
    orc.build()
    w = gen.prefill()
    _, dt, _, _ = oracle_prefill_sample(w, 512, seed=99)
    n_rows = int(min(w.tokens, max(512, 512 * 2.5 / max(dt, 1e-3))))  # ~2.5 s per step
    for s in range(args.warmup):
        oracle_prefill_sample(w, n_rows, seed=1000 + s)
    vals, times = [], []
    for s in range(args.steps):
        v, dt, _, thr = oracle_prefill_sample(w, n_rows, seed=s)
        vals.append(v)
        times.append(dt)
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill B=8 T=16384 H=16 Hkv=1 d=128 bf16 block=64 S=16",
                   "sample_rows_per_step": n_rows, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.threads(), "kind": "oracle",
                         "sample": f"{n_rows} random query tokens (all 16 heads) of the prefill workload per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- extras (N=1)
def bench_decode(torch, nsa, device, steps, warmup, flush, peaks):
    w = gen.decode()
    q, kc_, vc_ = dev(torch, w.q, device), dev(torch, w.k_cache, device), dev(torch, w.v_cache, device)
    sl = dev(torch, w.seqlens, device)
    n_c = nsa.num_cmp(w.max_len)
    kcmp = nsa.nsa_compress_k(kc_).view(w.batch, n_c, w.hkv, w.d)
    ws = torch.empty(nsa.nsa_sparse_decode_workspace_size(w.batch, w.max_len, w.h, w.hkv, w.d, k=w.topk),
                     dtype=torch.uint8, device=device)
    idx = torch.empty((w.batch, w.hkv, w.topk), dtype=torch.int32, device=device)
    out = torch.empty_like(q)

    def step():
        nsa.nsa_sparse_decode(q, kc_, vc_, kcmp, sl, k=w.topk, workspace=ws, idx_out=idx, out=out)

    # CUDA graph of the four launches
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        step()
    torch.cuda.current_stream().wait_stream(st)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    ms = timed(torch, g.replay, steps, warmup, flush)
    # algorithmic bytes: compressed keys of every (seq, kv-head), the chosen K/V rows, q and o
    ih = idx.cpu().numpy()
    t = (w.seqlens.astype(np.int64) - 1)[:, None, None]
    i = ih.astype(np.int64)
    keys = np.where(i >= 0, np.clip(t - i * 64 + 1, 0, 64), 0).sum()
    byts = w.batch * w.hkv * n_c * w.d * 2 + keys * w.d * 2 * 2 + 2 * w.batch * w.h * w.d * 2
    ms_step = float(np.mean(ms))
    gbs = byts / (ms_step * 1e-3) / 1e9
    # the NOSA decode step: CIS-weighted attention and two-stage selection (k = 64 of
    # qk_select = 64, so stage 2 keeps every stage-1 block; the weights change the output)
    cis = dev(torch, gen.cis_scores(gen.rng_for(3, 77), w.batch * w.max_len, w.hkv), device)
    nbs = -(-w.max_len // 64)
    cb = nsa.nsa_cis_block_scores(cis, batch=w.batch, seqlen=w.max_len, nb_stride=nbs)
    cis3 = cis.view(w.batch, w.max_len, w.hkv)
    ms_nosa = float(np.mean(timed(torch, lambda: nsa.nsa_sparse_decode_cis(
        q, kc_, vc_, kcmp, cis3, sl, cb, 64, k=w.topk, workspace=ws, idx_out=idx, out=out), steps, warmup, flush)))
    del cis, cb, cis3
    # compressing the cache (timed separately: one HBM pass over 537 MB)
    msc = timed(torch, lambda: nsa.nsa_compress_k(kc_, out=kcmp.view(-1, w.hkv, w.d)), steps, warmup, flush)
    cbytes = kc_.numel() * 2 + kcmp.numel() * 2
    cgbs = cbytes / (float(np.mean(msc)) * 1e-3) / 1e9
    return {"workload": "decode B=32 L=32768 H=16 Hkv=2 d=128 bf16 top-k 64 (blocks of 64)",
            "ms_per_step": ms_step, "kv_gbs": gbs, "tokens_per_s": w.batch / (ms_step * 1e-3),
            "bytes_per_step": int(byts), "hbm_frac": gbs / peaks["hbm_gbs"],
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"] + " copy"},
            "kernels_per_step": 1, "memsets_per_step": 1, "cuda_graph": True,
            "nosa_step_ms": ms_nosa,
            "compress_cache": {"ms": float(np.mean(msc)), "gbs": cgbs, "hbm_frac": cgbs / peaks["hbm_gbs"],
                               "bytes": int(cbytes)}}


def bench_prefill_bwd(torch, nsa, device, steps, warmup, flush, peaks, batch=8):
    """Backward of the selected branch on the prefill workload: dq, dk, dv from the
    forward's o and lse and a seeded upstream gradient (batch 8 is the workload; smaller
    batches for profiler captures)."""
    from sparse_attention_compress_gb300 import _lib
    w = gen.prefill(B=batch)
    q = dev(torch, w.q, device).view(w.batch, w.seqlen, w.h, w.d)
    k, v, idx = dev(torch, w.k, device), dev(torch, w.v, device), dev(torch, w.idx, device)
    do = dev(torch, gen.normal(gen.rng_for(1, 99), (w.tokens, w.h, w.d), "bf16"), device)
    lse = torch.empty((w.tokens, w.h), dtype=torch.float32, device=device)
    o = nsa.nsa_sparse_fwd(q, k, v, idx, w.block_size, lse=lse).view(w.tokens, w.h, w.d)
    shp = _lib.make_shape(w.tokens, w.h, w.hkv, w.d, _lib.NSA_BF16, batch=w.batch, seqlen=w.seqlen)
    ws = torch.empty(nsa.nsa_sparse_bwd_workspace_size(shp, w.S), dtype=torch.uint8, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        nsa.nsa_sparse_bwd(q, k, v, idx, o, lse, do, w.block_size, workspace=ws, dq=dq, dk=dk, dv=dv)

    ms_step = float(np.mean(timed(torch, step, steps, warmup, flush)))
    # five products per attended (row, key) pair: S and dP recomputed, dQ, dK, dV
    flops = prefill_flops(w) * 10 / 4
    tf = flops / (ms_step * 1e-3) / 1e12
    return {"workload": f"backward of selected attention, prefill B={batch} T=16384 H=16 Hkv=1 d=128 bf16, block 64, "
                        "S=16", "ms_per_step": ms_step, "tflops": tf, "flops_per_step": flops,
            "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "workspace_bytes": int(ws.numel()),
            "launches_per_step": 4}  # dq, list inversion, dK / dV, reduce


def bench_cmp_bwd(torch, nsa, device, steps, warmup, flush, peaks, T=65536):
    """Backward of the compressed branch at the layer shape: dq, d k_cmp, d v_cmp from the
    forward's o and lse, then the pooling backward to the token rows of K and V."""
    from sparse_attention_compress_gb300 import _lib
    w = gen.layer(T=T)
    q, k, v = dev(torch, w.q, device), dev(torch, w.k, device), dev(torch, w.v, device)
    kc, vc = nsa.nsa_compress_k(k), nsa.nsa_compress_k(v)
    do = dev(torch, gen.normal(gen.rng_for(4, 99), (w.tokens, w.h, w.d), "bf16"), device)
    lse = torch.empty((w.tokens, w.h), dtype=torch.float32, device=device)
    o = nsa.nsa_cmp_attn_fwd(q, kc, vc, w.hkv, lse=lse)
    shp = _lib.make_shape(w.tokens, w.h, w.hkv, w.d, _lib.NSA_BF16, batch=1, seqlen=w.tokens)
    ws = torch.empty(nsa.nsa_cmp_attn_bwd_workspace_size(shp), dtype=torch.uint8, device=device)
    dq, dkc, dvc = torch.empty_like(q), torch.empty_like(kc), torch.empty_like(vc)
    dk, dv = torch.empty_like(k), torch.empty_like(v)

    def step():
        nsa.nsa_cmp_attn_bwd(q, kc, vc, o, lse, do, w.hkv, workspace=ws, dq=dq, dk_cmp=dkc, dv_cmp=dvc)
        nsa.nsa_compress_bwd(dkc, w.tokens, out=dk)
        nsa.nsa_compress_bwd(dvc, w.tokens, out=dv)

    ms = float(np.mean(timed(torch, step, steps, warmup, flush)))
    t = np.arange(w.tokens)
    ncaus = np.clip((t - 31) // 16 + 1, 0, None)
    flops = float(ncaus.sum()) * w.h * 2 * w.d * 5  # S and dP recomputed, dQ, dK, dV
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": f"backward of the compressed branch + pooling, layer T={T} H=64 Hkv=4 d=128 bf16 "
                        "(32/16 windows)", "ms_per_step": ms, "tflops": tf, "flops_per_step": flops,
            "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "workspace_bytes": int(ws.numel()),
            "launches_per_step": 5}


def bench_swa_bwd(torch, nsa, device, steps, warmup, flush, peaks, T=65536):
    """Backward of the sliding-window branch (window 512) and of the gate, layer shape."""
    from sparse_attention_compress_gb300 import _lib
    w = gen.layer(T=T)
    q, k, v = dev(torch, w.q, device), dev(torch, w.k, device), dev(torch, w.v, device)
    do = dev(torch, gen.normal(gen.rng_for(4, 98), (w.tokens, w.h, w.d), "bf16"), device)
    lse = torch.empty((w.tokens, w.h), dtype=torch.float32, device=device)
    o = nsa.nsa_swa_fwd(q, k, v, 512, lse=lse)
    shp = _lib.make_shape(w.tokens, w.h, w.hkv, w.d, _lib.NSA_BF16, batch=1, seqlen=w.tokens)
    ws = torch.empty(nsa.nsa_swa_bwd_workspace_size(shp, 512), dtype=torch.uint8, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ms = float(np.mean(timed(torch, lambda: nsa.nsa_swa_bwd(q, k, v, o, lse, do, 512, workspace=ws, dq=dq, dk=dk,
                                                             dv=dv), steps, warmup, flush)))
    t = np.arange(w.tokens)
    flops = float(np.minimum(t + 1, 512).sum()) * w.h * 2 * w.d * 5
    logits = dev(torch, w.gates, device)
    msg = float(np.mean(timed(torch, lambda: nsa.nsa_gate_combine_bwd(do, o, o, o, logits), steps, warmup, flush)))
    gbytes = w.tokens * w.h * (w.d * 2 * 7 + 3 * 4 * 2)
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": f"backward of the sliding window (512) and of the gate, layer T={T} H=64 Hkv=4 d=128 bf16",
            "swa_ms": ms, "swa_tflops": tf, "swa_frac_of_bf16_peak": tf / peaks["bf16_tflops"],
            "gate_ms": msg, "gate_gbs": gbytes / (msg * 1e-3) / 1e9,
            "gate_hbm_frac": gbytes / (msg * 1e-3) / 1e9 / peaks["hbm_gbs"], "launches_per_step": 4}


def bench_layer_train(torch, nsa, device, steps, warmup, flush, peaks):
    """One training step of the layer at T=65536, H=64, Hkv=4: the training forward (keeps
    the branch outputs) and the layer backward (gate, three branches, pooling, sums)."""
    w = gen.layer()
    q, k, v = dev(torch, w.q, device), dev(torch, w.k, device), dev(torch, w.v, device)
    gl = dev(torch, w.gates, device)
    do = dev(torch, gen.normal(gen.rng_for(4, 97), (w.tokens, w.h, w.d), "bf16"), device)
    saved = nsa.nsa_layer_saved_buffers(w.tokens, nsa.num_cmp(w.tokens), w.h, w.hkv, w.d, 16, device)
    from sparse_attention_compress_gb300 import _lib
    shp = _lib.make_shape(w.tokens, w.h, w.hkv, w.d, _lib.NSA_BF16, batch=1, seqlen=w.tokens)
    wsf = torch.empty(nsa.nsa_layer_fwd_workspace_size(shp), dtype=torch.uint8, device=device)
    wsb = torch.empty(int(nsa.load().nsa_layer_bwd_workspace_size(_lib.ctypes.byref(shp), 32, 16, 64, 16, 512)),
                      dtype=torch.uint8, device=device)
    out = torch.empty_like(q)

    def fwd():
        nsa.nsa_layer_fwd_train(q, k, v, gl, saved, workspace=wsf, out=out)

    def bwd():
        nsa.nsa_layer_bwd(q, k, v, gl, saved, do, workspace=wsb)

    ms_f = float(np.mean(timed(torch, fwd, steps, warmup, flush)))
    ms_b = float(np.mean(timed(torch, bwd, steps, warmup, flush)))
    t = np.arange(w.tokens)
    ncaus = np.clip((t - 31) // 16 + 1, 0, None)
    r = w.h // w.hkv
    idx = saved["idx"].cpu().numpy().astype(np.int64)
    blk = np.where(idx >= 0, np.clip(t[:, None, None] - idx * 64 + 1, 0, 64), 0).sum()
    pairs_h = ncaus.sum() * w.h + float(blk) * r + np.minimum(t + 1, 512).sum() * w.h
    fwd_flops, bwd_flops = 4 * w.d * pairs_h, 10 * w.d * pairs_h
    return {"workload": "layer training step T=65536 H=64 Hkv=4 d=128 bf16 (training forward + backward)",
            "fwd_ms": ms_f, "bwd_ms": ms_b, "step_ms": ms_f + ms_b,
            "step_tflops": (fwd_flops + bwd_flops) / ((ms_f + ms_b) * 1e-3) / 1e12,
            "bwd_tflops": bwd_flops / (ms_b * 1e-3) / 1e12, "bwd_workspace_bytes": int(wsb.numel())}


def bench_nosa(torch, nsa, device, steps, warmup, flush, peaks):
    """NOSA stage 2: CIS-weighted selected attention on the prefill workload, and the
    block CIS scores plus two-stage selection on the varlen selection workload."""
    w = gen.prefill()
    q = dev(torch, w.q, device).view(w.batch, w.seqlen, w.h, w.d)
    k, v, idx = dev(torch, w.k, device), dev(torch, w.v, device), dev(torch, w.idx, device)
    cis = dev(torch, gen.cis_scores(gen.rng_for(1, 77), w.tokens, w.hkv), device)
    out = torch.empty_like(q)
    ms_att = float(np.mean(timed(torch, lambda: nsa.nsa_sparse_cis_fwd(q, k, v, cis, idx, 64, out=out), steps,
                                 warmup, flush)))
    flops = prefill_flops(w)
    del q, k, v, idx, out, cis
    sw = gen.selection()
    cu = dev(torch, sw.cu_seqlens, device)
    lens = np.diff(sw.cu_seqlens)
    nb = ((-(-sw.max_len // 64)) + 3) // 4 * 4
    sc = torch.rand((sw.tokens, sw.hkv, nb), dtype=torch.float32, device=device)
    scis = dev(torch, gen.cis_scores(gen.rng_for(2, 77), sw.tokens, sw.hkv), device)
    cs = torch.empty((len(lens), sw.hkv, nb), dtype=torch.float32, device=device)
    sel = torch.empty((sw.tokens, sw.hkv, 16), dtype=torch.int32, device=device)

    def select():
        nsa.nsa_cis_block_scores(scis, cu_seqlens=cu, max_seqlen=sw.max_len, nb_stride=nb, out=cs)
        nsa.nsa_topk_two_stage(sc, cs, 32, 16, cu_seqlens=cu, max_seqlen=sw.max_len, out=sel)

    ms_sel = float(np.mean(timed(torch, select, steps, warmup, flush)))
    tf = flops / (ms_att * 1e-3) / 1e12
    return {"cis_attention": {"workload": "CIS-weighted selected attention, prefill B=8 T=16384 H=16 Hkv=1 d=128 "
                                          "bf16, block 64, S=16", "ms": ms_att, "tflops": tf,
                              "frac_of_bf16_peak": tf / peaks["bf16_tflops"]},
            "cis_selection": {"workload": "block CIS scores + two-stage top-16 of 32, selection workload "
                                          f"({sw.tokens} tokens, Hkv=2)", "ms": ms_sel,
                              "tokens_per_s": sw.tokens / (ms_sel * 1e-3)},
            "launches_per_step": 3}


def bench_decode_offload(torch, nsa, device, steps, warmup, flush):
    """The decode workload with its K/V cache in page-locked host memory (the offloaded
    cache of the NOSA inference system); compressed keys, q and o stay in HBM."""
    w = gen.decode()
    n_c = nsa.num_cmp(w.max_len)
    kcmp = nsa.nsa_compress_k(dev(torch, w.k_cache, device)).view(w.batch, n_c, w.hkv, w.d)
    torch.cuda.empty_cache()
    hk = pinned(torch, w.k_cache).view(torch.bfloat16)
    hv = pinned(torch, w.v_cache).view(torch.bfloat16)
    q, sl = dev(torch, w.q, device), dev(torch, w.seqlens, device)
    ws = torch.empty(nsa.nsa_sparse_decode_workspace_size(w.batch, w.max_len, w.h, w.hkv, w.d, k=w.topk),
                     dtype=torch.uint8, device=device)
    idx = torch.empty((w.batch, w.hkv, w.topk), dtype=torch.int32, device=device)
    out = torch.empty_like(q)

    def step():
        nsa.nsa_sparse_decode(q, hk, hv, kcmp, sl, k=w.topk, workspace=ws, idx_out=idx, out=out)

    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        step()
    torch.cuda.current_stream().wait_stream(st)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    ms_step = float(np.mean(timed(torch, g.replay, steps, warmup, flush)))
    ih = idx.cpu().numpy().astype(np.int64)
    t = (w.seqlens.astype(np.int64) - 1)[:, None, None]
    keys = np.where(ih >= 0, np.clip(t - ih * 64 + 1, 0, 64), 0).sum()
    link_bytes = int(keys * w.d * 2 * 2)  # chosen K and V rows, read from host memory
    full_bytes = int(w.seqlens.astype(np.int64).sum() * w.hkv * w.d * 2 * 2)  # every cached K and V row
    del hk, hv
    return {"workload": "decode B=32 L=32768 H=16 Hkv=2 d=128 bf16 top-k 64 (blocks of 64), K/V cache "
                        "(1.07 GB) in page-locked host memory, compressed keys in HBM",
            "ms_per_step": ms_step, "tokens_per_s": w.batch / (ms_step * 1e-3),
            "link_bytes_per_step": link_bytes, "link_gbs": link_bytes / (ms_step * 1e-3) / 1e9,
            "full_cache_bytes": full_bytes, "kernels_per_step": 1, "memsets_per_step": 1, "cuda_graph": True}


def bench_selection(torch, nsa, device, steps, warmup, flush, peaks):
    """Varlen selection stage: compress -> block scores -> top-16, each call timed on its own
    (CUDA events between the calls of one step) against its own bound."""
    w = gen.selection()
    q, k = dev(torch, w.q, device), dev(torch, w.k, device)
    cu = dev(torch, w.cu_seqlens, device)
    lens = np.diff(w.cu_seqlens)
    n_cmp = int(sum(nsa.num_cmp(int(L)) for L in lens))
    kc = torch.empty((n_cmp, w.hkv, w.d), dtype=torch.bfloat16, device=device)
    nb = -(-w.max_len // 64)
    nb = (nb + 3) // 4 * 4
    sc = torch.empty((w.tokens, w.hkv, nb), dtype=torch.float32, device=device)
    idx = torch.empty((w.tokens, w.hkv, 16), dtype=torch.int32, device=device)
    calls = [lambda: nsa.nsa_compress_k(k, cu_seqlens=cu, max_seqlen=w.max_len, out=kc),
             lambda: nsa.nsa_cmp_scores_pool(q, kc, w.hkv, cu_seqlens=cu, max_seqlen=w.max_len, nb_stride=nb, out=sc),
             lambda: nsa.nsa_topk_select(sc, 16, cu_seqlens=cu, max_seqlen=w.max_len, out=idx)]
    for _ in range(warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in ev:
        flush()
        e[0].record()
        for i, c in enumerate(calls):
            c()
            e[i + 1].record()
    torch.cuda.synchronize()
    seg = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev]).mean(axis=0)
    ms = float(np.mean([e[0].elapsed_time(e[3]) for e in ev]))
    t = np.concatenate([np.arange(L) for L in lens])
    ncaus = np.where(t >= 31, (t - 31) // 16 + 1, 0)
    pass_flops = float(ncaus.sum()) * w.h * 2 * w.d  # one pass of scores over the causal compressed keys
    # the block scores take two passes over the keys (the softmax normaliser, then the
    # probabilities pooled to blocks): twice the contraction, one exponential per (head, key) each
    score_flops, score_exps = 2 * pass_flops, 2 * float(ncaus.sum()) * w.h
    comp_bytes = w.tokens * w.hkv * w.d * 2 + n_cmp * w.hkv * w.d * 2  # K in, compressed keys out
    own = np.concatenate([np.arange(L) // 64 for L in lens])
    topk_bytes = float(np.minimum(own + 1, nb).sum()) * w.hkv * 4 + w.tokens * w.hkv * 16 * 4  # causal scores in, lists out
    ms_c, ms_s, ms_k = (float(x) for x in seg)
    return {"workload": f"selection varlen lengths {lens.tolist()} H=16 Hkv=2 d=128 bf16 (compress 32/16, "
                        "pool to 64-token blocks, top-16 with 1 init + 2 local)",
            "ms_per_step": ms, "tokens_per_s": w.tokens / (ms * 1e-3), "qk_tflops": pass_flops / (ms * 1e-3) / 1e12,
            "launches_per_step": 3,
            "compress": {"ms": ms_c, "bytes": comp_bytes, "gbs": comp_bytes / (ms_c * 1e-3) / 1e9,
                         "hbm_frac": comp_bytes / (ms_c * 1e-3) / 1e9 / peaks["hbm_gbs"]},
            "scores": {"ms": ms_s, "flops": score_flops, "exps": score_exps,
                       "tflops": score_flops / (ms_s * 1e-3) / 1e12,
                       "tensor_frac": score_flops / (ms_s * 1e-3) / 1e12 / peaks["bf16_tflops"],
                       "exps_per_s": score_exps / (ms_s * 1e-3)},
            "topk": {"ms": ms_k, "bytes": topk_bytes, "gbs": topk_bytes / (ms_k * 1e-3) / 1e9,
                     "hbm_frac": topk_bytes / (ms_k * 1e-3) / 1e9 / peaks["hbm_gbs"]}}


def bench_block_sparse(torch, nsa, device, steps, warmup, flush, peaks, lengths=(1024, 4096, 16384)):
    """Block-mask sparse attention at the pages' block-sparse table shape (batch 8, 16
    heads, d 128, 64x64 tiles, half of the tiles active, not causal)."""
    res = {"workload": "block-mask attention B=8 H=16 d=128 bf16, 64x64 tiles, 50% active, not causal",
           "launches_per_step": 2}
    for T in lengths:
        w = gen.block_sparse(B=8, T=T, H=16, density=0.5, causal=False)
        q, k, v = (dev(torch, a, device).view(8, T, 16, 128) for a in (w.q, w.k, w.v))
        m = dev(torch, w.idx, device)
        out = torch.empty_like(q)
        ws = torch.empty(nsa.nsa_block_sparse_workspace_size(nsa.make_shape(8 * T, 16, 16, 128, 1, batch=8,
                                                                              seqlen=T)),
                         dtype=torch.uint8, device=device)

        def step():
            nsa.nsa_block_sparse_fwd(q, k, v, m, causal=False, workspace=ws, out=out)

        ms = float(np.mean(timed(torch, step, steps, warmup, flush)))
        flops = 4.0 * 128 * float(w.idx.astype(np.int64).sum()) * 64 * 64
        tf = flops / (ms * 1e-3) / 1e12
        res[f"T{T}"] = {"ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "flops": flops}
        del q, k, v, m, out, ws
        torch.cuda.empty_cache()
    return res


# kernels of one layer call: compress K, compress V, transpose V_cmp, transpose V,
# compressed branch + block scores, top-k, selected branch, sliding branch, gated sum
LAYER_LAUNCHES = 9


def bench_layer(torch, nsa, device, steps, warmup, flush, T=65536):
    w = gen.layer(T=T)
    q, k, v = dev(torch, w.q, device), dev(torch, w.k, device), dev(torch, w.v, device)
    gates = dev(torch, w.gates, device)
    shp = nsa.make_shape(w.tokens, w.h, w.hkv, w.d, 1, batch=1, seqlen=w.tokens)
    ws = torch.empty(nsa.nsa_layer_fwd_workspace_size(shp), dtype=torch.uint8, device=device)
    idx = torch.empty((w.tokens, w.hkv, 16), dtype=torch.int32, device=device)
    out = torch.empty_like(q)

    def step():
        nsa.nsa_layer_fwd(q, k, v, gates, workspace=ws, idx_out=idx, out=out)

    ms = float(np.mean(timed(torch, step, steps, warmup, flush)))
    t = np.arange(w.tokens)
    ncaus = np.where(t >= 31, (t - 31) // 16 + 1, 0).astype(np.float64)
    ih = idx.cpu().numpy().astype(np.int64)
    sel = np.where(ih >= 0, np.clip(t[:, None, None] - ih * 64 + 1, 0, 64), 0).sum()
    r = w.h // w.hkv
    flops = 4 * w.d * (ncaus.sum() * w.h + float(sel) * r + np.minimum(t + 1, 512).sum() * w.h)
    return {"workload": f"layer B=1 T={w.tokens} H=64 Hkv=4 d=128 bf16 (compressed 32/16 + selected 64x16 + window 512 "
                        "+ sigmoid gates)",
            "ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12, "tokens_per_s": w.tokens / (ms * 1e-3),
            "flops_per_step": flops, "launches_per_step": LAYER_LAUNCHES}


# ----------------------------------------------------------------------------- main arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-sample-rows", type=int, default=0, help="0: size the oracle sample to ~15 s")
    ap.add_argument("--batch", type=int, default=8, help="prefill batch (8 is the benchmark; smaller for ncu)")
    ap.add_argument("--layer-tokens", type=int, default=65536, help="layer workload length (65536 is the benchmark; also the branch backwards' length)")
    ap.add_argument("--only", default="", choices=["", "prefill", "prefill_bwd", "cmp_bwd", "swa_bwd", "layer_train", "nosa", "decode",
                                                    "decode_offload",
                                                    "selection", "layer", "block_sparse"],
                    help="time one workload only, with no e2e or CPU arm (for profiler captures)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import sparse_attention_compress_gb300 as nsa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        barrier = dist.barrier
    nsa.load()
    peaks = load_peaks()
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    flush_src = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=device)

    def flush():
        # write a buffer twice the L2 size, then copy another one into it: the L2 ends up
        # holding clean unrelated lines, so no write-back of the flush lands in a timed step
        flush_buf.zero_()
        flush_buf.copy_(flush_src)

    if args.only in ("prefill_bwd", "cmp_bwd", "swa_bwd", "layer_train", "nosa", "decode", "decode_offload",
                     "selection", "layer", "block_sparse"):
        fn = {"layer_train": lambda: bench_layer_train(torch, nsa, device, args.steps, args.warmup, flush, peaks),
              "swa_bwd": lambda: bench_swa_bwd(torch, nsa, device, args.steps, args.warmup, flush, peaks,
                                               args.layer_tokens),
              "cmp_bwd": lambda: bench_cmp_bwd(torch, nsa, device, args.steps, args.warmup, flush, peaks,
                                               args.layer_tokens),
              "nosa": lambda: bench_nosa(torch, nsa, device, args.steps, args.warmup, flush, peaks),
              "prefill_bwd": lambda: bench_prefill_bwd(torch, nsa, device, args.steps, args.warmup, flush, peaks,
                                                       batch=args.batch),
              "decode": lambda: bench_decode(torch, nsa, device, args.steps, args.warmup, flush, peaks),
              "decode_offload": lambda: bench_decode_offload(torch, nsa, device, args.steps, args.warmup, flush),
              "selection": lambda: bench_selection(torch, nsa, device, args.steps, args.warmup, flush, peaks),
              "block_sparse": lambda: bench_block_sparse(torch, nsa, device, args.steps, args.warmup, flush, peaks),
              "layer": lambda: bench_layer(torch, nsa, device, args.steps, args.warmup, flush,
                                           args.layer_tokens)}[args.only]
        print(json.dumps({"only": args.only, **fn()}), flush=True)
        return

    w = gen.prefill(B=args.batch, salt=rank)  # every rank processes its own batch
    flops = prefill_flops(w)
    q, k, v = dev(torch, w.q, device), dev(torch, w.k, device), dev(torch, w.v, device)
    idx = dev(torch, w.idx, device)
    out = torch.empty_like(q)
    qv = q.view(w.batch, w.seqlen, w.h, w.d)

    def step():
        nsa.nsa_sparse_fwd(qv, k, v, idx, w.block_size, out=out)

    clocks = Clocks(local)
    clocks.start()
    ms = timed(torch, step, args.steps, args.warmup, flush, barrier)
    clk = clocks.stop()
    ms_step = float(np.mean(ms))
    ms_step = max_over_ranks(ms_step, device)
    value = flops * world / (ms_step * 1e-3) / 1e12
    kernel_tflops = flops / (ms_step * 1e-3) / 1e12
    # K and V rows each attended (token, kv-head) pulls from L2 (2 * d bf16 per key)
    gathered = flops / (w.h // w.hkv) / (4 * w.d) * (2 * w.d * 2)
    if args.only == "prefill":
        print(json.dumps({"only": "prefill", "batch": w.batch, "ms_per_step": ms_step, "tflops": kernel_tflops}),
              flush=True)
        return

    # end to end through the public call with host buffers: inputs in, output out
    hq, hk, hv, hi = pinned(torch, w.q), pinned(torch, w.k), pinned(torch, w.v), pinned(torch, w.idx)
    ho = torch.empty((w.tokens, w.h, w.d), dtype=torch.int16).pin_memory()
    q16, k16, v16 = q.view(torch.int16), k.view(torch.int16), v.view(torch.int16)

    # Sequence by sequence on three streams: the copy engines move sequence b+1 in and
    # sequence b-1 out while the SMs attend over sequence b (same calls, same bytes).
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(w.batch)]
    ev_done = [torch.cuda.Event() for _ in range(w.batch)]
    o16 = out.view(torch.int16).view(w.tokens, w.h, w.d)

    def e2e_step():
        comp = torch.cuda.current_stream()
        s_in.wait_stream(comp)
        for b in range(w.batch):
            rows = slice(b * w.seqlen, (b + 1) * w.seqlen)
            with torch.cuda.stream(s_in):
                q16[rows].copy_(hq[rows], non_blocking=True)
                k16[rows].copy_(hk[rows], non_blocking=True)
                v16[rows].copy_(hv[rows], non_blocking=True)
                idx[rows].copy_(hi[rows], non_blocking=True)
                ev_in[b].record(s_in)
            comp.wait_event(ev_in[b])
            nsa.nsa_sparse_fwd(qv[b:b + 1], k[rows], v[rows], idx[rows], w.block_size, out=out[rows])
            ev_done[b].record(comp)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                ho[rows].copy_(o16[rows], non_blocking=True)
        comp.wait_stream(s_out)  # the step ends when the last output is on the host

    e2e_steps = max(3, args.steps // 2)
    e2e_ms = float(np.mean(timed(torch, e2e_step, e2e_steps, 1, None, barrier)))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hi))
    d2h = ho.numel() * ho.element_size()

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill B=8 T=16384 H=16 Hkv=1 d=128 bf16, block 64, S=16 random causal blocks "
                               "(block 0 and own block always listed)", "global_batch": w.batch * world,
                   "seq_len": 16384, "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (258 MB written, then 258 MB copied; outside the event pair)",
                   "flops_per_step": flops},
        "roofline": {"kernel": "sparse_fwd_tma<2>", "bound": "tensor", "achieved": kernel_tflops,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": kernel_tflops / peaks["bf16_tflops"],
                     "peak_source": peaks["source"] + " bf16 dense (cuBLAS burst)",
                     "traffic": PREFILL_NCU_TRAFFIC if args.batch == 8 else None,
                     "gathered_bytes": gathered, "gather_gbs": gathered / (ms_step * 1e-3) / 1e9},
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": args.steps + w.batch * e2e_steps,  # the e2e step launches one kernel per sequence
        "clocks": clk,
    }
    del hq, hk, hv, hi, ho

    if world == 1 and not args.no_extras:
        del q, k, v, out, qv
        torch.cuda.empty_cache()
        try:
            line["prefill_bwd"] = bench_prefill_bwd(torch, nsa, device, max(3, args.steps // 2), args.warmup, flush,
                                                    peaks)
            line["gpu_launches"] += 4 * max(3, args.steps // 2)
        except Exception as e:
            line["prefill_bwd"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["cmp_bwd"] = bench_cmp_bwd(torch, nsa, device, max(3, args.steps // 2), args.warmup, flush, peaks)
            line["gpu_launches"] += 5 * max(3, args.steps // 2)
        except Exception as e:
            line["cmp_bwd"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["swa_bwd"] = bench_swa_bwd(torch, nsa, device, max(3, args.steps // 2), args.warmup, flush, peaks)
            line["gpu_launches"] += 4 * max(3, args.steps // 2)
        except Exception as e:
            line["swa_bwd"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["layer_train"] = bench_layer_train(torch, nsa, device, 3, args.warmup, flush, peaks)
            line["gpu_launches"] += 3 * 9 + 3 * 16  # training forward 9 kernels, backward 16
        except Exception as e:
            line["layer_train"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["nosa"] = bench_nosa(torch, nsa, device, max(3, args.steps // 2), args.warmup, flush, peaks)
            line["gpu_launches"] += 3 * max(3, args.steps // 2)
        except Exception as e:
            line["nosa"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["decode"] = bench_decode(torch, nsa, device, args.steps, args.warmup, flush, peaks)
            line["gpu_launches"] += 3 * args.steps  # decode kernel, NOSA decode kernel, cache compression
        except Exception as e:  # report, never hide
            line["decode"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["decode_offload"] = bench_decode_offload(torch, nsa, device, args.steps, args.warmup, flush)
            line["gpu_launches"] += args.steps
        except Exception as e:
            line["decode_offload"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["selection"] = bench_selection(torch, nsa, device, args.steps, args.warmup, flush, peaks)
            line["gpu_launches"] += 3 * args.steps
        except Exception as e:
            line["selection"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["block_sparse"] = bench_block_sparse(torch, nsa, device, max(3, args.steps // 2), args.warmup,
                                                      flush, peaks)
            line["gpu_launches"] += 2 * 3 * max(3, args.steps // 2)
        except Exception as e:
            line["block_sparse"] = {"error": repr(e)}
        torch.cuda.empty_cache()
        try:
            line["layer"] = bench_layer(torch, nsa, device, max(3, args.steps // 2), args.warmup, flush)
            line["gpu_launches"] += LAYER_LAUNCHES * max(3, args.steps // 2)
        except Exception as e:
            line["layer"] = {"error": repr(e)}

    if rank == 0 and world == 1 and not args.no_extras:
        try:  # live ceilings of this GPU for the secondary rooflines
            from sparse_attention_compress_gb300 import probe
            pr = probe.run()
            line["probes"] = pr
            rf = line["roofline"]
            rf["l2_read_peak_gbs"] = pr["l2_read_gbs"]
            rf["l2_gather_peak_gbs"] = pr["l2_gather_gbs"]  # random 4 KB slices into shared memory, no compute
            rf["gather_frac_of_l2_gather"] = rf["gather_gbs"] / pr["l2_gather_gbs"]
            rf["mma_sync_peak_tflops"] = pr["mma_sync_bf16_tflops"]
            rf["frac_of_mma_sync"] = kernel_tflops / pr["mma_sync_bf16_tflops"]
            off = line.get("decode_offload", {})
            if "link_gbs" in off and pr.get("c2c_gather_gbs"):
                # the chosen blocks are random 4 KB slices of host memory: the gather probe bounds them
                off["roofline"] = {"bound": "cpu-gpu link", "achieved": off["link_gbs"], "peak": pr["c2c_gather_gbs"],
                                   "unit": "GB/s", "frac": off["link_gbs"] / pr["c2c_gather_gbs"],
                                   "peak_source": "live probe: random 4 KB host-memory slices into shared memory"}
                # no kernel can attend over the whole offloaded cache faster than it streams over the link
                off["full_attention_floor_ms"] = off["full_cache_bytes"] / (pr["c2c_read_gbs"] * 1e9) * 1e3
                off["speedup_vs_full_attention_floor"] = off["full_attention_floor_ms"] / off["ms_per_step"]
            sel = line.get("selection", {})
            if "scores" in sel and pr.get("ex2_per_sm_per_clk"):
                # the block-score kernel against both of its units: the tensor cores (two
                # passes of q.k) and the special-function unit (one ex2 per head and key per
                # pass) at the probe's ex2 rate x SMs x clock
                sco = sel["scores"]
                ex2_peak = pr["ex2_per_sm_per_clk"] * pr["sms"] * pr["clock_mhz"] * 1e6
                sco["mufu_peak_exps_per_s"] = ex2_peak
                sco["mufu_frac"] = sco["exps_per_s"] / ex2_peak
                mufu = sco["mufu_frac"] >= sco["tensor_frac"]
                sel["roofline"] = {"kernel": "block scores (tc::attn_kernel, scores only)",
                                   "bound": "alu" if mufu else "tensor",
                                   "achieved": sco["exps_per_s"] / 1e9 if mufu else sco["tflops"],
                                   "peak": ex2_peak / 1e9 if mufu else peaks["bf16_tflops"],
                                   "unit": "Gexp/s" if mufu else "TFLOP/s",
                                   "frac": sco["mufu_frac"] if mufu else sco["tensor_frac"],
                                   "peak_source": ("live probe: ex2.approx per SM per clock x SMs x clock" if mufu
                                                   else peaks["source"] + " bf16 dense (cuBLAS burst)"),
                                   "traffic": None}
            if "tflops" in line.get("layer", {}):
                line["layer"]["frac_of_bf16_peak"] = line["layer"]["tflops"] / peaks["bf16_tflops"]
        except Exception as e:
            line["probes"] = {"error": repr(e)}
    if rank == 0 and world == 1:
        n_rows = args.cpu_sample_rows
        if n_rows <= 0:  # size the sample to ~15 s of oracle work
            _, dt, _, _ = oracle_prefill_sample(w, 512, seed=7)
            n_rows = int(min(w.tokens, max(512, 512 * 15.0 / max(dt, 1e-3))))
        val, dt, _, thr = oracle_prefill_sample(w, n_rows, seed=11)
        line["cpu_baseline"] = {"value": val, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": f"{n_rows} random query tokens (all heads) of the prefill workload, "
                                          f"{dt:.1f} s"}
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
