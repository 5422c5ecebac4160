"""Write tests/golden/oracle_regression.json: small oracle results on seeded inputs.

The pages print no worked numeric example, so no stored value here is a printed one.
These values freeze what the oracle computes today: a later change to its arithmetic
makes tests/test_golden.py fail until the change (and the passage that justifies it) is
recorded and this file is regenerated.  Calls only oracle/ and the seeded input
generators.  Run from the repository root: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import oracle as orc  # noqa: E402
from sparse_attention_compress_gb300 import inputs as gen  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")


def summary(a):
    """Sum, sum of squares and eight values at fixed flat positions."""
    a = np.asarray(a, np.float64).ravel()
    pos = np.linspace(0, a.size - 1, 8).astype(int) if a.size else []
    return {"n": int(a.size), "sum": float(a.sum()), "sumsq": float((a * a).sum()),
            "samples": [float(a[i]) for i in pos], "positions": [int(i) for i in pos]}


def compute():
    rng = np.random.default_rng(20261203)
    lengths = [200, 131, 70]
    cu = gen.varlen_cu_seqlens(lengths)
    h, hkv, d = 4, 2, 32
    q, do = gen.normal(rng, (cu[-1], h, d), "bf16"), gen.normal(rng, (cu[-1], h, d), "bf16")
    k, v = gen.normal(rng, (cu[-1], hkv, d), "bf16"), gen.normal(rng, (cu[-1], hkv, d), "bf16")
    kc_exact, kc = orc.compress(k, cu)
    _, vc = orc.compress(v, cu)
    sc = orc.cmp_scores_pool(q, kc, cu)
    idx = orc.topk(sc, cu, k=3)
    o_s, l_s = orc.sparse_attn(q, k, v, idx, cu, 64)
    o_c, l_c = orc.cmp_attn(q, kc, vc, cu)
    o_w, l_w = orc.swa(q, k, v, cu, 40)
    gates = rng.standard_normal((int(cu[-1]), h, 3)).astype(np.float32)
    lay = orc.layer(q, k, v, gates, cu, S=3, window=40)
    dq, dk, dv = orc.sparse_attn_bwd(q, k, v, idx, do, cu, 64)
    cis = gen.cis_scores(rng, int(cu[-1]), hkv)
    cb = orc.cis_block_scores(cis, cu)
    o_cis, _ = orc.sparse_attn_cis(q, k, v, cis, idx, cu, 64)
    ldq, ldk, ldv, ldg = orc.layer_bwd(q, k, v, gates, idx, do, cu, window=40)
    res = {"compress_exact": summary(kc_exact), "scores": summary(sc), "topk": summary(idx),
           "sparse_o": summary(o_s), "sparse_lse": summary(l_s), "cmp_o": summary(o_c), "cmp_lse": summary(l_c[np.isfinite(l_c)]),
           "swa_o": summary(o_w), "layer_o": summary(lay["o"]), "layer_idx": summary(lay["idx"]),
           "sparse_dq": summary(dq), "sparse_dk": summary(dk), "sparse_dv": summary(dv),
           "cis_blocks": summary(cb), "cis_o": summary(o_cis), "layer_dq": summary(ldq), "layer_dk": summary(ldk),
           "layer_dv": summary(ldv), "layer_dgates": summary(ldg)}
    return res


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(compute(), f, indent=1)
    print(OUT)
