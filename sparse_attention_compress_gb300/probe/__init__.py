"""Roofline micro-benchmarks (L2, HBM and host-memory read bandwidth, mma.sync bf16 and ex2 rates).

run() compiles rooflines.cu with nvcc for sm_103a and returns its JSON result; the
benchmark uses it for the secondary ceilings of its roofline report.
"""
from __future__ import annotations

import json
import os
import subprocess

from ..build import ARCH, BUILD, nvcc

_SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rooflines.cu")


def run(timeout: float = 120.0) -> dict:
    os.makedirs(BUILD, exist_ok=True)
    exe = os.path.join(BUILD, "rooflines")
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(_SRC):
        subprocess.check_call([nvcc(), *ARCH, "-O3", "-o", exe, _SRC])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=timeout)
    if out.returncode != 0:
        raise RuntimeError(f"roofline probe failed: {out.stdout} {out.stderr}")
    return json.loads(out.stdout.strip().splitlines()[-1])
