"""Seeded synthetic workloads for the native-sparse-attention hot path.

This module only draws random numbers and lays them out: it holds none of the
method's arithmetic, so the CUDA path and the CPU oracle can both consume the
very same bytes.  NumPy ``Generator(PCG64(seed))``; draw order: sequence lengths
(when they size the tensors), Q, K, V, block indices, gate logits.  fp32 N(0,1) draws are
rounded to bf16 (nearest, ties to even) here on the host; bf16 tensors are carried
as ``uint16`` bit patterns.

Workloads (shapes of the pages' own settings: NOSA-1B's 16 heads / 2 kv-heads and
32k context, the H100 block-sparse table's batch 8 / heads 16 / dim 128, the 64k NSA
speed claim):

  tiny    B=1  T=256    H=4  Hkv=1 d=64  fp32, block 32, S=4 random causal indices
  prefill B=8  T=16384  H=16 Hkv=1 d=128 bf16, block 64, S=16 random causal indices
  select  4 varlen sequences, L ~ U[4096, 32768], H=16 Hkv=2 d=128 bf16
  decode  B=32, context 32768, H=16 Hkv=2 d=128 bf16 cache, top-k 64
  layer   B=1  T=65536  H=64 Hkv=4 d=128 bf16 + gate logits [T, H, 3] fp32
"""
from __future__ import annotations

import dataclasses

import numpy as np

SEED_BASE = 20261200


def rng_for(config_number: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + config_number + 1000 * salt))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) draws in fp32, rounded to bf16 bits when dtype == 'bf16'."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def cis_scores(rng: np.random.Generator, tokens: int, hkv: int) -> np.ndarray:
    """Synthetic per-key importance scores [tokens, hkv] fp32 in (0, 1): the logistic
    sigmoid of N(0,1) draws (the scorer that produces them is learned)."""
    x = rng.standard_normal(size=(tokens, hkv), dtype=np.float32)
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def dense_cu_seqlens(batch: int, seqlen: int) -> np.ndarray:
    return (np.arange(batch + 1, dtype=np.int64) * seqlen).astype(np.int32)


def varlen_cu_seqlens(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, np.int64))]).astype(np.int32)


def random_block_indices(rng: np.random.Generator, cu_seqlens: np.ndarray, hkv: int, S: int,
                         block_size: int, force_first: bool) -> np.ndarray:
    """Random causal block lists [tokens, hkv, S] int32.

    Each list holds the query's own block (and block 0 when force_first), plus
    distinct uniform draws from the remaining causal blocks (those starting at or
    before the query), sorted ascending and padded with -1 when fewer exist.
    """
    cu = np.asarray(cu_seqlens, np.int64)
    tot = int(cu[-1])
    t = np.concatenate([np.arange(cu[i + 1] - cu[i]) for i in range(len(cu) - 1)]) if tot else \
        np.zeros(0, np.int64)
    own = (t // block_size).astype(np.int64)
    nb = int(own.max()) + 1 if tot else 1
    out = np.full((tot, hkv, S), -1, np.int32)
    rows = tot * hkv
    own_r = np.repeat(own, hkv)
    # random priority for every candidate block; forced blocks get -1 (first), non-causal +2
    key = rng.random((rows, nb), dtype=np.float32)
    j = np.arange(nb)[None, :]
    key = np.where(j > own_r[:, None], 2.0, key)
    key = np.where(j == own_r[:, None], -1.0, key)
    if force_first:
        key[:, 0] = -1.0
    order = np.argsort(key, axis=1, kind="stable")[:, :S]
    chosen = np.take_along_axis(key, order, axis=1)
    order = np.where(chosen <= 1.0, order, np.iinfo(np.int32).max)
    order.sort(axis=1)
    order = np.where(order == np.iinfo(np.int32).max, -1, order)
    out[:] = order.reshape(tot, hkv, S).astype(np.int32)
    return out


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str
    cu_seqlens: np.ndarray
    h: int
    hkv: int
    d: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    block_size: int = 64
    S: int = 16
    kernel: int = 32
    stride: int = 16
    n_init: int = 1
    n_local: int = 2
    window: int = 512
    idx: np.ndarray | None = None
    gates: np.ndarray | None = None
    batch: int = 0
    seqlen: int = 0

    @property
    def tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_len(self) -> int:
        return int(np.max(np.diff(self.cu_seqlens)))


def attention_workload(name: str, config_number: int, B: int, T: int, H: int, HKV: int, D: int,
                       dtype: str, block_size: int, S: int, force_first: bool, salt: int = 0) -> Workload:
    rng = rng_for(config_number, salt)
    q = normal(rng, (B * T, H, D), dtype)
    k = normal(rng, (B * T, HKV, D), dtype)
    v = normal(rng, (B * T, HKV, D), dtype)
    cu = dense_cu_seqlens(B, T)
    idx = random_block_indices(rng, cu, HKV, S, block_size, force_first)
    return Workload(name, dtype, cu, H, HKV, D, q, k, v, block_size=block_size, S=S, idx=idx,
                    batch=B, seqlen=T)


def tiny(T: int = 256) -> Workload:
    """B=1, T=256, H=4, Hkv=1, d=64, fp32, block 32, S=4, own block always listed."""
    return attention_workload("tiny", 0, 1, T, 4, 1, 64, "f32", 32, 4, force_first=False)


def prefill(B: int = 8, T: int = 16384, salt: int = 0) -> Workload:
    """B=8, T=16384, H=16, Hkv=1, d=128, bf16, block 64, S=16, blocks 0 and own listed.
    `salt` draws an independent batch (one per rank when the work is sharded)."""
    return attention_workload("prefill", 1, B, T, 16, 1, 128, "bf16", 64, 16, force_first=True, salt=salt)


def selection(n_seqs: int = 4, lo: int = 4096, hi: int = 32768, H: int = 16, HKV: int = 2,
              D: int = 128) -> Workload:
    """Varlen selection stage: lengths ~ U[lo, hi] (inclusive), packed with cu_seqlens."""
    rng = rng_for(2)
    # lengths are drawn first so that the tensors can be sized; Q, K, V follow
    lengths = rng.integers(lo, hi, size=n_seqs, endpoint=True)
    tot = int(lengths.sum())
    q = normal(rng, (tot, H, D), "bf16")
    k = normal(rng, (tot, HKV, D), "bf16")
    v = normal(rng, (tot, HKV, D), "bf16")
    return Workload("selection", "bf16", varlen_cu_seqlens(lengths), H, HKV, D, q, k, v, S=16,
                    seqlen=int(lengths.max()))


@dataclasses.dataclass
class DecodeWorkload:
    q: np.ndarray        # [B, H, d] bf16 bits
    k_cache: np.ndarray  # [B, L, Hkv, d]
    v_cache: np.ndarray
    seqlens: np.ndarray  # [B] int32
    h: int
    hkv: int
    d: int
    topk: int = 64
    block_size: int = 64
    kernel: int = 32
    stride: int = 16
    n_init: int = 1
    n_local: int = 2

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def max_len(self) -> int:
        return self.k_cache.shape[1]


def decode(B: int = 32, L: int = 32768, H: int = 16, HKV: int = 2, D: int = 128, topk: int = 64,
           seqlens=None) -> DecodeWorkload:
    """Decode step: one new query per sequence; the bf16 N(0,1) cache holds L tokens."""
    rng = rng_for(3)
    q = normal(rng, (B, H, D), "bf16")
    kc = normal(rng, (B, L, HKV, D), "bf16")
    vc = normal(rng, (B, L, HKV, D), "bf16")
    sl = np.full(B, L, np.int32) if seqlens is None else np.asarray(seqlens, np.int32)
    return DecodeWorkload(q, kc, vc, sl, H, HKV, D, topk=topk)


def layer(T: int = 65536, H: int = 64, HKV: int = 4, D: int = 128, B: int = 1, lengths=None) -> Workload:
    """Three-branch layer: bf16 Q/K/V N(0,1) and fp32 N(0,1) gate logits [tokens, H, 3].

    lengths: packed varlen sequences (cu_seqlens) instead of B dense sequences of T tokens."""
    rng = rng_for(4, 0 if lengths is None else 1)
    cu = dense_cu_seqlens(B, T) if lengths is None else varlen_cu_seqlens(lengths)
    n = int(cu[-1])
    q = normal(rng, (n, H, D), "bf16")
    k = normal(rng, (n, HKV, D), "bf16")
    v = normal(rng, (n, HKV, D), "bf16")
    gates = rng.standard_normal(size=(n, H, 3), dtype=np.float32)
    if lengths is None:
        return Workload("layer", "bf16", cu, H, HKV, D, q, k, v, S=16, gates=gates, batch=B, seqlen=T)
    return Workload("layer", "bf16", cu, H, HKV, D, q, k, v, S=16, gates=gates)


def block_mask(rng: np.random.Generator, B: int, H: int, T: int, density: float = 0.5, causal: bool = True,
               block: int = 64) -> np.ndarray:
    """uint8 [B, H, nb, nb] block mask: each (query block, key block) tile active with
    probability `density`; the diagonal tile is always active (every query keeps its own
    block); with causal, tiles above the diagonal are cleared."""
    nb = -(-T // block)
    m = (rng.random((B, H, nb, nb)) < density).astype(np.uint8)
    i = np.arange(nb)
    m[:, :, i, i] = 1
    if causal:
        m &= np.tril(np.ones((nb, nb), np.uint8))
    return m


def block_sparse(B: int = 8, T: int = 16384, H: int = 16, D: int = 128, density: float = 0.5, causal: bool = True,
                 salt: int = 0) -> Workload:
    """Block-mask sparse attention (64 x 64 tiles, multi-head K/V): bf16 Q/K/V N(0,1)
    [B*T, H, D] and the mask in Workload.idx."""
    rng = rng_for(6, salt)
    q = normal(rng, (B * T, H, D), "bf16")
    k = normal(rng, (B * T, H, D), "bf16")
    v = normal(rng, (B * T, H, D), "bf16")
    m = block_mask(rng, B, H, T, density, causal)
    return Workload("block_sparse", "bf16", dense_cu_seqlens(B, T), H, H, D, q, k, v, block_size=64, idx=m,
                    batch=B, seqlen=T)
