"""Seeded synthetic inputs for the paged attention hot path.

This module only draws random numbers and lays them out: per-sequence
lengths, the assignment of physical KV blocks to sequences (block tables),
the contents of the KV-cache pool that stands for already-cached history, and
the new tokens' Q/K/V.  It contains none of the method's arithmetic (no RoPE,
no slot computation, no attention), so both the CUDA path and the CPU oracle
can consume its output without sharing any code with each other.

The five workloads follow the shapes of the Llama-2-style engine described on
the pages "Meta Llama source deep-dive" (ModelArgs / KV-cache sizing sections)
and "nano-vllm notes - Llama" (allocate_kv_cache, prepare_prefill,
prepare_decode):

  tiny           4 Q heads / 2 KV heads, d=64, prompts of 3, 5 and 2 tokens,
                 then 4 single-token decode steps per sequence, 16-block pool
  mha_decode_7b  32/32 heads, d=128, batch 32, 2048 cached tokens each
  gqa_decode_70b 64/8 heads, d=128, batch 32, 4096 cached tokens each
  prefill_13b    40/40 heads, d=128, 16 sequences, cached prefix 16*U{0..64},
                 new tokens U{128..2048}
  ragged_decode  32/8 heads, d=128, 256 sequences, cached lengths
                 log-uniform in [16, 32768], K/V ~ N(0, 0.5) with 1% outliers
                 ~ N(0, 8), pool sized to need + 10% in random order

Normal distributions N(mu, s) take s as the standard deviation.  Seeds are
20260 + workload index (1..5).
"""

from __future__ import annotations

import math
import os
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
ROPE_THETA = 10000.0


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    n_heads: int
    n_kv_heads: int
    head_dim: int
    batch: int
    kind: str  # "decode", "prefill" or "prefill+decode"
    block_size: int = BLOCK_SIZE
    rope_theta: float = ROPE_THETA
    kv_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_std: float = 0.0
    decode_steps: int = 1

    @property
    def seed(self) -> int:
        return 20260 + self.index

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads


WORKLOADS = {
    "tiny": Workload(1, "tiny", 4, 2, 64, 3, "prefill+decode", decode_steps=4),
    "mha_decode_7b": Workload(2, "mha_decode_7b", 32, 32, 128, 32, "decode"),
    "gqa_decode_70b": Workload(3, "gqa_decode_70b", 64, 8, 128, 32, "decode"),
    "prefill_13b": Workload(4, "prefill_13b", 40, 40, 128, 16, "prefill"),
    "ragged_decode": Workload(5, "ragged_decode", 32, 8, 128, 256, "decode",
                              kv_std=0.5, outlier_frac=0.01, outlier_std=8.0),
}


@dataclass
class Case:
    """One batch of synthetic input.

    num_cached[s]   tokens of sequence s already in the cache before this call
    num_new[s]      new tokens of sequence s in this call (1 for decode)
    block_tables    [B, max_blocks] int32, physical block of each logical
                    block, -1 where a sequence has no block
    num_blocks      physical blocks in the pool
    q, k, v         new tokens, flattened in sequence order:
                    [T, H, d], [T, Hk, d], [T, Hk, d] float16
    """

    wl: Workload
    num_cached: np.ndarray
    num_new: np.ndarray
    block_tables: np.ndarray
    num_blocks: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    extra_steps: list = field(default_factory=list)  # later decode steps (tiny)

    @property
    def total_new(self) -> int:
        return int(self.num_new.sum())


def _normal16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x.astype(np.float16)


def _assign_blocks(rng, blocks_needed, pool_blocks):
    """Hand out physical blocks of a pool of `pool_blocks` in seeded random
    order; sequence s receives the next blocks_needed[s] of them."""
    order = rng.permutation(pool_blocks).astype(np.int32)
    max_blocks = int(max(blocks_needed)) if len(blocks_needed) else 0
    table = np.full((len(blocks_needed), max(max_blocks, 1)), -1, dtype=np.int32)
    at = 0
    for s, nb in enumerate(blocks_needed):
        table[s, :nb] = order[at:at + nb]
        at += nb
    return table


def _ceil_div(a, b):
    return -(-a // b)


def make_case(name: str, *, batch: int | None = None, max_context: int | None = None) -> Case:
    """Draw the lengths, block tables and new tokens of workload `name`.

    `batch` / `max_context` shrink a workload for quick tests (same recipe,
    fewer sequences or shorter histories); the defaults give the full size.
    """
    wl = WORKLOADS[name]
    rng = np.random.default_rng(wl.seed)
    B = wl.batch if batch is None else batch
    bs = wl.block_size
    extra = []

    if wl.name == "tiny":
        num_cached = np.zeros(3, np.int64)
        num_new = np.array([3, 5, 2], np.int64)[:B]
        num_cached = num_cached[:B]
        final = num_new + wl.decode_steps
        need = [_ceil_div(int(n), bs) for n in final]
        table = _assign_blocks(rng, need, 16)
        pool = 16
    elif wl.kind == "decode":
        if wl.name == "ragged_decode":
            lo, hi = math.log(16.0), math.log(32768.0)
            c = np.rint(np.exp(rng.uniform(lo, hi, size=wl.batch))).astype(np.int64)
            c = c[:B]
        else:
            c = np.full(B, 2048 if wl.name == "mha_decode_7b" else 4096, np.int64)
        if max_context is not None:
            c = np.minimum(c, max_context - 1)
        num_cached = c
        num_new = np.ones(B, np.int64)
        need = [_ceil_div(int(x) + 1, bs) for x in c]
        if wl.name == "ragged_decode":
            pool = int(math.ceil(1.1 * sum(need)))
        else:
            pool = int(sum(need))
        table = _assign_blocks(rng, need, pool)
    else:  # prefill_13b
        p = bs * rng.integers(0, 65, size=wl.batch).astype(np.int64)
        L = rng.integers(128, 2049, size=wl.batch).astype(np.int64)
        p, L = p[:B], L[:B]
        if max_context is not None:
            L = np.minimum(L, np.maximum(max_context - p, 1))
        num_cached, num_new = p, L
        need = [_ceil_div(int(a + b), bs) for a, b in zip(p, L)]
        pool = int(sum(need))
        table = _assign_blocks(rng, need, pool)

    T = int(num_new.sum())
    H, Hk, d = wl.n_heads, wl.n_kv_heads, wl.head_dim
    q = _normal16(rng, (T, H, d))
    k = _normal16(rng, (T, Hk, d))
    v = _normal16(rng, (T, Hk, d))
    if wl.name == "tiny":
        for _ in range(wl.decode_steps):
            extra.append((_normal16(rng, (B, H, d)), _normal16(rng, (B, Hk, d)),
                          _normal16(rng, (B, Hk, d))))
    return Case(wl, num_cached, num_new, table, pool, q, k, v, extra)


def block_contents(wl: Workload, block: int) -> np.ndarray:
    """Synthetic history held in physical block `block` of the pool:
    float16 [2 (K,V), block_size, Hk, d].  Drawn from its own counter-based
    stream (seed, block), so any subset of blocks can be regenerated."""
    rng = np.random.default_rng([wl.seed, 7, int(block)])
    shape = (2, wl.block_size, wl.n_kv_heads, wl.head_dim)
    x = rng.standard_normal(shape, dtype=np.float32)
    if wl.kv_std != 1.0:
        x *= np.float32(wl.kv_std)
    if wl.outlier_frac > 0.0:
        # outliers: a binomial count of entries (indices drawn with
        # replacement) replaced by N(0, outlier_std)
        flat = x.reshape(-1)
        n_out = int(rng.binomial(flat.size, wl.outlier_frac))
        idx = rng.integers(0, flat.size, size=n_out)
        flat[idx] = rng.standard_normal(n_out, dtype=np.float32) * np.float32(wl.outlier_std)
    return x.astype(np.float16)


def initial_cache(case: Case, blocks=None) -> np.ndarray:
    """The pool before this call: float16 [2, 1, NB, bs, Hk, d] (one layer).
    Every block holds its synthetic history; `blocks` restricts the fill to a
    subset (the rest stay zero), which is enough for sampled checks."""
    wl = case.wl
    cache = np.zeros((2, 1, case.num_blocks, wl.block_size, wl.n_kv_heads, wl.head_dim),
                     np.float16)
    todo = list(range(case.num_blocks)) if blocks is None else sorted(set(int(b) for b in blocks))

    def fill(lo_hi):
        for b in todo[lo_hi[0]:lo_hi[1]]:
            cache[:, 0, b] = block_contents(wl, b)

    step = 512
    spans = [(i, min(i + step, len(todo))) for i in range(0, len(todo), step)]
    if len(spans) > 1:
        import concurrent.futures as cf
        with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, spans))
    else:
        for sp in spans:
            fill(sp)
    return cache
