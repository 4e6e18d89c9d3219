"""GPU parity of step a3 (varlen causal prefill over the paged cache, with a
cached prefix read through block_tables) through the C ABI against the
oracle, on the seeded workloads and on edge cases: prefixes that are not a
multiple of the block size, query lengths around the 128-row tile, GQA
groups, head_dim 64 and 128, NaN bits in unwritten slots."""

import math

import numpy as np
import pytest
import torch

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from paged_kv_gqa_rope_gb300 import workloads as W
from tests.gpu_helpers import assert_attention_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    assert pa.check_device() == pa.PA_OK
    return libpa


def custom_prefill_case(H, Hk, d, cached, new, seed, extra_blocks=3):
    wl = W.Workload(80 + seed % 9, f"pcustom{seed}", H, Hk, d, len(new), "prefill")
    rng = np.random.default_rng(seed)
    need = [-(-(c + n) // 16) for c, n in zip(cached, new)]
    pool = sum(need) + extra_blocks
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((len(new), max(need)), -1, np.int32)
    at = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[at:at + nb]
        at += nb
    T = sum(new)
    q = rng.standard_normal((T, H, d), dtype=np.float32).astype(np.float16)
    k = rng.standard_normal((T, Hk, d), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((T, Hk, d), dtype=np.float32).astype(np.float16)
    case = W.Case(wl, np.asarray(cached, np.int64), np.asarray(new, np.int64), table, pool, q, k, v)
    init = rng.standard_normal((2, 1, pool, 16, Hk, d), dtype=np.float32).astype(np.float16)
    return case, init


class PrefillRun:
    def __init__(self, case, init):
        wl = case.wl
        self.case = case
        md = pa.prepare_prefill(case.num_cached, case.num_new, case.block_tables)
        self.md = md
        self.table = pa.rope_table(max(int(md["max_seqlen_k"]), 1), wl.head_dim, wl.rope_theta)
        self.cache = pa.Cache(1, case.num_blocks, wl.n_kv_heads, wl.head_dim)
        self.cache.tensor.copy_(torch.from_numpy(init))
        self.q, self.k, self.v = (torch.from_numpy(x).cuda() for x in (case.q, case.k, case.v))
        self.pos = torch.from_numpy(md["positions"]).cuda()
        self.slots = torch.from_numpy(md["slot_mapping"]).cuda()
        self.cuq = torch.from_numpy(md["cu_seqlens_q"]).cuda()
        self.cuk = torch.from_numpy(md["cu_seqlens_k"]).cuda()
        self.bt = torch.from_numpy(case.block_tables).cuda()
        self.status = pa.new_status()

    def run(self):
        wl = self.case.wl
        pa.rope_kv_write(self.q, self.k, self.v, self.pos, self.slots, self.table, self.cache,
                         status=self.status)
        out = pa.prefill_varlen(self.q, self.cache, self.cuq, self.cuk, self.bt,
                                self.md["max_seqlen_q"], wl.n_kv_heads, status=self.status)
        torch.cuda.synchronize()
        return out


def oracle_prefill(case, init, seqs=None):
    wl = case.wl
    md = orc.prefill_metadata(case.num_cached, case.num_new, case.block_tables, 16)
    q_rot = orc.rope_pinned(case.q, md["positions"], wl.head_dim, wl.rope_theta)
    k_rot = orc.rope_pinned(case.k, md["positions"], wl.head_dim, wl.rope_theta)
    cache = init.copy()
    orc.kv_write(cache, 0, k_rot, case.v, md["slot_mapping"])
    out = orc.attention_prefill(q_rot, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"],
                                case.block_tables, wl.n_heads, wl.n_kv_heads,
                                1.0 / math.sqrt(wl.head_dim), seqs=seqs)
    return q_rot, cache, out, md


def check(case, init, seqs=None):
    run = PrefillRun(case, init)
    out = run.run()
    q_rot, cache, want, md = oracle_prefill(case, init, seqs=seqs)
    assert int(run.status.item()) == 0, f"device status {int(run.status.item())}"
    assert np.array_equal(bits(run.q), bits(q_rot))
    assert torch.equal(run.cache.tensor, torch.from_numpy(cache).cuda())
    if seqs is None:
        rows = np.arange(out.shape[0])
    else:
        cq = md["cu_seqlens_q"]
        rows = np.concatenate([np.arange(cq[s], cq[s + 1]) for s in seqs])
    return assert_attention_close(out, want, rows=rows), run, out, want


def test_tiny_workload_prefill():
    case = W.make_case("tiny")
    init = W.initial_cache(case)
    check(case, init)


@pytest.mark.parametrize("H,Hk,d", [(4, 4, 128), (8, 2, 128), (4, 1, 64), (6, 3, 64)])
def test_prefill_edge_lengths(H, Hk, d):
    cached = [0, 0, 5, 16, 37, 128, 300, 0, 1000]
    new = [1, 2, 127, 128, 129, 300, 17, 513, 64]
    case, init = custom_prefill_case(H, Hk, d, cached, new, seed=H * 17 + Hk + d)
    check(case, init)


def test_prefill_gqa_group_of_8():
    case, init = custom_prefill_case(32, 4, 128, [64, 0, 200], [700, 257, 90], seed=3)
    check(case, init)


def test_prefill_13b_workload_full_size():
    case = W.make_case("prefill_13b")
    init = W.initial_cache(case)
    (max_abs, rel), *_ = check(case, init)
    print(f"prefill_13b: max_abs={max_abs:.2e} rel_l2={rel:.2e}")


def test_prefill_ignores_nan_in_unwritten_slots():
    case, init = custom_prefill_case(4, 2, 128, [0, 3, 20], [13, 30, 7], seed=4)
    poisoned = init.copy()
    for s in range(3):
        n = int(case.num_cached[s] + case.num_new[s])
        blk = case.block_tables[s][(n - 1) // 16]
        if n % 16:
            poisoned[:, 0, blk, n % 16:] = np.float16(np.nan)
    run = PrefillRun(case, poisoned)
    out = run.run()
    _, _, want, _ = oracle_prefill(case, init)
    assert_attention_close(out, want)


def test_prefill_constant_v_returns_v():
    case, init = custom_prefill_case(8, 4, 128, [40, 0], [200, 129], seed=5)
    init[1] = np.float16(0.3125)
    case.v[:] = np.float16(0.3125)
    out = PrefillRun(case, init).run()
    assert float((out.float() - 0.3125).abs().max()) < 1e-3


def test_decode_matches_last_prefill_row_on_gpu():
    """A decode step equals the last row of a causal prefill of the same
    sequence ("personal chatgpt 22", sections 2-3), on the GPU path."""
    case, init = custom_prefill_case(16, 4, 128, [100, 0], [333, 70], seed=6)
    run = PrefillRun(case, init)
    out = run.run()
    cq = run.md["cu_seqlens_q"]
    last = torch.tensor([cq[1] - 1, cq[2] - 1], device="cuda")
    ctx = torch.tensor([433, 70], dtype=torch.int32, device="cuda")
    ws = pa.decode_workspace(2, 16, 4, 128)
    dec = pa.decode(run.q[last].contiguous(), run.cache, run.bt, ctx, ws, 4)
    torch.cuda.synchronize()
    assert float((dec.float() - out[last].float()).abs().max()) < 2e-3


def test_prefill_bad_lengths_are_reported():
    case, init = custom_prefill_case(4, 2, 64, [0, 10], [20, 20], seed=7)
    run = PrefillRun(case, init)
    run.run()
    run.status.zero_()
    bad = run.cuk.clone()
    bad[2] = bad[1] + 5          # seqlen_k < seqlen_q for sequence 1
    pa.prefill_varlen(run.q, run.cache, run.cuq, bad, run.bt, 20, 2, status=run.status)
    torch.cuda.synchronize()
    assert int(run.status.item()) & pa.PA_DEV_BAD_LENGTH


def test_prefill_many_sequences():
    """300 sequences: a 300-row sequence table in shared memory and many
    short units handed out by the work counter."""
    rng = np.random.default_rng(41)
    B = 300
    cached = rng.integers(0, 60, size=B).tolist()
    new = rng.integers(1, 40, size=B).tolist()
    case, init = custom_prefill_case(4, 2, 128, cached, new, seed=42)
    check(case, init)


def test_prefill_more_sequences_than_threads():
    """Past 512 sequences the kernel keeps the batch order instead of ranking
    the sequences by cost in its prologue (one sequence per thread)."""
    rng = np.random.default_rng(43)
    B = 700
    cached = rng.integers(0, 40, size=B).tolist()
    new = rng.integers(1, 24, size=B).tolist()
    case, init = custom_prefill_case(4, 2, 64, cached, new, seed=44)
    check(case, init)


def test_prefill_rising_maximum_rescales():
    """Keys whose norm grows with their position make later key tiles, and the
    second half of a tile, raise a row's running maximum past the rescale
    threshold, so the paths that rescale P (already written for a tile's
    first half) and O run on most tiles instead of almost never."""
    H, Hk, d = 8, 2, 128
    cached, new = [0, 48], [700, 300]
    case, init = custom_prefill_case(H, Hk, d, cached, new, seed=91)
    grow = lambda p: 1.0 + np.asarray(p, np.float32) / 16.0  # noqa: E731
    at = 0
    for s, (c, n) in enumerate(zip(cached, new)):
        pos = c + np.arange(n)
        case.k[at:at + n] = (case.k[at:at + n].astype(np.float32)
                             * grow(pos)[:, None, None]).astype(np.float16)
        at += n
        for p in range(c):  # the cached prefix, through the block table
            blk, row = case.block_tables[s][p // 16], p % 16
            init[0, 0, blk, row] = (init[0, 0, blk, row].astype(np.float32) * grow(p)).astype(np.float16)
    check(case, init)


@pytest.mark.parametrize("shape", ["prefill_13b", "skips"])
def test_prefill_repeats_bit_for_bit(shape):
    """The same launch thirty times gives the same bits.  The two query
    tiles of a unit share K/V stages; a tile skips the key tiles only the
    other one reads (the last key tile of a pair, every key tile of a first
    pair whose second tile is empty), and a stage it skipped must have been
    seen to land before it waits for the stage's next load.  "skips" makes
    such pairs common: query lengths that leave L_q mod 256 in 1..128, with
    prefixes of one to three key tiles."""
    if shape == "prefill_13b":
        case = W.make_case("prefill_13b")
        init = W.initial_cache(case)
    else:
        rng = np.random.default_rng(61)
        B = 24
        new = (256 * rng.integers(0, 4, size=B) + rng.integers(1, 129, size=B)).tolist()
        cached = (16 * rng.integers(8, 24, size=B)).tolist()
        case, init = custom_prefill_case(16, 4, 128, cached, new, seed=62)
    run = PrefillRun(case, init)
    first = run.run().clone()
    assert int(run.status.item()) == 0
    wl = case.wl
    for i in range(30):
        out = pa.prefill_varlen(run.q, run.cache, run.cuq, run.cuk, run.bt,
                                run.md["max_seqlen_q"], wl.n_kv_heads, status=run.status)
        torch.cuda.synchronize()
        assert torch.equal(out, first), f"launch {i + 1} differs from the first"
    assert int(run.status.item()) == 0
    if shape == "skips":
        _, _, want, _ = oracle_prefill(case, init)
        assert_attention_close(first, want)


def test_prefill_step_equals_separate_calls():
    """pa_prefill_step (RoPE/append and the prefill chained in one call) gives
    the bits of the two calls made one after the other, and the oracle's
    attention within the tolerance."""
    case, init = custom_prefill_case(16, 4, 128, [0, 37, 300], [513, 129, 1], seed=63)
    sep = PrefillRun(case, init)
    want = sep.run()
    one = PrefillRun(case, init)
    got = pa.prefill_step(one.q, one.k, one.v, one.pos, one.slots, one.table, one.cache, one.cuq,
                          one.cuk, one.bt, one.md["max_seqlen_q"], case.wl.n_kv_heads,
                          status=one.status)
    torch.cuda.synchronize()
    assert int(one.status.item()) == 0
    assert torch.equal(got, want)
    assert torch.equal(one.cache.tensor, sep.cache.tensor)
    assert torch.equal(one.q, sep.q)
    _, _, want64, _ = oracle_prefill(case, init)
    assert_attention_close(got, want64)
