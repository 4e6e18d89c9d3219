"""GPU parity of steps a1 (RoPE), a2 (paged K/V write) and a4 (decode)
through the C ABI against the oracle, on the seeded workloads at full size
and on small edge cases.  Cache writes and rotated Q/K must be bit-exact;
attention within max-abs 3e-3 and relative L2 1e-3."""

import math

import numpy as np
import pytest
import torch

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from paged_kv_gqa_rope_gb300 import workloads as W
from tests.gpu_helpers import DecodeRun, assert_attention_close, bits, oracle_decode_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    assert pa.check_device() == pa.PA_OK
    return libpa


def custom_case(H, Hk, d, ctxs, seed, kv_std=1.0, extra_blocks=3):
    """A decode case with the given cached lengths (+1 new token each)."""
    wl = W.Workload(90 + seed % 9, f"custom{seed}", H, Hk, d, len(ctxs), "decode", kv_std=kv_std)
    rng = np.random.default_rng(seed)
    need = [-(-(c + 1) // 16) for c in ctxs]
    pool = sum(need) + extra_blocks
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((len(ctxs), max(need)), -1, np.int32)
    at = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[at:at + nb]
        at += nb
    B = len(ctxs)
    q = rng.standard_normal((B, H, d), dtype=np.float32).astype(np.float16)
    k = rng.standard_normal((B, Hk, d), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((B, Hk, d), dtype=np.float32).astype(np.float16)
    case = W.Case(wl, np.asarray(ctxs, np.int64), np.ones(B, np.int64), table, pool, q, k, v)
    init = (rng.standard_normal((2, 1, pool, 16, Hk, d), dtype=np.float32) * kv_std).astype(np.float16)
    return case, init


def check_step(case, init, seqs=None):
    run = DecodeRun(case, init)
    out = run.run()
    q_rot, k_rot, cache, want = oracle_decode_step(case, init, seqs=seqs)
    assert int(run.status.item()) == 0
    assert np.array_equal(bits(run.q), bits(q_rot)), "rotated Q differs"
    assert np.array_equal(bits(run.k), bits(k_rot)), "rotated K differs"
    assert torch.equal(run.cache.tensor, torch.from_numpy(cache).cuda()), "cache differs"
    rows = list(range(len(case.num_cached))) if seqs is None else list(seqs)
    return assert_attention_close(out, want, rows=rows), run, out, want


@pytest.mark.parametrize("name", ["mha_decode_7b", "gqa_decode_70b", "ragged_decode"])
def test_decode_workload_full_size(name):
    case = W.make_case(name)
    init = W.initial_cache(case)
    (max_abs, rel), *_ = check_step(case, init)
    print(f"{name}: max_abs={max_abs:.2e} rel_l2={rel:.2e}")


@pytest.mark.parametrize("H,Hk,d", [(8, 8, 128), (16, 8, 64), (32, 8, 128), (64, 8, 128),
                                    (4, 2, 64), (8, 1, 64)])
def test_decode_edge_lengths(H, Hk, d):
    ctxs = [0, 1, 14, 15, 16, 17, 254, 255, 256, 257, 511, 512, 1000, 4100]
    case, init = custom_case(H, Hk, d, ctxs, seed=H * 131 + Hk * 7 + d)
    check_step(case, init)


def test_decode_single_sequence_long():
    case, init = custom_case(32, 8, 128, [32767], seed=5)
    check_step(case, init)


def test_decode_is_repeatable_and_resets_counters():
    case, init = custom_case(16, 4, 128, [300, 5, 1025, 64], seed=6)
    run = DecodeRun(case, init)
    out1 = run.run().clone()
    out2 = pa.decode(run.q, run.cache, run.bt, run.ctx, run.ws, case.wl.n_kv_heads)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    ncnt = len(case.num_cached) * case.wl.n_kv_heads
    assert int(run.ws[:4 * ncnt].view(torch.int32).abs().sum().item()) == 0
    # a workspace smaller than one CTA's records is refused on the host
    with pytest.raises(pa.PAError):
        pa.decode(run.q, run.cache, run.bt, run.ctx, run.ws[:256], case.wl.n_kv_heads)


def test_decode_constant_v_returns_v():
    case, init = custom_case(16, 2, 128, [700, 33], seed=7)
    init[1] = np.float16(-0.8125)
    case.v[:] = np.float16(-0.8125)
    run = DecodeRun(case, init)
    out = run.run()
    assert float((out.float() + 0.8125).abs().max()) < 1e-3


def test_decode_ignores_nan_in_unwritten_slots():
    """Slots past a sequence's context (the tail of its last block) may hold
    any bits; NaN there must not reach the output."""
    case, init = custom_case(16, 2, 128, [20, 300, 4], seed=12)
    md = orc.decode_metadata(case.num_cached, case.block_tables, 16)
    poisoned = init.copy()
    for s, c in enumerate(case.num_cached):
        n = int(c) + 1
        blk = case.block_tables[s][(n - 1) // 16]
        poisoned[:, 0, blk, n % 16 if n % 16 else 16:] = np.float16(np.nan)
    run = DecodeRun(case, poisoned)
    out = run.run()
    _, _, _, want = oracle_decode_step(case, init)
    assert_attention_close(out, want)


def test_decode_bad_block_is_reported_not_read():
    case, init = custom_case(8, 2, 64, [40, 300], seed=8)
    run = DecodeRun(case, init)
    run.run()
    run.status.zero_()
    bad = run.bt.clone()
    bad[0, 1] = case.num_blocks + 5
    out = pa.decode(run.q, run.cache, bad, run.ctx, run.ws, 2, status=run.status)
    torch.cuda.synchronize()
    assert int(run.status.item()) & pa.PA_DEV_BAD_BLOCK
    # the other sequence is unaffected
    _, _, _, want = oracle_decode_step(case, init)
    assert_attention_close(out, want, rows=[1])


def test_decode_bad_context_is_reported():
    case, init = custom_case(8, 2, 64, [40, 300], seed=9)
    run = DecodeRun(case, init)
    run.run()
    run.status.zero_()
    ctx = run.ctx.clone()
    ctx[0] = 0
    ctx[1] = run.bt.shape[1] * 16 + 1
    pa.decode(run.q, run.cache, run.bt, ctx, run.ws, 2, status=run.status)
    torch.cuda.synchronize()
    assert int(run.status.item()) & pa.PA_DEV_BAD_LENGTH


@pytest.mark.parametrize("ctxs,Hk,ctas,g,d", [
    ([2000, 3000], 2, 3, 4, 64), ([5000], 1, 5, 4, 64), ([3, 7000, 40, 900, 16], 2, 7, 4, 64),
    ([300, 20], 2, 1, 4, 64), ([1], 1, 2, 4, 64),
    # head_dim 128, full groups: 2, 4 (the merge of up to four pieces, their
    # records' loads in one pass at fp16) and 5 pieces (element by element)
    ([3000], 1, 2, 8, 128), ([5000], 1, 4, 8, 128), ([5000], 1, 5, 8, 128),
    ([4100, 100], 8, 3, 8, 128)])
def test_decode_narrow_grid_merges_pieces(ctxs, Hk, ctas, g, d):
    """A workspace with record slots for only a few CTAs narrows the grid, so
    one (sequence, KV head) pair is cut into pieces across several CTAs and
    merged; results must not change."""
    H = g * Hk
    case, init = custom_case(H, Hk, d, ctxs, seed=sum(ctxs) + ctas)
    run = DecodeRun(case, init)
    full = pa.decode_workspace_bytes(len(ctxs), H, Hk, d)
    slot_bytes = 2 * 8 * (d + 4) * 4
    counters = (len(ctxs) * Hk * 4 + 255) // 256 * 256
    assert full == counters + 608 * slot_bytes  # record slots for 4 CTAs per SM
    run.ws = pa.decode_workspace(len(ctxs), H, Hk, d, nbytes=counters + ctas * slot_bytes)
    out = run.run()
    _, _, _, want = oracle_decode_step(case, init)
    assert int(run.status.item()) == 0
    assert_attention_close(out, want)
    out2 = pa.decode(run.q, run.cache, run.bt, run.ctx, run.ws, Hk)   # counters were reset
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_rope_kv_write_prefill_workload_bit_exact():
    """RoPE + append of the 13B prefill workload's ~17k new tokens."""
    case = W.make_case("prefill_13b")
    wl = case.wl
    md = pa.prepare_prefill(case.num_cached, case.num_new, case.block_tables)
    table = pa.rope_table(int(md["max_seqlen_k"]), wl.head_dim)
    cache = pa.Cache(1, case.num_blocks, wl.n_kv_heads, wl.head_dim)
    cache.tensor.zero_()
    q, k, v = (torch.from_numpy(x).cuda() for x in (case.q, case.k, case.v))
    st = pa.new_status()
    pa.rope_kv_write(q, k, v, torch.from_numpy(md["positions"]).cuda(),
                     torch.from_numpy(md["slot_mapping"]).cuda(), table, cache, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    omd = orc.prefill_metadata(case.num_cached, case.num_new, case.block_tables, 16)
    q_rot = orc.rope_pinned(case.q, omd["positions"], wl.head_dim)
    k_rot = orc.rope_pinned(case.k, omd["positions"], wl.head_dim)
    assert np.array_equal(bits(q), bits(q_rot))
    assert np.array_equal(bits(k), bits(k_rot))
    want = orc.new_cache(1, case.num_blocks, 16, wl.n_kv_heads, wl.head_dim)
    orc.kv_write(want, 0, k_rot, case.v, omd["slot_mapping"])
    assert torch.equal(cache.tensor, torch.from_numpy(want).cuda())


def test_rope_table_matches_oracle_entries():
    t = pa.rope_table(32769, 128).cpu().numpy()
    for m in (0, 1, 2, 1000, 4096, 32768):
        c, s = orc.rope_cos_sin(m, 128)
        assert np.array_equal(t[m, :, 0], c) and np.array_equal(t[m, :, 1], s)
    t = pa.rope_table(10, 64, theta=1e6).cpu().numpy()
    c, s = orc.rope_cos_sin(9, 64, theta=1e6)
    assert np.array_equal(t[9, :, 0], c) and np.array_equal(t[9, :, 1], s)


def test_rope_bad_position_and_slot():
    H, Hk, d = 4, 2, 64
    cache = pa.Cache(1, 4, Hk, d)
    cache.tensor.fill_(1.0)
    table = pa.rope_table(64, d)
    rng = np.random.default_rng(11)
    q = torch.from_numpy(rng.standard_normal((4, H, d)).astype(np.float16)).cuda()
    k = torch.from_numpy(rng.standard_normal((4, Hk, d)).astype(np.float16)).cuda()
    v = torch.from_numpy(rng.standard_normal((4, Hk, d)).astype(np.float16)).cuda()
    q0, k0 = q.clone(), k.clone()
    pos = torch.tensor([3, 64, -1, 5], dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 1, 2, 4 * 16], dtype=torch.int32, device="cuda")
    st = pa.new_status()
    pa.rope_kv_write(q, k, v, pos, slots, table, cache, status=st)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & pa.PA_DEV_BAD_POSITION and s & pa.PA_DEV_BAD_SLOT
    # tokens 1, 2 (bad positions) untouched; token 3 rotated but not written
    assert torch.equal(q[1:3], q0[1:3]) and torch.equal(k[1:3], k0[1:3])
    assert not torch.equal(q[3], q0[3])
    flat = cache.tensor.view(2, -1, Hk, d)
    assert torch.equal(flat[0, 0], k[0]) and torch.equal(flat[1, 0], v[0])
    assert bool((flat[:, 1:] == 1.0).all())
    # a negative slot is a padding token: rotated, not written, no error
    st.zero_()
    pa.rope_kv_write(q[:1].clone(), k[:1].clone(), v[:1], pos[:1],
                     torch.tensor([-1], dtype=torch.int32, device="cuda"), table, cache, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_binding_rejects_mismatched_buffers_before_launch():
    """Buffers whose sizes disagree with q are refused on the host (the
    kernels would index past them): nothing is launched."""
    case, init = custom_case(4, 2, 64, [5, 40], seed=12)
    run = DecodeRun(case, init)
    T, Hk, d = run.k.shape
    with pytest.raises(ValueError):
        pa.rope_kv_write(run.q, run.k, run.v[:T - 1].contiguous(), run.positions, run.slots,
                         run.table, run.cache)
    with pytest.raises(ValueError):
        pa.rope_kv_write(run.q, run.k, run.v, run.positions[:T - 1], run.slots, run.table,
                         run.cache)
    with pytest.raises(ValueError):
        pa.decode(run.q, run.cache, run.bt, run.ctx[:1], run.ws, Hk)
    with pytest.raises(ValueError):
        pa.decode(run.q, run.cache, run.bt, run.ctx, run.ws, Hk,
                  out=torch.empty(1, 1, d, dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        pa.decode(run.q, run.cache, run.bt, run.ctx, run.ws, Hk,
                  status=torch.zeros(2, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    out = run.run()  # the same buffers, well formed, still go through
    assert_attention_close(out, oracle_decode_step(case, init)[3])
