"""GPU parity of the int8 KV cache (the quantised cache "Meta Llama source
deep-dive", 8.4 lists; the scheme is the library's reading, oracle
kv_quantize_int8): RoPE + quantised append, then decode against the codes
and scales, through the C ABI against the oracle.  Rotated Q/K, codes and
scales bit-exact; attention against the decode formula on code * scale
within the same tolerance as the fp16 path."""

import math

import numpy as np
import pytest
import torch

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from paged_kv_gqa_rope_gb300 import workloads as W
from tests.gpu_helpers import assert_attention_close, bits
from tests.test_gpu_decode import custom_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    assert pa.check_device() == pa.PA_OK
    return libpa


def quantize_cache(init16, chunk=2048):
    """The int8 form of an fp16 pool (oracle quantisation, block by block)."""
    two, L, NB, bs, Hk, d = init16.shape
    codes, scales = orc.new_cache_i8(L, NB, bs, Hk, d)
    for b0 in range(0, NB, chunk):
        c, s = orc.kv_quantize_int8(init16[:, :, b0:b0 + chunk])
        codes[:, :, b0:b0 + chunk] = c
        scales[:, :, b0:b0 + chunk] = np.swapaxes(s, -1, -2)
    return codes, scales


class I8Run:
    def __init__(self, case, codes, scales):
        wl = case.wl
        self.case, self.wl = case, wl
        md = pa.prepare_decode(case.num_cached, case.block_tables)
        self.md = md
        self.table = pa.rope_table(int(md["positions"].max()) + 1, wl.head_dim, wl.rope_theta)
        self.cache = pa.CacheI8(1, case.num_blocks, wl.n_kv_heads, wl.head_dim)
        self.cache.codes.copy_(torch.from_numpy(codes))
        self.cache.scales.copy_(torch.from_numpy(scales))
        dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
        self.q, self.k, self.v = dev(case.q), dev(case.k), dev(case.v)
        self.pos, self.slots = dev(md["positions"]), dev(md["slot_mapping"])
        self.ctx, self.bt = dev(md["context_lens"]), dev(case.block_tables)
        self.ws = pa.decode_workspace(len(case.num_cached), wl.n_heads, wl.n_kv_heads,
                                      wl.head_dim)
        self.status = pa.new_status()

    def run(self):
        wl = self.wl
        pa.rope_kv_write_i8(self.q, self.k, self.v, self.pos, self.slots, self.table, self.cache,
                            status=self.status)
        out = pa.decode_i8(self.q, self.cache, self.bt, self.ctx, self.ws, wl.n_kv_heads,
                           status=self.status)
        torch.cuda.synchronize()
        return out


def oracle_step(case, codes, scales):
    wl = case.wl
    md = orc.decode_metadata(case.num_cached, case.block_tables, wl.block_size)
    q_rot = orc.rope_pinned(case.q, md["positions"], wl.head_dim, wl.rope_theta)
    k_rot = orc.rope_pinned(case.k, md["positions"], wl.head_dim, wl.rope_theta)
    codes, scales = codes.copy(), scales.copy()
    orc.kv_write_i8(codes, scales, 0, k_rot, case.v, md["slot_mapping"])
    out = orc.attention_decode_i8(q_rot, codes, scales, 0, case.block_tables, md["context_lens"],
                                  wl.n_heads, wl.n_kv_heads, 1.0 / math.sqrt(wl.head_dim))
    return q_rot, k_rot, codes, scales, out


def check(case, codes, scales):
    run = I8Run(case, codes, scales)
    out = run.run()
    q_rot, k_rot, c_want, s_want, want = oracle_step(case, codes, scales)
    assert int(run.status.item()) == 0
    assert np.array_equal(bits(run.q), bits(q_rot)), "rotated Q"
    assert np.array_equal(bits(run.k), bits(k_rot)), "rotated K"
    assert np.array_equal(run.cache.codes.cpu().numpy(), c_want), "codes"
    assert np.array_equal(run.cache.scales.cpu().numpy().view(np.uint32),
                          s_want.view(np.uint32)), "scales"
    return assert_attention_close(out, want)


@pytest.mark.parametrize("name", ["mha_decode_7b", "gqa_decode_70b"])
def test_int8_decode_workload_full_size(name):
    case = W.make_case(name)
    codes, scales = quantize_cache(W.initial_cache(case))
    max_abs, rel = check(case, codes, scales)
    print(f"{name} int8: max_abs={max_abs:.2e} rel_l2={rel:.2e}")


@pytest.mark.parametrize("H,Hk,d", [(8, 8, 128), (32, 8, 128), (64, 8, 128), (16, 8, 64),
                                    (8, 1, 64)])
def test_int8_decode_edge_lengths(H, Hk, d):
    ctxs = [0, 1, 14, 15, 16, 17, 254, 255, 256, 257, 511, 1000, 4100]
    case, init = custom_case(H, Hk, d, ctxs, seed=700 + H + Hk + d)
    codes, scales = quantize_cache(init)
    check(case, codes, scales)


@pytest.mark.parametrize("ctxs,Hk,ctas,g,d", [([5000], 1, 2, 8, 128), ([5000], 1, 4, 8, 128),
                                              ([5000], 1, 5, 8, 128), ([2000, 3000], 2, 3, 4, 64),
                                              ([4100, 100], 8, 3, 8, 128)])
def test_int8_narrow_grid_merges_pieces(ctxs, Hk, ctas, g, d):
    """The int8 kernel's merges (a pair cut into 2, 4 or 5 pieces by a
    workspace with record slots for only a few CTAs) give the same result as
    the decode formula on code * scale."""
    H = g * Hk
    case, init = custom_case(H, Hk, d, ctxs, seed=900 + sum(ctxs) + ctas)
    codes, scales = quantize_cache(init)
    run = I8Run(case, codes, scales)
    slot_bytes = 2 * 8 * (d + 4) * 4
    counters = (len(ctxs) * Hk * 4 + 255) // 256 * 256
    run.ws = pa.decode_workspace(len(ctxs), H, Hk, d, nbytes=counters + ctas * slot_bytes)
    out = run.run()
    *_, want = oracle_step(case, codes, scales)
    assert int(run.status.item()) == 0
    assert_attention_close(out, want)


def test_int8_ignores_garbage_in_unwritten_slots():
    """Codes and scales past a sequence's context may hold anything (NaN
    scales included): the output must not see them."""
    case, init = custom_case(16, 4, 128, [20, 300, 4, 47], seed=71)
    codes, scales = quantize_cache(init)
    rng = np.random.default_rng(72)
    poisoned_c, poisoned_s = codes.copy(), scales.copy()
    for s, c in enumerate(case.num_cached):
        n = int(c) + 1
        blk = case.block_tables[s][(n - 1) // 16]
        r0 = n % 16 if n % 16 else 16
        poisoned_c[:, 0, blk, r0:] = rng.integers(-127, 128, size=poisoned_c[:, 0, blk, r0:].shape)
        poisoned_s[:, 0, blk, :, r0:] = np.float32(np.nan)
    run = I8Run(case, poisoned_c, poisoned_s)
    out = run.run()
    *_, want = oracle_step(case, codes, scales)
    assert_attention_close(out, want)


def test_int8_zero_rows_and_bad_block():
    """An all-zero K/V row stores scale 0 and zero codes; a block id past the
    pool is reported and not read."""
    case, init = custom_case(8, 2, 64, [40, 3], seed=73)
    case.k[0] = 0
    case.v[1] = 0
    codes, scales = quantize_cache(init)
    check(case, codes, scales)
    run = I8Run(case, codes, scales)
    run.bt[1, 0] = case.num_blocks + 5
    run.run()
    assert int(run.status.item()) & pa.PA_DEV_BAD_BLOCK


def test_int8_bytes_are_about_half():
    assert pa.lib().pa_cache_i8_bytes(1, 100, 16, 8, 128) < 0.52 * pa.cache_bytes(1, 100, 16, 8, 128)
