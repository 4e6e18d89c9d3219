"""RoPE + append (steps a1, a2) of many tokens.  The int8 RoPE/append kernel
runs one row of CTAs per token (blockIdx.y, and blockIdx.z past 65535
tokens), so 70000 tokens exercise the third grid dimension; the fp16 one
takes batches of at least eight tokens per SM in its staged kernel (each
CTA walks many tokens, bringing each token's rows into shared memory with
bulk copies), which the same 70000 tokens and a 2000-token batch with bad
positions and slots exercise.  Rotated Q/K, the fp16 cache and the int8
codes and scales are compared with the oracle bit for bit."""

import math

import numpy as np
import pytest
import torch

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from tests.gpu_helpers import bits

pytestmark = pytest.mark.gpu

T, H, HK, D, BS = 70000, 1, 1, 64, 16


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    return libpa


def _inputs(seed):
    rng = np.random.default_rng(seed)
    mk = lambda *s: rng.standard_normal(s, dtype=np.float32).astype(np.float16)  # noqa: E731
    q, k, v = mk(T, H, D), mk(T, HK, D), mk(T, HK, D)
    positions = rng.integers(0, 4096, size=T).astype(np.int32)
    nb = math.ceil(T / BS) + 8
    slots = rng.permutation(nb * BS)[:T].astype(np.int32)
    return q, k, v, positions, slots, nb


def test_rope_kv_write_past_65535_tokens():
    q, k, v, positions, slots, nb = _inputs(81)
    dq, dk, dv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    cache = pa.Cache(1, nb, HK, D)
    cache.tensor.zero_()
    table = pa.rope_table(4096, D)
    status = pa.new_status()
    pa.rope_kv_write(dq, dk, dv, torch.from_numpy(positions).cuda(),
                     torch.from_numpy(slots).cuda(), table, cache, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    q_rot = orc.rope_pinned(q, positions, D)
    k_rot = orc.rope_pinned(k, positions, D)
    want = orc.new_cache(1, nb, BS, HK, D)
    orc.kv_write(want, 0, k_rot, v, slots)
    assert np.array_equal(bits(dq), bits(q_rot))
    assert np.array_equal(bits(dk), bits(k_rot))
    assert np.array_equal(bits(cache.tensor), bits(want))


def test_rope_kv_write_i8_past_65535_tokens():
    q, k, v, positions, slots, nb = _inputs(82)
    dq, dk, dv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    cache = pa.CacheI8(1, nb, HK, D)
    cache.codes.zero_()
    cache.scales.zero_()
    table = pa.rope_table(4096, D)
    status = pa.new_status()
    pa.rope_kv_write_i8(dq, dk, dv, torch.from_numpy(positions).cuda(),
                        torch.from_numpy(slots).cuda(), table, cache, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    q_rot = orc.rope_pinned(q, positions, D)
    k_rot = orc.rope_pinned(k, positions, D)
    codes, scales = orc.new_cache_i8(1, nb, BS, HK, D)
    orc.kv_write_i8(codes, scales, 0, k_rot, v, slots)
    assert np.array_equal(bits(dq), bits(q_rot))
    assert np.array_equal(bits(dk), bits(k_rot))
    assert np.array_equal(cache.codes.cpu().numpy(), codes)
    assert np.array_equal(cache.scales.cpu().numpy().view(np.uint32), scales.view(np.uint32))


def test_rope_kv_write_staged_bad_position_and_slot():
    """The staged kernel's checks, as the per-token one's: a token with a
    position outside the table is neither rotated nor written and reports
    PA_DEV_BAD_POSITION; a slot past the pool is rotated, not written, and
    reports PA_DEV_BAD_SLOT; a negative slot is a padding token (rotated, not
    written, no report).  Everything else bit for bit as the oracle."""
    Tn, Hn, Hkn, d = 2000, 8, 2, 128
    rng = np.random.default_rng(12)
    mk = lambda *s: rng.standard_normal(s, dtype=np.float32).astype(np.float16)  # noqa: E731
    q, k, v = mk(Tn, Hn, d), mk(Tn, Hkn, d), mk(Tn, Hkn, d)
    nb = Tn // BS + 8
    pos = rng.integers(0, 512, size=Tn).astype(np.int32)
    slots = rng.permutation(nb * BS)[:Tn].astype(np.int32)
    pos[5], pos[77] = 512, -3          # outside the 512-position table
    slots[9] = nb * BS                 # past the pool
    slots[11] = -1                     # padding
    table = pa.rope_table(512, d)
    cache = pa.Cache(1, nb, Hkn, d)
    cache.tensor.fill_(1.0)
    dq, dk, dv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    st = pa.new_status()
    assert Tn >= 8 * torch.cuda.get_device_properties(0).multi_processor_count
    pa.rope_kv_write(dq, dk, dv, torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(),
                     table, cache, status=st)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & pa.PA_DEV_BAD_POSITION and s & pa.PA_DEV_BAD_SLOT

    good = (pos >= 0) & (pos < 512)
    q_rot = orc.rope_pinned(q[good], pos[good], d)
    k_rot = orc.rope_pinned(k[good], pos[good], d)
    assert np.array_equal(bits(dq)[good], bits(torch.from_numpy(q_rot)))
    assert np.array_equal(bits(dk)[good], bits(torch.from_numpy(k_rot)))
    assert np.array_equal(bits(dq)[~good], q[~good].view(np.uint16))
    assert np.array_equal(bits(dk)[~good], k[~good].view(np.uint16))
    want = np.ones((2, 1, nb, BS, Hkn, d), np.float16)
    oslots = slots[good].copy()
    oslots[oslots >= nb * BS] = -1
    orc.kv_write(want, 0, k_rot, v[good], oslots)
    assert torch.equal(cache.tensor, torch.from_numpy(want).cuda())
