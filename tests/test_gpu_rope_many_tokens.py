"""RoPE + append (steps a1, a2) of more tokens than one grid dimension
holds: the RoPE/append kernels run one row of CTAs per token (blockIdx.y,
and blockIdx.z past 65535 tokens), so 70000 tokens exercise the third grid
dimension.  Rotated Q/K, the fp16 cache and the int8 codes and scales are
compared with the oracle bit for bit."""

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
