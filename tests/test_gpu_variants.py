"""GPU parity of the whole path (RoPE, paged write, prefill and decode) on
the model shapes and RoPE bases the pages name besides the headline
workloads:

* TinyLlama: 32 Q heads over 4 KV heads, head_dim 64 (hidden 2048 / 32),
  rope_theta 1e4 ("nano-vllm notes - Llama", the TinyLlama config record);
* Qwen3: 16 Q heads over 8 KV heads, head_dim 128, rope_theta 1e6 (same page,
  the Qwen3 config record);
* Llama 3's RoPE base 500000 ("Meta Llama source deep-dive", 3.3 and 9.4) on
  a 32 / 8, d = 128 shape.

Positions reach past 20000 so that the larger bases' slow pairs turn by
more than a rounding error.  Same bars as the headline tests: rotated Q/K and
the cache bit-exact, attention within the stated tolerance."""

import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_gqa_rope_gb300 import pa
from tests.gpu_helpers import assert_attention_close
from tests.test_gpu_decode import check_step, custom_case
from tests.test_gpu_prefill import check, custom_prefill_case

pytestmark = pytest.mark.gpu

VARIANTS = {
    "tinyllama": (32, 4, 64, 1e4),
    "qwen3": (16, 8, 128, 1e6),
    "llama3_theta": (32, 8, 128, 5e5),
}


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    assert pa.check_device() == pa.PA_OK
    return libpa


def with_theta(case, theta):
    return dataclasses.replace(case, wl=dataclasses.replace(case.wl, rope_theta=theta))


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_decode_step_variant(name):
    H, Hk, d, theta = VARIANTS[name]
    case, init = custom_case(H, Hk, d, [0, 15, 16, 300, 4097, 20000], seed=300 + H + d)
    (max_abs, rel), *_ = check_step(with_theta(case, theta), init)
    print(f"{name} decode: max_abs={max_abs:.2e} rel_l2={rel:.2e}")


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_prefill_variant(name):
    H, Hk, d, theta = VARIANTS[name]
    case, init = custom_prefill_case(H, Hk, d, [0, 37, 1000, 20000], [300, 129, 64, 40],
                                     seed=400 + H + d)
    (max_abs, rel), *_ = check(with_theta(case, theta), init)
    print(f"{name} prefill: max_abs={max_abs:.2e} rel_l2={rel:.2e}")


def test_theta_changes_the_rotation():
    """The base reaches the kernel: the same token at position 20000 rotates
    differently under 1e4 and 1e6."""
    q = torch.ones(1, 1, 128, dtype=torch.float16, device="cuda")
    outs = []
    for theta in (1e4, 1e6):
        qq, kk = q.clone(), q.clone()
        v = torch.zeros_like(q)
        table = pa.rope_table(20001, 128, theta)
        cache = pa.Cache(1, 2, 1, 128)
        pos = torch.tensor([20000], dtype=torch.int32, device="cuda")
        slot = torch.tensor([-1], dtype=torch.int32, device="cuda")
        pa.rope_kv_write(qq, kk, v, pos, slot, table, cache)
        torch.cuda.synchronize()
        outs.append(qq.float().cpu().numpy())
    assert not np.array_equal(outs[0], outs[1])
