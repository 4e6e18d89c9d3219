"""The tiny workload end to end on the GPU: a prefill of three prompts
(3, 5 and 2 tokens, cu_seqlens_q = [0, 3, 8, 10]) followed by four
single-token decode steps of every sequence, the generate loop of
"personal chatgpt 22 - llama2 generate" section 1 (one prompt window, then
windows of one token) over the paged cache of "nano-vllm notes - Llama"
(prepare_prefill, then prepare_decode: positions p, context_lens p + 1).

The oracle carries its own cache across the five steps.  After every step:
the rotated Q and K bits, the whole 16-block pool bit for bit, and every
output row within the attention tolerance (max-abs beyond the fp16 rounding
and relative L2).  The decode steps run once as separate pa_rope_kv_write +
pa_decode calls and once through the fused pa_decode_step."""

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


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused_step"])
def test_tiny_prefill_then_four_decode_steps(fused):
    case = W.make_case("tiny")
    wl = case.wl
    H, Hk, d, bs = wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.block_size
    scale = 1.0 / math.sqrt(d)
    assert list(case.num_new) == [3, 5, 2] and len(case.extra_steps) == 4
    init = W.initial_cache(case)  # the pool's prior contents (never read by a sequence)

    # --- prefill ----------------------------------------------------------
    md = pa.prepare_prefill(case.num_cached, case.num_new, case.block_tables)
    assert list(md["cu_seqlens_q"]) == [0, 3, 8, 10]
    table = pa.rope_table(16, d, wl.rope_theta)
    cache = pa.Cache(1, case.num_blocks, Hk, d)
    cache.tensor.copy_(torch.from_numpy(init))
    st = pa.new_status()
    q, k, v = _dev(case.q), _dev(case.k), _dev(case.v)
    bt = _dev(case.block_tables)
    pa.rope_kv_write(q, k, v, _dev(md["positions"]), _dev(md["slot_mapping"]), table, cache,
                     status=st)
    out = pa.prefill_varlen(q, cache, _dev(md["cu_seqlens_q"]), _dev(md["cu_seqlens_k"]), bt,
                            md["max_seqlen_q"], Hk, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    omd = orc.prefill_metadata(case.num_cached, case.num_new, case.block_tables, bs)
    q_rot = orc.rope_pinned(case.q, omd["positions"], d, wl.rope_theta)
    k_rot = orc.rope_pinned(case.k, omd["positions"], d, wl.rope_theta)
    ocache = init.copy()
    orc.kv_write(ocache, 0, k_rot, case.v, omd["slot_mapping"])
    want = orc.attention_prefill(q_rot, ocache, 0, omd["cu_seqlens_q"], omd["cu_seqlens_k"],
                                 case.block_tables, H, Hk, scale)
    assert np.array_equal(bits(q), bits(q_rot)), "prefill: rotated Q"
    assert np.array_equal(bits(k), bits(k_rot)), "prefill: rotated K"
    assert torch.equal(cache.tensor, torch.from_numpy(ocache).cuda()), "prefill: pool"
    assert_attention_close(out, want)

    # --- four decode steps --------------------------------------------------
    cached = case.num_new.copy()
    ws = pa.decode_workspace(3, H, Hk, d)
    for step, (dq, dk, dv) in enumerate(case.extra_steps):
        dmd = pa.prepare_decode(cached, case.block_tables)
        omd = orc.decode_metadata(cached, case.block_tables, bs)
        assert list(dmd["context_lens"]) == list(omd["context_lens"])
        q, k, v = _dev(dq), _dev(dk), _dev(dv)
        pos, slots, ctx = _dev(dmd["positions"]), _dev(dmd["slot_mapping"]), \
            _dev(dmd["context_lens"])
        if fused:
            out = pa.decode_step(q, k, v, pos, slots, table, cache, bt, ctx, ws, Hk, status=st)
        else:
            pa.rope_kv_write(q, k, v, pos, slots, table, cache, status=st)
            out = pa.decode(q, cache, bt, ctx, ws, Hk, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"step {step}: device status"

        q_rot = orc.rope_pinned(dq, omd["positions"], d, wl.rope_theta)
        k_rot = orc.rope_pinned(dk, omd["positions"], d, wl.rope_theta)
        orc.kv_write(ocache, 0, k_rot, dv, omd["slot_mapping"])
        want = orc.attention_decode(q_rot, ocache, 0, case.block_tables, omd["context_lens"],
                                    H, Hk, scale)
        assert np.array_equal(bits(q), bits(q_rot)), f"step {step}: rotated Q"
        assert np.array_equal(bits(k), bits(k_rot)), f"step {step}: rotated K"
        assert torch.equal(cache.tensor, torch.from_numpy(ocache).cuda()), f"step {step}: pool"
        assert_attention_close(out, want)
        cached = cached + 1

    # after the fourth step the sequences hold 7, 9 and 6 tokens, each in
    # its own block of the shuffled 16-block pool
    assert list(cached) == [7, 9, 6]
    assert len(set(int(b) for b in case.block_tables[:, 0])) == 3
