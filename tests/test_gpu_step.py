"""GPU tests of the fused decode step (pa_decode_step: RoPE/append and
decode chained by programmatic dependent launch) and of its CUDA-graph form
(pa_step_graph_*), replayed over consecutive steps of a serving loop with
the buffers refilled in place ("nano-vllm notes - Llama": prepare_decode
each step, the decode step captured in a CUDA graph)."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from tests.gpu_helpers import DecodeRun, assert_attention_close, bits, oracle_decode_step
from tests.test_gpu_decode import custom_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    assert pa.check_device() == pa.PA_OK
    return libpa


def fused(run):
    wl = run.wl
    return pa.decode_step(run.q, run.k, run.v, run.positions, run.slots, run.table, run.cache,
                          run.bt, run.ctx, run.ws, wl.n_kv_heads, status=run.status)


def test_decode_step_equals_separate_calls():
    case, init = custom_case(32, 8, 128, [5, 100, 1000, 2999, 40000], seed=21)
    sep = DecodeRun(case, init)
    want_out = sep.run()
    one = DecodeRun(case, init)
    got = fused(one)
    torch.cuda.synchronize()
    assert int(one.status.item()) == 0
    assert torch.equal(got, want_out)
    assert torch.equal(one.cache.tensor, sep.cache.tensor)
    assert torch.equal(one.q, sep.q)
    _, _, _, want = oracle_decode_step(case, init)
    assert_attention_close(got, want)


def next_step(case, rng):
    """The same sequences one token later: new q/k/v, one more cached token."""
    wl = case.wl
    B = len(case.num_cached)
    q = rng.standard_normal((B, wl.n_heads, wl.head_dim), dtype=np.float32).astype(np.float16)
    k = rng.standard_normal((B, wl.n_kv_heads, wl.head_dim), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((B, wl.n_kv_heads, wl.head_dim), dtype=np.float32).astype(np.float16)
    return dataclasses.replace(case, num_cached=case.num_cached + 1, q=q, k=k, v=v)


def test_step_graph_replays_a_serving_loop():
    ctxs = [5, 100, 1000, 2999]  # (c + 3) stays inside each sequence's blocks
    case, init = custom_case(16, 4, 128, ctxs, seed=22)
    run = DecodeRun(case, init, table_rows=4096)
    g = pa.StepGraph(run.q, run.k, run.v, run.positions, run.slots, run.table, run.cache,
                     run.bt, run.ctx, run.ws, case.wl.n_kv_heads, status=run.status)
    rng = np.random.default_rng(23)
    cache_np = init
    try:
        for step in range(3):
            out = g.launch()
            torch.cuda.synchronize()
            assert int(run.status.item()) == 0
            q_rot, k_rot, cache_np, want = oracle_decode_step(case, cache_np)
            assert np.array_equal(bits(run.q), bits(q_rot)), f"step {step}: rotated Q"
            assert torch.equal(run.cache.tensor, torch.from_numpy(cache_np).cuda()), \
                f"step {step}: cache"
            assert_attention_close(out, want)
            # refill the captured buffers in place for the next step
            case = next_step(case, rng)
            md = orc.decode_metadata(case.num_cached, case.block_tables, 16)
            run.q.copy_(torch.from_numpy(case.q))
            run.k.copy_(torch.from_numpy(case.k))
            run.v.copy_(torch.from_numpy(case.v))
            run.positions.copy_(torch.from_numpy(md["positions"].astype(np.int32)))
            run.slots.copy_(torch.from_numpy(md["slot_mapping"].astype(np.int32)))
            run.ctx.copy_(torch.from_numpy(md["context_lens"].astype(np.int32)))
    finally:
        g.close()


def test_step_graph_launches_on_any_stream():
    case, init = custom_case(8, 8, 64, [17, 300], seed=24)
    a = DecodeRun(case, init)
    want = a.run()
    b = DecodeRun(case, init)
    g = pa.StepGraph(b.q, b.k, b.v, b.positions, b.slots, b.table, b.cache, b.bt, b.ctx, b.ws,
                     case.wl.n_kv_heads, status=b.status)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = g.launch(stream=s)
    s.synchronize()
    g.close()
    assert torch.equal(out, want)


def _packed(arrays, host_offset=0):
    """Host arrays laid out in one pinned uint8 buffer (256-byte aligned
    offsets, the buffer itself starting host_offset bytes into a pinned
    allocation) and device views of a device buffer of the same layout."""
    off, lay = 0, {}
    for k, a in arrays.items():
        lay[k] = (off, a)
        off = (off + a.nbytes + 255) // 256 * 256
    host = torch.zeros(off + 16, dtype=torch.uint8).pin_memory()[host_offset:host_offset + off]
    dev = torch.zeros(off, dtype=torch.uint8, device="cuda")
    views = {k: dev[o:o + a.nbytes].view(torch.from_numpy(a).dtype).view(a.shape)
             for k, (o, a) in lay.items()}

    def fill(new):
        hv = host.numpy()
        for k, a in new.items():
            o, ref = lay[k]
            a = np.ascontiguousarray(a, ref.dtype)
            hv[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
    return host, dev, views, fill


@pytest.mark.parametrize("host_offset", [0, 4], ids=["copy-kernels", "copy-engine"])
def test_step_graph_with_host_io_replays_a_serving_loop(host_offset):
    """pa_step_graph_create_io: each replay copies the step's inputs from
    pinned host memory, runs RoPE/append + decode and copies the output
    back; the device input buffers are never written any other way.  With
    16-byte aligned host buffers the copies are kernels reading and writing
    the mapped host memory; 4 bytes off that alignment they are copy-engine
    copies."""
    ctxs = [5, 100, 1000, 2999]
    case, init = custom_case(16, 4, 128, ctxs, seed=25)
    run = DecodeRun(case, init, table_rows=4096)
    md = orc.decode_metadata(case.num_cached, case.block_tables, 16)
    step_in = lambda c, m: dict(q=c.q, k=c.k, v=c.v,  # noqa: E731
                                positions=m["positions"].astype(np.int32),
                                slots=m["slot_mapping"].astype(np.int32),
                                ctx=m["context_lens"].astype(np.int32),
                                bt=c.block_tables.astype(np.int32))
    host, dev, d, fill = _packed(step_in(case, md), host_offset)
    n_out = run.q.numel()
    host_out = torch.zeros(n_out + 8, dtype=torch.float16).pin_memory()[
        host_offset // 2:host_offset // 2 + n_out].view(tuple(run.q.shape))
    assert (host.data_ptr() % 16 == 0) == (host_offset == 0)
    assert (host_out.data_ptr() % 16 == 0) == (host_offset == 0)
    g = pa.StepGraph(d["q"], d["k"], d["v"], d["positions"], d["slots"], run.table, run.cache,
                     d["bt"], d["ctx"], run.ws, case.wl.n_kv_heads, status=run.status,
                     host_in=host, dev_in=dev, host_out=host_out)
    rng = np.random.default_rng(26)
    cache_np = init
    try:
        for step in range(3):
            fill(step_in(case, md))
            g.launch()
            torch.cuda.synchronize()
            assert int(run.status.item()) == 0
            q_rot, _, cache_np, want = oracle_decode_step(case, cache_np)
            assert np.array_equal(bits(d["q"]), bits(q_rot)), f"step {step}: rotated Q"
            assert torch.equal(run.cache.tensor, torch.from_numpy(cache_np).cuda()), \
                f"step {step}: cache"
            assert torch.equal(host_out, g.out.cpu()), f"step {step}: output copied back"
            assert_attention_close(host_out.cuda(), want)
            case = next_step(case, rng)
            md = orc.decode_metadata(case.num_cached, case.block_tables, 16)
    finally:
        g.close()


def test_step_graph_io_refuses_pageable_host_memory(libpa):
    import ctypes
    case, init = custom_case(8, 8, 64, [17, 300], seed=27)
    b = DecodeRun(case, init)
    args = pa._step_args(b.q, b.k, b.v, b.positions, b.slots, b.table, b.cache, b.bt, b.ctx,
                         b.ws, case.wl.n_kv_heads, 0, 0.0, torch.empty_like(b.q), b.status)
    pageable = np.zeros(1024, np.uint8)
    dev = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p()
    rc = libpa.pa_step_graph_create_io(ctypes.byref(h), *args, pa._p(pageable), pa._p(dev), 1024,
                                       None)
    assert rc == pa.PA_ERR_INVALID and not h.value
    out_pageable = np.zeros(tuple(b.q.shape), np.float16)
    rc = libpa.pa_step_graph_create_io(ctypes.byref(h), *args, None, None, 0,
                                       pa._p(out_pageable))
    assert rc == pa.PA_ERR_INVALID and not h.value
