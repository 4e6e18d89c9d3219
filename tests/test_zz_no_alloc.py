"""pa_decode_noalloc: decode for callers that cannot give the library any
device memory (a plugin whose host framework owns all device allocations, a
caller that must not call cudaMalloc while running).  Its scratch lives in a
fixed array inside libpa.  Called here through the C ABI twice in a row (the
second call must not be disturbed by what the first left in the shared
array); each result must be bit for bit pa_decode's (the same kernel on the
same inputs) and within the attention tolerance of the fp64 oracle.

The file name makes pytest collect it last."""

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_gqa_rope_gb300 import pa
from paged_kv_gqa_rope_gb300 import workloads as W
from tests.gpu_helpers import DecodeRun, assert_attention_close, oracle_decode_step

pytestmark = pytest.mark.gpu


def _case(seed=31):
    rng = np.random.default_rng(seed)
    H, Hk, d = 32, 8, 128
    ctxs = [5, 300, 4097, 1, 1500, 64]
    wl = W.Workload(70, "noalloc", H, Hk, d, len(ctxs), "decode")
    need = [-(-(c + 1) // 16) for c in ctxs]
    pool = sum(need) + 2
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((len(ctxs), max(need)), -1, np.int32)
    at = 0
    for s, nb in enumerate(need):
        table[s, :nb] = perm[at:at + nb]
        at += nb
    B = len(ctxs)
    mk = lambda *sh: rng.standard_normal(sh, dtype=np.float32).astype(np.float16)  # noqa: E731
    case = W.Case(wl, np.asarray(ctxs, np.int64), np.ones(B, np.int64), table, pool,
                  mk(B, H, d), mk(B, Hk, d), mk(B, Hk, d))
    return case, mk(2, 1, pool, 16, Hk, d)


def _noalloc(lib, run, out, status):
    wl = run.case.wl
    return lib.pa_decode_noalloc(
        ctypes.c_void_p(run.q.data_ptr()), ctypes.byref(run.cache.desc), 0,
        ctypes.c_void_p(run.bt.data_ptr()), run.bt.shape[1], ctypes.c_void_p(run.ctx.data_ptr()),
        run.bt.shape[0], wl.n_heads, wl.n_kv_heads, wl.head_dim, 0.0,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_decode_noalloc_matches_decode(libpa):
    assert torch.cuda.is_available()
    case, init = _case()
    run = DecodeRun(case, init)
    ref = run.run()                      # RoPE + append + pa_decode (caller workspace)
    assert int(run.status.item()) == 0
    _, _, _, want = oracle_decode_step(case, init)
    assert_attention_close(ref, want)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        status = pa.new_status()
        rc = _noalloc(libpa, run, out, status)
        assert rc == pa.PA_OK, pa.strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref)     # same kernel, same inputs: same bits
        assert_attention_close(out, want)


def test_decode_noalloc_rejects_too_large(libpa):
    """4096 sequences x 256 KV heads need 4 MiB of counters on top of the
    4.9 MiB of records: more than the 8 MiB array.  Refused before anything
    is enqueued (the descriptor wraps an address that is never touched)."""
    d = pa.PaCache()
    fake = ctypes.c_void_p(1 << 20)
    assert libpa.pa_alloc_cache(ctypes.byref(d), 1, 10, 16, 256, 128, fake) == pa.PA_OK
    buf = ctypes.c_void_p(1 << 24)
    assert pa.decode_workspace_bytes(4096, 512, 256, 128) > (8 << 20)
    assert pa.decode_workspace_bytes(4096, 512, 195, 128) <= (8 << 20)
    rc = libpa.pa_decode_noalloc(buf, ctypes.byref(d), 0, buf, 4, buf, 4096, 512, 256, 128, 0.0,
                                 buf, None, None)
    assert rc == pa.PA_ERR_WORKSPACE
