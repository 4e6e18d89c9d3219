"""Host side of the C ABI, no GPU needed: the library loads and exports every
symbol the headers under include/ declare; the metadata builders agree bit for bit with
the oracle; invalid arguments are rejected before anything is enqueued."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from paged_kv_gqa_rope_gb300 import workloads as W

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(INCLUDE, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(pa_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_exports_every_declared_symbol(libpa):
    names = declared_functions()
    assert len(names) >= 12
    assert set(names) == set(pa.EXPORTS)
    for n in names:
        assert hasattr(libpa, n), n


def test_sizes(libpa):
    assert pa.cache_bytes(1, 16, 16, 2, 64) == 2 * 16 * 16 * 2 * 64 * 2
    assert pa.cache_bytes(0, 16, 16, 2, 64) == 0
    assert libpa.pa_rope_table_bytes(100, 128) == 100 * 64 * 8
    assert libpa.pa_rope_table_bytes(100, 7) == 0
    assert libpa.pa_decode_workspace_bytes(32, 64, 8, 128) > 0
    assert libpa.pa_decode_workspace_bytes(0, 64, 8, 128) == 0


def test_cache_descriptor_wraps_caller_memory(libpa):
    d = pa.PaCache()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced on the host
    assert libpa.pa_alloc_cache(ctypes.byref(d), 3, 10, 16, 8, 128, fake) == pa.PA_OK
    assert d.owns == 0 and d.layer_stride == 10 * 16 * 8 * 128 and d.kv_stride == 3 * d.layer_stride
    assert libpa.pa_free_cache(ctypes.byref(d)) == pa.PA_OK and not d.base
    assert libpa.pa_alloc_cache(ctypes.byref(d), 1, 10, 8, 8, 128, fake) == pa.PA_ERR_UNSUPPORTED
    assert libpa.pa_alloc_cache(ctypes.byref(d), 1, 10, 16, 8, 96, fake) == pa.PA_ERR_UNSUPPORTED
    assert libpa.pa_alloc_cache(ctypes.byref(d), 1, 10, 16, 8, 128, ctypes.c_void_p(1 << 20 | 16)) == pa.PA_ERR_INVALID
    assert libpa.pa_alloc_cache(None, 1, 10, 16, 8, 128, fake) == pa.PA_ERR_INVALID
    assert libpa.pa_alloc_cache(ctypes.byref(d), 0, 10, 16, 8, 128, fake) == pa.PA_ERR_INVALID


@pytest.mark.parametrize("name", ["tiny", "prefill_13b"])
def test_prepare_prefill_matches_oracle(libpa, name):
    c = W.make_case(name)
    got = pa.prepare_prefill(c.num_cached, c.num_new, c.block_tables)
    want = orc.prefill_metadata(c.num_cached, c.num_new, c.block_tables, 16)
    for key in ("positions", "slot_mapping", "cu_seqlens_q", "cu_seqlens_k"):
        assert np.array_equal(got[key], want[key]), key
    assert got["max_seqlen_q"] == want["max_seqlen_q"]
    assert got["max_seqlen_k"] == want["max_seqlen_k"]


@pytest.mark.parametrize("name", ["mha_decode_7b", "gqa_decode_70b", "ragged_decode"])
def test_prepare_decode_matches_oracle(libpa, name):
    c = W.make_case(name)
    got = pa.prepare_decode(c.num_cached, c.block_tables)
    want = orc.decode_metadata(c.num_cached, c.block_tables, 16)
    for key in ("positions", "slot_mapping", "context_lens"):
        assert np.array_equal(got[key], want[key]), key


def test_prepare_rejects_bad_metadata(libpa):
    bt = np.array([[3, -1]], np.int32)
    with pytest.raises(pa.PAError):
        pa.prepare_prefill([10], [10], bt)        # needs logical block 1 (-1)
    with pytest.raises(pa.PAError):
        pa.prepare_prefill([0], [33], bt)         # table row too short
    with pytest.raises(pa.PAError):
        pa.prepare_prefill([-1], [3], bt)
    with pytest.raises(pa.PAError):
        pa.prepare_decode([16], bt)               # position 16 -> block 1 = -1
    md = pa.prepare_prefill([0, 4], [0, 3], np.array([[1, -1], [2, -1]], np.int32))
    assert md["cu_seqlens_q"].tolist() == [0, 0, 3] and md["cu_seqlens_k"].tolist() == [0, 0, 7]


def test_kernel_entry_points_validate_before_launch(libpa):
    d = pa.PaCache()
    fake = ctypes.c_void_p(1 << 20)
    assert libpa.pa_alloc_cache(ctypes.byref(d), 1, 10, 16, 2, 64, fake) == pa.PA_OK
    buf = ctypes.c_void_p(1 << 24)
    # head_dim 96 unsupported; H % Hk != 0 invalid; wrong cache head count invalid
    assert libpa.pa_rope_kv_write(buf, buf, buf, buf, buf, 4, 4, 2, 96, buf, 8, ctypes.byref(d), 0, None, None) == pa.PA_ERR_UNSUPPORTED
    assert libpa.pa_rope_kv_write(buf, buf, buf, buf, buf, 4, 5, 2, 64, buf, 8, ctypes.byref(d), 0, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_rope_kv_write(buf, buf, buf, buf, buf, 4, 4, 4, 64, buf, 8, ctypes.byref(d), 0, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_rope_kv_write(buf, buf, buf, buf, buf, 4, 4, 2, 64, buf, 8, ctypes.byref(d), 1, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_rope_kv_write(None, buf, buf, buf, buf, 4, 4, 2, 64, buf, 8, ctypes.byref(d), 0, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_rope_kv_write(ctypes.c_void_p((1 << 24) + 2), buf, buf, buf, buf, 4, 4, 2, 64, buf, 8, ctypes.byref(d), 0, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_rope_kv_write(None, None, None, None, None, 0, 4, 2, 64, None, 8, ctypes.byref(d), 0, None, None) == pa.PA_OK
    # decode: group of 16 unsupported; too-small workspace; zero sequences is a no-op
    assert libpa.pa_decode(buf, ctypes.byref(d), 0, buf, 4, buf, 2, 32, 2, 64, 0.0, buf, 1 << 20, buf, None, None) == pa.PA_ERR_UNSUPPORTED
    assert libpa.pa_decode(buf, ctypes.byref(d), 0, buf, 4, buf, 2, 4, 2, 64, 0.0, buf, 16, buf, None, None) == pa.PA_ERR_WORKSPACE
    assert libpa.pa_decode(buf, ctypes.byref(d), 0, buf, 4, buf, 0, 4, 2, 64, 0.0, buf, 16, buf, None, None) == pa.PA_OK
    assert libpa.pa_decode(buf, ctypes.byref(d), 0, buf, 4, buf, 2, 4, 2, 64, -1.0, buf, 1 << 20, buf, None, None) == pa.PA_ERR_INVALID
    # prefill: H % Hk, head_dim
    assert libpa.pa_prefill_varlen(buf, 8, ctypes.byref(d), 0, buf, buf, buf, 4, 2, 16, 5, 2, 64, 0.0, buf, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_prefill_varlen(buf, 8, ctypes.byref(d), 0, buf, buf, buf, 4, 2, 16, 4, 2, 96, 0.0, buf, None, None) == pa.PA_ERR_UNSUPPORTED
    assert libpa.pa_prefill_varlen(buf, 8, ctypes.byref(d), 0, buf, buf, buf, 4, 2, 16, 4, 4, 64, 0.0, buf, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_prefill_varlen(buf, 0, ctypes.byref(d), 0, buf, buf, buf, 4, 2, 16, 4, 2, 64, 0.0, buf, None, None) == pa.PA_OK
    assert libpa.pa_prefill_varlen(ctypes.c_void_p((1 << 24) + 8), 8, ctypes.byref(d), 0, buf, buf, buf, 4, 2, 16, 4, 2, 64, 0.0, buf, None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_strerror(pa.PA_ERR_WORKSPACE) == b"decode workspace too small"


def test_step_graph_rejects_null_handles(libpa):
    assert libpa.pa_step_graph_create_io(None, *([None] * 6), 0, None, 0, None, 0, None, 1, 8, 8,
                                         128, 0.0, None, 0, None, None, None, None, 0,
                                         None) == pa.PA_ERR_INVALID
    h = ctypes.c_void_p()
    # an input copy needs both buffers
    assert libpa.pa_step_graph_create_io(ctypes.byref(h), *([None] * 6), 0, None, 0, None, 0,
                                         None, 1, 8, 8, 128, 0.0, None, 0, None, None, None,
                                         None, 64, None) == pa.PA_ERR_INVALID
    assert libpa.pa_step_graph_launch(None, None) == pa.PA_ERR_INVALID
    assert libpa.pa_step_graph_destroy(None) == pa.PA_ERR_INVALID
    assert libpa.pa_step_graph_create(None, *([None] * 6), 0, None, 0, None, 0, None,
                                      1, 8, 8, 128, 0.0, None, 0, None, None) == pa.PA_ERR_INVALID


def _prefill_raw(libpa, num_cached, num_new, table, block_size):
    nc, nn = (np.ascontiguousarray(x, np.int32) for x in (num_cached, num_new))
    bt = np.ascontiguousarray(table, np.int32)
    t = max(int(nn.astype(np.int64).sum()), 1)
    out = [np.full(t, -7, np.int32), np.full(t, -7, np.int32),
           np.full(len(nn) + 1, -7, np.int32), np.full(len(nn) + 1, -7, np.int32)]
    rc = libpa.pa_prepare_prefill(len(nn), pa._p(nc), pa._p(nn), pa._p(bt), bt.shape[1], block_size,
                                  *(pa._p(a) for a in out), None, None)
    return rc, out


def test_prepare_rejects_int32_overflow(libpa):
    # Two sequences of ~1.1e9 keys each: each fits int32, cu_seqlens_k's sum
    # does not.  A block size of 2^28 keeps the tables tiny.
    bs = 1 << 28
    table = np.tile(np.arange(8, dtype=np.int32), (2, 1))
    big = 1_100_000_000
    rc, out = _prefill_raw(libpa, [big], [1], table[:1], bs)
    assert rc == pa.PA_OK and out[3].tolist() == [0, big + 1]
    rc, out = _prefill_raw(libpa, [big, big], [1, 1], table, bs)
    assert rc == pa.PA_ERR_INVALID
    assert all((a == -7).all() for a in out)  # nothing written on error
    # Slots are int32: block id b covers slots b*16 .. b*16+15.
    last_ok = (2**31 - 1) // 16
    rc, out = _prefill_raw(libpa, [0], [16], [[last_ok]], 16)
    assert rc == pa.PA_OK and int(out[1][-1]) == 2**31 - 1
    rc, _ = _prefill_raw(libpa, [0], [1], [[last_ok + 1]], 16)
    assert rc == pa.PA_ERR_INVALID
    with pytest.raises(pa.PAError):
        pa.prepare_decode([3], np.array([[last_ok + 1]], np.int32))
    assert pa.prepare_decode([3], np.array([[last_ok]], np.int32))["slot_mapping"].tolist() == [last_ok * 16 + 3]


def test_prepare_prefill_no_sequences_accepts_null_outputs(libpa):
    assert libpa.pa_prepare_prefill(0, None, None, None, 0, 16, None, None, None, None, None,
                                    None) == pa.PA_OK
    md = pa.prepare_prefill([], [], np.zeros((0, 1), np.int32))
    assert md["cu_seqlens_q"].tolist() == [0] and md["cu_seqlens_k"].tolist() == [0]
    assert md["max_seqlen_q"] == 0 and md["max_seqlen_k"] == 0


def test_binding_shape_rule():
    """The binding's size check (the library sees only pointers): exact
    extents, None entries free, rank must match."""
    import torch
    t = torch.empty(4, 2, 64)
    pa._check_shape(t, (4, None, 64), "x")
    for bad in ((3, None, 64), (4, 2), (4, 2, 64, 1), (None, 3, None)):
        with pytest.raises(ValueError):
            pa._check_shape(t, bad, "x")
    with pytest.raises(TypeError):
        pa._dev(t.half(), torch.float16, "x", (4, 2, 64))  # a host tensor


C_CLIENT = r"""
#include <stdio.h>
#include "pa.h"
#include "pa_block_manager.h"

int main(void) {
    /* two sequences: 5 and 17 tokens cached, blocks {3} and {7, 2} */
    const int32_t cached[2] = {5, 17};
    const int32_t tables[4] = {3, -1, 7, 2};
    int32_t pos[2], slot[2], ctx[2];
    int rc = pa_prepare_decode(2, cached, tables, 2, 16, pos, slot, ctx);
    pa_bm_t bm = pa_bm_create(4, 16);
    int32_t toks[20];
    int i, hit = -1;
    for (i = 0; i < 20; ++i) toks[i] = i;
    if (bm) pa_bm_allocate(bm, 1, toks, 20, &hit);
    printf("%d %d %d %d %d %d %d %lu %d %s\n", rc, pos[0], slot[0], ctx[0], pos[1], slot[1],
           ctx[1], (unsigned long)pa_cache_bytes(1, 4, 16, 2, 64),
           bm ? pa_bm_num_free(bm) : -1, pa_strerror(PA_ERR_WORKSPACE));
    pa_bm_destroy(bm);
    return 0;
}
"""


def test_c_client_links_and_calls_the_library(libpa, tmp_path):
    """The boundary is plain C: a C99 program that includes the headers,
    links libpa.so and calls host-side entry points (no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not installed")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    libdir = os.path.dirname(pa.LIB_PATH)
    exe = tmp_path / "client"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE,
                    str(src), "-o", str(exe), "-L", libdir, "-lpa", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    # position 5 -> block 3 slot 53; position 17 -> logical block 1 = 2, slot 33
    assert out[:7] == ["0", "5", "53", "6", "17", "33", "18"]
    assert int(out[7]) == 2 * 4 * 16 * 2 * 64 * 2
    assert out[8] == "2"  # 20 tokens took two of the four blocks
    assert " ".join(out[9:]) == "decode workspace too small"


def test_binding_bounds_the_block_table_width():
    import torch
    ok = torch.empty(0, (2**31 - 1) // 16, dtype=torch.int32)
    assert pa._table_width(ok) == (2**31 - 1) // 16
    with pytest.raises(ValueError):
        pa._table_width(torch.empty(0, (2**31 - 1) // 16 + 1, dtype=torch.int32))


def test_prepare_metadata_random_batches_match_oracle(libpa):
    """Seeded random batches (empty sequences, block-aligned and ragged
    boundaries, long cached prefixes, permuted tables with padding) give the
    oracle's metadata bit for bit."""
    rng = np.random.default_rng(77)
    for trial in range(60):
        B = int(rng.integers(1, 12))
        bs = 16
        cached = rng.integers(0, 3 * bs, size=B) * rng.integers(0, 2, size=B)
        cached += rng.integers(0, 5, size=B) * bs * (trial % 3 == 0)
        new = rng.integers(0, 70, size=B)
        need = np.maximum((cached + new + bs - 1) // bs, 1)
        width = int(need.max()) + int(rng.integers(0, 3))
        perm = rng.permutation(int(need.sum()) + 5).astype(np.int32)
        table = np.full((B, width), -1, np.int32)
        at = 0
        for s in range(B):
            table[s, :need[s]] = perm[at:at + need[s]]
            at += need[s]
        got = pa.prepare_prefill(cached, new, table)
        want = orc.prefill_metadata(cached, new, table, bs)
        for key in ("positions", "slot_mapping", "cu_seqlens_q", "cu_seqlens_k"):
            assert np.array_equal(got[key], want[key]), (trial, key)
        assert got["max_seqlen_q"] == want["max_seqlen_q"]
        assert got["max_seqlen_k"] == want["max_seqlen_k"]
        dec = np.minimum(cached + new, need * bs - 1)  # a position inside the table
        got = pa.prepare_decode(dec, table)
        want = orc.decode_metadata(dec, table, bs)
        for key in ("positions", "slot_mapping", "context_lens"):
            assert np.array_equal(got[key], want[key]), (trial, key)


def test_c_entry_points_bound_the_block_table_width(libpa):
    """max_blocks_per_seq * 16 must fit in int32 (the kernels' length bound):
    every attention entry point refuses a wider table through the C ABI, not
    only the Python binding."""
    d = pa.PaCache()
    fake = ctypes.c_void_p(1 << 20)
    assert libpa.pa_alloc_cache(ctypes.byref(d), 1, 10, 16, 2, 64, fake) == pa.PA_OK
    buf = ctypes.c_void_p(1 << 24)
    widest = (2**31 - 1) // 16
    for maxb, want in ((widest + 1, pa.PA_ERR_INVALID), (2**31 - 1, pa.PA_ERR_INVALID)):
        assert libpa.pa_decode(buf, ctypes.byref(d), 0, buf, maxb, buf, 2, 4, 2, 64, 0.0, buf,
                               1 << 24, buf, None, None) == want
        assert libpa.pa_decode_noalloc(buf, ctypes.byref(d), 0, buf, maxb, buf, 2, 4, 2, 64,
                                       0.0, buf, None, None) == want
        assert libpa.pa_prefill_varlen(buf, 8, ctypes.byref(d), 0, buf, buf, buf, maxb, 2, 16, 4,
                                       2, 64, 0.0, buf, None, None) == want
        assert libpa.pa_decode_i8(buf, None, 0, buf, maxb, buf, 2, 4, 2, 64, 0.0, buf, 1 << 24,
                                  buf, None, None) == want
    # the widest accepted table passes this check (and stops at the next one:
    # a workspace of 16 bytes is too small)
    assert libpa.pa_decode(buf, ctypes.byref(d), 0, buf, widest, buf, 2, 4, 2, 64, 0.0, buf, 16,
                           buf, None, None) == pa.PA_ERR_WORKSPACE


def test_decode_noalloc_checks_arguments_like_decode(libpa):
    """pa_decode_noalloc makes pa_decode's argument checks, in the same order
    and before it touches its array: the same arguments give the same codes,
    num_seqs == 0 included (a no-op only once the cache descriptor and the
    shape are valid)."""
    d = pa.PaCache()
    fake = ctypes.c_void_p(1 << 20)
    assert libpa.pa_alloc_cache(ctypes.byref(d), 1, 10, 16, 2, 64, fake) == pa.PA_OK
    buf = ctypes.c_void_p(1 << 24)
    odd = ctypes.c_void_p((1 << 24) + 8)
    bad = pa.PaCache()  # all zero: no base pointer
    cases = [
        # (q, cache, layer, maxb, B, H, Hk, D, scale, out)
        (buf, d, 0, 4, 2, 32, 2, 64, 0.0, buf),      # group of 16: unsupported
        (buf, d, 0, 4, 2, 5, 2, 64, 0.0, buf),       # H % Hk != 0
        (buf, d, 0, 4, 2, 4, 2, 96, 0.0, buf),       # head_dim 96
        (buf, d, 0, 4, 5000, 4, 2, 64, 0.0, buf),    # more than 4096 sequences
        (buf, d, 1, 4, 2, 4, 2, 64, 0.0, buf),       # layer out of range
        (buf, bad, 0, 4, 2, 4, 2, 64, 0.0, buf),     # no cache
        (buf, bad, 0, 4, 0, 4, 2, 64, 0.0, buf),     # no cache, no sequences
        (buf, d, 0, 4, 0, 4, 2, 64, 0.0, buf),       # no sequences: no-op
        (buf, d, 0, 0, 2, 4, 2, 64, 0.0, buf),       # empty table
        (buf, d, 0, 4, 2, 4, 2, 64, -1.0, buf),      # negative scale
        (None, d, 0, 4, 2, 4, 2, 64, 0.0, buf),      # no q
        (odd, d, 0, 4, 2, 4, 2, 64, 0.0, buf),       # q not 16-byte aligned
        (buf, d, 0, 4, 2, 4, 2, 64, 0.0, odd),       # out not 16-byte aligned
    ]
    for q, c, layer, maxb, B, H, Hk, D, scale, out in cases:
        want = libpa.pa_decode(q, ctypes.byref(c), layer, buf, maxb, buf, B, H, Hk, D, scale, buf,
                               1 << 24, out, None, None)
        got = libpa.pa_decode_noalloc(q, ctypes.byref(c), layer, buf, maxb, buf, B, H, Hk, D,
                                      scale, out, None, None)
        assert want != pa.PA_ERR_WORKSPACE
        assert got == want, (q, layer, maxb, B, H, Hk, D, scale, out, got, want)
