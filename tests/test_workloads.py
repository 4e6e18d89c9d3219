"""The seeded input recipe: deterministic, and shaped like the five
workloads (lengths, pool sizes, block tables)."""

import numpy as np

from paged_kv_gqa_rope_gb300 import workloads as W


def test_deterministic():
    a = W.make_case("tiny")
    b = W.make_case("tiny")
    assert np.array_equal(a.q, b.q) and np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(W.block_contents(a.wl, 3), W.block_contents(b.wl, 3))


def test_tiny_shape():
    c = W.make_case("tiny")
    assert c.num_new.tolist() == [3, 5, 2] and c.num_cached.tolist() == [0, 0, 0]
    assert c.num_blocks == 16 and c.q.shape == (10, 4, 64) and c.k.shape == (10, 2, 64)
    assert len(c.extra_steps) == 4
    used = c.block_tables[c.block_tables >= 0]
    assert len(set(used.tolist())) == len(used) == 3


def test_decode_pools():
    c2 = W.make_case("mha_decode_7b")
    assert c2.num_blocks == 32 * 129 and c2.block_tables.shape == (32, 129)
    assert sorted(c2.block_tables.ravel().tolist()) == list(range(32 * 129))
    assert np.all(c2.num_cached == 2048)
    c3 = W.make_case("gqa_decode_70b")
    assert c3.num_blocks == 32 * 257 and np.all(c3.num_cached == 4096)
    c5 = W.make_case("ragged_decode")
    assert c5.num_cached.min() >= 16 and c5.num_cached.max() <= 32768
    need = sum(-(-(int(x) + 1) // 16) for x in c5.num_cached)
    assert c5.num_blocks == int(np.ceil(1.1 * need))
    used = c5.block_tables[c5.block_tables >= 0]
    assert len(used) == need and len(set(used.tolist())) == need


def test_prefill_lengths():
    c = W.make_case("prefill_13b")
    assert np.all(c.num_cached % 16 == 0) and c.num_cached.max() <= 1024
    assert c.num_new.min() >= 128 and c.num_new.max() <= 2048
    assert c.q.shape == (int(c.num_new.sum()), 40, 128)


def test_outliers_present():
    wl = W.WORKLOADS["ragged_decode"]
    x = np.concatenate([W.block_contents(wl, b).ravel() for b in range(8)]).astype(np.float32)
    big = np.mean(np.abs(x) > 4.0)   # N(0,0.5) alone almost never exceeds 4
    assert 0.003 < big < 0.02
