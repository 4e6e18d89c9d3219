"""Pins of the CPU oracle against things other than itself: the worked
examples printed on the pages (tests/golden/*.json, each with its source),
closed forms, invariants, and brute force against torch's float64
scaled_dot_product_attention.  CPU only."""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import reference as orc
from tests.conftest import GOLDEN


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- metadata

def test_cu_seqlens_worked_example():
    g = golden("nano_vllm_cu_seqlens.json")
    assert orc.cu_seqlens(g["q_lengths"]).tolist() == g["cu_seqlens_q"]


def test_prefill_metadata_two_prompts():
    g = golden("nano_vllm_prefill_two_prompts.json")
    tables = np.array([[3], [7]], np.int32)
    md = orc.prefill_metadata(g["num_cached"], g["num_new"], tables, 16)
    assert md["positions"].tolist() == g["positions"]
    assert md["cu_seqlens_q"].tolist() == g["cu_seqlens_q"]
    assert md["cu_seqlens_k"].tolist() == g["cu_seqlens_k"]
    assert md["max_seqlen_q"] == 5 and md["max_seqlen_k"] == 5


def test_decode_metadata_worked_example():
    g = golden("nano_vllm_decode_example.json")
    tables = np.array([[2], [9]], np.int32)
    md = orc.decode_metadata(g["num_cached"], tables, 16)
    assert md["positions"].tolist() == g["positions"]
    assert md["context_lens"].tolist() == g["context_lens"]


def test_generate_windows():
    """Prompt of 8 tokens, then single-token steps: windows 0:8, 8:9, 9:10."""
    g = golden("llama2_generate_windows.json")
    tables = np.array([[5]], np.int32)
    seen = []
    md = orc.prefill_metadata([0], [8], tables, 16)
    seen.append([int(md["positions"][0]), int(md["positions"][-1]) + 1])
    for cached in (8, 9):
        md = orc.decode_metadata([cached], tables, 16)
        seen.append([int(md["positions"][0]), int(md["context_lens"][0])])
    assert seen == g["windows"]


def _slots_by_enumeration(tables, n_tokens, bs):
    """(seq, logical position) -> physical slot, by walking each sequence's
    blocks in order and numbering their rows."""
    out = {}
    for s, row in enumerate(tables):
        pos = 0
        for blk in row:
            for r in range(bs):
                if pos >= n_tokens[s]:
                    break
                out[(s, pos)] = int(blk) * bs + r
                pos += 1
    return out


@pytest.mark.parametrize("bs", [16, 4])
def test_slot_mapping_matches_enumeration(bs):
    rng = np.random.default_rng(1)
    cached = [0, 17, 32, 5]
    new = [3, 20, 1, 16]
    need = [-(-(c + n) // bs) for c, n in zip(cached, new)]
    perm = rng.permutation(sum(need) + 3)
    tables = np.full((4, max(need)), -1, np.int32)
    at = 0
    for s, nb in enumerate(need):
        tables[s, :nb] = perm[at:at + nb]
        at += nb
    want = _slots_by_enumeration(tables, [c + n for c, n in zip(cached, new)], bs)
    md = orc.prefill_metadata(cached, new, tables, bs)
    got, t = {}, 0
    for s in range(4):
        for pos in range(cached[s], cached[s] + new[s]):
            assert md["positions"][t] == pos
            got[(s, pos)] = int(md["slot_mapping"][t])
            t += 1
    for key, slot in got.items():
        assert want[key] == slot
    assert len(set(got.values())) == len(got)
    assert md["cu_seqlens_k"].tolist() == orc.cu_seqlens([c + n for c, n in zip(cached, new)]).tolist()
    dm = orc.decode_metadata([c + n - 1 for c, n in zip(cached, new)], tables, bs)
    for s in range(4):
        assert dm["slot_mapping"][s] == want[(s, cached[s] + new[s] - 1)]
        assert dm["context_lens"][s] == cached[s] + new[s]


# ---------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 4, 64)).astype(np.float16)
    y = orc.rope_pinned(x, [0, 0, 0], 64)
    assert np.array_equal(y.view(np.uint16), x.view(np.uint16))


def test_rope_closed_form_angles():
    """d=4: pair 0 turns at 1 rad per position, pair 1 at theta^(-1/2) =
    0.01 rad per position.  A unit vector on the first axis of a pair turns
    counter-clockwise to (cos a, sin a) and leaves the other pair alone."""
    e0 = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    e2 = np.array([[[0.0, 0.0, 1.0, 0.0]]])
    y = orc.rope_exact(e0, [3], 4)[0, 0]
    assert np.allclose(y, [math.cos(3.0), math.sin(3.0), 0.0, 0.0], atol=1e-15)
    y = orc.rope_exact(e2, [100], 4)[0, 0]
    assert np.allclose(y, [0.0, 0.0, math.cos(1.0), math.sin(1.0)], atol=1e-14)
    # the pinned fp16 path lands on the fp16 rounding of the same values
    y16 = orc.rope_pinned(e2.astype(np.float16), [100], 4)[0, 0]
    assert np.array_equal(y16, np.array([0, 0, math.cos(1.0), math.sin(1.0)]).astype(np.float16))
    # theta as a parameter: theta=1e6, d=4 -> pair 1 turns at 1e-3 rad/pos
    y = orc.rope_exact(e2, [1000], 4, theta=1e6)[0, 0]
    assert np.allclose(y, [0.0, 0.0, math.cos(1.0), math.sin(1.0)], atol=1e-13)


def test_rope_pairs_are_adjacent():
    d = 8
    for i in range(d // 2):
        x = np.zeros((1, 1, d))
        x[0, 0, 2 * i] = 1.0
        y = orc.rope_exact(x, [7], d)[0, 0]
        touched = set(np.nonzero(np.abs(y) > 1e-12)[0].tolist())
        assert touched <= {2 * i, 2 * i + 1}
        assert abs(y[2 * i + 1]) > 1e-3  # really rotated


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 3, 128))
    pos = [0, 1, 77, 4096, 32768]
    y = orc.rope_exact(x, pos, 128)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(nx, ny, rtol=1e-12, atol=1e-12)


def test_rope_dot_depends_on_relative_position():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    base = None
    for shift in (0, 1, 1000, 30000):
        m, n = 5 + shift, 17 + shift
        qr = orc.rope_exact(q, [m], 128)
        kr = orc.rope_exact(k, [n], 128)
        dot = float((qr * kr).sum())
        if base is None:
            base = dot
        # angles grow with the shift, so allow for their float64 rounding
        assert abs(dot - base) < 1e-9 * max(1.0, abs(base))


def test_rope_pinned_within_one_ulp_of_exact():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 2, 128)).astype(np.float16)
    pos = rng.integers(0, 32769, size=64)
    pinned = orc.rope_pinned(x, pos, 128).astype(np.float64)
    exact = orc.rope_exact(x.astype(np.float64), pos, 128)
    # one fp16 ulp of the exact value, plus the fp32 cancellation allowance
    ulp = np.spacing(np.abs(exact).astype(np.float16)).astype(np.float64)
    mag = np.repeat(np.maximum(np.abs(x[..., 0::2]), np.abs(x[..., 1::2])), 2, axis=-1)
    assert np.all(np.abs(pinned - exact) <= ulp + 4 * 2.0 ** -24 * mag.astype(np.float64))
    # and the vast majority are the correctly rounded fp16 value
    same = np.mean(pinned == exact.astype(np.float16).astype(np.float64))
    assert same > 0.99


def test_rope_table_entries_are_rounded_libm():
    c, s = orc.rope_cos_sin(12345, 128)
    inv = 10000.0 ** (-np.arange(0, 128, 2) / 128.0)
    ang = 12345.0 * inv
    assert np.all(np.abs(c.astype(np.float64) - np.cos(ang)) <= np.spacing(np.float32(1.0)))
    assert np.all(np.abs(s.astype(np.float64) - np.sin(ang)) <= np.spacing(np.float32(1.0)))
    # rounded once: the entry is the nearest float32 to the double value
    assert np.all(np.abs(c - np.cos(ang)) <= 0.5 * np.spacing(np.abs(c)) * (1 + 1e-6) + 1e-15)


# ---------------------------------------------------------------- KV write

def test_kv_write_round_trip_and_untouched():
    rng = np.random.default_rng(6)
    bs, Hk, d = 16, 2, 8
    cached, new = [3, 0], [20, 5]
    need = [2, 1]
    tables = np.array([[4, 1], [2, -1]], np.int32)
    cache = orc.new_cache(1, 6, bs, Hk, d)
    sentinel = np.float16(7.0)
    cache[:] = sentinel
    md = orc.prefill_metadata(cached, new, tables, bs)
    T = sum(new)
    k = rng.standard_normal((T, Hk, d)).astype(np.float16)
    v = rng.standard_normal((T, Hk, d)).astype(np.float16)
    orc.kv_write(cache, 0, k, v, md["slot_mapping"])
    t = 0
    for s in range(2):
        K, V = orc.gather_kv(cache, 0, tables[s], cached[s] + new[s])
        for pos in range(cached[s], cached[s] + new[s]):
            assert np.array_equal(K[pos].astype(np.float16).view(np.uint16), k[t].view(np.uint16))
            assert np.array_equal(V[pos].astype(np.float16).view(np.uint16), v[t].view(np.uint16))
            t += 1
    # exactly T rows per K/V plane changed; blocks 0, 3, 5 untouched
    changed = np.any(cache != sentinel, axis=(4, 5))
    assert changed[0].sum() == T and changed[1].sum() <= T
    for blk in (0, 3, 5):
        assert np.all(cache[:, 0, blk] == sentinel)
    # negative slots are skipped
    before = cache.copy()
    orc.kv_write(cache, 0, k[:2], v[:2], np.array([-1, -5], np.int32))
    assert np.array_equal(before, cache)


# ---------------------------------------------------------------- attention

def _sdpa_prefill(q, K, V, p, H, Hk, scale):
    """torch float64 SDPA with repeat_kv as repeat_interleave and the
    page's mask: a zero block of width p, then triu(-inf, diagonal=1)."""
    g = H // Hk
    lq = q.shape[0]
    Kt = torch.from_numpy(K).repeat_interleave(g, dim=1)   # [lk, H, d]
    Vt = torch.from_numpy(V).repeat_interleave(g, dim=1)
    qt = torch.from_numpy(q)
    mask = torch.triu(torch.full((lq, lq), float("-inf"), dtype=torch.float64), diagonal=1)
    mask = torch.hstack([torch.zeros((lq, p), dtype=torch.float64), mask])
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.transpose(0, 1), Kt.transpose(0, 1), Vt.transpose(0, 1),
        attn_mask=mask, scale=scale)
    return o.transpose(0, 1).numpy()


def _random_paged(rng, cached, new, H, Hk, d, bs=16, extra_blocks=2, scale_kv=1.0):
    need = [-(-(c + n) // bs) for c, n in zip(cached, new)]
    nb = sum(need) + extra_blocks
    perm = rng.permutation(nb)
    tables = np.full((len(new), max(need)), -1, np.int32)
    at = 0
    for s, k in enumerate(need):
        tables[s, :k] = perm[at:at + k]
        at += k
    cache = (rng.standard_normal((2, 1, nb, bs, Hk, d)) * scale_kv).astype(np.float16)
    T = sum(new)
    q = rng.standard_normal((T, H, d)).astype(np.float16)
    k = rng.standard_normal((T, Hk, d)).astype(np.float16)
    v = rng.standard_normal((T, Hk, d)).astype(np.float16)
    md = orc.prefill_metadata(cached, new, tables, bs)
    orc.kv_write(cache, 0, k, v, md["slot_mapping"])
    return cache, tables, q, md


@pytest.mark.parametrize("H,Hk,d", [(4, 2, 64), (4, 4, 32), (8, 1, 16), (6, 3, 8)])
def test_prefill_matches_sdpa_brute_force(H, Hk, d):
    rng = np.random.default_rng(10 + H + Hk + d)
    cached, new = [0, 16, 5, 32], [3, 7, 1, 18]
    cache, tables, q, md = _random_paged(rng, cached, new, H, Hk, d)
    scale = 1.0 / math.sqrt(d)
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"],
                                tables, H, Hk)
    cq = md["cu_seqlens_q"]
    for s in range(4):
        K, V = orc.gather_kv(cache, 0, tables[s], cached[s] + new[s])
        want = _sdpa_prefill(q[cq[s]:cq[s + 1]].astype(np.float64), K, V, cached[s], H, Hk, scale)
        assert np.max(np.abs(out[cq[s]:cq[s + 1]] - want)) < 1e-12


def test_gqa_uses_contiguous_groups():
    """Q head h reads KV head h // g (repeat_kv), not h % Hk: on a case
    where the two conventions differ the oracle must match the former."""
    rng = np.random.default_rng(11)
    H, Hk, d = 4, 2, 16
    cache, tables, q, md = _random_paged(rng, [8], [4], H, Hk, d)
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, H, Hk)
    K, V = orc.gather_kv(cache, 0, tables[0], 12)
    want = _sdpa_prefill(q.astype(np.float64), K, V, 8, H, Hk, 1 / math.sqrt(d))
    perm = [0, 2, 1, 3]  # h % Hk grouping of heads 0..3 onto kv heads 0,1,0,1
    other = _sdpa_prefill(q.astype(np.float64)[:, perm], K, V, 8, H, Hk, 1 / math.sqrt(d))[:, np.argsort(perm)]
    assert np.max(np.abs(out - want)) < 1e-12
    assert np.max(np.abs(out - other)) > 1e-2


def test_mha_reduction():
    rng = np.random.default_rng(12)
    H = Hk = 3
    d = 16
    cache, tables, q, md = _random_paged(rng, [16], [9], H, Hk, d)
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, H, Hk)
    K, V = orc.gather_kv(cache, 0, tables[0], 25)
    # plain per-head attention, no head broadcast at all
    for h in range(H):
        sc = q[:, h].astype(np.float64) @ K[:, h].T / math.sqrt(d)
        for i in range(9):
            row = sc[i, :16 + i + 1]
            w = np.exp(row - row.max())
            assert np.allclose(out[i, h], w @ V[:16 + i + 1, h] / w.sum(), atol=1e-13)


def test_constant_v_returns_v():
    rng = np.random.default_rng(13)
    H, Hk, d = 4, 2, 32
    cache, tables, q, md = _random_paged(rng, [32, 0], [5, 9], H, Hk, d)
    cache[1] = np.float16(0.375)
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, H, Hk)
    assert np.max(np.abs(out - 0.375)) < 1e-14
    dm = orc.decode_metadata([36, 8], tables, 16)
    od = orc.attention_decode(q[[4, 13]], cache, 0, tables, dm["context_lens"], H, Hk)
    assert np.max(np.abs(od - 0.375)) < 1e-14


def test_single_key_returns_its_value():
    rng = np.random.default_rng(14)
    cache, tables, q, md = _random_paged(rng, [0], [1], 2, 1, 8)
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, 2, 1)
    v = cache[1, 0, tables[0, 0], 0, 0].astype(np.float64)
    assert np.array_equal(out[0, 0], v) and np.array_equal(out[0, 1], v)
    od = orc.attention_decode(q, cache, 0, tables, [1], 2, 1)
    assert np.array_equal(od[0, 0], v)


def test_decode_equals_last_row_of_prefill():
    rng = np.random.default_rng(15)
    H, Hk, d = 8, 2, 32
    cache, tables, q, md = _random_paged(rng, [0, 0], [21, 40], H, Hk, d)
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, H, Hk)
    last = [20, 60]
    od = orc.attention_decode(q[last], cache, 0, tables, [21, 40], H, Hk)
    assert np.max(np.abs(od - out[last])) < 1e-13


def test_decode_matches_sdpa_without_mask():
    rng = np.random.default_rng(16)
    H, Hk, d = 8, 2, 64
    cache, tables, q, md = _random_paged(rng, [0], [50], H, Hk, d)
    od = orc.attention_decode(q[[49]], cache, 0, tables, [50], H, Hk)
    K, V = orc.gather_kv(cache, 0, tables[0], 50)
    qt = torch.from_numpy(q[[49]].astype(np.float64)).transpose(0, 1)  # [H,1,d]
    Kt = torch.from_numpy(K).repeat_interleave(4, dim=1).transpose(0, 1)
    Vt = torch.from_numpy(V).repeat_interleave(4, dim=1).transpose(0, 1)
    want = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt).transpose(0, 1).numpy()
    assert np.max(np.abs(od - want)) < 1e-12


def test_block_permutation_invariance():
    rng = np.random.default_rng(17)
    H, Hk, d = 4, 2, 16
    cache, tables, q, md = _random_paged(rng, [16, 3], [12, 30], H, Hk, d, extra_blocks=5)
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, H, Hk)
    nb = cache.shape[2]
    perm = rng.permutation(nb)
    cache2 = np.empty_like(cache)
    cache2[:, :, perm] = cache
    tables2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = orc.attention_prefill(q, cache2, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables2, H, Hk)
    assert np.array_equal(out, out2)
    ctx = [28, 33]
    d1 = orc.attention_decode(q[[11, 41]], cache, 0, tables, ctx, H, Hk)
    d2 = orc.attention_decode(q[[11, 41]], cache2, 0, tables2, ctx, H, Hk)
    assert np.array_equal(d1, d2)


def test_prefix_prefill_equals_rows_of_full_prefill():
    rng = np.random.default_rng(18)
    H, Hk, d = 4, 4, 32
    cache, tables, q, md = _random_paged(rng, [0], [45], H, Hk, d)
    full = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, H, Hk)
    for p in (16, 32, 44):
        cq = orc.cu_seqlens([45 - p])
        ck = orc.cu_seqlens([45])
        part = orc.attention_prefill(q[p:], cache, 0, cq, ck, tables, H, Hk)
        assert np.max(np.abs(part - full[p:])) < 1e-13


def test_softmax_is_stable_for_large_logits():
    rng = np.random.default_rng(19)
    H, Hk, d = 2, 1, 16
    cache, tables, q, md = _random_paged(rng, [0], [20], H, Hk, d)
    q = (q.astype(np.float32) * 4000).astype(np.float16)  # logits ~1e4
    out = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, H, Hk)
    assert np.all(np.isfinite(out))
    od = orc.attention_decode(q[[19]], cache, 0, tables, [20], H, Hk)
    assert np.all(np.isfinite(od)) and np.max(np.abs(od - out[[19]])) < 1e-12


def test_scale_argument():
    rng = np.random.default_rng(20)
    cache, tables, q, md = _random_paged(rng, [0], [6], 2, 1, 8)
    a = orc.attention_prefill(q, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], tables, 2, 1, scale=0.0)
    K, V = orc.gather_kv(cache, 0, tables[0], 6)
    # scale 0: uniform weights over the visible keys
    for i in range(6):
        assert np.allclose(a[i, 0], V[:i + 1, 0].mean(axis=0), atol=1e-14)


# ---------------------------------------------------------------- int8 KV cache

def test_int8_quantize_worked_example():
    """absmax 1 -> scale fl32(1/127); 0.5 / scale lands on 63.5 in float32
    and rounds to the even 64; 0.25 -> 31.75 -> 32; zeros stay zero; a zero
    row has scale 0 and zero codes."""
    x = np.array([[0.5, -1.0, 0.25, 0.0], [0.0, 0.0, 0.0, 0.0]], np.float16)
    codes, scale = orc.kv_quantize_int8(x)
    assert codes.tolist() == [[64, -127, 32, 0], [0, 0, 0, 0]]
    assert scale[0] == np.float32(1.0) / np.float32(127.0) and scale[1] == 0.0


def test_int8_quantize_error_bound_and_extremes():
    rng = np.random.default_rng(40)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.01, 30, size=(500, 1))).astype(np.float16)
    codes, scale = orc.kv_quantize_int8(x)
    back = codes.astype(np.float64) * scale[:, None].astype(np.float64)
    err = np.abs(back - x.astype(np.float64))
    # half a step, plus the float32 rounding of the quotient (|q| <= 127
    # units of 2^-24 each) that the rounding decision is made on
    assert np.all(err <= scale[:, None] * (0.5 + 127 * 2.0 ** -24))
    assert np.all(np.abs(codes).max(axis=1) == 127)     # the largest entry maps to +-127
    assert codes.min() >= -127


def test_int8_lossless_inputs_give_the_fp16_attention():
    """Rows whose values are k / 128 with integer |k| <= 127 and a +-127 entry
    quantise exactly (scale = 2^-7), so decode on the int8 cache equals
    decode on the fp16 cache holding the same values."""
    rng = np.random.default_rng(41)
    bs, Hk, H, d, n = 16, 2, 4, 32, 37
    k = rng.integers(-127, 128, size=(n, Hk, d))
    v = rng.integers(-127, 128, size=(n, Hk, d))
    k[..., 0], v[..., 3] = 127, -127
    k16 = (k / 128.0).astype(np.float16)
    v16 = (v / 128.0).astype(np.float16)
    nb = -(-n // bs)
    table = np.arange(nb, dtype=np.int32)[None, :]
    slots = np.arange(n)
    codes, scales = orc.new_cache_i8(1, nb, bs, Hk, d)
    orc.kv_write_i8(codes, scales, 0, k16, v16, slots)
    assert np.all(scales[:, 0, :, :, :][..., :n % bs or bs] >= 0)
    assert np.array_equal(codes[0, 0].reshape(-1, Hk, d)[:n], k.astype(np.int8))
    cache = orc.new_cache(1, nb, bs, Hk, d)
    orc.kv_write(cache, 0, k16, v16, slots)
    q = rng.standard_normal((1, H, d)).astype(np.float16)
    a = orc.attention_decode_i8(q, codes, scales, 0, table, [n], H, Hk)
    b = orc.attention_decode(q, cache, 0, table, [n], H, Hk)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_int8_write_places_codes_and_scales_by_slot():
    rng = np.random.default_rng(42)
    bs, Hk, d = 16, 3, 8
    k16 = rng.standard_normal((3, Hk, d)).astype(np.float16)
    v16 = rng.standard_normal((3, Hk, d)).astype(np.float16)
    codes, scales = orc.new_cache_i8(2, 4, bs, Hk, d)
    orc.kv_write_i8(codes, scales, 1, k16, v16, [5, -1, 3 * bs + 15])
    kq, ks = orc.kv_quantize_int8(k16)
    vq, vs = orc.kv_quantize_int8(v16)
    assert np.array_equal(codes[0, 1, 0, 5], kq[0]) and np.array_equal(codes[1, 1, 3, 15], vq[2])
    assert np.array_equal(scales[0, 1, 0, :, 5], ks[0]) and np.array_equal(scales[1, 1, 3, :, 15], vs[2])
    assert not codes[:, 0].any() and not scales[:, 0].any()   # other layer untouched
    assert np.count_nonzero(scales[0, 1]) == 2 * Hk            # padding token not written
