"""CPU oracle for the paged-KV / GQA / RoPE attention hot path.

TEST INFRASTRUCTURE ONLY.  This module is imported by the tests, by the
smoke check and by the CPU-baseline leg of the benchmark, never by the
product path.  It shares no code with the CUDA library: it restates, in plain
numpy (float64 for the attention arithmetic), what the pages define:

* "nano-vllm notes - Llama", sections prepare_prefill / prepare_decode:
  the flattened token stream, positions, cu_seqlens_q/k, slot_mapping,
  block_tables, context_lens (the worked examples 3,5,2 -> [0,3,8,10];
  prompts of 5 and 3 -> positions [0,1,2,3,4,0,1,2]; decode positions [5,3]
  with context_lens [6,4]).
* "nano-vllm notes - Llama", section allocate_kv_cache: the pool
  [2, layers, blocks, block_size, n_kv_heads, head_dim].
* "Meta Llama source deep-dive", section 3.3 (precompute_freqs_cis,
  apply_rotary_emb) and section 9 (RoPE derivation): adjacent pairs
  (x_2i, x_2i+1) rotated counter-clockwise by m * theta^(-2i/d).
* "Meta Llama source deep-dive", sections 3.4 (repeat_kv: Q head h reads KV
  head h // n_rep), 3.5 (scores = q k^T / sqrt(d), softmax, times V) and
  3.8 (causal mask with a cached prefix: zeros of width start_pos, then the
  upper triangle at -inf); "personal chatgpt 22 - llama2 generate",
  sections 2-3 (M_ij = 0 for j <= i, -inf otherwise; decode needs no mask).
* "llama2.zig", section 5.4: softmax subtracts the row maximum.

Every function here has a pin in tests/test_oracle_pins.py (worked examples,
closed forms, invariants, brute force against a library routine).

Pinned rounding of the RoPE step (the pages compute it in fp32 and store the
result back in the input dtype, "type_as"; they do not fix the order of the
fp32 operations, so this module fixes one and the CUDA path must match it bit
for bit):
  angle  = m * inv_freq_i           in float64, inv_freq_i = 1 / theta**(2i/d)
  c, s   = cos(angle), sin(angle)   in float64, each rounded once to float32
  x'     = fl32(fl32(x*c) - fl32(y*s))
  y'     = fl32(fl32(x*s) + fl32(y*c))          (no fused multiply-add)
  stored = round-to-nearest-even float16 of x', y'
"""

from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# Step a0: metadata of the flattened token stream
# ---------------------------------------------------------------------------

def cu_seqlens(lengths) -> np.ndarray:
    """Cumulative sequence lengths starting at 0 ("nano-vllm notes - Llama",
    prepare_prefill: cu_seqlens_q.append(cu_seqlens_q[-1] + seqlen_q))."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return np.asarray(out, dtype=np.int32)


def prefill_metadata(num_cached, num_new, block_tables, block_size):
    """Metadata for one prefill call ("nano-vllm notes - Llama",
    prepare_prefill).  For sequence s with `start` tokens cached and
    `seqlen_q` new ones: end = start + seqlen_q, seqlen_k = end, the new
    tokens sit at positions start..end-1, and each one is written to the slot
    block_table[s][pos // block_size] * block_size + pos % block_size.

    Returns dict(positions, cu_seqlens_q, cu_seqlens_k, slot_mapping,
    max_seqlen_q, max_seqlen_k)."""
    positions, slots, lq, lk = [], [], [], []
    for s in range(len(num_new)):
        start = int(num_cached[s])
        end = start + int(num_new[s])
        lq.append(end - start)
        lk.append(end)
        for pos in range(start, end):
            positions.append(pos)
            blk = int(block_tables[s][pos // block_size])
            slots.append(blk * block_size + pos % block_size)
    return dict(
        positions=np.asarray(positions, np.int32),
        cu_seqlens_q=cu_seqlens(lq),
        cu_seqlens_k=cu_seqlens(lk),
        slot_mapping=np.asarray(slots, np.int32),
        max_seqlen_q=max(lq) if lq else 0,
        max_seqlen_k=max(lk) if lk else 0,
    )


def decode_metadata(num_cached, block_tables, block_size):
    """Metadata for one decode step ("nano-vllm notes - Llama",
    prepare_decode): each sequence feeds its last token, at position
    num_cached[s]; after its K/V is appended the sequence holds
    context_lens[s] = num_cached[s] + 1 tokens (the page's example: positions
    [5,3], context_lens [6,4])."""
    positions, slots, ctx = [], [], []
    for s in range(len(num_cached)):
        pos = int(num_cached[s])
        positions.append(pos)
        ctx.append(pos + 1)
        blk = int(block_tables[s][pos // block_size])
        slots.append(blk * block_size + pos % block_size)
    return dict(
        positions=np.asarray(positions, np.int32),
        slot_mapping=np.asarray(slots, np.int32),
        context_lens=np.asarray(ctx, np.int32),
    )


# ---------------------------------------------------------------------------
# Step a1: rotary position embedding
# ---------------------------------------------------------------------------

def rope_inv_freq(head_dim: int, theta: float = 10000.0) -> list:
    """theta_i = 1 / theta**(2i/d) for i < d/2 ("Meta Llama source
    deep-dive", 3.3 precompute_freqs_cis; 9.2 theta_i = 10000^(-2i/d)).
    Python floats (IEEE double, C library pow)."""
    return [1.0 / (theta ** ((2 * i) / head_dim)) for i in range(head_dim // 2)]


def rope_cos_sin(position: int, head_dim: int, theta: float = 10000.0):
    """float64 angle m * theta_i, cos and sin from the C library, each rounded
    once to float32 (the pinned table entry for one position)."""
    inv = rope_inv_freq(head_dim, theta)
    c = np.empty(head_dim // 2, np.float32)
    s = np.empty(head_dim // 2, np.float32)
    for i, f in enumerate(inv):
        ang = float(position) * f
        c[i] = math.cos(ang)
        s[i] = math.sin(ang)
    return c, s


def rope_pinned(x16: np.ndarray, positions, head_dim: int, theta: float = 10000.0) -> np.ndarray:
    """Rotate each adjacent pair (x_2i, x_2i+1) of every head of token t by
    positions[t] * theta_i with the pinned float32 arithmetic of the module
    docstring; returns float16 of the same shape [T, n_heads, d]."""
    x16 = np.asarray(x16, np.float16)
    out = np.empty_like(x16)
    cache = {}
    for t in range(x16.shape[0]):
        m = int(positions[t])
        if m not in cache:
            cache[m] = rope_cos_sin(m, head_dim, theta)
        c, s = cache[m]
        xe = x16[t, :, 0::2].astype(np.float32)
        xo = x16[t, :, 1::2].astype(np.float32)
        re = (xe * c) - (xo * s)          # each op rounds to float32
        im = (xe * s) + (xo * c)
        out[t, :, 0::2] = re.astype(np.float16)
        out[t, :, 1::2] = im.astype(np.float16)
    return out


def rope_exact(x, positions, head_dim: int, theta: float = 10000.0) -> np.ndarray:
    """The same rotation entirely in float64, no rounding of the result:
    (x + i y) * e^{i m theta_i} ("Meta Llama source deep-dive", 9.3)."""
    x = np.asarray(x, np.float64)
    inv = np.asarray(rope_inv_freq(head_dim, theta), np.float64)
    out = np.empty_like(x)
    for t in range(x.shape[0]):
        ang = float(positions[t]) * inv
        c, s = np.cos(ang), np.sin(ang)
        xe, xo = x[t, :, 0::2], x[t, :, 1::2]
        out[t, :, 0::2] = xe * c - xo * s
        out[t, :, 1::2] = xe * s + xo * c
    return out


# ---------------------------------------------------------------------------
# Step a2: K/V write into the paged cache
# ---------------------------------------------------------------------------

def new_cache(layers, num_blocks, block_size, n_kv_heads, head_dim) -> np.ndarray:
    """The pool of "nano-vllm notes - Llama", allocate_kv_cache:
    [2, layers, num_blocks, block_size, n_kv_heads, head_dim] float16."""
    return np.zeros((2, layers, num_blocks, block_size, n_kv_heads, head_dim), np.float16)


def kv_write(cache: np.ndarray, layer: int, k16, v16, slot_mapping) -> None:
    """Store token t's K and V at physical slot slot_mapping[t]: block
    slot // block_size, row slot % block_size.  A negative slot means "no
    write" (a padding token).  In place, bit for bit."""
    bs = cache.shape[3]
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        cache[0, layer, slot // bs, slot % bs] = k16[t]
        cache[1, layer, slot // bs, slot % bs] = v16[t]


def gather_kv(cache: np.ndarray, layer: int, table_row, n_tokens: int):
    """Logical tokens 0..n_tokens-1 of one sequence, read through its block
    table: K, V float64 [n_tokens, n_kv_heads, d]."""
    bs = cache.shape[3]
    K = np.empty((n_tokens,) + cache.shape[4:], np.float64)
    V = np.empty_like(K)
    for lb in range((n_tokens + bs - 1) // bs):      # logical block lb
        blk = int(table_row[lb])
        rows = min(bs, n_tokens - lb * bs)
        K[lb * bs:lb * bs + rows] = cache[0, layer, blk, :rows]
        V[lb * bs:lb * bs + rows] = cache[1, layer, blk, :rows]
    return K, V


# ---------------------------------------------------------------------------
# Steps a3 / a4: attention
# ---------------------------------------------------------------------------

def _softmax_rows(scores: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted first ("llama2.zig" 5.4).
    Entries at -inf get weight 0."""
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / e.sum(axis=-1, keepdims=True)


def attention_prefill(q16, cache, layer, cu_seqlens_q, cu_seqlens_k, block_tables,
                      n_heads, n_kv_heads, scale=None, seqs=None) -> np.ndarray:
    """Varlen causal attention over a flattened stream.

    Sequence s owns query rows cu_seqlens_q[s]..cu_seqlens_q[s+1]-1 and has
    seqlen_k = cu_seqlens_k[s+1]-cu_seqlens_k[s] keys, of which the first
    p = seqlen_k - seqlen_q are a cached prefix.  Query row i sits at
    absolute position p + i and sees keys j <= p + i: the prefix block of
    zeros followed by the causal triangle ("Meta Llama source deep-dive",
    3.8; M_ij of "personal chatgpt 22", section 2).  Q head h uses KV head
    h // (n_heads / n_kv_heads) (repeat_kv, 3.4).  scores = q.k * scale with
    scale = 1/sqrt(d) by default, softmax, times V (3.5).  float64.

    q16: [T, n_heads, d] (already rotated).  Returns float64 [T, n_heads, d];
    rows of sequences not in `seqs` (when given) are left NaN."""
    T, H, d = q16.shape
    assert H == n_heads and n_heads % n_kv_heads == 0
    g = n_heads // n_kv_heads
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.full((T, H, d), np.nan)
    B = len(cu_seqlens_q) - 1
    for s in (range(B) if seqs is None else seqs):
        q0, q1 = int(cu_seqlens_q[s]), int(cu_seqlens_q[s + 1])
        lq = q1 - q0
        lk = int(cu_seqlens_k[s + 1]) - int(cu_seqlens_k[s])
        if lq == 0:
            continue
        p = lk - lq
        K, V = gather_kv(cache, layer, block_tables[s], lk)
        i = np.arange(lq)[:, None]
        j = np.arange(lk)[None, :]
        mask = np.where(j <= p + i, 0.0, -np.inf)
        Q = q16[q0:q1].astype(np.float64)
        for h in range(H):
            kv = h // g
            scores = (Q[:, h, :] @ K[:, kv, :].T) * scale + mask
            out[q0:q1, h, :] = _softmax_rows(scores) @ V[:, kv, :]
    return out


def attention_decode(q16, cache, layer, block_tables, context_lens,
                     n_heads, n_kv_heads, scale=None, seqs=None) -> np.ndarray:
    """Single-token decode: the query of sequence s (at position
    context_lens[s]-1, its K/V already appended) attends to all
    context_lens[s] cached keys; no mask is needed because every cached key
    is in its past ("personal chatgpt 22", section 3; "Meta Llama source
    deep-dive", 3.8 decode branch).  Written out per head as a plain weighted
    sum, independently of attention_prefill.

    q16: [B, n_heads, d].  Returns float64 [B, n_heads, d] (NaN rows for
    sequences not in `seqs`)."""
    B, H, d = q16.shape
    g = n_heads // n_kv_heads
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.full((B, H, d), np.nan)
    for s in (range(B) if seqs is None else seqs):
        n = int(context_lens[s])
        K, V = gather_kv(cache, layer, block_tables[s], n)
        for h in range(H):
            kv = h // g
            qv = q16[s, h].astype(np.float64)
            sc = (K[:, kv, :] @ qv) * scale          # [n]
            w = np.exp(sc - sc.max())
            out[s, h] = (w @ V[:, kv, :]) / w.sum()
    return out


# ---------------------------------------------------------------------------
# NEXT-4: int8 KV cache ("Meta Llama source deep-dive", 8.4: a quantised KV
# cache stored as int8 saves memory; the page gives no scheme, so this is
# the reading the CUDA path also follows)
# ---------------------------------------------------------------------------
#
# Each (token, KV head) row x of head_dim fp16 values (K after the pinned
# RoPE, V as given) is stored as int8 codes and one float32 scale:
#   amax  = max_i |x_i|                       (exact in float32)
#   scale = fl32(amax / 127)                  (0 when amax is 0)
#   q_i   = clamp(rint(fl32(x_i / scale)), -127, 127)   rint: ties to even
# and read back as q_i * scale.  Layout: codes [2, layers, blocks,
# block_size, n_kv_heads, head_dim] int8; scales [2, layers, blocks,
# n_kv_heads, block_size] float32 (a block's 16 scales of one head are
# contiguous).

def kv_quantize_int8(x16):
    """Rows of the last axis -> (codes int8, scales float32 [...])."""
    x = np.asarray(x16, np.float16).astype(np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    r = np.rint((x / safe[..., None]).astype(np.float32))
    codes = np.clip(r, -127, 127).astype(np.int8)
    codes[scale == 0] = 0
    return codes, scale


def new_cache_i8(layers, num_blocks, block_size, n_kv_heads, head_dim):
    codes = np.zeros((2, layers, num_blocks, block_size, n_kv_heads, head_dim), np.int8)
    scales = np.zeros((2, layers, num_blocks, n_kv_heads, block_size), np.float32)
    return codes, scales


def kv_write_i8(codes, scales, layer: int, k16, v16, slot_mapping) -> None:
    """Quantise token t's K and V rows and store them at slot
    slot_mapping[t] (negative: no write)."""
    bs = codes.shape[3]
    kq, ks = kv_quantize_int8(k16)
    vq, vs = kv_quantize_int8(v16)
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        b, r = slot // bs, slot % bs
        codes[0, layer, b, r], codes[1, layer, b, r] = kq[t], vq[t]
        scales[0, layer, b, :, r], scales[1, layer, b, :, r] = ks[t], vs[t]


def dequantize_cache_i8(codes, scales) -> np.ndarray:
    """The float64 cache the int8 one stands for: q * scale."""
    s = np.swapaxes(scales, -1, -2)[..., None].astype(np.float64)  # [..., bs, Hk, 1]
    return codes.astype(np.float64) * s


def attention_decode_i8(q16, codes, scales, layer, block_tables, context_lens,
                        n_heads, n_kv_heads, scale=None, seqs=None) -> np.ndarray:
    """Decode against the int8 cache: the decode formula on the values the
    codes and scales stand for."""
    return attention_decode(q16, dequantize_cache_i8(codes, scales), layer, block_tables,
                            context_lens, n_heads, n_kv_heads, scale=scale, seqs=seqs)
