"""A small serving loop on the GPU driven by the host block manager: two
requests share a prompt prefix (the second reuses the first's full blocks
and prefills only the rest), prompts are prefilled in chunks under a token
budget, then both decode a few tokens ("nano-vllm notes - Llama":
scheduler.py and model_runner.py; prefill with a cached prefix read through
block_tables).  Every attention row is checked against the oracle run from
scratch on the whole sequence with no sharing and no chunking.

Activations stand in for a model: the pre-RoPE q/k/v of a token are drawn
from a generator seeded by (token id, position), so equal prefixes give equal
K/V, as a real model's would."""

import math

import numpy as np
import pytest
import torch

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from tests.gpu_helpers import assert_attention_close

pytestmark = pytest.mark.gpu

H, HK, D, BS = 8, 2, 128, 16


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    assert pa.check_device() == pa.PA_OK
    return libpa


def act(token, pos):
    rng = np.random.default_rng([int(token), int(pos), 77])
    f = lambda *s: rng.standard_normal(s, dtype=np.float32).astype(np.float16)  # noqa: E731
    return f(H, D), f(HK, D), f(HK, D)


def oracle_rows(tokens, rows):
    """Attention of rows `rows` of the whole sequence, computed from scratch."""
    n = len(tokens)
    q, k, v = (np.stack(x) for x in zip(*(act(t, i) for i, t in enumerate(tokens))))
    pos = np.arange(n)
    qr = orc.rope_pinned(q, pos, D)
    kr = orc.rope_pinned(k, pos, D)
    nb = -(-n // BS)
    table = np.arange(nb, dtype=np.int32)[None, :]
    cache = orc.new_cache(1, nb, BS, HK, D)
    md = orc.prefill_metadata([0], [n], table, BS)
    orc.kv_write(cache, 0, kr, v, md["slot_mapping"])
    out = orc.attention_prefill(qr, cache, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], table,
                                H, HK, 1.0 / math.sqrt(D))
    return out[rows]


class Engine:
    def __init__(self, num_blocks):
        self.bm = pa.BlockManager(num_blocks, BS)
        self.cache = pa.Cache(1, num_blocks, HK, D)
        self.cache.tensor.fill_(float("nan"))  # nothing may read a slot never written
        self.table = pa.rope_table(4096, D)
        self.status = pa.new_status()
        self.tokens = {}

    def tables(self, sids):
        ts = [self.bm.block_table(s) for s in sids]
        bt = np.full((len(sids), max(len(t) for t in ts)), -1, np.int32)
        for i, t in enumerate(ts):
            bt[i, :len(t)] = t
        return bt

    def prefill(self, chunks):
        """chunks: [(sid, num_cached, num_new)] -> {sid: output rows}."""
        sids = [c[0] for c in chunks]
        cached = np.array([c[1] for c in chunks], np.int64)
        new = np.array([c[2] for c in chunks], np.int64)
        bt = self.tables(sids)
        md = pa.prepare_prefill(cached, new, bt)
        acts = [act(self.tokens[s][p], p) for s, c, n in chunks for p in range(c, c + n)]
        q, k, v = (torch.from_numpy(np.stack(x)).cuda() for x in zip(*acts))
        dev = lambda x: torch.from_numpy(x).cuda()  # noqa: E731
        pa.rope_kv_write(q, k, v, dev(md["positions"]), dev(md["slot_mapping"]), self.table,
                         self.cache, status=self.status)
        out = pa.prefill_varlen(q, self.cache, dev(md["cu_seqlens_q"]), dev(md["cu_seqlens_k"]),
                                dev(bt), md["max_seqlen_q"], HK, status=self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        res, at = {}, 0
        for s, c, n in chunks:
            res[s] = out[at:at + n]
            at += n
            self.bm.mark_computed(s, n)
        return res

    def decode(self, new_tokens):
        """new_tokens: {sid: token} -> {sid: output row}."""
        sids = list(new_tokens)
        slots = []
        for s in sids:
            assert self.bm.can_append(s)
            slots.append(self.bm.append(s, new_tokens[s]))
            self.tokens[s].append(new_tokens[s])
        cached = np.array([len(self.tokens[s]) - 1 for s in sids], np.int64)
        bt = self.tables(sids)
        md = pa.prepare_decode(cached, bt)
        assert md["slot_mapping"].tolist() == slots
        acts = [act(new_tokens[s], len(self.tokens[s]) - 1) for s in sids]
        q, k, v = (torch.from_numpy(np.stack(x)).cuda() for x in zip(*acts))
        dev = lambda x: torch.from_numpy(x).cuda()  # noqa: E731
        ws = pa.decode_workspace(len(sids), H, HK, D)
        out = pa.decode_step(q, k, v, dev(md["positions"]), dev(md["slot_mapping"]), self.table,
                             self.cache, dev(bt), dev(md["context_lens"]), ws, HK,
                             status=self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        return {s: out[i:i + 1] for i, s in enumerate(sids)}


def test_prefix_shared_chunked_prefill_then_decode():
    rng = np.random.default_rng(5)
    eng = Engine(64)
    a = rng.integers(0, 32000, size=150).tolist()
    b = a[:128] + rng.integers(0, 32000, size=30).tolist()
    eng.tokens = {1: list(a), 2: list(b)}
    assert eng.bm.allocate(1, a) == 0
    # B is admitted after A's prefill is under way; its first 8 blocks match
    budget = 64
    c, n = eng.bm.next_chunk(1, budget)
    outs = eng.prefill([(1, c, n)])
    got = {1: [outs[1]], 2: []}
    assert eng.bm.allocate(2, b) == 128
    assert np.array_equal(eng.bm.block_table(1)[:8], eng.bm.block_table(2)[:8])
    while True:
        chunks, left = [], budget
        for s in (1, 2):
            c, n = eng.bm.next_chunk(s, max(left, 1))
            n = min(n, left)
            if n > 0:
                chunks.append((s, c, n))
                left -= n
        if not chunks:
            break
        outs = eng.prefill(chunks)
        for s in outs:
            got[s].append(outs[s])
    # B computed only its 30 own tokens
    assert sum(x.shape[0] for x in got[2]) == 30
    assert_attention_close(torch.cat(got[1]), oracle_rows(a, slice(0, 150)))
    assert_attention_close(torch.cat(got[2]), oracle_rows(b, slice(128, 158)))
    for step in range(5):
        toks = {1: int(rng.integers(0, 32000)), 2: int(rng.integers(0, 32000))}
        outs = eng.decode(toks)
        for s in (1, 2):
            seq = eng.tokens[s]
            assert_attention_close(outs[s], oracle_rows(seq, slice(len(seq) - 1, len(seq))))
    eng.bm.free(1)
    eng.bm.free(2)
    assert eng.bm.num_free() == 64
