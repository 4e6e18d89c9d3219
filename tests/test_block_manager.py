"""Host block manager (include/pa_block_manager.h), no GPU needed: block
ownership and reference counts, prefix-cache reuse of full blocks matched by
a chained hash ("nano-vllm notes - Llama", scheduler.py: the BlockManager
reports how many blocks a prefix-cache hit lets a request reuse, those
tokens are not prefilled again; a finished or preempted request returns its
blocks), decode appends, chunked-prefill progress, and a random sequence of
operations replayed against a small Python model of the same rules."""

import numpy as np
import pytest

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa

BS = 16


@pytest.fixture(autouse=True)
def _lib(libpa):
    return libpa


def toks(n, seed):
    return np.random.default_rng(seed).integers(0, 32000, size=n).astype(np.int32)


def test_fresh_prompt_takes_new_blocks():
    bm = pa.BlockManager(10)
    assert bm.num_free() == 10
    assert bm.allocate(1, toks(40, 1)) == 0
    t = bm.block_table(1)
    assert len(t) == 3 and len(set(t.tolist())) == 3
    assert bm.num_free() == 7
    assert bm.num_tokens(1) == 40
    assert bm.blocks_needed(40) == 3


def test_prefix_hit_shares_full_blocks_only():
    bm = pa.BlockManager(20)
    a = toks(40, 2)
    assert bm.allocate(1, a) == 0
    b = np.concatenate([a[:32], toks(9, 3)])  # same two full blocks, new tail
    assert bm.allocate(2, b) == 32             # prefill starts at token 32
    ta, tb = bm.block_table(1), bm.block_table(2)
    assert np.array_equal(ta[:2], tb[:2]) and ta[2] != tb[2]
    assert bm.num_free() == 20 - 3 - 1
    # a partial block is never shared, even with equal tokens
    c = a[:40].copy()
    assert bm.allocate(3, c) == 32
    assert bm.block_table(3)[2] not in (ta[2], tb[2])


def test_a_block_matches_only_with_its_whole_prefix():
    bm = pa.BlockManager(20)
    a = toks(48, 4)
    bm.allocate(1, a)
    b = np.concatenate([toks(16, 5), a[16:48]])  # blocks 1, 2 equal, block 0 not
    assert bm.allocate(2, b) == 0
    assert len(set(bm.block_table(1).tolist()) & set(bm.block_table(2).tolist())) == 0


def test_fully_cached_prompt_recomputes_its_last_token():
    bm = pa.BlockManager(8)
    a = toks(32, 6)
    bm.allocate(1, a)
    assert bm.allocate(2, a) == 31
    assert np.array_equal(bm.block_table(1), bm.block_table(2))
    assert bm.num_free() == 6


def test_freed_blocks_stay_matchable_until_reused():
    bm = pa.BlockManager(6)
    a = toks(48, 7)
    bm.allocate(1, a)
    ta = bm.block_table(1).copy()
    bm.free(1)
    assert bm.num_free() == 6
    assert bm.allocate(2, np.concatenate([a[:32], toks(5, 8)])) == 32
    assert np.array_equal(bm.block_table(2)[:2], ta[:2])
    bm.free(2)
    # fill the pool with unrelated prompts: the old blocks are handed out anew
    bm.allocate(3, toks(96, 9))
    bm.free(3)
    assert bm.allocate(4, a) == 0


def test_out_of_blocks_changes_nothing():
    bm = pa.BlockManager(4)
    bm.allocate(1, toks(40, 10))
    with pytest.raises(pa.PAError) as e:
        bm.allocate(2, toks(40, 11))
    assert e.value.code == pa.PA_ERR_WORKSPACE
    assert bm.num_free() == 1 and bm.num_tokens(2) == -1
    with pytest.raises(pa.PAError):
        bm.allocate(1, toks(5, 12))  # duplicate id


def test_decode_appends_fill_blocks_and_register_them():
    bm = pa.BlockManager(8)
    a = toks(20, 13)
    bm.allocate(1, a)
    bm.mark_computed(1, 20)
    t0 = bm.block_table(1)
    extra = toks(13, 14)
    slots = [bm.append(1, int(x)) for x in extra]
    assert slots[:12] == [int(t0[1]) * BS + o for o in range(4, 16)]
    t1 = bm.block_table(1)
    assert len(t1) == 3 and slots[12] == int(t1[2]) * BS
    # the block filled by decode now matches a prompt with the same 32 tokens
    full = np.concatenate([a, extra])[:32]
    assert bm.allocate(2, np.concatenate([full, toks(3, 15)])) == 32
    assert np.array_equal(bm.block_table(2)[:2], t1[:2])


def test_chunked_prefill_progress():
    bm = pa.BlockManager(64)
    a = toks(300, 16)
    assert bm.allocate(1, a) == 0
    done = []
    while True:
        c, n = bm.next_chunk(1, 128)
        if n == 0:
            break
        done.append((c, n))
        with pytest.raises(pa.PAError):
            bm.append(1, 5)  # not before the prompt is computed
        bm.mark_computed(1, n)
    assert done == [(0, 128), (128, 128), (256, 44)]
    assert bm.can_append(1)
    bm.append(1, 7)
    with pytest.raises(pa.PAError):
        bm.mark_computed(1, 1)  # nothing left to compute


def test_can_append_needs_a_free_block_only_at_a_block_boundary():
    bm = pa.BlockManager(2)
    bm.allocate(1, toks(17, 17))
    bm.mark_computed(1, 17)
    assert bm.can_append(1)
    for _ in range(15):
        bm.append(1, 1)
    assert bm.num_tokens(1) == 32 and bm.num_free() == 0
    assert not bm.can_append(1)
    with pytest.raises(pa.PAError):
        bm.append(1, 1)


def test_tables_feed_the_metadata_builders():
    """slot_mapping built from the manager's tables places every new token in
    its own block, as the oracle's metadata builder does."""
    bm = pa.BlockManager(40)
    a = toks(70, 18)
    bm.allocate(1, a)
    c2 = bm.allocate(2, np.concatenate([a[:64], toks(10, 19)]))
    cached = np.array([0, c2], np.int64)
    new = np.array([70, 74 - c2], np.int64)
    tables = [bm.block_table(1), bm.block_table(2)]
    width = max(len(t) for t in tables)
    bt = np.full((2, width), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    got = pa.prepare_prefill(cached, new, bt)
    want = orc.prefill_metadata(cached, new, bt, BS)
    assert np.array_equal(got["slot_mapping"], want["slot_mapping"])
    assert np.array_equal(got["positions"], want["positions"])


class Model:
    """The manager's rules restated in Python (test infrastructure)."""

    def __init__(self, nb):
        self.free = list(range(nb))          # oldest-freed first
        self.ref = [0] * nb
        self.key = {}                         # block -> full-token prefix tuple
        self.by_key = {}                      # full-token prefix tuple -> block
        self.seqs = {}

    def _take(self):
        b = self.free.pop(0)
        k = self.key.pop(b, None)
        if k is not None and self.by_key.get(k) == b:
            del self.by_key[k]
        self.ref[b] = 1
        return b

    def _register(self, b, k):
        if k not in self.by_key:
            self.by_key[k] = b
            self.key[b] = k

    def allocate(self, sid, t):
        n, full = len(t), len(t) // BS
        hits = []
        for i in range(full):
            b = self.by_key.get(tuple(t[:(i + 1) * BS]))
            if b is None:
                break
            hits.append(b)
        need = -(-n // BS)
        if need - len(hits) + sum(self.ref[b] == 0 for b in hits) > len(self.free):
            return None
        blocks = []
        for b in hits:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
            blocks.append(b)
        for i in range(len(hits), need):
            b = self._take()
            blocks.append(b)
            if i < full:
                self._register(b, tuple(t[:(i + 1) * BS]))
        self.seqs[sid] = (list(t), blocks)
        return min(len(hits) * BS, n - 1)

    def append(self, sid, x):
        t, blocks = self.seqs[sid]
        if len(t) % BS == 0:
            if not self.free:
                return None
            blocks.append(self._take())
        t.append(x)
        if len(t) % BS == 0:
            self._register(blocks[-1], tuple(t))
        return blocks[(len(t) - 1) // BS] * BS + (len(t) - 1) % BS

    def release(self, sid):
        _, blocks = self.seqs.pop(sid)
        for b in reversed(blocks):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)


def test_random_operations_match_the_model():
    rng = np.random.default_rng(20)
    nb = 48
    bm, m = pa.BlockManager(nb), Model(nb)
    bases = [toks(200, 100 + i) for i in range(4)]  # shared prompt stems
    live, next_id = [], 1
    for step in range(1500):
        op = rng.random()
        if op < 0.35 or not live:
            stem = bases[rng.integers(0, 4)]
            keep = int(rng.integers(0, 200))
            t = np.concatenate([stem[:keep], toks(int(rng.integers(1, 40)), 1000 + step)])
            want = m.allocate(next_id, t.tolist())
            if want is None:
                with pytest.raises(pa.PAError):
                    bm.allocate(next_id, t)
            else:
                assert bm.allocate(next_id, t) == want, step
                bm.mark_computed(next_id, len(t) - want)
                live.append(next_id)
            next_id += 1
        elif op < 0.8:
            sid = live[int(rng.integers(0, len(live)))]
            x = int(rng.integers(0, 32000))
            want = m.append(sid, x)
            if want is None:
                assert not bm.can_append(sid)
                with pytest.raises(pa.PAError):
                    bm.append(sid, x)
            else:
                assert bm.append(sid, x) == want, step
        else:
            sid = live.pop(int(rng.integers(0, len(live))))
            m.release(sid)
            bm.free(sid)
        assert bm.num_free() == len(m.free), step
    for sid in live:
        assert bm.block_table(sid).tolist() == m.seqs[sid][1]


def test_create_refuses_pools_past_int32_slots(libpa):
    with pytest.raises(ValueError):
        pa.BlockManager(2**27, 16)  # 2^31 slots: their count is past INT32_MAX
    with pytest.raises(ValueError):
        pa.BlockManager(0, 16)


def test_mark_computed_rejects_overflowing_counts(libpa):
    bm = pa.BlockManager(8, 16)
    bm.allocate(1, list(range(20)))
    with pytest.raises(pa.PAError):
        bm.mark_computed(1, 2**31 - 1)
    bm.mark_computed(1, 20)
