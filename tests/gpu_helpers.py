"""Shared set-up of the GPU parity tests: run a workload through the C ABI
and through the oracle on the same seeded inputs."""

import math

import numpy as np
import torch

from oracle import reference as orc
from paged_kv_gqa_rope_gb300 import pa
from paged_kv_gqa_rope_gb300 import workloads as W

# Tolerance of attention outputs against the fp64 oracle: max-abs 3e-3 and
# relative L2 1e-3.  The output is stored in fp16, so no result can be closer
# to the exact value than half an fp16 ulp of it (7.8e-3 for outputs in
# [16, 32), which the 8-sigma V outliers of the ragged workload produce); the
# max-abs bound therefore applies to the error beyond that rounding.
MAX_ABS = 3e-3
REL_L2 = 1e-3


def half_ulp16(x):
    a = np.abs(x).astype(np.float16)
    return 0.5 * np.spacing(a).astype(np.float64)


def assert_attention_close(got16, want64, rows=None):
    got = got16.float().cpu().numpy().astype(np.float64) if isinstance(got16, torch.Tensor) else got16
    if rows is not None:
        got, want64 = got[rows], want64[rows]
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - want64)
    beyond = float(np.max(err - half_ulp16(want64)))
    rel = float(np.linalg.norm(got - want64) / max(np.linalg.norm(want64), 1e-30))
    assert beyond <= MAX_ABS and rel <= REL_L2, \
        f"max_abs={float(err.max()):.3e} beyond_fp16_rounding={beyond:.3e} rel_l2={rel:.3e}"
    return float(err.max()), rel


def bits(x):
    a = x.cpu().numpy() if isinstance(x, torch.Tensor) else x
    return a.view(np.uint16)


class DecodeRun:
    """One decode step (RoPE + append + decode) of a workload on the GPU,
    plus the oracle's view of the same step."""

    def __init__(self, case: W.Case, init_cache: np.ndarray, table_rows=None):
        wl = case.wl
        self.case, self.wl = case, wl
        md = pa.prepare_decode(case.num_cached, case.block_tables)
        self.md = md
        max_pos = int(md["positions"].max()) + 1 if table_rows is None else table_rows
        self.table = pa.rope_table(max_pos, wl.head_dim, wl.rope_theta)
        self.cache = pa.Cache(1, case.num_blocks, wl.n_kv_heads, wl.head_dim)
        self.cache.tensor.copy_(torch.from_numpy(init_cache))
        dev = "cuda"
        self.q = torch.from_numpy(case.q).to(dev)
        self.k = torch.from_numpy(case.k).to(dev)
        self.v = torch.from_numpy(case.v).to(dev)
        self.positions = torch.from_numpy(md["positions"]).to(dev)
        self.slots = torch.from_numpy(md["slot_mapping"]).to(dev)
        self.ctx = torch.from_numpy(md["context_lens"]).to(dev)
        self.bt = torch.from_numpy(case.block_tables).to(dev)
        self.ws = pa.decode_workspace(len(case.num_cached), wl.n_heads, wl.n_kv_heads,
                                      wl.head_dim)
        self.status = pa.new_status()

    def run(self):
        wl = self.wl
        pa.rope_kv_write(self.q, self.k, self.v, self.positions, self.slots, self.table,
                         self.cache, status=self.status)
        out = pa.decode(self.q, self.cache, self.bt, self.ctx, self.ws, wl.n_kv_heads,
                        status=self.status)
        torch.cuda.synchronize()
        return out


def oracle_decode_step(case: W.Case, init_cache: np.ndarray, seqs=None):
    """Oracle: rotate, append, attend.  Returns (q_rot, k_rot, cache, out)."""
    wl = case.wl
    md = orc.decode_metadata(case.num_cached, case.block_tables, wl.block_size)
    q_rot = orc.rope_pinned(case.q, md["positions"], wl.head_dim, wl.rope_theta)
    k_rot = orc.rope_pinned(case.k, md["positions"], wl.head_dim, wl.rope_theta)
    cache = init_cache.copy()
    orc.kv_write(cache, 0, k_rot, case.v, md["slot_mapping"])
    out = orc.attention_decode(q_rot, cache, 0, case.block_tables, md["context_lens"],
                               wl.n_heads, wl.n_kv_heads, 1.0 / math.sqrt(wl.head_dim), seqs=seqs)
    return q_rot, k_rot, cache, out
