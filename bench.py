"""Benchmark of the paged-KV GQA attention hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-extra] [--int8]

A step is one pass of the hot path over one batch of synthetic input.  For a
decode workload: RoPE of the new tokens' Q/K + append of their K/V through
slot_mapping (pa_rope_kv_write) and decode attention of every sequence
against its whole cache (pa_decode), as the one call pa_decode_step (the two
kernels chained by programmatic dependent launch).  For the prefill
workload: RoPE + append of the new tokens and varlen causal prefill reading
the cached prefix through block_tables (pa_prefill_varlen), as the one call
pa_prefill_step.  The int8 cache has no one-call step: its steps are the two
calls.

The headline workload is the Llama-2-70B-shaped GQA decode (64 Q heads over
8 KV heads, d=128, batch 32, 4096 cached tokens + 1); its metric is decode
throughput in GB/s of KV bytes read (sum of context lengths x n_kv_heads x
head_dim x 2 (K, V) x 2 B).  The line also carries the other workloads (MHA
decode, ragged GQA decode, prefill in TFLOP/s, the int8 cache; for fp16
decode also the graph-captured step, and for every workload the RoPE/append
kernel's own time and bandwidth) under "per_workload" unless --no-extra; the
ragged GQA decode there is instrumented like the headline (roofline with
ncu traffic, e2e, cpu_baseline).

Timing: W untimed warm-up steps, then exactly K steps between a barrier +
synchronize on each side, CUDA events on the launching stream; the KV bytes
a step reads (0.54 to 5.0 GB; 0.28 GB and up for the int8 cache) are larger
than the 129 MB L2 (inputs larger than L2; no flush between steps).  The
line gives the mean and the median step time.  Per-kernel durations (the
dominant kernel against its roofline, the RoPE/append kernel's bandwidth)
come from a second timed loop of the same K steps made of the two separate
calls with events around each kernel.  `e2e` repeats the step through the
library's calls with the step's inputs copied from pinned host memory (one
copy of a buffer that holds them all) and the output copied back inside the
timed region; for fp16 decode the step runs as the captured step graph with
both copies inside it (pa_step_graph_create_io), as a serving loop would
replay it: one launch per step.

    --int8   decode workloads: the int8 KV cache path (pa_rope_kv_write_i8 +
             pa_decode_i8) as the timed step.

--impl reference times the CPU oracle (the only implementation the source
pages define) on a bounded sample of the same workload.  Under torchrun with
N > 1 every rank runs the same workload on its own GPU (replicas; the path
has no exchange step) and rank 0 prints one line with the max over ranks.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_gqa_rope_gb300 import workloads as W  # noqa: E402

HEADLINE = "gqa_decode_70b"
METRIC = "paged GQA decode KV GB/s (% of HBM peak); prefill attention TFLOP/s (% peak)"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- work units

def kv_bytes(case) -> int:
    wl = case.wl
    ctx = case.num_cached.astype(np.int64) + 1
    return int(ctx.sum()) * wl.n_kv_heads * wl.head_dim * 2 * 2


def kv_bytes_i8(case) -> int:
    """Bytes an int8-cache decode step reads: K and V codes plus one float32
    scale per (token, KV head) for each."""
    wl = case.wl
    ctx = case.num_cached.astype(np.int64) + 1
    return int(ctx.sum()) * wl.n_kv_heads * (wl.head_dim + 4) * 2


def rope_bytes(case) -> int:
    """Algorithmic bytes of pa_rope_kv_write: Q, K, V of the new tokens read;
    rotated Q and K written back in place; K and V written into the pool
    (the cos/sin table rows are not counted)."""
    wl = case.wl
    T, H, Hk, d = case.total_new, wl.n_heads, wl.n_kv_heads, wl.head_dim
    return T * (H + 2 * Hk) * d * 2 + T * (H + 3 * Hk) * d * 2


def rope_bytes_i8(case) -> int:
    """pa_rope_kv_write_i8: the same reads and in-place writes; K and V go
    into the pool as int8 codes plus one fp32 scale per (token, KV head)."""
    wl = case.wl
    T, H, Hk, d = case.total_new, wl.n_heads, wl.n_kv_heads, wl.head_dim
    return T * (H + 2 * Hk) * d * 2 + T * (H + Hk) * d * 2 + 2 * T * Hk * (d + 4)


def prefill_flops(case) -> int:
    wl = case.wl
    tot = 0
    for p, n in zip(case.num_cached.tolist(), case.num_new.tolist()):
        tot += n * (p + 1) + n * (n - 1) // 2
    return 4 * wl.head_dim * wl.n_heads * tot


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.err = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception as e:  # nvidia-smi missing
            self.err = str(e)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.err or not self.lines:
            return {"error": self.err or "no samples"}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"error": "unparsed samples"}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

class PackedInputs:
    """A step's host inputs laid out in one buffer (each array at a 256-byte
    aligned offset): one pinned host copy, one device copy, and device views
    that the library calls take.  An end-to-end step then moves its inputs
    with a single host-to-device copy."""

    def __init__(self, host, dev):
        import torch
        self.layout, off = {}, 0
        arrays = {k: np.ascontiguousarray(v) for k, v in host.items()}
        for k, a in arrays.items():
            self.layout[k] = (off, a)
            off = (off + a.nbytes + 255) // 256 * 256
        self.nbytes = off
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        hv = self.host.numpy()
        for k, (o, a) in self.layout.items():
            hv[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
        self.device = self.host.to(dev)
        self.views = {}
        for k, (o, a) in self.layout.items():
            t = torch.from_numpy(a)
            self.views[k] = self.device[o:o + a.nbytes].view(t.dtype).view(t.shape)

    def upload(self):
        self.device.copy_(self.host, non_blocking=True)


class DecodeBench:
    rope_kernel = "rope_kv_write_kernel"

    def __init__(self, name, dev, int8=False, batch=None):
        import torch
        from paged_kv_gqa_rope_gb300 import pa
        self.pa, self.torch = pa, torch
        case = W.make_case(name, batch=batch)
        self.case = case
        wl = case.wl
        md = pa.prepare_decode(case.num_cached, case.block_tables)
        self.md = md
        self.table = pa.rope_table(int(md["positions"].max()) + 1, wl.head_dim, wl.rope_theta)
        if not int8:
            self.cache = pa.Cache(1, case.num_blocks, wl.n_kv_heads, wl.head_dim, device=dev)
            self.cache.tensor.copy_(torch.from_numpy(W.initial_cache(case)))
        self.host = dict(q=case.q, k=case.k, v=case.v, positions=md["positions"],
                         slots=md["slot_mapping"], bt=case.block_tables, ctx=md["context_lens"])
        self.packed = PackedInputs(self.host, dev)
        self.d = self.packed.views
        self.ws = pa.decode_workspace(len(case.num_cached), wl.n_heads, wl.n_kv_heads,
                                      wl.head_dim, device=dev)
        self.out = torch.empty_like(self.d["q"])
        self.status = pa.new_status(dev)
        self.units = kv_bytes(case)
        self.unit = "GB/s"
        self.rope_units = rope_bytes(case)
        self.launches_per_step = 2

    def step(self, ev=None):
        """One step; `ev` = three CUDA events recorded before the RoPE/append
        kernel, between it and the attention kernel, and after that."""
        pa, d, wl = self.pa, self.d, self.case.wl
        if ev is not None:
            ev[0].record()
        pa.rope_kv_write(d["q"], d["k"], d["v"], d["positions"], d["slots"], self.table,
                         self.cache, status=self.status)
        if ev is not None:
            ev[1].record()
        pa.decode(d["q"], self.cache, d["bt"], d["ctx"], self.ws, wl.n_kv_heads, out=self.out,
                  status=self.status)
        if ev is not None:
            ev[2].record()

    def fused_step(self):
        """The step as one call (pa_decode_step: the two kernels chained)."""
        pa, d, wl = self.pa, self.d, self.case.wl
        pa.decode_step(d["q"], d["k"], d["v"], d["positions"], d["slots"], self.table, self.cache,
                       d["bt"], d["ctx"], self.ws, wl.n_kv_heads, out=self.out, status=self.status)

    def e2e_setup(self):
        """Inputs from pinned host memory (one copy), the step, output back
        to pinned host memory.  Where there is a captured step graph, both
        copies are inside it (pa_step_graph_create_io): one replay per
        step."""
        torch = self.torch
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.e2e_graph = None
        if getattr(self, "graph_setup", None) is not None:
            pa, d, wl = self.pa, self.d, self.case.wl
            self.e2e_graph = pa.StepGraph(d["q"], d["k"], d["v"], d["positions"], d["slots"],
                                          self.table, self.cache, d["bt"], d["ctx"], self.ws,
                                          wl.n_kv_heads, out=self.out, status=self.status,
                                          host_in=self.packed.host, dev_in=self.packed.device,
                                          host_out=self.out_host)
        return self.packed.nbytes, self.out_host.numel() * self.out_host.element_size()

    def e2e_step(self):
        if self.e2e_graph is not None:
            self.e2e_graph.launch()
            return
        self.packed.upload()
        self.fused_step()
        self.out_host.copy_(self.out, non_blocking=True)

    def e2e_close(self):
        if self.e2e_graph is not None:
            self.e2e_graph.close()

    def kernel_name(self):
        return "decode_kernel"

    def graph_setup(self):
        """The same step as pa_step_graph: captured once, replayed per step."""
        pa, d, wl = self.pa, self.d, self.case.wl
        self.graph = pa.StepGraph(d["q"], d["k"], d["v"], d["positions"], d["slots"], self.table,
                                  self.cache, d["bt"], d["ctx"], self.ws, wl.n_kv_heads,
                                  out=self.out, status=self.status)

    def graph_step(self):
        self.graph.launch()


class DecodeI8Bench(DecodeBench):
    """The same decode step against the int8 cache (codes + scales)."""

    def __init__(self, name, dev, batch=None):
        super().__init__(name, dev, int8=True, batch=batch)
        import torch
        pa, case, wl = self.pa, self.case, self.case.wl
        self.cache8 = pa.CacheI8(1, case.num_blocks, wl.n_kv_heads, wl.head_dim, device=dev)
        # Any codes and positive scales will do for timing: fill them on the GPU.
        g = torch.Generator(device=dev).manual_seed(wl.seed)
        self.cache8.codes.copy_(torch.randint(-127, 128, self.cache8.codes.shape, generator=g,
                                              device=dev, dtype=torch.int8))
        self.cache8.scales.copy_(torch.rand(self.cache8.scales.shape, generator=g, device=dev) /
                                 64 + 1e-3)
        self.units = kv_bytes_i8(case)
        self.rope_units = rope_bytes_i8(case)

    def step(self, ev=None):
        """One step; `ev` = three CUDA events recorded before the RoPE/append
        kernel, between it and the attention kernel, and after that."""
        pa, d, wl = self.pa, self.d, self.case.wl
        if ev is not None:
            ev[0].record()
        pa.rope_kv_write_i8(d["q"], d["k"], d["v"], d["positions"], d["slots"], self.table,
                            self.cache8, status=self.status)
        if ev is not None:
            ev[1].record()
        pa.decode_i8(d["q"], self.cache8, d["bt"], d["ctx"], self.ws, wl.n_kv_heads, out=self.out,
                     status=self.status)
        if ev is not None:
            ev[2].record()

    def fused_step(self):
        """No one-call int8 step: the two calls."""
        self.step()

    def kernel_name(self):
        return "decode_kernel (int8 cache)"

    rope_kernel = "rope_kv_write_i8_kernel"

    graph_setup = None  # the captured step is the fp16 cache's


class PrefillBench:
    rope_kernel = "rope_kv_write_kernel"
    graph_setup = None

    def __init__(self, name, dev, batch=None):
        import torch
        from paged_kv_gqa_rope_gb300 import pa
        self.pa, self.torch = pa, torch
        case = W.make_case(name, batch=batch)
        self.case = case
        wl = case.wl
        md = pa.prepare_prefill(case.num_cached, case.num_new, case.block_tables)
        self.md = md
        self.table = pa.rope_table(int(md["max_seqlen_k"]), wl.head_dim, wl.rope_theta)
        self.cache = pa.Cache(1, case.num_blocks, wl.n_kv_heads, wl.head_dim, device=dev)
        self.cache.tensor.copy_(torch.from_numpy(W.initial_cache(case)))
        self.host = dict(q=case.q, k=case.k, v=case.v, positions=md["positions"],
                         slots=md["slot_mapping"], bt=case.block_tables,
                         cuq=md["cu_seqlens_q"], cuk=md["cu_seqlens_k"])
        self.packed = PackedInputs(self.host, dev)
        self.d = self.packed.views
        # the library's choice of RoPE/append kernel (a label only): the
        # staged kernel for at least eight tokens per SM when two stages of
        # a token's rows fit in its 100 KB of shared memory
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        stage = (wl.n_heads + 2 * wl.n_kv_heads) * wl.head_dim * 2
        if len(case.q) >= 8 * sms and 2 * stage + 16 <= 100 * 1024:
            self.rope_kernel = "rope_kv_write_staged_kernel"
        self.out = torch.empty_like(self.d["q"])
        self.status = pa.new_status(dev)
        self.units = prefill_flops(case)
        self.unit = "TFLOP/s"
        self.rope_units = rope_bytes(case)
        self.launches_per_step = 2

    def step(self, ev=None):
        """One step; `ev` = three CUDA events recorded before the RoPE/append
        kernel, between it and the attention kernel, and after that."""
        pa, d, wl = self.pa, self.d, self.case.wl
        if ev is not None:
            ev[0].record()
        pa.rope_kv_write(d["q"], d["k"], d["v"], d["positions"], d["slots"], self.table,
                         self.cache, status=self.status)
        if ev is not None:
            ev[1].record()
        pa.prefill_varlen(d["q"], self.cache, d["cuq"], d["cuk"], d["bt"], self.md["max_seqlen_q"],
                          wl.n_kv_heads, out=self.out, status=self.status)
        if ev is not None:
            ev[2].record()

    def fused_step(self):
        """The step as one call (pa_prefill_step: the two kernels chained)."""
        pa, d, wl = self.pa, self.d, self.case.wl
        pa.prefill_step(d["q"], d["k"], d["v"], d["positions"], d["slots"], self.table, self.cache,
                        d["cuq"], d["cuk"], d["bt"], self.md["max_seqlen_q"], wl.n_kv_heads,
                        out=self.out, status=self.status)

    def e2e_setup(self):
        torch = self.torch
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        return self.packed.nbytes, self.out_host.numel() * self.out_host.element_size()

    def e2e_step(self):
        self.packed.upload()
        self.fused_step()
        self.out_host.copy_(self.out, non_blocking=True)

    def e2e_close(self):
        pass

    def kernel_name(self):
        return "prefill_kernel"


def make_bench(name, dev, int8=False, batch=None):
    if int8:
        return DecodeI8Bench(name, dev, batch=batch)
    return (PrefillBench if W.WORKLOADS[name].kind == "prefill" else DecodeBench)(name, dev,
                                                                                  batch=batch)


def committed_traffic(kernel, workload, units=None):
    """DRAM bytes per launch (read + write) of `kernel` on `workload` from
    the committed ncu summaries, or None when there is no capture of that
    kernel on that workload made from the kernel's current source.  A
    capture of a smaller case of the same workload (fewer sequences) is
    scaled to a full launch by the algorithmic units (`units` = a full
    launch's), since the traffic of these kernels grows in proportion."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)
    except Exception:
        return None
    for rec in recs if isinstance(recs, list) else []:
        if not isinstance(rec, dict) or rec.get("kernel") != kernel or \
                rec.get("workload") != workload:
            continue
        try:
            with open(os.path.join(ROOT, rec["source"]), "rb") as f:
                sha = hashlib.sha256(f.read()).hexdigest()
        except OSError:
            return None
        if not sha.startswith(rec["sha256_prefix"]):
            return None
        t = rec["dram_bytes_read"] + rec["dram_bytes_write"]
        cap = rec.get("units_captured")
        if cap and units and cap != units:
            t = int(round(t * units / cap))
        return t
    return None


def rate(units, seconds, unit):
    return units / seconds / (1e9 if unit == "GB/s" else 1e12)


def time_bench(b, steps, warmup, dist_ctx):
    """Times `steps` steps after `warmup` untimed ones, twice.  First the step
    as a user runs it (one call: RoPE/append and the attention kernel
    chained), with CUDA events only between steps: ms per step over the whole
    timed region (max over ranks) and the mean and median of each step's own
    duration.  Then the same steps made of the two separate calls with
    events around each kernel (which keeps the kernels from overlapping):
    the attention kernel's and the RoPE/append kernel's durations.  Returns
    those and the device status word."""
    torch = b.torch
    for _ in range(warmup):
        b.fused_step()
    torch.cuda.synchronize()
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    starts = [E() for _ in range(steps + 1)]
    dist_ctx.barrier()
    torch.cuda.synchronize()
    for i in range(steps):
        starts[i].record()
        b.fused_step()
    starts[steps].record()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    ms = starts[0].elapsed_time(starts[steps]) / steps
    step_ms = [starts[i].elapsed_time(starts[i + 1]) for i in range(steps)]
    # the kernels one at a time
    for _ in range(warmup):
        b.step()
    kev = [(E(), E(), E()) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        b.step(kev[i])
    torch.cuda.synchronize()
    kern = [z.elapsed_time(w) for _, z, w in kev]
    rope = [a.elapsed_time(z) for a, z, _ in kev]
    st = int(b.status.item())
    return dict(ms=dist_ctx.max(ms), ms_median=dist_ctx.max(float(np.median(step_ms))),
                kernel_ms=dist_ctx.max(float(np.mean(kern))),
                kernel_ms_median=dist_ctx.max(float(np.median(kern))),
                rope_ms=dist_ctx.max(float(np.mean(rope))),
                rope_ms_median=dist_ctx.max(float(np.median(rope))), status=st)


def time_e2e(b, steps, warmup, dist_ctx):
    torch = b.torch
    h2d, d2h = b.e2e_setup()
    for _ in range(warmup):
        b.e2e_step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_ctx.barrier()
    torch.cuda.synchronize()
    start.record()
    for _ in range(steps):
        b.e2e_step()
    stop.record()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    b.e2e_close()
    return dist_ctx.max(start.elapsed_time(stop) / steps), h2d, d2h


def time_graph(b, steps, warmup, dist_ctx):
    """ms per step of the graph-captured decode step (RoPE/append + decode)."""
    torch = b.torch
    b.graph_setup()
    for _ in range(warmup):
        b.graph_step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_ctx.barrier()
    torch.cuda.synchronize()
    start.record()
    for _ in range(steps):
        b.graph_step()
    stop.record()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    b.graph.close()
    return dist_ctx.max(start.elapsed_time(stop) / steps)


class DistCtx:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x):
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())


# ---------------------------------------------------------------- CPU oracle

THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _sequence_pool(case, s):
    """Sequence s's KV blocks alone, as a compact pool (blocks relabelled
    0..n-1, the same contents), and its one-row block table."""
    from paged_kv_gqa_rope_gb300.workloads import block_contents
    wl = case.wl
    blocks = [int(b) for b in case.block_tables[s] if b >= 0]
    pool = np.zeros((2, 1, max(len(blocks), 1), wl.block_size, wl.n_kv_heads, wl.head_dim),
                    np.float16)
    for j, b in enumerate(blocks):
        pool[:, 0, j] = block_contents(wl, b)
    return pool, np.arange(len(blocks), dtype=np.int32)[None, :]


def _oracle_decode_seq(orc, case, s, pool, table):
    """One sequence's decode step on the oracle: (seconds, KV bytes)."""
    wl = case.wl
    t0 = time.perf_counter()
    md = orc.decode_metadata(case.num_cached[s:s + 1], table, wl.block_size)
    q = orc.rope_pinned(case.q[s:s + 1], md["positions"], wl.head_dim, wl.rope_theta)
    k = orc.rope_pinned(case.k[s:s + 1], md["positions"], wl.head_dim, wl.rope_theta)
    orc.kv_write(pool, 0, k, case.v[s:s + 1], md["slot_mapping"])
    orc.attention_decode(q, pool, 0, table, md["context_lens"], wl.n_heads, wl.n_kv_heads)
    dt = time.perf_counter() - t0
    return dt, (int(case.num_cached[s]) + 1) * wl.n_kv_heads * wl.head_dim * 4


def _oracle_prefill_seq(orc, case, s, pool, table):
    """One sequence's prefill on the oracle: (seconds, FLOPs)."""
    wl = case.wl
    t0 = time.perf_counter()
    nc, nn = case.num_cached[s:s + 1], case.num_new[s:s + 1]
    md = orc.prefill_metadata(nc, nn, table, wl.block_size)
    lo = int(case.num_new[:s].sum())
    hi = lo + int(nn[0])
    q = orc.rope_pinned(case.q[lo:hi], md["positions"], wl.head_dim, wl.rope_theta)
    k = orc.rope_pinned(case.k[lo:hi], md["positions"], wl.head_dim, wl.rope_theta)
    orc.kv_write(pool, 0, k, case.v[lo:hi], md["slot_mapping"])
    orc.attention_prefill(q, pool, 0, md["cu_seqlens_q"], md["cu_seqlens_k"], table,
                          wl.n_heads, wl.n_kv_heads)
    dt = time.perf_counter() - t0
    p, n = int(nc[0]), int(nn[0])
    return dt, 4 * wl.head_dim * wl.n_heads * (n * (p + 1) + n * (n - 1) // 2)


def _oracle_worker(name, w, stride, inq, outq):
    """Worker process: owns sequences w, w + stride, ... of workload `name`
    (their KV blocks drawn once, on first use).  For each request (tag, n)
    it evaluates the next n of them in turn and answers (tag, oracle
    seconds, units, n, w)."""
    from oracle import reference as orc
    case = W.make_case(name)
    fn = _oracle_prefill_seq if case.wl.kind == "prefill" else _oracle_decode_seq
    mine = list(range(w, case.wl.batch, stride))
    kept, i = {}, 0
    while True:
        msg = inq.get()
        if msg is None:
            return
        tag, n = msg
        dt_sum, units = 0.0, 0
        for _ in range(n):
            s = mine[i % len(mine)]
            i += 1
            if s not in kept:
                kept[s] = _sequence_pool(case, s)
            dt, u = fn(orc, case, s, *kept[s])
            dt_sum += dt
            units += u
        outq.put((tag, dt_sum, units, n, w))


class OracleSampler:
    """The oracle, as it stands, on bounded samples of a workload: one
    single-threaded worker process per host core (at most one per sequence;
    `cores` caps the count), started once.  A step hands every worker
    `per_worker` whole-sequence evaluations; its throughput is the units
    done over the oracle seconds spent per worker (the workers run side by
    side).  Only the oracle's arithmetic is on the clock (drawing the
    synthetic inputs is not)."""

    # the first answer of a worker includes drawing its inputs and starting
    # the interpreter: it gets this long; later ones ten times their
    # expected oracle time, but at least two minutes
    FIRST_LIMIT_S = 1800.0

    def __init__(self, name, cores=None):
        import multiprocessing as mp
        self.name = name
        self.B = W.WORKLOADS[name].batch
        self.cores = max(1, min(cores or os.cpu_count() or 1, self.B))
        ctx = mp.get_context("spawn")
        # The workers import numpy before any initializer runs: the thread
        # limits go in through the environment they inherit.
        saved = {v: os.environ.get(v) for v in THREAD_VARS}
        os.environ.update({v: "1" for v in THREAD_VARS})
        try:
            self.inq = [ctx.Queue() for _ in range(self.cores)]
            self.outq = ctx.Queue()
            self.procs = [ctx.Process(target=_oracle_worker,
                                      args=(name, w, self.cores, self.inq[w], self.outq),
                                      daemon=True) for w in range(self.cores)]
            for p in self.procs:
                p.start()
        finally:
            for v, x in saved.items():
                if x is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = x
        self.items = 0
        self.item_s = None  # mean oracle seconds per item, once measured
        self.pending = [0] * self.cores  # requests each worker has not answered

    def _limit(self, items_per_worker):
        if self.item_s is None:
            return self.FIRST_LIMIT_S
        return max(120.0, 10.0 * self.item_s * items_per_worker)

    def _put(self, w, tag, n):
        self.pending[w] += 1
        self.inq[w].put((tag, n))

    def _get(self, deadline, limit):
        """The next answer.  Raises at once if a worker has died, and once
        time.monotonic() passes `deadline`, naming the workers that still
        owe an answer."""
        import queue
        while True:
            try:
                ans = self.outq.get(timeout=2.0)
                self.pending[ans[4]] -= 1
                return ans
            except queue.Empty:
                dead = [w for w, p in enumerate(self.procs) if p.exitcode is not None]
                if dead:
                    raise RuntimeError(f"oracle worker(s) {dead} exited with code "
                                       f"{self.procs[dead[0]].exitcode}")
                if time.monotonic() > deadline:
                    late = [w for w, k in enumerate(self.pending) if k > 0]
                    raise RuntimeError(f"oracle worker(s) {late} gave no answer within "
                                       f"{limit:.0f} s")

    def step(self, per_worker):
        """Every worker evaluates `per_worker` sequences.  Returns (units,
        oracle seconds per worker, items)."""
        limit = self._limit(per_worker)
        deadline = time.monotonic() + limit
        for w in range(self.cores):
            self._put(w, 0, per_worker)
        cpu_s, units, n = 0.0, 0, 0
        for _ in range(self.cores):
            _, dt, u, k, _ = self._get(deadline, limit)
            cpu_s, units, n = cpu_s + dt, units + u, n + k
        self.items += n
        self.item_s = cpu_s / n
        return units, cpu_s / self.cores, n

    def samples(self, count, per_sample):
        """`count` independent samples of `per_sample` sequences each, sample
        i on worker i mod cores, all in flight together.  Returns per sample
        (units, oracle seconds), in order."""
        limit = self._limit(-(-count // self.cores) * per_sample)
        deadline = time.monotonic() + limit
        for i in range(count):
            self._put(i % self.cores, i, per_sample)
        out = [None] * count
        for _ in range(count):
            tag, dt, u, _, _ = self._get(deadline, limit)
            out[tag] = (u, dt)
        self.items += count * per_sample
        return out

    def per_worker_for(self, wall_s):
        """Items per worker that take about `wall_s` seconds."""
        return max(1, int(wall_s / self.item_s)) if self.item_s else 1

    def close(self):
        for q in self.inq:
            q.put(None)
        for p in self.procs:
            p.join(30)
            if p.is_alive():
                p.terminate()


def oracle_baseline(name, budget_s=15.0, cores=None):
    """The `cpu_baseline` key: one sample of about `budget_s` CPU-seconds of
    oracle arithmetic (after two untimed rounds: the first draws the inputs,
    the second, warm, sizes the sample), on one single-threaded worker per
    host core, or on `cores` of them."""
    smp = OracleSampler(name, cores=cores)
    try:
        smp.step(1)
        smp.step(1)
        k = smp.per_worker_for(budget_s / smp.cores)
        units, wall, n = smp.step(k)
    finally:
        smp.close()
    unit = "TFLOP/s" if W.WORKLOADS[name].kind == "prefill" else "GB/s"
    return dict(value=rate(units, wall, unit), unit=unit, cores=smp.cores, kind="oracle",
                sample=f"{n} sequence evaluations cycling through the {smp.B} sequences of "
                       f"{name}, {k} per single-threaded worker, {wall * smp.cores:.1f} CPU-s "
                       f"of oracle arithmetic")


def reference_arm(name, steps, warmup, wall_budget_s=45.0):
    """`--impl reference`: the oracle timed over `warmup` untimed and `steps`
    timed steps.  A step is a bounded sample (whole sequences on one
    single-threaded worker) and its value is that worker's rate times the
    number of workers, which run side by side; the samples are independent,
    so the workers take them in turn, and each is sized so that the whole
    run spends about `wall_budget_s` seconds on every worker (at least one
    sequence per sample).  Returns (median value, unit, info)."""
    smp = OracleSampler(name)
    unit = "TFLOP/s" if W.WORKLOADS[name].kind == "prefill" else "GB/s"
    try:
        smp.step(1)  # draws every worker's inputs; also the per-item estimate
        k = smp.per_worker_for(wall_budget_s * smp.cores / (steps + warmup))
        res = smp.samples(warmup + steps, k)[warmup:]
    finally:
        smp.close()
    vals = [rate(u, dt / smp.cores, unit) for u, dt in res]
    cpu = sum(dt for _, dt in res)
    info = dict(cores=smp.cores, kind="oracle",
                sample=f"per step {k} sequence evaluation(s) on one of {smp.cores} "
                       f"single-threaded workers (taken in turn, value = its rate x "
                       f"{smp.cores}), cycling through the {smp.B} sequences of {name}; "
                       f"{cpu:.1f} CPU-s of oracle arithmetic over {steps} timed steps")
    return float(np.median(vals)), unit, info


# ---------------------------------------------------------------- main

def workload_config(name, batch, int8=False, world=1):
    """The `config` object of a line: the workload and its shape."""
    wl = W.WORKLOADS[name]
    return {"workload": name, "n_heads": wl.n_heads, "n_kv_heads": wl.n_kv_heads,
            "head_dim": wl.head_dim, "block_size": wl.block_size, "batch": batch,
            "kv_cache": "int8 codes + fp32 scales" if int8 else "fp16",
            "l2": "inputs larger than L2 (KV bytes or prefill Q/K/V/O per step > 129 MB); "
                  "no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


INPUT_NOTE = ("every timed step runs on the same device buffers: RoPE rotates the step's "
              "q/k in place again each step (its cost does not depend on the values); "
              "the int8 cache of the timed int8 steps holds seeded random codes and "
              "scales, not the quantised fp16 history (decode cost does not depend on "
              "the code values)")


def measure(b, name, steps, warmup, dctx, peaks, with_e2e=True, with_graph=True):
    """Time workload `name` on bench `b`: the step (mean and median), the
    dominant kernel against its roofline, the RoPE/append kernel on its own,
    and optionally the end-to-end step (host I/O inside the timed region)
    and the graph-captured decode step."""
    r = time_bench(b, steps, warmup, dctx)
    world = dctx.world
    if b.unit == "GB/s":
        peak, bound = peaks[0], "hbm"
    else:
        peak, bound = peaks[1], "tensor"
    achieved = rate(b.units, r["kernel_ms"] / 1e3, b.unit)
    rope_gbs = rate(b.rope_units, r["rope_ms"] / 1e3, "GB/s")
    out = {
        "value": rate(b.units * world, r["ms"] / 1e3, b.unit), "unit": b.unit,
        "ms_per_step": r["ms"], "ms_per_step_median": r["ms_median"], "steps": steps,
        "roofline": {"bound": bound, "kernel": b.kernel_name(), "achieved": achieved,
                     "peak": peak, "peak_source": peaks[3], "unit": b.unit,
                     "frac": achieved / peak,
                     "traffic": committed_traffic(b.kernel_name(), name, b.units),
                     "kernel_ms": r["kernel_ms"], "kernel_ms_median": r["kernel_ms_median"],
                     "units_per_launch": b.units},
        "rope_kv_write": {"kernel": b.rope_kernel, "ms": r["rope_ms"],
                          "ms_median": r["rope_ms_median"], "bytes_per_launch": b.rope_units,
                          "GB/s": rope_gbs, "frac_of_hbm": rope_gbs / peaks[0]},
        "device_status": r["status"],
    }
    if b.unit != "GB/s" and peaks[2]:
        # the same against the sustained cuBLAS figure, which was measured
        # with the clocks held down by the power cap
        out["roofline_sustained"] = {"peak": peaks[2], "frac": achieved / peaks[2],
                                     "note": "peak of a seconds-long cuBLAS loop at "
                                             "power-capped clocks; this kernel runs at "
                                             "the clocks in 'clocks'"}
    if with_e2e:
        e2e_ms, h2d, d2h = time_e2e(b, max(10, steps // 4), warmup, dctx)
        out["e2e"] = {"value": rate(b.units * world, e2e_ms / 1e3, b.unit), "unit": b.unit,
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": e2e_ms}
    if with_graph and getattr(b, "graph_setup", None) is not None:
        g_ms = time_graph(b, steps, warmup, dctx)
        out["step_graph"] = {"value": rate(b.units * world, g_ms / 1e3, b.unit),
                             "unit": b.unit, "ms_per_step": g_ms, "steps": steps,
                             "kernels_per_step": 2,
                             "how": "pa_step_graph: RoPE/append + decode captured once "
                                    "(programmatic dependent launch between them), replayed"}
    return out


# workloads reported under per_workload, and whether each gets the headline's
# whole instrumentation (e2e, cpu_baseline)
EXTRA = (("mha_decode_7b", False), ("ragged_decode", True), ("gqa_decode_70b", False),
         ("prefill_13b", False), ("mha_decode_7b:int8", False), ("gqa_decode_70b:int8", False),
         ("ragged_decode:int8", False))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(W.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer sequences of the same workload (profiling a smaller case)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--int8", action="store_true",
                    help="decode workloads: time the int8 KV cache path instead (our arm)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    dctx = DistCtx()
    peaks = load_peaks()
    wl = W.WORKLOADS[args.workload]
    batch = wl.batch if args.batch is None else min(args.batch, wl.batch)

    if args.impl == "reference":
        if dctx.rank != 0:
            return
        steps = args.steps or 3
        v, unit, info = reference_arm(args.workload, steps, warmup)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit,
                "n_gpus": args.gpus, "steps": steps, "warmup": warmup,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic (seeded; shapes of the pages' workloads)",
                "config": workload_config(args.workload, batch, args.int8, args.gpus),
                "cpu_baseline": dict(info, value=v, unit=unit),
                "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    torch.cuda.set_device(dctx.local)
    dev = f"cuda:{dctx.local}"
    from paged_kv_gqa_rope_gb300 import pa
    pa.lib()
    if args.int8 and wl.kind != "decode":
        raise SystemExit("--int8 applies to decode workloads")
    b = make_bench(args.workload, dev, int8=args.int8, batch=args.batch)
    steps = args.steps or (4000 if wl.kind != "prefill" else 2000)
    with ClockSampler(dctx.local) as clk:
        r = time_bench(b, steps, warmup, dctx)
    clocks = clk.summary()
    # the timed loop above is the headline; e2e and the step graph follow it
    value = rate(b.units * dctx.world, r["ms"] / 1e3, b.unit)
    achieved = rate(b.units, r["kernel_ms"] / 1e3, b.unit)
    peak, bound = (peaks[0], "hbm") if b.unit == "GB/s" else (peaks[1], "tensor")
    e2e_ms, h2d, d2h = time_e2e(b, max(10, steps // 4), warmup, dctx)
    rope_gbs = rate(b.rope_units, r["rope_ms"] / 1e3, "GB/s")
    line = {
        "metric": METRIC, "value": value, "unit": b.unit, "n_gpus": dctx.world,
        "steps": steps, "warmup": warmup, "ms_per_step": r["ms"],
        "ms_per_step_median": r["ms_median"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16 (fp32 accumulate)",
        "data": "synthetic (seeded; shapes of the pages' workloads)",
        "inputs": INPUT_NOTE,
        "config": workload_config(args.workload, batch, args.int8, dctx.world),
        "roofline": {"bound": bound, "kernel": b.kernel_name(), "achieved": achieved,
                     "peak": peak, "peak_source": peaks[3], "unit": b.unit,
                     "frac": achieved / peak,
                     "traffic": committed_traffic(b.kernel_name(), args.workload, b.units),
                     "kernel_ms": r["kernel_ms"], "kernel_ms_median": r["kernel_ms_median"],
                     "units_per_launch": b.units},
        "e2e": {"value": rate(b.units * dctx.world, e2e_ms / 1e3, b.unit), "unit": b.unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "rope_kv_write": {"kernel": b.rope_kernel, "ms": r["rope_ms"],
                          "ms_median": r["rope_ms_median"], "bytes_per_launch": b.rope_units,
                          "GB/s": rope_gbs, "frac_of_hbm": rope_gbs / peaks[0]},
        "gpu_launches": b.launches_per_step * steps,
        "clocks": clocks,
        "device_status": r["status"],
    }
    if b.unit != "GB/s" and peaks[2]:
        line["roofline_sustained"] = {"peak": peaks[2], "frac": achieved / peaks[2],
                                      "note": "peak of a seconds-long cuBLAS loop at "
                                              "power-capped clocks; this kernel runs at "
                                              "the clocks in 'clocks'"}
    if getattr(b, "graph_setup", None) is not None:
        g_ms = time_graph(b, steps, warmup, dctx)
        line["step_graph"] = {"value": rate(b.units * dctx.world, g_ms / 1e3, b.unit),
                              "unit": b.unit, "ms_per_step": g_ms, "steps": steps,
                              "kernels_per_step": 2,
                              "how": "pa_step_graph: RoPE/append + decode captured once "
                                     "(programmatic dependent launch between them), replayed"}
    full_extra = []
    if not args.no_extra and dctx.world == 1 and args.batch is None:
        extra = {}
        del b
        torch.cuda.empty_cache()
        for name, full in EXTRA:
            if name == args.workload + (":int8" if args.int8 else ""):
                continue
            try:
                base, _, kind = name.partition(":")
                eb = make_bench(base, dev, int8=(kind == "int8"))
                n = 1000 if eb.unit == "GB/s" else 400
                extra[name] = measure(eb, base, n, warmup, dctx, peaks, with_e2e=full)
                if full:
                    full_extra.append(name)
                del eb
                torch.cuda.empty_cache()
            except Exception as e:  # report, keep the headline
                extra[name] = {"error": f"{type(e).__name__}: {e}"}
        line["per_workload"] = extra
    if dctx.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(args.workload)
        line["cpu_baseline"]["single_thread"] = oracle_baseline(args.workload, budget_s=6.0,
                                                                cores=1)
        for name in full_extra:
            line["per_workload"][name]["cpu_baseline"] = oracle_baseline(name)
    if dctx.rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
