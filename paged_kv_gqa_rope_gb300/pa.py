"""Thin ctypes binding of libpa (include/pa.h): the same entry points, with
torch tensors in and out.  It only checks dtypes/devices and marshals
pointers; every step of the computation runs in the library's kernels.  If
libpa.so has not been built, every call raises (there is no fallback).
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_WORKSPACE = 0, 1, 2, 3, 4
PA_DEV_BAD_SLOT, PA_DEV_BAD_POSITION, PA_DEV_BAD_BLOCK = 1, 2, 4
PA_DEV_BAD_LENGTH, PA_DEV_TIMEOUT, PA_DEV_WORKSPACE = 8, 16, 32

# every symbol include/pa.h declares
EXPORTS = (
    "pa_cache_bytes", "pa_alloc_cache", "pa_free_cache", "pa_prepare_prefill",
    "pa_prepare_decode", "pa_rope_table_bytes", "pa_rope_table_init", "pa_rope_kv_write",
    "pa_prefill_varlen", "pa_decode_workspace_bytes", "pa_decode", "pa_strerror",
    "pa_check_device", "pa_decode_noalloc", "pa_decode_step", "pa_prefill_step",
    "pa_step_graph_create",
    "pa_step_graph_launch", "pa_step_graph_destroy", "pa_step_graph_create_io",
    "pa_bm_create", "pa_bm_destroy", "pa_bm_num_free", "pa_bm_blocks_needed", "pa_bm_allocate",
    "pa_bm_next_chunk", "pa_bm_mark_computed", "pa_bm_can_append", "pa_bm_append",
    "pa_bm_num_tokens", "pa_bm_block_table", "pa_bm_free", "pa_selftest_wait_timeout",
    "pa_cache_i8_bytes", "pa_alloc_cache_i8", "pa_free_cache_i8", "pa_rope_kv_write_i8",
    "pa_decode_i8",
)


class PaCache(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("layers", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("owns", ctypes.c_int32), ("layer_stride", ctypes.c_int64),
                ("kv_stride", ctypes.c_int64)]


class PaCacheI8(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("layers", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("owns", ctypes.c_int32)]


class PAError(RuntimeError):
    def __init__(self, name, code):
        super().__init__(f"{name} failed: {strerror(code)} (code {code})")
        self.code = code


_lib = None

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGS = {
    "pa_cache_bytes": (_sz, [_i32] * 5),
    "pa_alloc_cache": (_i32, [ctypes.POINTER(PaCache)] + [_i32] * 5 + [_vp]),
    "pa_free_cache": (_i32, [ctypes.POINTER(PaCache)]),
    "pa_prepare_prefill": (_i32, [_i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "pa_prepare_decode": (_i32, [_i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp]),
    "pa_rope_table_bytes": (_sz, [_i32, _i32]),
    "pa_rope_table_init": (_i32, [_vp, _i32, _i32, ctypes.c_double, _vp]),
    "pa_rope_kv_write": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32,
                                ctypes.POINTER(PaCache), _i32, _vp, _vp]),
    "pa_prefill_varlen": (_i32, [_vp, _i32, ctypes.POINTER(PaCache), _i32, _vp, _vp, _vp, _i32,
                                 _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _vp, _vp]),
    "pa_decode_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "pa_decode": (_i32, [_vp, ctypes.POINTER(PaCache), _i32, _vp, _i32, _vp, _i32, _i32, _i32,
                         _i32, ctypes.c_float, _vp, _sz, _vp, _vp, _vp]),
    "pa_decode_noalloc": (_i32, [_vp, ctypes.POINTER(PaCache), _i32, _vp, _i32, _vp, _i32, _i32,
                                 _i32, _i32, ctypes.c_float, _vp, _vp, _vp]),
    "pa_decode_step": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, ctypes.POINTER(PaCache), _i32,
                              _vp, _i32, _vp, _i32, _i32, _i32, _i32, ctypes.c_float, _vp, _sz,
                              _vp, _vp, _vp]),
    "pa_prefill_step": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, ctypes.POINTER(PaCache), _i32,
                               _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                               ctypes.c_float, _vp, _vp, _vp]),
    "pa_step_graph_create": (_i32, [ctypes.POINTER(_vp), _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                    ctypes.POINTER(PaCache), _i32, _vp, _i32, _vp, _i32, _i32,
                                    _i32, _i32, ctypes.c_float, _vp, _sz, _vp, _vp]),
    "pa_step_graph_create_io": (_i32, [ctypes.POINTER(_vp), _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                       ctypes.POINTER(PaCache), _i32, _vp, _i32, _vp, _i32, _i32,
                                       _i32, _i32, ctypes.c_float, _vp, _sz, _vp, _vp, _vp, _vp,
                                       _sz, _vp]),
    "pa_step_graph_launch": (_i32, [_vp, _vp]),
    "pa_step_graph_destroy": (_i32, [_vp]),
    "pa_bm_create": (_vp, [_i32, _i32]),
    "pa_bm_destroy": (None, [_vp]),
    "pa_bm_num_free": (_i32, [_vp]),
    "pa_bm_blocks_needed": (_i32, [_vp, _i32]),
    "pa_bm_allocate": (_i32, [_vp, _i64, _vp, _i32, ctypes.POINTER(_i32)]),
    "pa_bm_next_chunk": (_i32, [_vp, _i64, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]),
    "pa_bm_mark_computed": (_i32, [_vp, _i64, _i32]),
    "pa_bm_can_append": (_i32, [_vp, _i64]),
    "pa_bm_append": (_i32, [_vp, _i64, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "pa_bm_num_tokens": (_i32, [_vp, _i64]),
    "pa_bm_block_table": (_i32, [_vp, _i64, _vp, _i32, ctypes.POINTER(_i32)]),
    "pa_bm_free": (_i32, [_vp, _i64]),
    "pa_selftest_wait_timeout": (_i32, [_vp, _vp]),
    "pa_cache_i8_bytes": (_sz, [_i32] * 5),
    "pa_alloc_cache_i8": (_i32, [ctypes.POINTER(PaCacheI8)] + [_i32] * 5 + [_vp]),
    "pa_free_cache_i8": (_i32, [ctypes.POINTER(PaCacheI8)]),
    "pa_rope_kv_write_i8": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32,
                                   ctypes.POINTER(PaCacheI8), _i32, _vp, _vp]),
    "pa_decode_i8": (_i32, [_vp, ctypes.POINTER(PaCacheI8), _i32, _vp, _i32, _vp, _i32, _i32,
                            _i32, _i32, ctypes.c_float, _vp, _sz, _vp, _vp, _vp]),
    "pa_strerror": (ctypes.c_char_p, [_i32]),
    "pa_check_device": (_i32, []),
}


def lib() -> ctypes.CDLL:
    """Load libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_gqa_rope_gb300.build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype, fn.argtypes = res, args
        _lib = l
    return _lib


def strerror(code: int) -> str:
    return lib().pa_strerror(int(code)).decode()


def _check(name, rc):
    if rc != PA_OK:
        raise PAError(name, rc)


def _p(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, name, shape=None):
    """A contiguous CUDA tensor of `dtype`; with `shape`, of exactly that shape
    (None entries free).  The library sees only pointers, so the sizes its
    kernels index by are checked here."""
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous CUDA {dtype} tensor")
    if shape is not None:
        _check_shape(t, shape, name)
    return t


def _check_shape(t, shape, name):
    if t.dim() != len(shape) or any(want is not None and got != want
                                    for got, want in zip(t.shape, shape)):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected "
                         f"{tuple('*' if w is None else w for w in shape)}")


def _table_width(block_tables):
    """max_blocks_per_seq; the kernels bound lengths by it * 16 in int32."""
    w = block_tables.shape[1]
    if w * 16 > 2**31 - 1:
        raise ValueError(f"block_tables rows of {w} entries: max_blocks_per_seq * 16 "
                         "must stay within int32")
    return w


def _opt(t, dtype, name, shape):
    return None if t is None else _dev(t, dtype, name, shape)


def _out(out, like, name="out"):
    if out is None:
        return torch.empty_like(like)
    return _dev(out, like.dtype, name, tuple(like.shape))


def check_device() -> int:
    return lib().pa_check_device()


# ------------------------------------------------------------------ host metadata

def prepare_prefill(num_cached, num_new, block_tables, block_size=16):
    nc = np.ascontiguousarray(num_cached, np.int32)
    nn = np.ascontiguousarray(num_new, np.int32)
    bt = np.ascontiguousarray(block_tables, np.int32)
    B = len(nn)
    T = int(nn.sum())
    pos = np.empty(max(T, 1), np.int32)
    slots = np.empty(max(T, 1), np.int32)
    cuq = np.empty(B + 1, np.int32)
    cuk = np.empty(B + 1, np.int32)
    mq, mk = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("pa_prepare_prefill", lib().pa_prepare_prefill(
        B, _p(nc), _p(nn), _p(bt), bt.shape[1] if bt.ndim == 2 else 0, block_size, _p(pos),
        _p(slots), _p(cuq), _p(cuk), ctypes.byref(mq), ctypes.byref(mk)))
    return dict(positions=pos[:T], slot_mapping=slots[:T], cu_seqlens_q=cuq, cu_seqlens_k=cuk,
                max_seqlen_q=mq.value, max_seqlen_k=mk.value)


def prepare_decode(num_cached, block_tables, block_size=16):
    nc = np.ascontiguousarray(num_cached, np.int32)
    bt = np.ascontiguousarray(block_tables, np.int32)
    B = len(nc)
    pos, slots, ctx = (np.empty(max(B, 1), np.int32) for _ in range(3))
    _check("pa_prepare_decode", lib().pa_prepare_decode(
        B, _p(nc), _p(bt), bt.shape[1], block_size, _p(pos), _p(slots), _p(ctx)))
    return dict(positions=pos[:B], slot_mapping=slots[:B], context_lens=ctx[:B])


# ------------------------------------------------------------------ cache and table

class Cache:
    """The block pool [2, layers, num_blocks, block_size, n_kv_heads, head_dim]
    fp16.  By default the memory is a torch tensor (``self.tensor``) that the
    library wraps; ``library_owned=True`` lets pa_alloc_cache allocate it."""

    def __init__(self, layers, num_blocks, n_kv_heads, head_dim, block_size=16, device="cuda",
                 library_owned=False):
        self.desc = PaCache()
        self.tensor = None
        if library_owned:
            base = None
        else:
            self.tensor = torch.empty((2, layers, num_blocks, block_size, n_kv_heads, head_dim),
                                      dtype=torch.float16, device=device)
            base = _p(self.tensor)
        _check("pa_alloc_cache", lib().pa_alloc_cache(
            ctypes.byref(self.desc), layers, num_blocks, block_size, n_kv_heads, head_dim, base))

    def free(self):
        if self.desc.base:
            _check("pa_free_cache", lib().pa_free_cache(ctypes.byref(self.desc)))
        self.tensor = None

    def __del__(self):
        try:
            if self.desc.owns and self.desc.base:
                lib().pa_free_cache(ctypes.byref(self.desc))
        except Exception:
            pass


def cache_bytes(layers, num_blocks, block_size, n_kv_heads, head_dim) -> int:
    return lib().pa_cache_bytes(layers, num_blocks, block_size, n_kv_heads, head_dim)


def rope_table(max_positions, head_dim, theta=10000.0, device="cuda", stream=None):
    nbytes = lib().pa_rope_table_bytes(max_positions, head_dim)
    if nbytes == 0:
        raise ValueError("bad RoPE table shape")
    t = torch.empty((max_positions, head_dim // 2, 2), dtype=torch.float32, device=device)
    _check("pa_rope_table_init", lib().pa_rope_table_init(
        _p(t), max_positions, head_dim, float(theta), _stream(stream)))
    return t


def new_status(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)


# ------------------------------------------------------------------ the hot path

def _rope_args(q, k, v, positions, slot_mapping, table, status):
    _dev(q, torch.float16, "q", (None, None, None))
    T, H, d = q.shape
    _dev(k, torch.float16, "k", (T, None, d))
    _dev(v, torch.float16, "v", tuple(k.shape))
    _dev(positions, torch.int32, "positions", (T,))
    _dev(slot_mapping, torch.int32, "slot_mapping", (T,))
    _dev(table, torch.float32, "table", (None, d // 2, 2))
    _opt(status, torch.int32, "status", (1,))
    return T, H, k.shape[1], d


def rope_kv_write(q, k, v, positions, slot_mapping, table, cache: Cache, layer=0, status=None,
                  stream=None):
    T, H, Hk, d = _rope_args(q, k, v, positions, slot_mapping, table, status)
    _check("pa_rope_kv_write", lib().pa_rope_kv_write(
        _p(q), _p(k), _p(v), _p(positions), _p(slot_mapping), T, H, Hk, d, _p(table),
        table.shape[0], ctypes.byref(cache.desc), layer, _p(status), _stream(stream)))


def prefill_varlen(q, cache: Cache, cu_seqlens_q, cu_seqlens_k, block_tables, max_seqlen_q,
                   n_kv_heads, layer=0, scale=0.0, out=None, status=None, stream=None):
    _dev(q, torch.float16, "q", (None, None, None))
    T, H, d = q.shape
    _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q", (None,))
    B = cu_seqlens_q.shape[0] - 1
    _dev(cu_seqlens_k, torch.int32, "cu_seqlens_k", (B + 1,))
    _dev(block_tables, torch.int32, "block_tables", (B, None))
    _table_width(block_tables)
    _opt(status, torch.int32, "status", (1,))
    out = _out(out, q)
    _check("pa_prefill_varlen", lib().pa_prefill_varlen(
        _p(q), T, ctypes.byref(cache.desc), layer, _p(cu_seqlens_q), _p(cu_seqlens_k),
        _p(block_tables), block_tables.shape[1], B, int(max_seqlen_q), H,
        n_kv_heads, d, float(scale), _p(out), _p(status), _stream(stream)))
    return out


def prefill_step(q, k, v, positions, slot_mapping, rope_table, cache: Cache, cu_seqlens_q,
                 cu_seqlens_k, block_tables, max_seqlen_q, n_kv_heads, layer=0, scale=0.0,
                 out=None, status=None, stream=None):
    """pa_prefill_step: RoPE + append of the new tokens, then the varlen prefill."""
    T, H, Hk, d = _rope_args(q, k, v, positions, slot_mapping, rope_table, status)
    _dev(cu_seqlens_q, torch.int32, "cu_seqlens_q", (None,))
    B = cu_seqlens_q.shape[0] - 1
    _dev(cu_seqlens_k, torch.int32, "cu_seqlens_k", (B + 1,))
    _dev(block_tables, torch.int32, "block_tables", (B, None))
    _table_width(block_tables)
    if Hk != n_kv_heads:
        raise ValueError(f"k has {Hk} KV heads, n_kv_heads is {n_kv_heads}")
    out = _out(out, q)
    _check("pa_prefill_step", lib().pa_prefill_step(
        _p(q), _p(k), _p(v), _p(positions), _p(slot_mapping), _p(rope_table),
        rope_table.shape[0], ctypes.byref(cache.desc), layer, _p(cu_seqlens_q), _p(cu_seqlens_k),
        _p(block_tables), block_tables.shape[1], B, T, int(max_seqlen_q), H, n_kv_heads, d,
        float(scale), _p(out), _p(status), _stream(stream)))
    return out


def decode_workspace_bytes(num_seqs, n_heads, n_kv_heads, head_dim) -> int:
    return lib().pa_decode_workspace_bytes(num_seqs, n_heads, n_kv_heads, head_dim)


def decode_workspace(num_seqs, n_heads, n_kv_heads, head_dim, device="cuda", nbytes=None):
    """A zeroed workspace for pa_decode (its counters must start at zero);
    `nbytes` overrides the size (a smaller one narrows the grid)."""
    n = decode_workspace_bytes(num_seqs, n_heads, n_kv_heads, head_dim) if nbytes is None else nbytes
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _decode_args(q, block_tables, context_lens, workspace, status):
    _dev(q, torch.float16, "q", (None, None, None))
    B = q.shape[0]
    _dev(block_tables, torch.int32, "block_tables", (B, None))
    _table_width(block_tables)
    _dev(context_lens, torch.int32, "context_lens", (B,))
    _dev(workspace, torch.uint8, "workspace", (None,))
    _opt(status, torch.int32, "status", (1,))
    return q.shape


def decode(q, cache: Cache, block_tables, context_lens, workspace, n_kv_heads, layer=0, scale=0.0,
           out=None, status=None, stream=None):
    B, H, d = _decode_args(q, block_tables, context_lens, workspace, status)
    out = _out(out, q)
    _check("pa_decode", lib().pa_decode(
        _p(q), ctypes.byref(cache.desc), layer, _p(block_tables), block_tables.shape[1],
        _p(context_lens), B, H, n_kv_heads, d, float(scale), _p(workspace), workspace.numel(),
        _p(out), _p(status), _stream(stream)))
    return out


def _step_args(q, k, v, positions, slot_mapping, rope_table, cache, block_tables, context_lens,
               workspace, n_kv_heads, layer, scale, out, status):
    _rope_args(q, k, v, positions, slot_mapping, rope_table, status)
    B, H, d = _decode_args(q, block_tables, context_lens, workspace, status)
    _dev(out, torch.float16, "out", (B, H, d))
    return [_p(q), _p(k), _p(v), _p(positions), _p(slot_mapping), _p(rope_table),
            rope_table.shape[0], ctypes.byref(cache.desc), layer, _p(block_tables),
            block_tables.shape[1], _p(context_lens), B, H, n_kv_heads, d, float(scale),
            _p(workspace), workspace.numel(), _p(out), _p(status)]


def decode_step(q, k, v, positions, slot_mapping, rope_table, cache: Cache, block_tables,
                context_lens, workspace, n_kv_heads, layer=0, scale=0.0, out=None, status=None,
                stream=None):
    """pa_decode_step: RoPE + append of the new tokens, then decode."""
    out = _out(out, q)
    args = _step_args(q, k, v, positions, slot_mapping, rope_table, cache, block_tables,
                      context_lens, workspace, n_kv_heads, layer, scale, out, status)
    _check("pa_decode_step", lib().pa_decode_step(*args, _stream(stream)))
    return out


class StepGraph:
    """pa_step_graph_*: a decode step captured once, replayed by launch().
    The tensors passed in are the step's buffers for every replay; refill
    them in place between replays.  References are kept so they outlive
    the graph.

    With `host_in` (a pinned uint8 host tensor) and `dev_in` (the device
    uint8 tensor of the same size that the input tensors are views of), a
    replay first copies host_in to dev_in; with `host_out` (a pinned host
    tensor shaped like q), it ends by copying the output there
    (pa_step_graph_create_io): one launch per step, I/O included."""

    def __init__(self, q, k, v, positions, slot_mapping, rope_table, cache: Cache, block_tables,
                 context_lens, workspace, n_kv_heads, layer=0, scale=0.0, out=None,
                 status=None, host_in=None, dev_in=None, host_out=None):
        self.out = _out(out, q)
        self._keep = (q, k, v, positions, slot_mapping, rope_table, cache, block_tables,
                      context_lens, workspace, status, host_in, dev_in, host_out)
        args = _step_args(q, k, v, positions, slot_mapping, rope_table, cache, block_tables,
                          context_lens, workspace, n_kv_heads, layer, scale, self.out, status)
        h = ctypes.c_void_p()
        if host_in is None and dev_in is None and host_out is None:
            _check("pa_step_graph_create", lib().pa_step_graph_create(ctypes.byref(h), *args))
        else:
            nin = 0
            if host_in is not None or dev_in is not None:
                if not (isinstance(host_in, torch.Tensor) and not host_in.is_cuda
                        and host_in.is_pinned() and host_in.dtype == torch.uint8
                        and host_in.is_contiguous()):
                    raise TypeError("host_in must be a contiguous pinned host uint8 tensor")
                _dev(dev_in, torch.uint8, "dev_in", (host_in.numel(),))
                nin = host_in.numel()
            if host_out is not None:
                if not (isinstance(host_out, torch.Tensor) and not host_out.is_cuda
                        and host_out.is_pinned() and host_out.dtype == torch.float16
                        and host_out.is_contiguous()):
                    raise TypeError("host_out must be a contiguous pinned host fp16 tensor")
                _check_shape(host_out, tuple(q.shape), "host_out")
            _check("pa_step_graph_create_io", lib().pa_step_graph_create_io(
                ctypes.byref(h), *args, _p(host_in), _p(dev_in), nin, _p(host_out)))
        self._h = h

    def launch(self, stream=None):
        _check("pa_step_graph_launch", lib().pa_step_graph_launch(self._h, _stream(stream)))
        return self.out

    def close(self):
        if self._h:
            _check("pa_step_graph_destroy", lib().pa_step_graph_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BlockManager:
    """pa_bm_*: the host block manager (block ownership, prefix-cache reuse,
    chunked-prefill progress); its tables feed prepare_prefill/decode."""

    def __init__(self, num_blocks, block_size=16):
        self._h = lib().pa_bm_create(num_blocks, block_size)
        if not self._h:
            raise ValueError("bad block manager sizes")
        self.block_size = block_size

    def num_free(self):
        return lib().pa_bm_num_free(self._h)

    def blocks_needed(self, num_tokens):
        return lib().pa_bm_blocks_needed(self._h, num_tokens)

    def allocate(self, seq_id, tokens):
        """Admit a prompt; returns the number of tokens already cached."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        n = ctypes.c_int()
        _check("pa_bm_allocate", lib().pa_bm_allocate(self._h, seq_id, _p(t), t.size,
                                                       ctypes.byref(n)))
        return n.value

    def next_chunk(self, seq_id, max_tokens):
        c, n = ctypes.c_int(), ctypes.c_int()
        _check("pa_bm_next_chunk", lib().pa_bm_next_chunk(self._h, seq_id, max_tokens,
                                                           ctypes.byref(c), ctypes.byref(n)))
        return c.value, n.value

    def mark_computed(self, seq_id, num_tokens):
        _check("pa_bm_mark_computed", lib().pa_bm_mark_computed(self._h, seq_id, num_tokens))

    def can_append(self, seq_id):
        r = lib().pa_bm_can_append(self._h, seq_id)
        if r < 0:
            raise PAError("pa_bm_can_append", -r)
        return bool(r)

    def append(self, seq_id, token):
        """Append a decoded token; returns its cache slot."""
        slot = ctypes.c_int32()
        _check("pa_bm_append", lib().pa_bm_append(self._h, seq_id, int(token), ctypes.byref(slot)))
        return slot.value

    def num_tokens(self, seq_id):
        return lib().pa_bm_num_tokens(self._h, seq_id)

    def block_table(self, seq_id):
        n = ctypes.c_int()
        lib().pa_bm_block_table(self._h, seq_id, None, 0, ctypes.byref(n))
        out = np.zeros(max(n.value, 1), np.int32)
        _check("pa_bm_block_table", lib().pa_bm_block_table(self._h, seq_id, _p(out), out.size,
                                                             ctypes.byref(n)))
        return out[:n.value]

    def free(self, seq_id):
        _check("pa_bm_free", lib().pa_bm_free(self._h, seq_id))

    def close(self):
        if self._h:
            lib().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def selftest_wait_timeout(status, stream=None):
    """pa_selftest_wait_timeout: a bounded wait that runs out (about 1 s)."""
    _dev(status, torch.int32, "status", (1,))
    _check("pa_selftest_wait_timeout", lib().pa_selftest_wait_timeout(_p(status), _stream(stream)))


class CacheI8:
    """The int8 pool: ``codes`` int8 [2, layers, num_blocks, block_size,
    n_kv_heads, head_dim] and ``scales`` float32 [2, layers, num_blocks,
    n_kv_heads, block_size], views of one torch allocation the library
    wraps."""

    def __init__(self, layers, num_blocks, n_kv_heads, head_dim, block_size=16, device="cuda"):
        self.desc = PaCacheI8()
        n = lib().pa_cache_i8_bytes(layers, num_blocks, block_size, n_kv_heads, head_dim)
        if n == 0:
            raise ValueError("bad int8 cache shape")
        self.buffer = torch.empty(n, dtype=torch.uint8, device=device)
        _check("pa_alloc_cache_i8", lib().pa_alloc_cache_i8(
            ctypes.byref(self.desc), layers, num_blocks, block_size, n_kv_heads, head_dim,
            _p(self.buffer)))
        nc = 2 * layers * num_blocks * block_size * n_kv_heads * head_dim
        off = self.desc.scales - self.desc.codes
        self.codes = self.buffer[:nc].view(torch.int8).view(
            2, layers, num_blocks, block_size, n_kv_heads, head_dim)
        self.scales = self.buffer[off:].view(torch.float32).view(
            2, layers, num_blocks, n_kv_heads, block_size)


def rope_kv_write_i8(q, k, v, positions, slot_mapping, table, cache: CacheI8, layer=0,
                     status=None, stream=None):
    T, H, Hk, d = _rope_args(q, k, v, positions, slot_mapping, table, status)
    _check("pa_rope_kv_write_i8", lib().pa_rope_kv_write_i8(
        _p(q), _p(k), _p(v), _p(positions), _p(slot_mapping), T, H, Hk, d, _p(table),
        table.shape[0], ctypes.byref(cache.desc), layer, _p(status), _stream(stream)))


def decode_i8(q, cache: CacheI8, block_tables, context_lens, workspace, n_kv_heads, layer=0,
              scale=0.0, out=None, status=None, stream=None):
    B, H, d = _decode_args(q, block_tables, context_lens, workspace, status)
    out = _out(out, q)
    _check("pa_decode_i8", lib().pa_decode_i8(
        _p(q), ctypes.byref(cache.desc), layer, _p(block_tables), block_tables.shape[1],
        _p(context_lens), B, H, n_kv_heads, d, float(scale), _p(workspace), workspace.numel(),
        _p(out), _p(status), _stream(stream)))
    return out
