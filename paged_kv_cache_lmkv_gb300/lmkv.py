"""Python binding of liblmkv.so (argument marshalling only).

Every function here maps one-to-one onto an ``extern "C"`` entry point of
``include/lmkv.h``; all data movement runs in the library's CUDA kernels.
PyTorch tensors are used only as carriers of device memory and streams.  If
the library has not been built, the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblmkv.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_MISALIGNED = 2
ERR_CUDA = 3
ERR_UNSUPPORTED = 4
ERR_BAD_BLOCK = 5
ERR_BAD_POINTER = 6
ERR_TIMEOUT = 7
ERR_SCRATCH_LIMIT = 8
ERR_BAD_DATA = 9
NOALLOC_STAGING_BYTES = 64 << 20
CACHEGEN_BATCH = 256
CACHEGEN_MAX_CHANNELS = 2048
CACHEGEN_MAX_TOKENS = 4096
CACHEGEN_MAX_LAYERS = 128

ENTRY_POINTS = (
    "lmkv_count_chunks", "lmkv_enumerate_chunks", "lmkv_gather_chunks", "lmkv_scatter_chunks",
    "lmkv_gather_layer", "lmkv_scatter_layer", "lmkv_gather_chunks_fp8e4m3",
    "lmkv_scatter_chunks_fp8e4m3", "lmkv_status_string", "lmkv_abi_version",
    "lmkv_launch_count", "lmkv_store_layers", "lmkv_retrieve_layers",
    "lmkv_store_layers_staged", "lmkv_retrieve_layers_staged",
    "lmkv_store_layers_staged_noalloc", "lmkv_decode_store_ranges",
    "lmkv_offload_init", "lmkv_offload_plan", "lmkv_offload_copied", "lmkv_offload_allocate",
    "lmkv_offload_add_free", "lmkv_cachegen_default_bins", "lmkv_cachegen_layout",
    "lmkv_cachegen_workspace_bytes", "lmkv_cachegen_encode", "lmkv_cachegen_decode",
    "lmkv_cachegen_store_chunks", "lmkv_cachegen_retrieve_chunks",
    "lmkv_last_cuda_error", "lmkv_cuda_error_name",
    "lmkv_store_layers_overlapped", "lmkv_retrieve_layers_overlapped",
)


class LmkvError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = f"{what}: lmkv status {code} ({status_string(code)})"
        if code == ERR_CUDA:
            err = last_cuda_error()
            msg += f"; last CUDA error {err} ({cuda_error_name(err)})"
        super().__init__(msg)


class OffloadState(ctypes.Structure):
    """lmkv_offload_t: positions in the free-page order, start <= current <= end."""
    _fields_ = [("start", ctypes.c_int64), ("current", ctypes.c_int64), ("end", ctypes.c_int64),
                ("limit", ctypes.c_int64), ("window", ctypes.c_int64)]

    def as_tuple(self):
        return (self.start, self.current, self.end, self.limit, self.window)


class CachegenLayout(ctypes.Structure):
    """lmkv_cachegen_layout_t: byte offsets of one chunk's encoded blob."""
    _fields_ = [("max1_offset", ctypes.c_uint64), ("cdf_offset", ctypes.c_uint64),
                ("lengths_offset", ctypes.c_uint64), ("bytes_offset", ctypes.c_uint64),
                ("max_bytes", ctypes.c_uint64)]


class _PoolT(ctypes.Structure):
    _fields_ = [
        ("layer_base", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("num_layers", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("elem_bytes", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    """Load liblmkv.so (raises if it is missing: build it with build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: the CUDA library must be built "
                               "(paged_kv_cache_lmkv_gb300.build.build()); there is no fallback")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        pool_p = ctypes.POINTER(_PoolT)
        lib.lmkv_count_chunks.argtypes = [P, P, i32, i32, i32, P]
        lib.lmkv_decode_store_ranges.argtypes = [P, P, i32, i32, P, P, P]
        off_p = ctypes.POINTER(OffloadState)
        lib.lmkv_offload_init.argtypes = [off_p, i64, i64]
        lib.lmkv_offload_plan.argtypes = [off_p, i64, P, P]
        lib.lmkv_offload_copied.argtypes = [off_p, i64]
        lib.lmkv_offload_allocate.argtypes = [off_p, i64, P, P]
        lib.lmkv_offload_add_free.argtypes = [off_p, i64]
        lib.lmkv_enumerate_chunks.argtypes = [P, P, i32, i32, i32, P, P, P, i32]
        move = [pool_p, P, i32, P, P, i32, i32, i32, P, P, P]
        lib.lmkv_gather_chunks.argtypes = move
        lib.lmkv_scatter_chunks.argtypes = move
        layer = [pool_p, P, i32, P, P, i32, i32, i32, P, i32, P, P]
        lib.lmkv_gather_layer.argtypes = layer
        lib.lmkv_scatter_layer.argtypes = layer
        layers = [pool_p, P, i32, P, P, i32, i32, i32, P, i32, i32, P, P, P, P]
        lib.lmkv_store_layers.argtypes = layers
        lib.lmkv_retrieve_layers.argtypes = layers
        staged = [pool_p, P, i32, P, P, i32, i32, i32, P, P, i64, i32, i32, P, P, P, P]
        lib.lmkv_store_layers_staged.argtypes = staged
        lib.lmkv_retrieve_layers_staged.argtypes = staged
        lib.lmkv_store_layers_staged_noalloc.argtypes = [pool_p, P, i32, P, P, i32, i32, i32, P,
                                                         i32, i32, P, P, P, P]
        overlapped = [pool_p, P, i32, P, P, i32, i32, i32, P, P, i64, i32, i32, P, P, P, P, P, P]
        lib.lmkv_store_layers_overlapped.argtypes = overlapped
        lib.lmkv_retrieve_layers_overlapped.argtypes = overlapped
        fp8 = [pool_p, P, i32, P, P, i32, i32, i32, P, P, P, P]
        lib.lmkv_gather_chunks_fp8e4m3.argtypes = fp8
        lib.lmkv_scatter_chunks_fp8e4m3.argtypes = fp8
        lib.lmkv_cachegen_default_bins.argtypes = [i32, P]
        lib.lmkv_cachegen_layout.argtypes = [i32, i32, i32, P, ctypes.POINTER(CachegenLayout)]
        lib.lmkv_cachegen_workspace_bytes.argtypes = [i32, i32, P, i32, P]
        lib.lmkv_cachegen_encode.argtypes = [P, P, i32, i32, i32, P, P, P, P, ctypes.c_uint64, P, P]
        lib.lmkv_cachegen_decode.argtypes = [P, P, P, i32, i32, i32, P, P, P, ctypes.c_uint64, P, P]
        cg_pool = [pool_p, P, i32, P, P, i32, i32, i32, P, P, P, P, ctypes.c_uint64, P, P]
        lib.lmkv_cachegen_store_chunks.argtypes = cg_pool
        lib.lmkv_cachegen_retrieve_chunks.argtypes = cg_pool
        for name in ("lmkv_count_chunks", "lmkv_enumerate_chunks", "lmkv_gather_chunks",
                     "lmkv_cachegen_default_bins", "lmkv_cachegen_layout",
                     "lmkv_cachegen_workspace_bytes", "lmkv_cachegen_encode", "lmkv_cachegen_decode",
                     "lmkv_cachegen_store_chunks", "lmkv_cachegen_retrieve_chunks",
                     "lmkv_decode_store_ranges", "lmkv_offload_init", "lmkv_offload_plan",
                     "lmkv_offload_copied", "lmkv_offload_allocate", "lmkv_offload_add_free",
                     "lmkv_scatter_chunks", "lmkv_gather_layer", "lmkv_scatter_layer",
                     "lmkv_gather_chunks_fp8e4m3", "lmkv_scatter_chunks_fp8e4m3",
                     "lmkv_abi_version", "lmkv_store_layers", "lmkv_retrieve_layers",
                     "lmkv_store_layers_staged", "lmkv_retrieve_layers_staged",
                     "lmkv_store_layers_staged_noalloc", "lmkv_store_layers_overlapped",
                     "lmkv_retrieve_layers_overlapped"):
            getattr(lib, name).restype = ctypes.c_int
        lib.lmkv_status_string.argtypes = [ctypes.c_int]
        lib.lmkv_status_string.restype = ctypes.c_char_p
        lib.lmkv_launch_count.argtypes = []
        lib.lmkv_launch_count.restype = ctypes.c_int64
        lib.lmkv_last_cuda_error.argtypes = []
        lib.lmkv_last_cuda_error.restype = ctypes.c_int
        lib.lmkv_cuda_error_name.argtypes = [ctypes.c_int]
        lib.lmkv_cuda_error_name.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().lmkv_status_string(int(code)).decode()


def launch_count() -> int:
    return int(load().lmkv_launch_count())


def last_cuda_error() -> int:
    return int(load().lmkv_last_cuda_error())


def cuda_error_name(err: int) -> str:
    return load().lmkv_cuda_error_name(int(err)).decode()


def _i64_array(values) -> np.ndarray:
    """Contiguous int64 host array (no copy when it already is one)."""
    if isinstance(values, np.ndarray) and values.dtype == np.int64 and values.flags.c_contiguous:
        return values
    return np.ascontiguousarray(values, dtype=np.int64)


def _stream_handle(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class Pool:
    """A paged KV pool: per-layer device tensors [2][num_blocks][block_size][heads*head_dim].

    Holds the DEVICE array of layer base pointers the ABI takes.
    """

    def __init__(self, layers: Sequence[torch.Tensor], num_kv_heads: int, head_dim: int):
        t0 = layers[0]
        if t0.dim() != 4 or t0.shape[0] != 2 or t0.shape[3] != num_kv_heads * head_dim:
            raise ValueError("pool layers must be [2][num_blocks][block_size][heads*head_dim]")
        for t in layers:
            if t.shape != t0.shape or t.dtype != t0.dtype or not t.is_contiguous() or not t.is_cuda:
                raise ValueError("pool layers must be contiguous CUDA tensors of one shape/dtype")
        self.layers = list(layers)
        self.num_kv_heads = num_kv_heads
        self.head_dim = head_dim
        self.block_size = t0.shape[2]
        self.num_blocks = t0.shape[1]
        self.elem_bytes = t0.element_size()
        self.ptrs = torch.tensor([t.data_ptr() for t in layers], dtype=torch.int64,
                                 device=t0.device)
        self._struct = _PoolT(self.ptrs.data_ptr(), self.num_blocks, len(layers), num_kv_heads,
                              head_dim, self.block_size, self.elem_bytes)

    @property
    def num_layers(self) -> int:
        return len(self.layers)

    @property
    def struct(self):
        return ctypes.byref(self._struct)


def pointer_array(tensors: Sequence[torch.Tensor], device) -> torch.Tensor:
    """DEVICE int64 array of the tensors' data pointers (chunk_ptrs / code_ptrs).

    The copy is queued on the current stream from pinned host memory, so the
    host does not wait for the device (the caching host allocator keeps the
    pinned block until the copy has run)."""
    host = torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64)
    if torch.device(device).type != "cuda":
        return host.to(device)
    return host.pin_memory().to(device, non_blocking=True)


def count_chunks(start, end, chunk_size: int, save_unfull: bool) -> int:
    lib = load()
    s, e = _i64_array(start), _i64_array(end)
    out = ctypes.c_int32(0)
    rc = lib.lmkv_count_chunks(s.ctypes.data, e.ctypes.data, len(s), chunk_size, int(save_unfull),
                               ctypes.byref(out))
    if rc != OK:
        raise LmkvError(rc, "lmkv_count_chunks")
    return out.value


def decode_store_ranges(stored_end, cur_end, chunk_size: int):
    """lmkv_decode_store_ranges -> (start, end, number of completed chunks)."""
    lib = load()
    s, e = _i64_array(stored_end), _i64_array(cur_end)
    out_s = np.zeros(len(s), np.int64)
    out_e = np.zeros(len(s), np.int64)
    n = ctypes.c_int32(0)
    rc = lib.lmkv_decode_store_ranges(s.ctypes.data, e.ctypes.data, len(s), chunk_size,
                                      out_s.ctypes.data, out_e.ctypes.data, ctypes.byref(n))
    if rc != OK:
        raise LmkvError(rc, "lmkv_decode_store_ranges")
    return out_s, out_e, n.value


class Offload:
    """Thin wrapper of the lmkv_offload_* calls on one caller-owned state."""

    def __init__(self, num_free: int, window: int):
        self.state = OffloadState()
        self._call("lmkv_offload_init", ctypes.byref(self.state), int(num_free), int(window))

    def _call(self, name, *args):
        rc = getattr(load(), name)(*args)
        if rc != OK:
            raise LmkvError(rc, name)

    def plan(self, max_pages: int):
        first, count = ctypes.c_int64(0), ctypes.c_int64(0)
        self._call("lmkv_offload_plan", ctypes.byref(self.state), int(max_pages),
                   ctypes.byref(first), ctypes.byref(count))
        return first.value, count.value

    def copied(self, count: int):
        self._call("lmkv_offload_copied", ctypes.byref(self.state), int(count))

    def allocate(self, want: int):
        g, s = ctypes.c_int64(0), ctypes.c_int64(0)
        self._call("lmkv_offload_allocate", ctypes.byref(self.state), int(want), ctypes.byref(g),
                   ctypes.byref(s))
        return g.value, s.value

    def add_free(self, n: int):
        self._call("lmkv_offload_add_free", ctypes.byref(self.state), int(n))


def enumerate_chunks(start, end, chunk_size: int, save_unfull: bool):
    """[(request, first token, n tokens)] in chunk order."""
    lib = load()
    n = count_chunks(start, end, chunk_size, save_unfull)
    s, e = _i64_array(start), _i64_array(end)
    req = (ctypes.c_int32 * max(n, 1))()
    tok0 = (ctypes.c_int64 * max(n, 1))()
    ntok = (ctypes.c_int32 * max(n, 1))()
    rc = lib.lmkv_enumerate_chunks(s.ctypes.data, e.ctypes.data, len(s), chunk_size,
                                   int(save_unfull), req, tok0, ntok, n)
    if rc != OK:
        raise LmkvError(rc, "lmkv_enumerate_chunks")
    return [(req[i], tok0[i], ntok[i]) for i in range(n)]


def _ptr(t):
    return None if t is None else t.data_ptr()


def _common(pool: Pool, block_table: torch.Tensor, start, end):
    """(pool, table, max_blocks, start, end, num_req) plus the host arrays to keep alive."""
    if block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32")
    s, e = _i64_array(start), _i64_array(end)
    if s.shape != e.shape:
        raise ValueError("start and end must have one entry per request")
    return (pool.struct, block_table.data_ptr(), block_table.shape[-1], s.ctypes.data,
            e.ctypes.data, len(s)), (s, e)


def gather_chunks(pool, block_table, start, end, chunk_size, save_unfull, chunk_ptrs,
                  status=None, stream=None) -> int:
    """lmkv_gather_chunks; returns the status code (0 = launched)."""
    a, _keep = _common(pool, block_table, start, end)
    return load().lmkv_gather_chunks(*a, chunk_size, int(save_unfull), _ptr(chunk_ptrs),
                                     _ptr(status), _stream_handle(stream))


def scatter_chunks(pool, block_table, start, end, chunk_size, save_unfull, chunk_ptrs,
                   status=None, stream=None) -> int:
    a, _keep = _common(pool, block_table, start, end)
    return load().lmkv_scatter_chunks(*a, chunk_size, int(save_unfull), _ptr(chunk_ptrs),
                                      _ptr(status), _stream_handle(stream))


def gather_layer(pool, block_table, start, end, chunk_size, save_unfull, chunk_ptrs, layer,
                 status=None, stream=None) -> int:
    a, _keep = _common(pool, block_table, start, end)
    return load().lmkv_gather_layer(*a, chunk_size, int(save_unfull), _ptr(chunk_ptrs),
                                    int(layer), _ptr(status), _stream_handle(stream))


def scatter_layer(pool, block_table, start, end, chunk_size, save_unfull, chunk_ptrs, layer,
                  status=None, stream=None) -> int:
    a, _keep = _common(pool, block_table, start, end)
    return load().lmkv_scatter_layer(*a, chunk_size, int(save_unfull), _ptr(chunk_ptrs),
                                     int(layer), _ptr(status), _stream_handle(stream))


def gather_chunks_fp8e4m3(pool, block_table, start, end, chunk_size, save_unfull, code_ptrs,
                          scales, status=None, stream=None) -> int:
    a, _keep = _common(pool, block_table, start, end)
    return load().lmkv_gather_chunks_fp8e4m3(*a, chunk_size, int(save_unfull), _ptr(code_ptrs),
                                             _ptr(scales), _ptr(status), _stream_handle(stream))


def scatter_chunks_fp8e4m3(pool, block_table, start, end, chunk_size, save_unfull, code_ptrs,
                           scales, status=None, stream=None) -> int:
    a, _keep = _common(pool, block_table, start, end)
    return load().lmkv_scatter_chunks_fp8e4m3(*a, chunk_size, int(save_unfull), _ptr(code_ptrs),
                                              _ptr(scales), _ptr(status), _stream_handle(stream))


def _event_array(events, n):
    """HOST array of n cudaEvent_t handles (0 = none) from torch.cuda.Event objects."""
    if events is None:
        return None
    if len(events) != n:
        raise ValueError("one event (or None) per layer")
    arr = (ctypes.c_void_p * max(n, 1))()
    for i, e in enumerate(events):
        if e is None:
            continue
        handle = e.cuda_event if isinstance(e, torch.cuda.Event) else int(e)
        if not handle:
            raise ValueError("event has no CUDA event yet: record it once first")
        arr[i] = handle
    return arr


def store_layers(pool, block_table, start, end, chunk_size, save_unfull, chunk_ptrs, layer_lo,
                 layer_n, layer_ready=None, layer_done=None, status=None, stream=None) -> int:
    """lmkv_store_layers: per layer, wait on layer_ready[i], gather, record layer_done[i]."""
    a, _keep = _common(pool, block_table, start, end)
    r, d = _event_array(layer_ready, layer_n), _event_array(layer_done, layer_n)
    return load().lmkv_store_layers(*a, chunk_size, int(save_unfull), _ptr(chunk_ptrs), int(layer_lo),
                                    int(layer_n), r, d, _ptr(status), _stream_handle(stream))


def retrieve_layers(pool, block_table, start, end, chunk_size, save_unfull, chunk_ptrs, layer_lo,
                    layer_n, layer_ready=None, layer_done=None, status=None, stream=None) -> int:
    """lmkv_retrieve_layers: per layer, wait on layer_ready[i], scatter, record layer_done[i]."""
    a, _keep = _common(pool, block_table, start, end)
    r, d = _event_array(layer_ready, layer_n), _event_array(layer_done, layer_n)
    return load().lmkv_retrieve_layers(*a, chunk_size, int(save_unfull), _ptr(chunk_ptrs),
                                       int(layer_lo), int(layer_n), r, d, _ptr(status),
                                       _stream_handle(stream))


def _host_ptr_array(tensors):
    """HOST array of the (pinned host) tensors' data pointers."""
    arr = (ctypes.c_void_p * max(len(tensors), 1))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr()
    return arr


def staging_bytes(pool, start, end, chunk_size, save_unfull) -> int:
    """Bytes of the one-layer staging buffer the staged pipeline needs."""
    n = sum(ntok for _, _, ntok in enumerate_chunks(start, end, chunk_size, save_unfull))
    return 2 * pool.num_kv_heads * pool.head_dim * pool.elem_bytes * n


def store_layers_staged(pool, block_table, start, end, chunk_size, save_unfull, host_chunks,
                        staging, layer_lo, layer_n, layer_ready=None, layer_done=None,
                        status=None, stream=None) -> int:
    """lmkv_store_layers_staged; host_chunks: pinned host tensors, staging: device tensor."""
    a, _keep = _common(pool, block_table, start, end)
    h = _host_ptr_array(host_chunks)
    r, d = _event_array(layer_ready, layer_n), _event_array(layer_done, layer_n)
    return load().lmkv_store_layers_staged(*a, chunk_size, int(save_unfull), h, _ptr(staging),
                                           staging.numel() * staging.element_size(), int(layer_lo),
                                           int(layer_n), r, d, _ptr(status), _stream_handle(stream))


def retrieve_layers_staged(pool, block_table, start, end, chunk_size, save_unfull, host_chunks,
                           staging, layer_lo, layer_n, layer_ready=None, layer_done=None,
                           status=None, stream=None) -> int:
    """lmkv_retrieve_layers_staged (host -> staging by 2-D copies, then scatter)."""
    a, _keep = _common(pool, block_table, start, end)
    h = _host_ptr_array(host_chunks)
    r, d = _event_array(layer_ready, layer_n), _event_array(layer_done, layer_n)
    return load().lmkv_retrieve_layers_staged(*a, chunk_size, int(save_unfull), h, _ptr(staging),
                                              staging.numel() * staging.element_size(),
                                              int(layer_lo), int(layer_n), r, d, _ptr(status),
                                              _stream_handle(stream))


def overlap_events(stream=None):
    """Four events for the overlapped pipeline (recorded once on `stream`, so
    that their CUDA handles exist)."""
    evs = [torch.cuda.Event() for _ in range(4)]
    for e in evs:
        e.record(stream)
    return evs


def _overlapped(fn, pool, block_table, start, end, chunk_size, save_unfull, host_chunks, staging,
                layer_lo, layer_n, sync_events, layer_ready, layer_done, status, stream, copy_stream):
    a, _keep = _common(pool, block_table, start, end)
    h = _host_ptr_array(host_chunks)
    r, d = _event_array(layer_ready, layer_n), _event_array(layer_done, layer_n)
    e = _event_array(sync_events, 4)
    if copy_stream is None:
        raise ValueError("the overlapped pipeline needs a copy stream")
    return fn(*a, chunk_size, int(save_unfull), h, _ptr(staging), staging.numel() * staging.element_size(),
              int(layer_lo), int(layer_n), r, d, e, _ptr(status), _stream_handle(stream),
              _stream_handle(copy_stream))


def store_layers_overlapped(pool, block_table, start, end, chunk_size, save_unfull, host_chunks,
                            staging, layer_lo, layer_n, sync_events, layer_ready=None,
                            layer_done=None, status=None, stream=None, copy_stream=None) -> int:
    """lmkv_store_layers_overlapped: two staging halves (staging holds 2 layers),
    kernels on `stream`, copies on `copy_stream`, 4 sync events (overlap_events())."""
    return _overlapped(load().lmkv_store_layers_overlapped, pool, block_table, start, end, chunk_size,
                       save_unfull, host_chunks, staging, layer_lo, layer_n, sync_events, layer_ready,
                       layer_done, status, stream, copy_stream)


def retrieve_layers_overlapped(pool, block_table, start, end, chunk_size, save_unfull, host_chunks,
                               staging, layer_lo, layer_n, sync_events, layer_ready=None,
                               layer_done=None, status=None, stream=None, copy_stream=None) -> int:
    """lmkv_retrieve_layers_overlapped (the inverse of store_layers_overlapped)."""
    return _overlapped(load().lmkv_retrieve_layers_overlapped, pool, block_table, start, end, chunk_size,
                       save_unfull, host_chunks, staging, layer_lo, layer_n, sync_events, layer_ready,
                       layer_done, status, stream, copy_stream)


def store_layers_staged_noalloc(pool, block_table, start, end, chunk_size, save_unfull,
                                host_chunks, layer_lo, layer_n, layer_ready=None, layer_done=None,
                                status=None, stream=None) -> int:
    """lmkv_store_layers_staged_noalloc: the staged store using the library's
    built-in 64 MiB device staging area instead of a caller buffer, for callers
    that cannot allocate device memory.  Make the first call on a device before
    any stream capture; calls that overlap on the GPU share the staging area."""
    a, _keep = _common(pool, block_table, start, end)
    h = _host_ptr_array(host_chunks)
    r, d = _event_array(layer_ready, layer_n), _event_array(layer_done, layer_n)
    return load().lmkv_store_layers_staged_noalloc(*a, chunk_size, int(save_unfull), h,
                                                   int(layer_lo), int(layer_n), r, d,
                                                   _ptr(status), _stream_handle(stream))


# ---- CacheGen codec ----

def _i32_array(values) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(values).reshape(-1), dtype=np.int32)


def cachegen_default_bins(num_layers: int) -> np.ndarray:
    """int32 [2][num_layers] bins (row 0 K, row 1 V)."""
    out = np.zeros(2 * num_layers, np.int32)
    check(load().lmkv_cachegen_default_bins(num_layers, out.ctypes.data), "lmkv_cachegen_default_bins")
    return out.reshape(2, num_layers)


def cachegen_layout(num_layers: int, num_tokens: int, channels: int, bins) -> CachegenLayout:
    b = _i32_array(bins)
    out = CachegenLayout()
    check(load().lmkv_cachegen_layout(num_layers, num_tokens, channels, b.ctypes.data,
                                      ctypes.byref(out)), "lmkv_cachegen_layout")
    return out


def cachegen_workspace_bytes(num_layers: int, channels: int, num_tokens) -> int:
    n = _i32_array(num_tokens)
    out = ctypes.c_uint64(0)
    check(load().lmkv_cachegen_workspace_bytes(num_layers, channels, n.ctypes.data, len(n),
                                               ctypes.byref(out)), "lmkv_cachegen_workspace_bytes")
    return out.value


def cachegen_encode(chunk_ptrs, num_tokens, num_layers, channels, bins, blob_ptrs, sizes,
                    workspace, status=None, stream=None) -> int:
    """chunk_ptrs / blob_ptrs: DEVICE int64 pointer arrays; sizes: DEVICE uint64
    (int64 tensor) [num_chunks]; workspace: a DEVICE uint8 tensor."""
    n, b = _i32_array(num_tokens), _i32_array(bins)
    return load().lmkv_cachegen_encode(_ptr(chunk_ptrs), n.ctypes.data, len(n), num_layers, channels,
                                       b.ctypes.data, _ptr(blob_ptrs), _ptr(sizes), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(status),
                                       _stream_handle(stream))


def cachegen_decode(blob_ptrs, sizes, num_tokens, num_layers, channels, bins, chunk_ptrs,
                    workspace, status=None, stream=None) -> int:
    n, b = _i32_array(num_tokens), _i32_array(bins)
    return load().lmkv_cachegen_decode(_ptr(blob_ptrs), _ptr(sizes), n.ctypes.data, len(n), num_layers,
                                       channels, b.ctypes.data, _ptr(chunk_ptrs), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(status),
                                       _stream_handle(stream))


def cachegen_store_chunks(pool, block_table, start, end, chunk_size, save_unfull, bins, blob_ptrs,
                          sizes, workspace, status=None, stream=None) -> int:
    """Encode a store call's chunks straight from the pool's pages."""
    a, _keep = _common(pool, block_table, start, end)
    b = _i32_array(bins)
    return load().lmkv_cachegen_store_chunks(*a, chunk_size, int(save_unfull), b.ctypes.data,
                                             _ptr(blob_ptrs), _ptr(sizes), _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _ptr(status),
                                             _stream_handle(stream))


def cachegen_retrieve_chunks(pool, block_table, start, end, chunk_size, save_unfull, bins, blob_ptrs,
                             sizes, workspace, status=None, stream=None) -> int:
    """Decode blobs straight into the pages of a retrieve call's chunks."""
    a, _keep = _common(pool, block_table, start, end)
    b = _i32_array(bins)
    return load().lmkv_cachegen_retrieve_chunks(*a, chunk_size, int(save_unfull), b.ctypes.data,
                                                _ptr(blob_ptrs), _ptr(sizes), _ptr(workspace),
                                                workspace.numel() * workspace.element_size(),
                                                _ptr(status), _stream_handle(stream))


class CachegenCodec:
    """Chunk buffers [2][L][n][H] bf16 <-> CacheGen blobs, through
    lmkv_cachegen_encode / lmkv_cachegen_decode, and pool pages <-> blobs
    through the fused store / retrieve.  Holds the bins and a device workspace
    that grows to the largest batch seen (PyTorch memory); calls that share
    one codec object must be ordered on one stream (they share the
    workspace)."""

    _POINTER_CACHE = 32      # pointer arrays kept for reuse

    def __init__(self, num_layers: int, channels: int, bins=None, device="cuda"):
        self.num_layers, self.channels = num_layers, channels
        self.bins = _i32_array(cachegen_default_bins(num_layers) if bins is None else bins)
        self.device = torch.device(device)
        self.workspace = torch.empty(0, dtype=torch.uint8, device=self.device)
        self._need = {}          # token counts -> workspace bytes
        self._ptrs = {}          # data pointers -> (device pointer array, event after its copy)

    def layout(self, num_tokens: int) -> CachegenLayout:
        return cachegen_layout(self.num_layers, num_tokens, self.channels, self.bins)

    def _workspace(self, ntok):
        key = tuple(ntok)
        need = self._need.get(key)
        if need is None:
            need = self._need[key] = cachegen_workspace_bytes(self.num_layers, self.channels, ntok)
        if self.workspace.numel() < need:
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self.workspace

    def _pointers(self, tensors):
        """The device pointer array of the tensors, reused while the same
        addresses come back (a serving loop with fixed buffers builds it once).
        The current stream waits for the copy that filled it (outside a
        stream capture; warm up before capturing)."""
        key = tuple(t.data_ptr() for t in tensors)
        hit = self._ptrs.pop(key, None)
        if hit is None:
            arr = pointer_array(tensors, self.device)
            ev = torch.cuda.Event()
            ev.record(torch.cuda.current_stream(self.device))
            hit = (arr, ev)
            if len(self._ptrs) >= self._POINTER_CACHE:
                self._ptrs.pop(next(iter(self._ptrs)))
        else:
            cur = torch.cuda.current_stream(self.device)
            if not torch.cuda.is_current_stream_capturing():
                cur.wait_event(hit[1])
            hit[0].record_stream(cur)    # evicted later: freed only after this stream's use
        self._ptrs[key] = hit            # most recently used last
        return hit[0]

    def encode(self, chunks, blobs=None, sizes=None, status=None, stream=None):
        """Encode the chunk tensors; returns (blobs, sizes): device uint8 tensors
        of each layout's max_bytes and a device int64 tensor of the sizes."""
        ntok = [int(c.shape[2]) for c in chunks]
        if blobs is None:
            blobs = [torch.empty(self.layout(n).max_bytes, dtype=torch.uint8, device=self.device)
                     for n in ntok]
        if sizes is None:
            sizes = torch.zeros(len(chunks), dtype=torch.int64, device=self.device)
        ws = self._workspace(ntok)
        cptr, bptr = self._pointers(chunks), self._pointers(blobs)
        self._order(stream, cptr, bptr)
        check(cachegen_encode(cptr, ntok, self.num_layers, self.channels, self.bins, bptr, sizes, ws,
                              status, stream), "lmkv_cachegen_encode")
        return blobs, sizes

    def _order(self, stream, *arrays):
        """The pointer arrays are written on the current stream: a different
        `stream` waits for them and keeps them alive until it has read them."""
        if stream is None:
            return
        cur = torch.cuda.current_stream(self.device)
        if isinstance(stream, torch.cuda.Stream) and stream != cur:
            stream.wait_stream(cur)
            for a in arrays:
                a.record_stream(stream)

    def store(self, pool, block_table, start, end, chunk_size, save_unfull, blobs=None, sizes=None,
              status=None, stream=None):
        """Encode a store call's chunks straight from the pool; returns (blobs, sizes)."""
        ntok = [n for _, _, n in enumerate_chunks(start, end, chunk_size, save_unfull)]
        if blobs is None:
            blobs = [torch.empty(self.layout(n).max_bytes, dtype=torch.uint8, device=self.device)
                     for n in ntok]
        if sizes is None:
            sizes = torch.zeros(len(ntok), dtype=torch.int64, device=self.device)
        ws = self._workspace(ntok)
        bptr = self._pointers(blobs)
        self._order(stream, bptr)
        check(cachegen_store_chunks(pool, block_table, start, end, chunk_size, save_unfull, self.bins,
                                    bptr, sizes, ws, status, stream), "lmkv_cachegen_store_chunks")
        return blobs, sizes

    def retrieve(self, pool, block_table, start, end, chunk_size, save_unfull, blobs, sizes,
                 status=None, stream=None):
        """Decode blobs straight into the pool's pages of a retrieve call's chunks."""
        ntok = [n for _, _, n in enumerate_chunks(start, end, chunk_size, save_unfull)]
        ws = self._workspace(ntok)
        bptr = self._pointers(blobs)
        self._order(stream, bptr)
        check(cachegen_retrieve_chunks(pool, block_table, start, end, chunk_size, save_unfull, self.bins,
                                       bptr, sizes, ws, status, stream), "lmkv_cachegen_retrieve_chunks")

    def decode(self, blobs, sizes, chunks, status=None, stream=None):
        """Decode into the chunk tensors (their token counts give n)."""
        ntok = [int(c.shape[2]) for c in chunks]
        ws = self._workspace(ntok)
        bptr, cptr = self._pointers(blobs), self._pointers(chunks)
        self._order(stream, bptr, cptr)
        check(cachegen_decode(bptr, sizes, ntok, self.num_layers, self.channels, self.bins, cptr, ws,
                              status, stream), "lmkv_cachegen_decode")
        return chunks


def check(rc: int, what: str = "lmkv") -> None:
    if rc != OK:
        raise LmkvError(rc, what)
