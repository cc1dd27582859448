"""CPU oracle for the paged-KV chunk gather / scatter (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it shares no code
with them.

The arithmetic lives in ``lmkv_oracle.c`` (plain C, built here with gcc); this
module only compiles that file on demand and marshals numpy arrays into it.
The functions follow:

* "LMCache: An Efficient KV Cache Layer for Enterprise-Scale LLM Inference",
  section on the configurable chunk size (pages are copied into a contiguous
  streaming buffer of 256-token chunks and split back on load) and section on
  the layer-wise pipeline (one layer per call);
* "LMCache 源码解析" (cache_engine.py walk-through), section "store()"
  (chunk_size, save_unfull_chunk, chunk-aligned prefix);
* "LMCache 分布式 KV Cache 序列化框架：Serde 双层接口设计与自定义扩展实战",
  section 7.1 (fp8 e4m3 cast, one byte per element).

Parity status: every function here is pinned by the tests in
``tests/test_oracle_*.py`` (a per-token dictionary model, closed forms,
torch's own float8/bfloat16 conversions, round-trip and bijection invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lmkv_oracle.c")
_LIB = os.path.join(_HERE, "liblmkv_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
INVALID = -1
BAD_BLOCK = 5


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fp contraction, no OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        move_args = [P, i32, i64, i32, i32, P, i32, P, P, i32, i32, i32, P, i32]
        lib.lmkvo_enumerate.argtypes = [P, P, i32, i32, i32, P, P, P, i64]
        lib.lmkvo_enumerate.restype = i64
        for name in ("lmkvo_gather", "lmkvo_scatter"):
            getattr(lib, name).argtypes = move_args
            getattr(lib, name).restype = ctypes.c_int
        fp8_args = [P, i32, i64, i32, i32, P, i32, P, P, i32, i32, i32, P, P]
        for name in ("lmkvo_gather_fp8", "lmkvo_scatter_fp8"):
            getattr(lib, name).argtypes = fp8_args
            getattr(lib, name).restype = ctypes.c_int
        lib.lmkvo_f32_to_e4m3_array.argtypes = [P, P, i64]
        lib.lmkvo_e4m3_to_f32_array.argtypes = [P, P, i64]
        lib.lmkvo_f32_to_bf16_array.argtypes = [P, P, i64]
        lib.lmkvo_div_f32_array.argtypes = [P, ctypes.c_float, P, i64]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _ptr_array(arrays) -> np.ndarray:
    return np.array([a.ctypes.data for a in arrays], dtype=np.uint64)


def _req_arrays(start, end):
    s = np.ascontiguousarray(np.asarray(start, dtype=np.int64))
    e = np.ascontiguousarray(np.asarray(end, dtype=np.int64))
    assert s.shape == e.shape and s.ndim == 1
    return s, e


def enumerate_chunks(start, end, chunk_size: int, save_unfull: bool):
    """Chunk list [(request, first token, n tokens)], or None if invalid."""
    lib = _load()
    s, e = _req_arrays(start, end)
    n = lib.lmkvo_enumerate(_ptr(s), _ptr(e), len(s), chunk_size, int(save_unfull),
                            None, None, None, 0)
    if n < 0:
        return None
    req = np.zeros(max(n, 1), np.int32)
    tok0 = np.zeros(max(n, 1), np.int64)
    ntok = np.zeros(max(n, 1), np.int32)
    n2 = lib.lmkvo_enumerate(_ptr(s), _ptr(e), len(s), chunk_size, int(save_unfull),
                             _ptr(req), _ptr(tok0), _ptr(ntok), n)
    assert n2 == n
    return [(int(req[i]), int(tok0[i]), int(ntok[i])) for i in range(n)]


class HostPool:
    """Per-layer host pool arrays, each shaped [2][num_blocks][block_size][row] (uint8 rows)."""

    def __init__(self, layers, block_size: int):
        self.layers = [np.ascontiguousarray(a) for a in layers]
        self.block_size = block_size
        a0 = self.layers[0]
        assert a0.ndim == 4 and a0.shape[0] == 2 and a0.shape[2] == block_size
        self.num_blocks = a0.shape[1]
        self.row_bytes = a0.shape[3] * a0.dtype.itemsize
        for a in self.layers:
            assert a.shape == a0.shape and a.dtype == a0.dtype
        self._ptrs = _ptr_array(self.layers)

    @property
    def num_layers(self):
        return len(self.layers)


def _move(fn_name, pool: HostPool, block_table, start, end, chunk_size, save_unfull,
          chunks, layer):
    lib = _load()
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim == 1:
        bt = bt[None, :]
    s, e = _req_arrays(start, end)
    cptr = _ptr_array(chunks) if len(chunks) else np.zeros(1, np.uint64)
    return getattr(lib, fn_name)(
        _ptr(pool._ptrs), pool.num_layers, pool.num_blocks, pool.block_size,
        pool.row_bytes, _ptr(bt), bt.shape[1], _ptr(s), _ptr(e), len(s), chunk_size,
        int(save_unfull), _ptr(cptr), layer)


def gather(pool: HostPool, block_table, start, end, chunk_size, save_unfull, chunks,
           layer: int = -1) -> int:
    """Gather pages into chunk buffers (each chunk array [2][L][n_g][row])."""
    return _move("lmkvo_gather", pool, block_table, start, end, chunk_size, save_unfull,
                 chunks, layer)


def scatter(pool: HostPool, block_table, start, end, chunk_size, save_unfull, chunks,
            layer: int = -1) -> int:
    """Scatter chunk buffers back into pages."""
    return _move("lmkvo_scatter", pool, block_table, start, end, chunk_size, save_unfull,
                 chunks, layer)


def _move_fp8(fn_name, pool: HostPool, block_table, start, end, chunk_size, save_unfull,
              codes, scales):
    lib = _load()
    assert pool.layers[0].dtype.itemsize == 2, "fp8 variant takes a bf16 (uint16) pool"
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim == 1:
        bt = bt[None, :]
    s, e = _req_arrays(start, end)
    cptr = _ptr_array(codes) if len(codes) else np.zeros(1, np.uint64)
    assert scales.dtype == np.float32 and scales.flags["C_CONTIGUOUS"]
    return getattr(lib, fn_name)(
        _ptr(pool._ptrs), pool.num_layers, pool.num_blocks, pool.block_size,
        pool.row_bytes // 2, _ptr(bt), bt.shape[1], _ptr(s), _ptr(e), len(s), chunk_size,
        int(save_unfull), _ptr(cptr), _ptr(scales) if scales.size else None)


def gather_fp8(pool, block_table, start, end, chunk_size, save_unfull, codes, scales) -> int:
    """Quantising gather: codes[g] [2][L][n_g][row] uint8, scales [G][2][L] float32."""
    return _move_fp8("lmkvo_gather_fp8", pool, block_table, start, end, chunk_size,
                     save_unfull, codes, scales)


def scatter_fp8(pool, block_table, start, end, chunk_size, save_unfull, codes, scales) -> int:
    """Dequantising scatter back into a bf16 pool."""
    return _move_fp8("lmkvo_scatter_fp8", pool, block_table, start, end, chunk_size,
                     save_unfull, codes, scales)


def f32_to_e4m3(v: np.ndarray) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib.lmkvo_f32_to_e4m3_array(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_to_f32(c: np.ndarray) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float32)
    lib.lmkvo_e4m3_to_f32_array(_ptr(c), _ptr(out), c.size)
    return out


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    lib.lmkvo_f32_to_bf16_array(_ptr(v), _ptr(out), v.size)
    return out


def div_f32(x: np.ndarray, s: float) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.float32)
    lib.lmkvo_div_f32_array(_ptr(x), ctypes.c_float(s), _ptr(out), x.size)
    return out
