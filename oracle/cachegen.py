"""CPU oracle for the CacheGen KV codec (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path never imports, links
or calls it, and it shares no code with it.

The arithmetic lives in ``cachegen_oracle.c`` (plain C, built here with gcc);
this module compiles it on demand and marshals numpy arrays.  It follows
"LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与源码解析",
sections 1-5 (bins per layer group, per-layer quantisation, CDF estimation
and 2^16 normalisation, arithmetic coding in 256-token batches, decoding and
dequantisation); the readings of the parts the page leaves open are listed at
the top of the C file.

Parity status: pinned by ``tests/test_oracle_cachegen.py`` (closed forms for
dyadic CDFs, exact-rational CDFs, hand-worked fixtures under
``tests/golden/``, code-length bounds, round trips and the quantisation error
bound) and by the planted mistakes in ``tests/test_oracle_mutants.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cachegen_oracle.c")
_LIB = os.path.join(_HERE, "libcachegen_oracle.so")
_lock = threading.Lock()
_lib = None

BATCH = 256


def build(force: bool = False) -> str:
    """Compile the codec oracle with gcc (-O2, no fp contraction)."""
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
        lib.cgo_default_bins.argtypes = [i32, P]
        lib.cgo_quantize.argtypes = [P, i32, i32, i32, P, P]
        lib.cgo_cdf.argtypes = [P, i32, i64, i32, P]
        lib.cgo_encode.argtypes = [P, i32, i64, P, i32, P, i64]
        lib.cgo_encode.restype = i64
        lib.cgo_decode.argtypes = [P, i64, i32, P, i32, P, i64]
        lib.cgo_dequantize.argtypes = [P, P, i32, i32, i32, P]
        lib.cgo_layout.argtypes = [i32, i32, i32, P, P]
        lib.cgo_layout.restype = ctypes.c_int
        lib.cgo_encode_chunk.argtypes = [P, i32, i32, i32, P, P, i64]
        lib.cgo_encode_chunk.restype = i64
        lib.cgo_decode_chunk.argtypes = [P, i64, i32, i32, i32, P, P]
        lib.cgo_decode_chunk.restype = ctypes.c_int
        _lib = lib
        return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    """bf16 data as a contiguous uint16 array (numpy uint16/int16, or a torch
    bfloat16 tensor on the CPU)."""
    if hasattr(x, "view") and hasattr(x, "numpy") and not isinstance(x, np.ndarray):
        import torch
        x = x.contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(np.asarray(x).view(np.uint16))


def nsym(bins: int) -> int:
    return 2 * (bins // 2 - 1) + 1


def default_bins(num_layers: int) -> np.ndarray:
    """int32 [2][num_layers]: row 0 K, row 1 V."""
    out = np.zeros(2 * num_layers, np.int32)
    _load().cgo_default_bins(num_layers, _p(out))
    return out.reshape(2, num_layers)


def quantize(x, bins: int):
    """x: bf16 [n][H] -> (symbols uint8 [n][H], max1 float32 [n])."""
    x = _u16(x)
    n, H = x.shape
    sym = np.zeros((n, H), np.uint8)
    max1 = np.zeros(n, np.float32)
    _load().cgo_quantize(_p(x), n, H, int(bins), _p(sym), _p(max1))
    return sym, max1


def cdf(symbols, num_symbols: int) -> np.ndarray:
    """One channel's symbols (uint8 [n]) -> C[0..num_symbols] as uint32."""
    s = np.ascontiguousarray(symbols, np.uint8)
    C = np.zeros(num_symbols + 1, np.uint32)
    _load().cgo_cdf(_p(s), len(s), 1, int(num_symbols), _p(C))
    return C


def encode(symbols, C) -> bytes:
    """Code one stream with the CDF C (uint32, C[-1] == 65536)."""
    s = np.ascontiguousarray(symbols, np.uint8)
    C = np.ascontiguousarray(C, np.uint32)
    cap = (18 * len(s) + 2 + 7) // 8 + 8
    out = np.zeros(cap, np.uint8)
    n = _load().cgo_encode(_p(s), len(s), 1, _p(C), len(C) - 1, _p(out), cap)
    if n < 0:
        raise ValueError(f"oracle encode failed ({n})")
    return out[:n].tobytes()


def decode(stream: bytes, n: int, C) -> np.ndarray:
    buf = np.frombuffer(bytes(stream) + b"\0", np.uint8).copy()
    C = np.ascontiguousarray(C, np.uint32)
    sym = np.zeros(max(n, 1), np.uint8)
    _load().cgo_decode(_p(buf), len(stream), n, _p(C), len(C) - 1, _p(sym), 1)
    return sym[:n]


def dequantize(symbols, max1, bins: int) -> np.ndarray:
    """symbols uint8 [n][H], max1 float32 [n] -> bf16 bits uint16 [n][H]."""
    s = np.ascontiguousarray(symbols, np.uint8)
    m = np.ascontiguousarray(max1, np.float32)
    n, H = s.shape
    out = np.zeros((n, H), np.uint16)
    _load().cgo_dequantize(_p(s), _p(m), n, H, int(bins), _p(out))
    return out


def layout(num_layers: int, n: int, H: int, bins) -> dict:
    """Byte offsets of the encoded chunk's parts and a bound on its size."""
    b = np.ascontiguousarray(np.asarray(bins, np.int32).reshape(-1))
    off = np.zeros(5, np.int64)
    rc = _load().cgo_layout(num_layers, n, H, _p(b), _p(off))
    if rc != 0:
        raise ValueError("invalid CacheGen layout arguments")
    return {"max1": int(off[0]), "cdf": int(off[1]), "lengths": int(off[2]),
            "bytes": int(off[3]), "bound": int(off[4])}


def encode_chunk(chunk, bins) -> bytes:
    """chunk: bf16 [2][L][n][H] -> the encoded blob."""
    x = _u16(chunk)
    _, L, n, H = x.shape
    b = np.ascontiguousarray(np.asarray(bins, np.int32).reshape(-1))
    cap = layout(L, n, H, b)["bound"]
    blob = np.zeros(cap, np.uint8)
    size = _load().cgo_encode_chunk(_p(x), L, n, H, _p(b), _p(blob), cap)
    if size < 0:
        raise ValueError(f"oracle encode failed ({size})")
    return blob[:size].tobytes()


def decode_chunk(blob: bytes, num_layers: int, n: int, H: int, bins) -> np.ndarray:
    """The encoded blob -> bf16 bits uint16 [2][L][n][H]."""
    buf = np.frombuffer(bytes(blob) + b"\0", np.uint8).copy()
    b = np.ascontiguousarray(np.asarray(bins, np.int32).reshape(-1))
    out = np.zeros((2, num_layers, n, H), np.uint16)
    rc = _load().cgo_decode_chunk(_p(buf), len(blob), num_layers, n, H, _p(b), _p(out))
    if rc != 0:
        raise ValueError(f"oracle decode failed ({rc})")
    return out


def parse(blob: bytes, num_layers: int, n: int, H: int, bins) -> dict:
    """Split a blob into its parts (numpy views), for tests."""
    lay = layout(num_layers, n, H, bins)
    raw = np.frombuffer(bytes(blob), np.uint8)
    b = np.asarray(bins, np.int32).reshape(-1)
    nb = (n + BATCH - 1) // BATCH
    max1 = raw[lay["max1"]:lay["cdf"]].view(np.float32).reshape(2, num_layers, n)
    cdfs, pos = [], lay["cdf"]
    for s in range(2 * num_layers):
        k = nsym(int(b[s])) - 1
        cdfs.append(raw[pos:pos + 2 * H * k].view(np.uint16).reshape(H, k))
        pos += 2 * H * k
    lengths = raw[lay["lengths"]:lay["bytes"]].view(np.uint32).reshape(nb, 2, num_layers, H)
    return {"max1": max1, "cdf": cdfs, "lengths": lengths, "bytes": raw[lay["bytes"]:],
            "layout": lay}
