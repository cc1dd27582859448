"""The C-ABI library loads, exports every symbol include/lmkv.h declares, and
rejects bad arguments on the host before any CUDA call (CPU only)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_lmkv_gb300 import build, lmkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "lmkv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return lmkv.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lmkv_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(lmkv.ENTRY_POINTS)


def test_abi_version_and_status_strings(lib):
    assert lib.lmkv_abi_version() == 1
    for code in range(8):
        assert lmkv.status_string(code) != "unknown status"
    assert lmkv.status_string(99) == "unknown status"


def test_count_and_enumerate_match_closed_form(lib):
    assert lmkv.count_chunks([0, 0, 0, 0], [4096, 9000, 20000, 32768], 256, True) == 259
    assert lmkv.count_chunks([0, 0, 0, 0], [4096, 9000, 20000, 32768], 256, False) == 257
    ch = lmkv.enumerate_chunks([0, 256], [300, 700], 256, True)
    assert ch == [(0, 0, 256), (0, 256, 44), (1, 256, 256), (1, 512, 188)]
    with pytest.raises(lmkv.LmkvError):
        lmkv.count_chunks([17], [300], 256, True)


class FakeTensor:
    """Stands in for a device tensor in host-validation tests (never dereferenced)."""

    def __init__(self, ptr=0x10000, dtype=None, shape=(1, 64)):
        import torch
        self._ptr = ptr
        self.dtype = dtype or torch.int32
        self.shape = shape

    def data_ptr(self):
        return self._ptr


def fake_pool(num_layers=2, heads=2, head_dim=64, block_size=16, num_blocks=64, elem=2):
    p = lmkv.Pool.__new__(lmkv.Pool)
    p._struct = lmkv._PoolT(0x20000, num_blocks, num_layers, heads, head_dim, block_size, elem)
    return p


def call(fn, pool, start, end, chunk=256, flag=1, bt_cols=64, **kw):
    bt = FakeTensor(shape=(1, bt_cols))
    if fn in (lmkv.gather_layer, lmkv.scatter_layer):
        return fn(pool, bt, start, end, chunk, flag, FakeTensor(0x30000), kw.get("layer", 0),
                  None, 0)
    if fn in (lmkv.gather_chunks_fp8e4m3, lmkv.scatter_chunks_fp8e4m3):
        return fn(pool, bt, start, end, chunk, flag, FakeTensor(0x30000), FakeTensor(0x40000),
                  None, 0)
    return fn(pool, bt, start, end, chunk, flag, FakeTensor(0x30000), None, 0)


ALL = [lmkv.gather_chunks, lmkv.scatter_chunks, lmkv.gather_layer, lmkv.scatter_layer,
       lmkv.gather_chunks_fp8e4m3, lmkv.scatter_chunks_fp8e4m3]


@pytest.mark.parametrize("fn", ALL)
def test_host_validation(lib, fn):
    ok_pool = fake_pool()
    assert call(fn, ok_pool, [17], [300]) == lmkv.ERR_INVALID_ARG          # unaligned start
    assert call(fn, ok_pool, [256], [100]) == lmkv.ERR_INVALID_ARG         # end < start
    assert call(fn, ok_pool, [0], [4096], bt_cols=64) == lmkv.ERR_INVALID_ARG  # table too short
    assert call(fn, ok_pool, [0], [512], chunk=24) == lmkv.ERR_INVALID_ARG  # C % B != 0
    assert call(fn, fake_pool(num_layers=0), [0], [512]) == lmkv.ERR_INVALID_ARG
    assert call(fn, fake_pool(block_size=0), [0], [512]) == lmkv.ERR_INVALID_ARG
    assert call(fn, fake_pool(heads=1, head_dim=3), [0], [512]) == lmkv.ERR_MISALIGNED
    if fn in (lmkv.gather_layer, lmkv.scatter_layer):
        assert call(fn, ok_pool, [0], [512], layer=2) == lmkv.ERR_INVALID_ARG
        assert call(fn, ok_pool, [0], [512], layer=-1) == lmkv.ERR_INVALID_ARG
    if fn in (lmkv.gather_chunks_fp8e4m3, lmkv.scatter_chunks_fp8e4m3):
        assert call(fn, fake_pool(elem=4), [0], [512]) == lmkv.ERR_UNSUPPORTED
        assert call(fn, fake_pool(heads=1, head_dim=8), [0], [512]) == lmkv.ERR_UNSUPPORTED


def test_empty_batch_launches_nothing(lib):
    before = lmkv.launch_count()
    assert call(lmkv.gather_chunks, fake_pool(), [0], [100], flag=0) == lmkv.OK
    assert call(lmkv.scatter_chunks, fake_pool(), [], []) == lmkv.OK
    assert lmkv.launch_count() == before


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(lmkv, "_lib", None)
    monkeypatch.setattr(lmkv, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        lmkv.load()
