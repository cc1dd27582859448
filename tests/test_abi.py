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
    for code in range(10):
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


def test_layer_pipeline_host_validation(lib):
    pool = fake_pool(num_layers=4)
    bt = FakeTensor(shape=(1, 64))
    for fn in (lmkv.store_layers, lmkv.retrieve_layers):
        ptrs = FakeTensor(0x30000)
        assert fn(pool, bt, [0], [512], 256, True, ptrs, 2, 3, None, None, None, 0) == lmkv.ERR_INVALID_ARG
        assert fn(pool, bt, [0], [512], 256, True, ptrs, -1, 1, None, None, None, 0) == lmkv.ERR_INVALID_ARG
        assert fn(pool, bt, [17], [512], 256, True, ptrs, 0, 4, None, None, None, 0) == lmkv.ERR_INVALID_ARG
        before = lmkv.launch_count()
        assert fn(pool, bt, [0], [512], 256, True, ptrs, 1, 0, None, None, None, 0) == lmkv.OK
        assert lmkv.launch_count() == before


def test_staged_pipeline_host_validation(lib):
    import ctypes as C
    pool = fake_pool(num_layers=4)
    bt = FakeTensor(shape=(1, 64))
    need = 2 * 2 * 64 * 2 * 512          # 2 * row_bytes * tokens
    for fn in (lib.lmkv_store_layers_staged, lib.lmkv_retrieve_layers_staged):
        s, e = (C.c_int64 * 1)(0), (C.c_int64 * 1)(512)
        h = (C.c_void_p * 2)(0x50000, 0x60000)
        args = lambda stage, nbytes, lo=0, n=4: fn(pool.struct, 0x10000, 64, s, e, 1, 256, 1, h,
                                                   stage, nbytes, lo, n, None, None, None, 0)
        assert args(0x70000, need - 16) == lmkv.ERR_INVALID_ARG        # staging too small
        assert args(None, need) == lmkv.ERR_INVALID_ARG                # no staging
        assert args(0x70008, need) == lmkv.ERR_MISALIGNED              # misaligned staging
        assert args(0x70000, need, 3, 2) == lmkv.ERR_INVALID_ARG       # layers out of range
        assert args(0x70000, need, 1, 0) == lmkv.OK                    # nothing to do


class FakeWorkspace(FakeTensor):
    def __init__(self, nbytes, ptr=0x50000):
        super().__init__(ptr)
        self.nbytes = nbytes

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1


def test_cachegen_layout_agrees_with_the_oracle(lib):
    """Two independent implementations of the blob layout (the library's and
    the oracle's) give the same offsets and bound, and the same bins rule."""
    from oracle import cachegen as cg
    for L in (1, 3, 9, 10, 11, 32, 80):
        assert lmkv.cachegen_default_bins(L).tolist() == cg.default_bins(L).tolist()
    for L, n, H in [(1, 1, 4), (2, 300, 40), (32, 256, 1024), (32, 768, 1024), (80, 4096, 2048)]:
        bins = cg.default_bins(L)
        a = lmkv.cachegen_layout(L, n, H, bins)
        b = cg.layout(L, n, H, bins)
        assert (a.max1_offset, a.cdf_offset, a.lengths_offset, a.bytes_offset, a.max_bytes) == \
            (b["max1"], b["cdf"], b["lengths"], b["bytes"], b["bound"])


def test_cachegen_host_validation(lib):
    bins = lmkv.cachegen_default_bins(2)
    for args in [(0, 10, 64, bins), (2, 0, 64, bins), (2, 4097, 64, bins), (2, 10, 66, bins),
                 (2, 10, 4096, bins), (2, 10, 64, [2, 16, 16, 16]), (2, 10, 64, [16, 16, 16, 34])]:
        with pytest.raises(lmkv.LmkvError):
            lmkv.cachegen_layout(*args)
    ws = lmkv.cachegen_workspace_bytes(2, 64, [10, 300])
    assert ws > 2 * 2 * 310 * 64
    before = lmkv.launch_count()
    ptrs, sizes = FakeTensor(0x30000), FakeTensor(0x40000)
    for fn in (lmkv.cachegen_encode, lmkv.cachegen_decode):
        def go(ntok=(10, 300), L=2, H=64, b=bins, w=FakeWorkspace(ws)):
            if fn is lmkv.cachegen_encode:
                return fn(ptrs, list(ntok), L, H, b, ptrs, sizes, w, None, 0)
            return fn(ptrs, sizes, list(ntok), L, H, b, ptrs, w, None, 0)
        assert go(w=FakeWorkspace(ws - 1)) == lmkv.ERR_INVALID_ARG       # workspace too small
        assert go(w=FakeWorkspace(ws, ptr=0x50008)) == lmkv.ERR_MISALIGNED
        assert go(ntok=(10, 0)) == lmkv.ERR_INVALID_ARG                    # empty chunk
        assert go(ntok=(5000,)) == lmkv.ERR_INVALID_ARG                    # beyond the token limit
        assert go(H=62) == lmkv.ERR_INVALID_ARG
        assert go(b=[16, 16, 16, 3]) == lmkv.ERR_INVALID_ARG
        assert go(ntok=()) == lmkv.OK                                      # nothing to do
    assert lmkv.launch_count() == before


def test_cachegen_pool_forms_host_validation(lib):
    """The fused store / retrieve validate like the gather and need bf16."""
    bins = lmkv.cachegen_default_bins(2)
    ws = FakeWorkspace(1 << 30)
    bt = FakeTensor(shape=(1, 64))
    for fn in (lmkv.cachegen_store_chunks, lmkv.cachegen_retrieve_chunks):
        args = (FakeTensor(0x30000), FakeTensor(0x40000), ws, None, 0)
        assert fn(fake_pool(), bt, [17], [300], 256, True, bins, *args) == lmkv.ERR_INVALID_ARG
        assert fn(fake_pool(), bt, [0], [4096], 256, True, bins, *args) == lmkv.ERR_INVALID_ARG
        assert fn(fake_pool(elem=4), bt, [0], [512], 256, True, bins, *args) == lmkv.ERR_UNSUPPORTED
        assert fn(fake_pool(), bt, [0], [512], 256, True, [16, 16, 16, 2], *args) == lmkv.ERR_INVALID_ARG
        assert fn(fake_pool(), bt, [0], [100], 256, False, bins, *args) == lmkv.OK   # no chunk


def test_overlapped_pipeline_host_validation(lib):
    """The two-stream staged pipeline needs two layers of staging, a copy
    stream other than the kernel stream and four events; all checked before
    anything is enqueued."""
    import ctypes as C
    pool = fake_pool(num_layers=4)
    need = 2 * 2 * 2 * 64 * 2 * 512      # two layers of 2 * row_bytes * tokens
    ev = (C.c_void_p * 4)(0x1000, 0x2000, 0x3000, 0x4000)
    ev_null = (C.c_void_p * 4)(0x1000, 0, 0x3000, 0x4000)
    for fn in (lib.lmkv_store_layers_overlapped, lib.lmkv_retrieve_layers_overlapped):
        s, e = (C.c_int64 * 1)(0), (C.c_int64 * 1)(512)
        h = (C.c_void_p * 2)(0x50000, 0x60000)

        def call(stage=0x70000, nbytes=need, events=ev, stream=0x111, copy=0x222, n=4):
            return fn(pool.struct, 0x10000, 64, s, e, 1, 256, 1, h, stage, nbytes, 0, n, None, None,
                      events, None, stream, copy)
        assert call(nbytes=need // 2) == lmkv.ERR_INVALID_ARG           # one layer of staging only
        assert call(events=None) == lmkv.ERR_INVALID_ARG
        assert call(events=ev_null) == lmkv.ERR_INVALID_ARG
        assert call(copy=None) == lmkv.ERR_INVALID_ARG
        assert call(copy=0x111) == lmkv.ERR_INVALID_ARG                 # the same stream twice
        assert call(stage=0x70008) == lmkv.ERR_MISALIGNED
        assert call(n=0) == lmkv.OK                                     # nothing to do
