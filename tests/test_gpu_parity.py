"""GPU parity of the copy kernels against the CPU oracle (bit-exact).

Movement rule: "LMCache: An Efficient KV Cache Layer for Enterprise-Scale LLM Inference", section on the
configurable chunk size (pages ->
contiguous chunk buffers and back) and layer-wise pipeline section (one layer
per call); chunking rule from the cache_engine.py walk-through, "store()".
All calls go through the C ABI (liblmkv.so) via the ctypes binding.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl
from gpu_util import (DEV, alloc_chunks, compact_subbatch, device_pool, host_bytes,
                      new_status, nonsentinel_rows, oracle_chunks_for, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def run_small_case(w, table, table2, flag, layer_wise=False, seed=0):
    """Gather + scatter on the GPU and on the oracle; compare every byte."""
    pool = device_pool(w, seed)
    bt = torch.from_numpy(table).to(DEV)
    bt2 = torch.from_numpy(table2).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, w.chunk_size, flag)
    assert chunks == oracle.enumerate_chunks(w.starts, w.ends, w.chunk_size, flag)
    dt = pool.layers[0].dtype
    bufs, ptrs = alloc_chunks(chunks, w, dtype=dt, fill=0x5A)
    st = new_status()
    if layer_wise:
        for l in range(w.num_layers):
            pkg.check(pkg.gather_layer(pool, bt, w.starts, w.ends, w.chunk_size, flag, ptrs, l, st))
    else:
        pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, w.chunk_size, flag, ptrs, st))
    pool2 = device_pool(w, None, fill="sentinel")
    if layer_wise:
        for l in range(w.num_layers):
            pkg.check(pkg.scatter_layer(pool2, bt2, w.starts, w.ends, w.chunk_size, flag, ptrs, l, st))
    else:
        pkg.check(pkg.scatter_chunks(pool2, bt2, w.starts, w.ends, w.chunk_size, flag, ptrs, st))
    torch.cuda.synchronize()
    assert st.item() == 0

    host = [host_bytes(t) for t in pool.layers]
    ref = [np.full((2, w.num_layers, n, w.row_bytes), 0x5A, np.uint8) for _, _, n in chunks]
    assert oracle.gather(oracle.HostPool(host, w.block_size), table, w.starts, w.ends,
                         w.chunk_size, flag, ref) == 0
    for g, (a, b) in enumerate(zip(bufs, ref)):
        np.testing.assert_array_equal(host_bytes(a), b, err_msg=f"gather chunk {g}")
    h2 = [np.full_like(a, wl.SENTINEL_BYTE) for a in host]
    assert oracle.scatter(oracle.HostPool(h2, w.block_size), table2, w.starts, w.ends,
                          w.chunk_size, flag, ref) == 0
    for l, (t, h) in enumerate(zip(pool2.layers, h2)):
        np.testing.assert_array_equal(host_bytes(t), h, err_msg=f"scatter layer {l}")
    return chunks


@pytest.mark.parametrize("layer_wise", [False, True])
def test_tiny_workload(layer_wise):
    w = wl.TINY
    run_small_case(w, wl.block_table(w, 0, tiny_subset=w.num_blocks), wl.block_table(w, 1),
                   True, layer_wise)


SHAPES = [
    # L, H, D, B, nb, ends, starts, C, elem, flag
    (3, 2, 64, 16, 96, (300, 1000, 17), (0, 256, 0), 256, 2, True),
    (3, 2, 64, 16, 96, (300, 1000, 17), (0, 256, 0), 256, 2, False),
    (2, 1, 8, 1, 700, (600,), (0,), 16, 2, True),         # one-token pages
    (2, 4, 32, 2, 300, (333, 64), (64, 0), 64, 4, True),  # fp32 rows
    (4, 1, 16, 4, 256, (255, 1, 700), (0, 0, 512), 128, 1, True),  # 16-byte rows
    (2, 8, 128, 32, 64, (900,), (0,), 256, 2, True),      # 64 KiB pages
    (2, 8, 128, 64, 32, (1100,), (256,), 256, 2, True),   # 128 KiB pages
    (2, 8, 128, 64, 40, (1000,), (0,), 256, 4, True),     # 256 KiB pages (fp32 rows): 8 items each
    (1, 2, 64, 16, 64, (0, 256, 256), (0, 0, 256), 256, 2, True),  # empty requests
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
@pytest.mark.parametrize("layer_wise", [False, True])
def test_random_shapes(shape, layer_wise):
    L, H, D, B, nb, ends, starts, C, elem, flag = shape
    w = wl.Workload("s", L, H, D, B, nb, ends, req_start=starts, chunk_size=C, elem_bytes=elem,
                    save_unfull=flag)
    run_small_case(w, wl.block_table(w, 3), wl.block_table(w, 4), flag, layer_wise, seed=5)


def test_many_requests_split_over_launches():
    """More requests than one launch's parameter block holds (256)."""
    rng = np.random.default_rng(8)
    n = 300
    ends = tuple(int(x) for x in rng.integers(0, 80, n))
    w = wl.Workload("many", 2, 1, 16, 4, 8000, ends, chunk_size=16)
    before = pkg.lmkv.launch_count()
    run_small_case(w, wl.block_table(w, 5), wl.block_table(w, 6), True)
    assert pkg.lmkv.launch_count() - before == 4      # 2 launches each for gather and scatter


def test_bad_block_ids_skip_and_report():
    w = wl.Workload("bad", 2, 1, 64, 4, 64, (40,), chunk_size=8)
    table = wl.block_table(w, 1)
    table[0, 2] = 64
    table[0, 5] = -7
    pool = device_pool(w, 0)
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 8, True)
    bufs, ptrs = alloc_chunks(chunks, w, fill=0x33)
    st = new_status()
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, 8, True, ptrs, st))
    torch.cuda.synchronize()
    assert st.item() == pkg.lmkv.ERR_BAD_BLOCK
    host = [host_bytes(t) for t in pool.layers]
    ref = [np.full((2, 2, n, w.row_bytes), 0x33, np.uint8) for _, _, n in chunks]
    assert oracle.gather(oracle.HostPool(host, 4), table, w.starts, w.ends, 8, True, ref) == \
        oracle.BAD_BLOCK
    for a, b in zip(bufs, ref):
        np.testing.assert_array_equal(host_bytes(a), b)
    st.zero_()
    pool2 = device_pool(w, None, fill="sentinel")
    pkg.check(pkg.scatter_chunks(pool2, bt, w.starts, w.ends, 8, True, ptrs, st))
    torch.cuda.synchronize()
    assert st.item() == pkg.lmkv.ERR_BAD_BLOCK


def test_null_chunk_pointer_reported():
    w = wl.TINY
    pool = device_pool(w, 0)
    bt = torch.from_numpy(wl.block_table(w, 0)).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 256, True)
    bufs, ptrs = alloc_chunks(chunks, w, fill=0)
    ptrs[1] = 0
    st = new_status()
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, 256, True, ptrs, st))
    torch.cuda.synchronize()
    assert st.item() == pkg.lmkv.ERR_BAD_POINTER
    assert (bufs[1] == 0).all()


def test_deterministic():
    w = wl.TINY
    pool = device_pool(w, 0)
    bt = torch.from_numpy(wl.block_table(w, 0)).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 256, True)
    a, pa = alloc_chunks(chunks, w, fill=1)
    b, pb = alloc_chunks(chunks, w, fill=2)
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, 256, True, pa))
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, 256, True, pb))
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


# ---------------------------------------------------------------------------
# Full-size workloads (the launch configuration the bench times), sampled.

def test_llama8b_full_gather_scatter_and_layer_wise():
    w = wl.LLAMA8B
    pool = device_pool(w, 0)
    t1 = wl.block_table(w, 1)
    t2 = wl.block_table(w, 2)
    bt, bt2 = torch.from_numpy(t1).to(DEV), torch.from_numpy(t2).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 256, True)
    assert len(chunks) == 40
    bufs, ptrs = alloc_chunks(chunks, w)
    st = new_status()
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, 256, True, ptrs, st))
    torch.cuda.synchronize()
    # every chunk against the oracle (the 640 referenced blocks copied to the host)
    ref = oracle_chunks_for(pool.layers, t1, chunks, list(range(40)), 256, 32, w.row_bytes)
    for g in range(40):
        np.testing.assert_array_equal(host_bytes(bufs[g]), ref[g], err_msg=f"chunk {g}")
    # layer-wise gather reproduces the full gather
    lbufs, lptrs = alloc_chunks(chunks, w, fill=0)
    for l in range(w.num_layers):
        pkg.check(pkg.gather_layer(pool, bt, w.starts, w.ends, 256, True, lptrs, l, st))
    torch.cuda.synchronize()
    for a, b in zip(bufs, lbufs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    del lbufs, lptrs
    # scatter into a second pool under another table
    pool2 = device_pool(w, None, fill="sentinel")
    pkg.check(pkg.scatter_chunks(pool2, bt2, w.starts, w.ends, 256, True, ptrs, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    assert nonsentinel_rows(pool2.layers) == 2 * 32 * 10240
    sample = [0, 17, 39]
    hp, tab, s, e, _ = compact_subbatch(pool2.layers, t2, chunks, sample)
    hs = [np.full_like(a, wl.SENTINEL_BYTE) for a in hp.layers]
    assert oracle.scatter(oracle.HostPool(hs, 16), tab, s, e, 256, True, [ref[g] for g in sample]) == 0
    for a, b in zip(hp.layers, hs):
        np.testing.assert_array_equal(a, b)
    # layer-wise scatter into a third pool equals the full scatter
    del hp, hs
    pool3 = device_pool(w, None, fill="sentinel")
    for l in range(w.num_layers):
        pkg.check(pkg.scatter_layer(pool3, bt2, w.starts, w.ends, 256, True, ptrs, l, st))
    torch.cuda.synchronize()
    for a, b in zip(pool2.layers, pool3.layers):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert st.item() == 0


@pytest.mark.parametrize("flag", [True, False])
def test_llama70b_batch_sampled(flag):
    """160 GiB pool, 4 requests with partial last chunks, interleaved tables;
    scatter into disjoint unused blocks of the same pool."""
    w = wl.LLAMA70B.with_(save_unfull=flag)
    t1 = wl.block_table(w, 1)
    used = set(int(x) for x in t1[t1 >= 0])
    t2 = wl.block_table(w, 2, exclude=used)
    assert not used & set(int(x) for x in t2[t2 >= 0])
    layers = wl.make_pool(w, DEV, None, fill="sentinel")
    ids = torch.as_tensor(sorted(used), dtype=torch.long, device=DEV)
    for l, t in enumerate(layers):
        vals = torch.empty((2, len(ids), w.block_size, w.row_elems), dtype=torch.bfloat16, device=DEV)
        wl.fill_normal_(vals, 1000 + l)
        t.index_copy_(1, ids, vals)
    del vals
    pool = pkg.Pool(layers, w.num_kv_heads, w.head_dim)
    bt, bt2 = torch.from_numpy(t1).to(DEV), torch.from_numpy(t2).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 256, flag)
    assert len(chunks) == (259 if flag else 257)
    bufs, ptrs = alloc_chunks(chunks, w)
    st = new_status()
    before = nonsentinel_rows(pool.layers)
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, 256, flag, ptrs, st))
    pkg.check(pkg.scatter_chunks(pool, bt2, w.starts, w.ends, 256, flag, ptrs, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    n_tok = sum(n for _, _, n in chunks)
    assert nonsentinel_rows(pool.layers) == before + 2 * w.num_layers * n_tok
    last = np.cumsum([len(pkg.enumerate_chunks([0], [e], 256, flag)) for e in w.ends]) - 1
    sample = sorted(set([0, 16, int(last[1]), int(last[2]), int(last[3])] +
                        list(np.random.default_rng(0).integers(0, len(chunks), 3))))
    ref = oracle_chunks_for(pool.layers, t1, chunks, sample, 256, w.num_layers, w.row_bytes)
    for g, r in zip(sample, ref):
        np.testing.assert_array_equal(host_bytes(bufs[g]), r, err_msg=f"chunk {g}")
    hp, tab, s, e, _ = compact_subbatch(pool.layers, t2, chunks, sample)
    hs = [np.full_like(a, wl.SENTINEL_BYTE) for a in hp.layers]
    # the compact copy of the scatter target holds only the sampled chunks' blocks; slots past
    # a partial chunk's end keep the sentinel on both sides
    assert oracle.scatter(oracle.HostPool(hs, 16), tab, s, e, 256, True, ref) == 0
    for a, b in zip(hp.layers, hs):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("block_size", [16, 32, 64])
def test_qwen32b_bf16_full_size_sampled(block_size):
    """Qwen2.5-32B shape (64 layers, one 16384-token request) on 16-, 32- and
    64-token pages, the launches the bench times for this shape: pages of
    64 / 128 KiB move as 32 KiB items.  Whole-batch gather against the oracle
    on sampled chunks; per-layer gather equal to it; whole-batch and per-layer
    scatter equal to each other and, on the sampled chunks, to the oracle."""
    w = wl.qwen_with_block_size(block_size)
    pool = device_pool(w, 0)
    t1, t2 = wl.block_table(w, 1), wl.block_table(w, 2)
    bt, bt2 = torch.from_numpy(t1).to(DEV), torch.from_numpy(t2).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 256, True)
    assert len(chunks) == 64
    bufs, ptrs = alloc_chunks(chunks, w)
    st = new_status()
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, 256, True, ptrs, st))
    torch.cuda.synchronize()
    sample = [0, 33, 63]
    ref = oracle_chunks_for(pool.layers, t1, chunks, sample, 256, w.num_layers, w.row_bytes)
    for g, r in zip(sample, ref):
        np.testing.assert_array_equal(host_bytes(bufs[g]), r, err_msg=f"chunk {g}")
    lbufs, lptrs = alloc_chunks(chunks, w, fill=0)
    for l in range(w.num_layers):
        pkg.check(pkg.gather_layer(pool, bt, w.starts, w.ends, 256, True, lptrs, l, st))
    torch.cuda.synchronize()
    for a, b in zip(bufs, lbufs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    del lbufs, lptrs, pool
    torch.cuda.empty_cache()
    pool2 = device_pool(w, None, fill="sentinel")
    pkg.check(pkg.scatter_chunks(pool2, bt2, w.starts, w.ends, 256, True, ptrs, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    assert nonsentinel_rows(pool2.layers) == 2 * w.num_layers * 16384
    hp, tab, s, e, _ = compact_subbatch(pool2.layers, t2, chunks, sample)
    hs = [np.full_like(a, wl.SENTINEL_BYTE) for a in hp.layers]
    assert oracle.scatter(oracle.HostPool(hs, block_size), tab, s, e, 256, True, ref) == 0
    for a, b in zip(hp.layers, hs):
        np.testing.assert_array_equal(a, b)
    del hp, hs
    pool3 = device_pool(w, None, fill="sentinel")
    for l in range(w.num_layers):
        pkg.check(pkg.scatter_layer(pool3, bt2, w.starts, w.ends, 256, True, ptrs, l, st))
    torch.cuda.synchronize()
    for a, b in zip(pool2.layers, pool3.layers):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert st.item() == 0


def test_llama70b_per_layer_and_fp8_sampled():
    """The 70B batch as the bench times it (160 GiB pool, interleaved tables,
    partial last chunks): the 80 per-layer gathers equal the whole-batch gather
    and, on sampled chunks, the oracle; the per-layer scatters into disjoint
    unused blocks of the same pool and the fp8 pair (dequantised into a third
    disjoint set of blocks) match the oracle on the sampled chunks."""
    w = wl.LLAMA70B
    L = w.num_layers
    t1 = wl.block_table(w, 1)
    used = set(int(x) for x in t1[t1 >= 0])
    t2 = wl.block_table(w, 2, exclude=used)
    used2 = used | set(int(x) for x in t2[t2 >= 0])
    t3 = wl.block_table(w, 3, exclude=used2)
    layers = wl.make_pool(w, DEV, None, fill="sentinel")
    ids = torch.as_tensor(sorted(used), dtype=torch.long, device=DEV)
    for l, t in enumerate(layers):
        vals = torch.empty((2, len(ids), w.block_size, w.row_elems), dtype=torch.bfloat16, device=DEV)
        wl.fill_normal_(vals, 1000 + l)
        t.index_copy_(1, ids, vals)
    del vals
    pool = pkg.Pool(layers, w.num_kv_heads, w.head_dim)
    bt, bt2, bt3 = (torch.from_numpy(t).to(DEV) for t in (t1, t2, t3))
    a = (w.starts, w.ends, 256, True)
    chunks = pkg.enumerate_chunks(*a)
    assert len(chunks) == 259
    bufs, ptrs = alloc_chunks(chunks, w)
    lbufs, lptrs = alloc_chunks(chunks, w, fill=0)
    st = new_status()
    pkg.check(pkg.gather_chunks(pool, bt, *a, ptrs, st))
    for l in range(L):
        pkg.check(pkg.gather_layer(pool, bt, *a, lptrs, l, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    for g, (x, y) in enumerate(zip(bufs, lbufs)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), f"per-layer gather, chunk {g}"
    last = np.cumsum([len(pkg.enumerate_chunks([0], [e], 256, True)) for e in w.ends]) - 1
    sample = sorted(set([0, 16, int(last[1]), int(last[2]), int(last[3]), 130]))
    ref = oracle_chunks_for(pool.layers, t1, chunks, sample, 256, L, w.row_bytes)
    for g, r in zip(sample, ref):
        np.testing.assert_array_equal(host_bytes(lbufs[g]), r, err_msg=f"chunk {g}")
    del lbufs, lptrs
    torch.cuda.empty_cache()
    # per-layer scatter into the second set of blocks
    for l in range(L):
        pkg.check(pkg.scatter_layer(pool, bt2, *a, ptrs, l, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    hp, tab, s, e, _ = compact_subbatch(pool.layers, t2, chunks, sample)
    hs = [np.full_like(x, wl.SENTINEL_BYTE) for x in hp.layers]
    assert oracle.scatter(oracle.HostPool(hs, 16), tab, s, e, 256, True, ref) == 0
    for x, y in zip(hp.layers, hs):
        np.testing.assert_array_equal(x, y)
    del bufs, ptrs, hp, hs
    torch.cuda.empty_cache()
    # fp8 pair: quantise from the first set, dequantise into the third
    codes, cptrs = alloc_chunks(chunks, w, dtype=torch.uint8, fill=0xEE)
    scales = torch.full((len(chunks), 2, L), -1.0, dtype=torch.float32, device=DEV)
    pkg.check(pkg.gather_chunks_fp8e4m3(pool, bt, *a, cptrs, scales, st))
    pkg.check(pkg.scatter_chunks_fp8e4m3(pool, bt3, *a, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    hp, tab, s, e, _ = compact_subbatch(pool.layers, t1, chunks, sample)
    hp16 = oracle.HostPool([x.view(np.uint16) for x in hp.layers], 16)
    rc = [np.zeros((2, L, chunks[g][2], w.row_elems), np.uint8) for g in sample]
    rs = np.zeros((len(sample), 2, L), np.float32)
    assert oracle.gather_fp8(hp16, tab, s, e, 256, True, rc, rs) == 0
    for i, g in enumerate(sample):
        np.testing.assert_array_equal(scales[g].cpu().numpy().view(np.uint32), rs[i].view(np.uint32))
        np.testing.assert_array_equal(codes[g].cpu().numpy(), rc[i], err_msg=f"codes chunk {g}")
    hq, tab3, s3, e3, _ = compact_subbatch(pool.layers, t3, chunks, sample)
    h3 = [np.full(x.shape[:3] + (x.shape[3] // 2,), wl.SENTINEL_BF16, np.uint16) for x in hq.layers]
    assert oracle.scatter_fp8(oracle.HostPool(h3, 16), tab3, s3, e3, 256, True, rc, rs) == 0
    for x, y in zip(hq.layers, h3):
        np.testing.assert_array_equal(x.view(np.uint16), y)
