"""Layer-wise pipeline entry points (lmkv_store_layers / lmkv_retrieve_layers).

LMCache paper, layer-wise pipeline section: compute and data movement run on
separate CUDA streams; layer i's KV moves while another layer computes.  Data
must equal the oracle; events must order each layer's movement against the
compute stream.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl
from gpu_util import DEV, alloc_chunks, device_pool, host_bytes, new_status, require_gpu

pytestmark = pytest.mark.gpu

W = wl.Workload("pipe", 6, 2, 64, 16, 160, (700, 300), chunk_size=256)


def host_chunks(chunks, w, arena=False):
    """Pinned host chunk buffers: separate allocations, or consecutive slices of
    one allocation (which the staged pipeline moves with one 3-D copy per run of
    full chunks)."""
    if arena:
        total = sum(2 * w.num_layers * n * w.row_elems for _, _, n in chunks)
        flat = torch.zeros(total, dtype=torch.bfloat16, pin_memory=True)
        bufs, off = [], 0
        for _, _, n in chunks:
            k = 2 * w.num_layers * n * w.row_elems
            bufs.append(flat[off:off + k].view(2, w.num_layers, n, w.row_elems))
            off += k
    else:
        bufs = [torch.zeros((2, w.num_layers, n, w.row_elems), dtype=torch.bfloat16, pin_memory=True)
                for _, _, n in chunks]
    return bufs, pkg.pointer_array(bufs, DEV)


@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_store_layers_gated_by_compute_events(where):
    require_gpu()
    w = W
    pool = device_pool(w, 0)
    table = wl.block_table(w, 1)
    bt = torch.from_numpy(table).to(DEV)
    a = (w.starts, w.ends, w.chunk_size, True)
    chunks = pkg.enumerate_chunks(*a)
    bufs, ptrs = alloc_chunks(chunks, w, fill=0) if where == "device" else host_chunks(chunks, w)
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    # the "compute" stream rewrites each layer (x2) and then marks it ready
    ready = [torch.cuda.Event() for _ in range(w.num_layers)]
    with torch.cuda.stream(compute):
        for l in range(w.num_layers):
            torch.cuda._sleep(200_000)
            pool.layers[l].mul_(2)
            ready[l].record(compute)
    st = new_status()
    pkg.check(pkg.store_layers(pool, bt, *a, ptrs, 0, w.num_layers, ready, None, st, copy))
    torch.cuda.synchronize()
    assert st.item() == 0
    host = [host_bytes(t) for t in pool.layers]        # the doubled values
    ref = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    assert oracle.gather(oracle.HostPool(host, w.block_size), table, *a, ref) == 0
    for g, (x, r) in enumerate(zip(bufs, ref)):
        np.testing.assert_array_equal(host_bytes(x), r, err_msg=f"chunk {g}")


@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_retrieve_layers_signals_each_layer(where):
    require_gpu()
    w = W
    src = device_pool(w, 0)
    t1, t2 = wl.block_table(w, 1), wl.block_table(w, 2)
    a = (w.starts, w.ends, w.chunk_size, True)
    chunks = pkg.enumerate_chunks(*a)
    bufs, ptrs = alloc_chunks(chunks, w, fill=0) if where == "device" else host_chunks(chunks, w)
    pkg.check(pkg.gather_chunks(src, torch.from_numpy(t1).to(DEV), *a, ptrs))
    dst = device_pool(w, None, fill="sentinel")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    done = [torch.cuda.Event() for _ in range(w.num_layers)]
    for e in done:
        e.record(copy)                                 # create the events
    st = new_status()
    pkg.check(pkg.retrieve_layers(dst, torch.from_numpy(t2).to(DEV), *a, ptrs, 0, w.num_layers,
                                  None, done, st, copy))
    snaps = []
    with torch.cuda.stream(compute):
        for l in range(w.num_layers):
            compute.wait_event(done[l])
            snaps.append(dst.layers[l].clone())        # what layer l's compute would read
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_chunks = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    assert oracle.gather(oracle.HostPool([host_bytes(t) for t in src.layers], w.block_size), t1, *a,
                         ref_chunks) == 0
    ref = [np.full((2, w.num_blocks, w.block_size, w.row_bytes), wl.SENTINEL_BYTE, np.uint8)
           for _ in range(w.num_layers)]
    assert oracle.scatter(oracle.HostPool(ref, w.block_size), t2, *a, ref_chunks) == 0
    for l in range(w.num_layers):
        np.testing.assert_array_equal(host_bytes(snaps[l]), ref[l], err_msg=f"layer {l}")


STAGED = [
    W,                                                                    # 2 requests, partial chunk
    wl.Workload("many", 3, 1, 16, 4, 24000, tuple(range(0, 600, 2)), chunk_size=16),  # 300 requests
    W.with_(save_unfull=False),
    # 64-token pages of 2 KiB rows: each page moves as four 32 KiB items
    wl.Workload("bigpage", 3, 8, 128, 64, 48, (900, 300), chunk_size=256),
]


@pytest.mark.parametrize("arena", [False, True], ids=["separate", "arena"])
@pytest.mark.parametrize("w", STAGED, ids=["two", "many", "no_tail", "big_pages"])
def test_staged_store_and_retrieve_vs_oracle(w, arena):
    require_gpu()
    pool = device_pool(w, 0)
    t1, t2 = wl.block_table(w, 1), wl.block_table(w, 2)
    a = (w.starts, w.ends, w.chunk_size, w.save_unfull)
    chunks = pkg.enumerate_chunks(*a)
    hbufs, _ = host_chunks(chunks, w, arena)
    staging = torch.empty(max(pkg.staging_bytes(pool, *a), 16), dtype=torch.uint8, device=DEV)
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    ready = [torch.cuda.Event() for _ in range(w.num_layers)]
    done = [torch.cuda.Event() for _ in range(w.num_layers)]
    for e in done:
        e.record(copy)
    with torch.cuda.stream(compute):
        for l in range(w.num_layers):
            torch.cuda._sleep(100_000)
            ready[l].record(compute)
    st = new_status()
    pkg.check(pkg.store_layers_staged(pool, torch.from_numpy(t1).to(DEV), *a, hbufs, staging, 0,
                                      w.num_layers, ready, None, st, copy))
    torch.cuda.synchronize()
    assert st.item() == 0
    host = [host_bytes(t) for t in pool.layers]
    ref = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    assert oracle.gather(oracle.HostPool(host, w.block_size), t1, *a, ref) == 0
    for g, (x, r) in enumerate(zip(hbufs, ref)):
        np.testing.assert_array_equal(host_bytes(x), r, err_msg=f"stored chunk {g}")
    # retrieve into a sentinel pool; the compute stream snapshots layer l after done[l]
    dst = device_pool(w, None, fill="sentinel")
    torch.cuda.synchronize()
    pkg.check(pkg.retrieve_layers_staged(dst, torch.from_numpy(t2).to(DEV), *a, hbufs, staging, 0,
                                         w.num_layers, None, done, st, copy))
    snaps = []
    with torch.cuda.stream(compute):
        for l in range(w.num_layers):
            compute.wait_event(done[l])
            snaps.append(dst.layers[l].clone())
    torch.cuda.synchronize()
    assert st.item() == 0
    exp = [np.full((2, w.num_blocks, w.block_size, w.row_bytes), wl.SENTINEL_BYTE, np.uint8)
           for _ in range(w.num_layers)]
    assert oracle.scatter(oracle.HostPool(exp, w.block_size), t2, *a, ref) == 0
    for l in range(w.num_layers):
        np.testing.assert_array_equal(host_bytes(snaps[l]), exp[l], err_msg=f"layer {l}")


def test_staged_layer_range():
    """A sub-range of layers moves only those layers' slices."""
    require_gpu()
    w = W
    pool = device_pool(w, 0)
    t1 = wl.block_table(w, 1)
    a = (w.starts, w.ends, w.chunk_size, True)
    chunks = pkg.enumerate_chunks(*a)
    hbufs, _ = host_chunks(chunks, w, arena=True)
    for h in hbufs:
        h.view(torch.uint8).fill_(0x77)
    staging = torch.empty(pkg.staging_bytes(pool, *a), dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    pkg.check(pkg.store_layers_staged(pool, torch.from_numpy(t1).to(DEV), *a, hbufs, staging, 2, 3))
    torch.cuda.synchronize()
    ref = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    oracle.gather(oracle.HostPool([host_bytes(t) for t in pool.layers], w.block_size), t1, *a, ref)
    for x, r in zip(hbufs, ref):
        got = host_bytes(x)
        np.testing.assert_array_equal(got[:, 2:5], r[:, 2:5])
        assert (got[:, :2] == 0x77).all() and (got[:, 5:] == 0x77).all()


@pytest.mark.parametrize("arena", [False, True], ids=["separate", "arena"])
@pytest.mark.parametrize("w", STAGED, ids=["two", "many", "no_tail", "big_pages"])
def test_overlapped_store_and_retrieve_vs_oracle(w, arena):
    """The two-stream form (two staging halves, copies on their own stream)
    stores and retrieves exactly what the oracle's gather / scatter give, with
    the per-layer ready / done events honoured: the compute stream reads layer
    l after done[l] of the retrieve."""
    require_gpu()
    pool = device_pool(w, 0)
    t1, t2 = wl.block_table(w, 1), wl.block_table(w, 2)
    a = (w.starts, w.ends, w.chunk_size, w.save_unfull)
    chunks = pkg.enumerate_chunks(*a)
    hbufs, _ = host_chunks(chunks, w, arena)
    staging = torch.empty(2 * max(pkg.staging_bytes(pool, *a), 16), dtype=torch.uint8, device=DEV)
    compute, kern, copy = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sync = pkg.overlap_events(kern)
    torch.cuda.synchronize()
    ready = [torch.cuda.Event() for _ in range(w.num_layers)]
    done = [torch.cuda.Event() for _ in range(w.num_layers)]
    for e in done:
        e.record(copy)
    with torch.cuda.stream(compute):
        for l in range(w.num_layers):
            torch.cuda._sleep(100_000)
            ready[l].record(compute)
    st = new_status()
    pkg.check(pkg.store_layers_overlapped(pool, torch.from_numpy(t1).to(DEV), *a, hbufs, staging, 0,
                                          w.num_layers, sync, ready, None, st, kern, copy))
    kern.synchronize()                       # the call's work ends on the kernel stream
    assert st.item() == 0
    host = [host_bytes(t) for t in pool.layers]
    ref = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    assert oracle.gather(oracle.HostPool(host, w.block_size), t1, *a, ref) == 0
    for g, (x, r) in enumerate(zip(hbufs, ref)):
        np.testing.assert_array_equal(host_bytes(x), r, err_msg=f"stored chunk {g}")
    dst = device_pool(w, None, fill="sentinel")
    torch.cuda.synchronize()
    pkg.check(pkg.retrieve_layers_overlapped(dst, torch.from_numpy(t2).to(DEV), *a, hbufs, staging, 0,
                                             w.num_layers, sync, None, done, st, kern, copy))
    snaps = []
    with torch.cuda.stream(compute):
        for l in range(w.num_layers):
            compute.wait_event(done[l])
            snaps.append(dst.layers[l].clone())
    torch.cuda.synchronize()
    assert st.item() == 0
    exp = [np.full((2, w.num_blocks, w.block_size, w.row_bytes), wl.SENTINEL_BYTE, np.uint8)
           for _ in range(w.num_layers)]
    assert oracle.scatter(oracle.HostPool(exp, w.block_size), t2, *a, ref) == 0
    for l in range(w.num_layers):
        np.testing.assert_array_equal(host_bytes(snaps[l]), exp[l], err_msg=f"layer {l}")


def test_overlapped_store_per_layer_done_events():
    """Store: done[l] fires only once layer l's rows are on the host (the host
    reads them after synchronising on the event alone)."""
    require_gpu()
    w = W
    pool = device_pool(w, 0)
    t1 = wl.block_table(w, 1)
    a = (w.starts, w.ends, w.chunk_size, True)
    chunks = pkg.enumerate_chunks(*a)
    hbufs, _ = host_chunks(chunks, w, arena=True)
    for h in hbufs:
        h.view(torch.uint8).fill_(0x77)
    staging = torch.empty(2 * pkg.staging_bytes(pool, *a), dtype=torch.uint8, device=DEV)
    kern, copy = torch.cuda.Stream(), torch.cuda.Stream()
    sync = pkg.overlap_events(kern)
    done = [torch.cuda.Event() for _ in range(w.num_layers)]
    for e in done:
        e.record(copy)
    torch.cuda.synchronize()
    pkg.check(pkg.store_layers_overlapped(pool, torch.from_numpy(t1).to(DEV), *a, hbufs, staging, 0,
                                          w.num_layers, sync, None, done, None, kern, copy))
    ref = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    oracle.gather(oracle.HostPool([host_bytes(t) for t in pool.layers], w.block_size), t1, *a, ref)
    for l in range(w.num_layers):
        done[l].synchronize()
        for x, r in zip(hbufs, ref):
            np.testing.assert_array_equal(host_bytes(x)[:, l], r[:, l], err_msg=f"layer {l}")
    torch.cuda.synchronize()
