"""The no-allocation staged store (lmkv_store_layers_staged_noalloc).

Some callers cannot allocate device memory at the point where they store KV
cache -- for example a runtime whose device memory is all owned by its own
pool, a process held to a strict memory budget, or a callback path where
cudaMalloc is not allowed.  For them the library offers one entry point that
uses its own built-in staging area instead of a caller buffer.  These tests
call it through the C ABI and compare what it writes with the CPU oracle's
gather of the same batch and with what the ordinary staged store
(caller-provided staging buffer) writes, on two calls in a row with different
batches; they also check the size limit.  This file is collected last so that
a failure here does not stop the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def host_arena(chunks, w):
    total = sum(2 * w.num_layers * n * w.row_elems for _, _, n in chunks)
    flat = torch.zeros(total, dtype=torch.bfloat16, pin_memory=True)
    out, off = [], 0
    for _, _, n in chunks:
        k = 2 * w.num_layers * n * w.row_elems
        out.append(flat[off:off + k].view(2, w.num_layers, n, w.row_elems))
        off += k
    return out


def store_both_ways(w, seed):
    """(no-alloc result, caller-buffer result, oracle result) as lists of host
    arrays of the chunks' bytes."""
    pool = pkg.Pool(wl.make_pool(w, DEV, seed), w.num_kv_heads, w.head_dim)
    table = wl.block_table(w, seed + 1)
    bt = torch.from_numpy(table).to(DEV)
    a = (w.starts, w.ends, w.chunk_size, w.save_unfull)
    chunks = pkg.enumerate_chunks(*a)
    mine, ref = host_arena(chunks, w), host_arena(chunks, w)
    staging = torch.empty(pkg.staging_bytes(pool, *a), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    pkg.check(pkg.lmkv.store_layers_staged_noalloc(pool, bt, *a, mine, 0, w.num_layers,
                                              status=status))
    pkg.check(pkg.store_layers_staged(pool, bt, *a, ref, staging, 0, w.num_layers,
                                      status=status))
    torch.cuda.synchronize()
    assert status.item() == 0
    host = [t.cpu().view(torch.uint8).numpy().reshape(t.shape[:3] + (w.row_bytes,)) for t in pool.layers]
    want = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    assert oracle.gather(oracle.HostPool(host, w.block_size), table, *a, want) == 0
    as_bytes = lambda ts: [t.view(torch.uint8).numpy().reshape(o.shape) for t, o in zip(ts, want)]
    return as_bytes(mine), as_bytes(ref), want


def test_two_calls_match_the_caller_buffer_form():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    first = wl.Workload("a", 6, 2, 64, 16, 160, (700, 300), chunk_size=256)
    second = wl.Workload("b", 4, 8, 128, 16, 1024, (10240,), chunk_size=256)   # 42 MB per layer
    for w, seed in ((first, 10), (second, 20)):
        mine, ref, want = store_both_ways(w, seed)
        for g, (x, y, z) in enumerate(zip(mine, ref, want)):
            np.testing.assert_array_equal(x, z, err_msg=f"{w.name} chunk {g} against the oracle")
            np.testing.assert_array_equal(x, y, err_msg=f"{w.name} chunk {g} against the staged store")
            assert (x != 0).any()


def test_batch_beyond_the_staging_area_is_rejected():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = wl.Workload("big", 2, 8, 128, 16, 2048, (16640,), chunk_size=256)   # 68 MB per layer
    pool = pkg.Pool(wl.make_pool(w, DEV, 0), w.num_kv_heads, w.head_dim)
    bt = torch.from_numpy(wl.block_table(w, 1)).to(DEV)
    a = (w.starts, w.ends, w.chunk_size, w.save_unfull)
    assert pkg.staging_bytes(pool, *a) > pkg.lmkv.NOALLOC_STAGING_BYTES
    chunks = pkg.enumerate_chunks(*a)
    host = host_arena(chunks, w)
    before = pkg.lmkv.launch_count()
    rc = pkg.lmkv.store_layers_staged_noalloc(pool, bt, *a, host, 0, w.num_layers)
    assert rc == pkg.lmkv.ERR_SCRATCH_LIMIT
    assert pkg.lmkv.launch_count() == before
    assert all(int((h.view(torch.int16) != 0).sum()) == 0 for h in host)
