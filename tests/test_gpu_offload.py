"""Backing up free pages on the GPU: the planned range of the free list is
stored with one page per chunk (block_size-token chunks whose block table is
the free list) through the staged store; the host copies equal the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl
from gpu_util import DEV, device_pool, host_bytes, new_status, require_gpu

pytestmark = pytest.mark.gpu


def test_backup_steps_copy_the_planned_pages():
    require_gpu()
    w = wl.Workload("free", 4, 2, 64, 16, 256, (16,), chunk_size=16)
    pool = device_pool(w, 0)
    rng = np.random.default_rng(2)
    free_list = rng.permutation(w.num_blocks)[:120].astype(np.int32)[None, :]   # engine's free order
    fl = torch.from_numpy(free_list).to(DEV)
    B = w.block_size
    o = pkg.Offload(num_free=120, window=48)
    page_bytes = 2 * w.num_layers * B * w.row_bytes
    backups = {}
    staging = torch.empty(2 * w.row_bytes * 10 * B, dtype=torch.uint8, device=DEV)
    st = new_status()
    torch.cuda.synchronize()
    for step in range(12):
        first, count = o.plan(10)
        if count:
            host = [torch.empty((2, w.num_layers, B, w.row_elems), dtype=torch.bfloat16,
                                pin_memory=True) for _ in range(count)]
            s, e = np.array([first * B]), np.array([(first + count) * B])
            pkg.check(pkg.store_layers_staged(pool, fl, s, e, B, False, host, staging, 0,
                                              w.num_layers, status=st))
            torch.cuda.synchronize()
            for i, h in enumerate(host):
                backups[first + i] = host_bytes(h)
            o.copied(count)
        o.allocate(int(rng.integers(0, 9)))
    assert st.item() == 0 and len(backups) == o.state.current
    # oracle: the same pages gathered as block_size-token chunks of the free list
    n = o.state.current
    ref = [np.zeros((2, w.num_layers, B, w.row_bytes), np.uint8) for _ in range(n)]
    host_pool = oracle.HostPool([host_bytes(t) for t in pool.layers], B)
    assert oracle.gather(host_pool, free_list, [0], [n * B], B, False, ref) == 0
    for pos in range(n):
        np.testing.assert_array_equal(backups[pos], ref[pos], err_msg=f"position {pos}")
    assert page_bytes == ref[0].nbytes
