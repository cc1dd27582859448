"""Deferred decode-KV store on the GPU: over a simulated decode run, storing
the chunks completed at each step (lmkv_decode_store_ranges + gather with
save_unfull_chunk = 0) yields exactly the oracle's chunks of every request's
final full-chunk prefix."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl
from gpu_util import DEV, device_pool, host_bytes, new_status, require_gpu

pytestmark = pytest.mark.gpu


def test_decode_run_stores_every_completed_chunk():
    require_gpu()
    rng = np.random.default_rng(3)
    C = 64
    final = rng.integers(300, 900, 5)
    w = wl.Workload("dec", 3, 2, 64, 16, 512, tuple(int(x) for x in final), chunk_size=C)
    pool = device_pool(w, 0)
    table = wl.block_table(w, 1)
    bt = torch.from_numpy(table).to(DEV)
    prompt = rng.integers(0, 200, 5)
    stored = (prompt // C) * C
    cur = prompt.copy()
    got = {}                                   # (request, first token) -> chunk tensor
    st = new_status()
    while (cur < final).any():
        cur = np.minimum(final, cur + rng.integers(1, 40, 5))
        s, e, n = pkg.decode_store_ranges(stored, cur, C)
        if n == 0:
            continue
        chunks = pkg.enumerate_chunks(s, e, C, False)
        bufs = [torch.zeros((2, w.num_layers, k, w.row_elems), dtype=torch.bfloat16, device=DEV)
                for _, _, k in chunks]
        pkg.check(pkg.gather_chunks(pool, bt, s, e, C, False, pkg.pointer_array(bufs, DEV), st))
        for (r, t0, k), b in zip(chunks, bufs):
            assert k == C and (r, t0) not in got
            got[(r, t0)] = b
        stored = e
    # chunks stored at prefill time (below the prompt's full prefix) are not part of this run
    first = (prompt // C) * C
    torch.cuda.synchronize()
    assert st.item() == 0
    ref_chunks = oracle.enumerate_chunks(first, final, C, False)
    assert sorted(got) == sorted((r, t0) for r, t0, _ in ref_chunks)
    ref = [np.zeros((2, w.num_layers, C, w.row_bytes), np.uint8) for _ in ref_chunks]
    host = [host_bytes(t) for t in pool.layers]
    assert oracle.gather(oracle.HostPool(host, w.block_size), table, first, final, C, False, ref) == 0
    for (r, t0, _), x in zip(ref_chunks, ref):
        np.testing.assert_array_equal(host_bytes(got[(r, t0)]), x)
