"""The entry points allocate nothing and never synchronise, so a sequence of
calls can be captured in a CUDA graph (the layer-wise pipeline's 32 calls per
direction are the launch-bound case).  Replays must equal eager calls."""
import numpy as np
import pytest
import torch

import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl
from gpu_util import DEV, alloc_chunks, device_pool, new_status, require_gpu

pytestmark = pytest.mark.gpu


def test_graph_capture_matches_eager():
    require_gpu()
    w = wl.Workload("g", 4, 2, 64, 16, 256, (700, 300), chunk_size=256)
    pool = device_pool(w, 0)
    bt = torch.from_numpy(wl.block_table(w, 1)).to(DEV)
    bt2 = torch.from_numpy(wl.block_table(w, 2)).to(DEV)
    a = (w.starts, w.ends, 256, True)
    chunks = pkg.enumerate_chunks(*a)
    eager, pe = alloc_chunks(chunks, w, fill=0)
    graph, pg = alloc_chunks(chunks, w, fill=0)
    codes_e, cpe = alloc_chunks(chunks, w, dtype=torch.uint8, fill=0)
    codes_g, cpg = alloc_chunks(chunks, w, dtype=torch.uint8, fill=0)
    sc_e = torch.zeros((len(chunks), 2, w.num_layers), dtype=torch.float32, device=DEV)
    sc_g = torch.zeros_like(sc_e)
    pool_e = device_pool(w, None, fill="sentinel")
    pool_g = device_pool(w, None, fill="sentinel")
    st = new_status()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()            # buffers were filled on the default stream

    def seq(bufs, ptrs, codes_ptrs, scales, target):
        with torch.cuda.stream(s):
            for l in range(w.num_layers):
                pkg.check(pkg.gather_layer(pool, bt, *a, ptrs, l, st, s))
            pkg.check(pkg.gather_chunks_fp8e4m3(pool, bt, *a, codes_ptrs, scales, st, s))
            pkg.check(pkg.scatter_chunks(target, bt2, *a, ptrs, st, s))
            for l in range(w.num_layers):
                pkg.check(pkg.scatter_layer(target, bt2, *a, ptrs, l, st, s))

    seq(eager, pe, cpe, sc_e, pool_e)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        seq(graph, pg, cpg, sc_g, pool_g)
    torch.cuda.synchronize()
    assert all(int((b != 0).sum()) == 0 for b in graph)      # capture itself ran nothing
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    for x, y in zip(eager, graph):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for x, y in zip(codes_e, codes_g):
        assert torch.equal(x, y)
    assert torch.equal(sc_e, sc_g)
    for x, y in zip(pool_e.layers, pool_g.layers):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
