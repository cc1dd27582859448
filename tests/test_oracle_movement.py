"""Pins for the oracle's gather / scatter (CPU only).

Each test checks the oracle against something other than itself: the
per-token dictionary model in brute.py, torch's strided copy for the
identity block table, and invariants that hold for any correct
implementation (round trip, bijection onto (block, slot), sentinels, layer
union).  Movement rule: "LMCache: An Efficient KV Cache Layer for Enterprise-Scale LLM Inference",
section on the configurable chunk size
(pages -> contiguous 256-token chunks and back) and layer-wise pipeline
section (one layer per call).
"""
import numpy as np
import pytest
import torch

import brute
import oracle
from paged_kv_cache_lmkv_gb300 import workloads as wl


def rand_pool(rng, L, nb, B, row_elems, dtype=np.uint16):
    info = np.iinfo(dtype)
    return [rng.integers(0, info.max, (2, nb, B, row_elems), dtype=dtype, endpoint=True)
            for _ in range(L)]


def sentinel_pool(L, nb, B, row_elems, dtype=np.uint16):
    val = wl.SENTINEL_BF16 if dtype == np.uint16 else wl.SENTINEL_BYTE
    return [np.full((2, nb, B, row_elems), val, dtype=dtype) for _ in range(L)]


def chunk_bufs(chunks, L, row_elems, dtype=np.uint16, fill=0):
    return [np.full((2, L, n, row_elems), fill, dtype=dtype) for _, _, n in chunks]


def random_case(rng):
    L = int(rng.integers(1, 4))
    B = int(rng.choice([1, 2, 4, 16]))
    C = B * int(rng.choice([1, 2, 4]))
    row = int(rng.choice([8, 64]))
    nreq = int(rng.integers(1, 4))
    starts = rng.integers(0, 3, nreq) * C
    ends = starts + rng.integers(0, 3 * C + 2, nreq)
    need = [int(-(-e // B)) for e in ends]
    nb = sum(need) + int(rng.integers(0, 6))
    perm = rng.permutation(nb)
    table = np.full((nreq, max(max(need), 1)), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[k:k + n]
        k += n
    flag = bool(rng.integers(0, 2))
    return L, B, C, row, starts, ends, nb, table, flag


def test_tiny_workload_matches_dict_model():
    w = wl.TINY
    rng = np.random.default_rng(0)
    layers = rand_pool(rng, w.num_layers, w.num_blocks, w.block_size, w.row_elems)
    table = wl.block_table(w, seed=0)
    chunks = oracle.enumerate_chunks(w.starts, w.ends, w.chunk_size, w.save_unfull)
    assert len(chunks) == 2
    got = chunk_bufs(chunks, w.num_layers, w.row_elems)
    ref = chunk_bufs(chunks, w.num_layers, w.row_elems)
    pool = oracle.HostPool(layers, w.block_size)
    assert oracle.gather(pool, table, w.starts, w.ends, w.chunk_size, w.save_unfull, got) == 0
    assert brute.gather(layers, table, w.starts, w.ends, w.chunk_size, w.save_unfull, ref) == 0
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("seed", range(40))
def test_random_shapes_gather_scatter_match_dict_model(seed):
    rng = np.random.default_rng(100 + seed)
    L, B, C, row, starts, ends, nb, table, flag = random_case(rng)
    dtype = np.uint16 if seed % 2 == 0 else np.uint8
    layers = rand_pool(rng, L, nb, B, row, dtype)
    chunks = oracle.enumerate_chunks(starts, ends, C, flag)
    got = chunk_bufs(chunks, L, row, dtype)
    ref = chunk_bufs(chunks, L, row, dtype)
    pool = oracle.HostPool(layers, B)
    assert oracle.gather(pool, table, starts, ends, C, flag, got) == 0
    brute.gather(layers, table, starts, ends, C, flag, ref)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)
    # scatter of fresh random chunk contents into a sentinel pool
    src = [rng.integers(0, np.iinfo(dtype).max, a.shape, dtype=dtype) for a in got]
    p_or = sentinel_pool(L, nb, B, row, dtype)
    p_br = sentinel_pool(L, nb, B, row, dtype)
    assert oracle.scatter(oracle.HostPool(p_or, B), table, starts, ends, C, flag, src) == 0
    brute.scatter(p_br, table, starts, ends, C, flag, src)
    for a, b in zip(p_or, p_br):
        np.testing.assert_array_equal(a, b)


def test_identity_table_equals_strided_copy():
    """One request, block table = 0,1,2,...: the gather is a plain strided slice."""
    rng = np.random.default_rng(3)
    L, nb, B, row, C = 3, 60, 16, 64, 256
    layers = rand_pool(rng, L, nb, B, row)
    s, e = 256, 256 + 2 * 256 + 77
    table = np.arange(nb, dtype=np.int32)[None, :]
    chunks = oracle.enumerate_chunks([s], [e], C, True)
    got = chunk_bufs(chunks, L, row)
    assert oracle.gather(oracle.HostPool(layers, B), table, [s], [e], C, True, got) == 0
    tl = [torch.from_numpy(a.view(np.int16)) for a in layers]
    for (r, t0, n), buf in zip(chunks, got):
        expect = torch.stack([torch.stack([t.view(2, nb * B, row)[kv, t0:t0 + n] for t in tl])
                              for kv in range(2)])
        np.testing.assert_array_equal(buf.view(np.int16), expect.numpy())


def test_round_trip_and_bijection():
    """gather(P,BT) -> scatter(P',BT') -> gather(P',BT') reproduces the chunks;
    exactly the enumerated (block, slot) rows of P' change, each once."""
    w = wl.Workload("rt", 2, 1, 16, 4, 64, (100, 37, 64), req_start=(0, 0, 64), chunk_size=16)
    rng = np.random.default_rng(11)
    layers = rand_pool(rng, w.num_layers, w.num_blocks, w.block_size, w.row_elems)
    t1 = wl.block_table(w, seed=1)
    t2 = wl.block_table(w, seed=2)
    for flag in (True, False):
        chunks = oracle.enumerate_chunks(w.starts, w.ends, w.chunk_size, flag)
        x = chunk_bufs(chunks, w.num_layers, w.row_elems)
        assert oracle.gather(oracle.HostPool(layers, w.block_size), t1, w.starts, w.ends,
                             w.chunk_size, flag, x) == 0
        p2 = sentinel_pool(w.num_layers, w.num_blocks, w.block_size, w.row_elems)
        assert oracle.scatter(oracle.HostPool(p2, w.block_size), t2, w.starts, w.ends,
                              w.chunk_size, flag, x) == 0
        y = chunk_bufs(chunks, w.num_layers, w.row_elems, fill=7)
        assert oracle.gather(oracle.HostPool(p2, w.block_size), t2, w.starts, w.ends,
                             w.chunk_size, flag, y) == 0
        for a, b in zip(x, y):
            np.testing.assert_array_equal(a, b)
        # bijection: the rows that left the sentinel are exactly the enumerated tokens
        n_tok = sum(n for _, _, n in chunks)
        changed = sum(int((a != wl.SENTINEL_BF16).any(axis=-1).sum()) for a in p2)
        assert changed == 2 * w.num_layers * n_tok
        image = set()
        for r, t0, n in chunks:
            for tok in range(t0, t0 + n):
                image.add((int(t2[r, tok // w.block_size]), tok % w.block_size))
        assert len(image) == n_tok
        for l in range(w.num_layers):
            for kv in range(2):
                for blk in range(w.num_blocks):
                    for slot in range(w.block_size):
                        touched = (blk, slot) in image
                        is_sent = bool((p2[l][kv, blk, slot] == wl.SENTINEL_BF16).all())
                        assert touched != is_sent


def test_layer_union_equals_full():
    rng = np.random.default_rng(5)
    for _ in range(5):
        L, B, C, row, starts, ends, nb, table, flag = random_case(rng)
        layers = rand_pool(rng, L, nb, B, row)
        chunks = oracle.enumerate_chunks(starts, ends, C, flag)
        full = chunk_bufs(chunks, L, row)
        per = chunk_bufs(chunks, L, row)
        pool = oracle.HostPool(layers, B)
        oracle.gather(pool, table, starts, ends, C, flag, full)
        for l in range(L):
            oracle.gather(pool, table, starts, ends, C, flag, per, layer=l)
        for a, b in zip(full, per):
            np.testing.assert_array_equal(a, b)
        pf = sentinel_pool(L, nb, B, row)
        pl = sentinel_pool(L, nb, B, row)
        oracle.scatter(oracle.HostPool(pf, B), table, starts, ends, C, flag, full)
        for l in range(L):
            oracle.scatter(oracle.HostPool(pl, B), table, starts, ends, C, flag, full, layer=l)
        for a, b in zip(pf, pl):
            np.testing.assert_array_equal(a, b)


def test_one_layer_touches_only_that_layer():
    rng = np.random.default_rng(9)
    L, nb, B, row, C = 3, 32, 4, 8, 16
    layers = rand_pool(rng, L, nb, B, row)
    table = rng.permutation(nb).astype(np.int32)[None, :]
    chunks = oracle.enumerate_chunks([0], [50], C, True)
    bufs = chunk_bufs(chunks, L, row, fill=3)
    oracle.gather(oracle.HostPool(layers, B), table, [0], [50], C, True, bufs, layer=1)
    for b in bufs:
        assert (b[:, [0, 2]] == 3).all()
        assert not (b[:, 1] == 3).all()


def test_bad_block_ids_are_skipped_and_flagged():
    rng = np.random.default_rng(2)
    L, nb, B, row, C = 2, 16, 4, 8, 8
    layers = rand_pool(rng, L, nb, B, row)
    table = rng.permutation(nb).astype(np.int32)[None, :]
    table[0, 1] = nb          # out of range
    table[0, 3] = -2          # negative
    chunks = oracle.enumerate_chunks([0], [30], C, True)
    got = chunk_bufs(chunks, L, row, fill=9)
    ref = chunk_bufs(chunks, L, row, fill=9)
    assert oracle.gather(oracle.HostPool(layers, B), table, [0], [30], C, True, got) == oracle.BAD_BLOCK
    assert brute.gather(layers, table, [0], [30], C, True, ref) > 0
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)
    p = sentinel_pool(L, nb, B, row)
    assert oracle.scatter(oracle.HostPool(p, B), table, [0], [30], C, True, got) == oracle.BAD_BLOCK


def test_invalid_arguments():
    rng = np.random.default_rng(1)
    layers = rand_pool(rng, 1, 8, 4, 8)
    pool = oracle.HostPool(layers, 4)
    table = np.arange(8, dtype=np.int32)[None, :]
    buf = [np.zeros((2, 1, 8, 8), np.uint16)]
    assert oracle.gather(pool, table, [4], [12], 8, True, buf) == oracle.INVALID    # unaligned start
    assert oracle.gather(pool, table, [0], [40], 8, True, buf) == oracle.INVALID    # table too short
    assert oracle.gather(pool, table, [8], [0], 8, True, buf) == oracle.INVALID     # end < start
    assert oracle.gather(pool, table, [0], [8], 8, True, buf, layer=1) == oracle.INVALID


def test_partial_chunks_are_compact():
    """A partial last chunk's buffer holds exactly its n rows per (kv, layer)."""
    rng = np.random.default_rng(4)
    L, nb, B, row, C = 2, 64, 16, 8, 256
    layers = rand_pool(rng, L, nb, B, row)
    table = rng.permutation(nb).astype(np.int32)[None, :]
    chunks = oracle.enumerate_chunks([0], [296], C, True)
    assert [n for _, _, n in chunks] == [256, 40]
    bufs = chunk_bufs(chunks, L, row)
    oracle.gather(oracle.HostPool(layers, B), table, [0], [296], C, True, bufs)
    for kv in range(2):
        for l in range(L):
            for t in range(40):
                tok = 256 + t
                np.testing.assert_array_equal(bufs[1][kv, l, t],
                                              layers[l][kv, table[0, tok // B], tok % B])
