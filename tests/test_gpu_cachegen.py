"""GPU parity of the CacheGen codec ("LMCache 中的 KV Cache 压缩：CacheGen
编解码原理、配置方式与源码解析", sections 1-5).

The blob (per-token max1, the 2^16 CDFs, the stream lengths and the coded
bytes) must equal the oracle's byte for byte: every symbol is an integer
decided by fp32 arithmetic that both sides take in fp32 (MAX / max1 by IEEE
division, x * factor and + MAX rounded separately, ties to even), the CDF
is exact integer arithmetic and the coder is integer-only.  Decoding must give
the oracle's bf16 rows bit for bit.  Shapes: the page's benchmark (32 layers
x 8 KV heads x 128, chunk sizes 64 / 128 / 256 / 768), odd sizes that leave a
ragged last batch and partial warps, the largest chunk and channel counts,
outlier channels, all-zero rows, and more chunks than one launch takes.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_lmkv_gb300 as pkg
from oracle import cachegen as cg
from paged_kv_cache_lmkv_gb300 import workloads as wl
from gpu_util import DEV, host_u16, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def gpu_encode(codec, chunks):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    blobs, sizes = codec.encode(chunks, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, pkg.lmkv.status_string(status.item())
    sz = sizes.cpu().tolist()
    return [b[:s].cpu().numpy().tobytes() for b, s in zip(blobs, sz)], blobs, sizes


def gpu_decode(codec, blobs_bytes, ntoks):
    blobs = [torch.from_numpy(np.frombuffer(b, np.uint8).copy()).to(DEV) for b in blobs_bytes]
    sizes = torch.tensor([len(b) for b in blobs_bytes], dtype=torch.int64, device=DEV)
    outs = [torch.full((2, codec.num_layers, n, codec.channels), 7.0, dtype=torch.bfloat16, device=DEV)
            for n in ntoks]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    codec.decode(blobs, sizes, outs, status=status)
    torch.cuda.synchronize()
    return [host_u16(o) for o in outs], status.item()


def check_against_oracle(L, H, ntoks, seed, bins=None, **kw):
    bins = cg.default_bins(L) if bins is None else np.asarray(bins, np.int32).reshape(2, L)
    chunks = wl.cachegen_chunks(L, H, ntoks, seed, **kw)
    codec = pkg.CachegenCodec(L, H, bins, device=DEV)
    got, _, _ = gpu_encode(codec, [c.to(DEV) for c in chunks])
    expect = [cg.encode_chunk(c, bins) for c in chunks]
    for g, (a, b) in enumerate(zip(got, expect)):
        assert len(a) == len(b), f"chunk {g}: size {len(a)} != oracle {len(b)}"
        if a != b:
            diff = np.flatnonzero(np.frombuffer(a, np.uint8) != np.frombuffer(b, np.uint8))
            lay = cg.layout(L, ntoks[g], H, bins)
            raise AssertionError(f"chunk {g}: {diff.size} bytes differ, first at {diff[0]} (layout {lay})")
    dec, st = gpu_decode(codec, expect, ntoks)
    assert st == 0
    for g, (c, d) in enumerate(zip(chunks, dec)):
        assert np.array_equal(d, cg.decode_chunk(expect[g], L, ntoks[g], H, bins)), f"chunk {g}"
    return expect


@pytest.mark.parametrize("L,H,ntoks", [
    (1, 4, [1]),                       # one token, one partial warp
    (2, 40, [5, 256, 300]),            # ragged last batch, 10 of 32 lanes
    (3, 128, [257, 513, 64]),          # three batches
    (2, 96, [1000]),
    (1, 512, [1, 3, 5]),               # chunks shorter than their CTAs per slice
    (2, 1024, [256, 767]),
])
def test_small_shapes_exact(L, H, ntoks):
    bins = cg.default_bins(L)
    bins[0, 0] = 8
    bins[1, -1] = 4
    check_against_oracle(L, H, ntoks, seed=L * 100 + H, bins=bins)


@pytest.mark.parametrize("n", wl.CACHEGEN_CHUNK_SIZES)
def test_benchmark_shape_exact(n):
    """The page's benchmark shape with the 7B/8B default bins."""
    check_against_oracle(wl.CACHEGEN_LAYERS, wl.CACHEGEN_CHANNELS, [n], seed=n)


def test_outliers_and_zero_rows_exact():
    check_against_oracle(4, 1024, [256, 100], seed=5, outliers=True, zero_rows=3)


def test_subnormal_rows_exact():
    """Rows of bf16 subnormals: MAX / max1 overflows to +inf, so the symbols
    are 2*MAX, 0, and 0 for the zero entries (0 * inf)."""
    check_against_oracle(2, 256, [40, 300], seed=6, zero_rows=1, tiny_rows=5)


def test_largest_sizes_exact():
    """The most channels per row and the most tokens per chunk."""
    check_against_oracle(1, pkg.lmkv.CACHEGEN_MAX_CHANNELS, [300], seed=9)
    check_against_oracle(1, 64, [pkg.lmkv.CACHEGEN_MAX_TOKENS], seed=10)


def test_more_chunks_than_one_launch():
    rng = np.random.default_rng(3)
    ntoks = [int(v) for v in rng.integers(1, 400, 70)]
    check_against_oracle(2, 32, ntoks, seed=11)


def test_round_trip_error_bound_and_determinism():
    """Two encodes give the same bytes; the decoded rows stay within half a
    quantisation step (max1 / MAX) of the input plus the bf16 rounding."""
    L, H, n = wl.CACHEGEN_LAYERS, wl.CACHEGEN_CHANNELS, 256
    bins = cg.default_bins(L)
    x = wl.cachegen_chunks(L, H, [n, n], seed=21, device=DEV)
    codec = pkg.CachegenCodec(L, H, bins, device=DEV)
    a, blobs, sizes = gpu_encode(codec, x)
    b, _, _ = gpu_encode(codec, x)
    assert a == b
    out = [torch.empty_like(t) for t in x]
    codec.decode(blobs, sizes, out)
    torch.cuda.synchronize()
    for xi, yi in zip(x, out):
        xf, yf = xi.float(), yi.float()
        max1 = xf.abs().amax(dim=3, keepdim=True)
        MAX = torch.tensor(bins // 2 - 1, dtype=torch.float32, device=DEV)[:, :, None, None]
        assert bool(((yf - xf).abs() <= max1 * (0.5 / MAX * (1 + 1e-5) + 2.0 ** -8)).all())
    raw = sum(t.numel() * 2 for t in x)
    assert raw / sum(len(v) for v in a) > 3.0


def test_inconsistent_blob_is_rejected():
    """A blob whose lengths do not add up to its size decodes to nothing and
    reports BAD_DATA; the output keeps its contents."""
    L, H, n = 2, 64, 300
    bins = cg.default_bins(L)
    x = wl.cachegen_chunks(L, H, [n], seed=4)
    blob = bytearray(cg.encode_chunk(x[0], bins))
    lay = cg.layout(L, n, H, bins)
    first = int.from_bytes(blob[lay["lengths"]:lay["lengths"] + 4], "little")
    blob[lay["lengths"]:lay["lengths"] + 4] = (first + 1).to_bytes(4, "little")
    codec = pkg.CachegenCodec(L, H, bins, device=DEV)
    dec, st = gpu_decode(codec, [bytes(blob)], [n])
    assert st == pkg.lmkv.ERR_BAD_DATA
    assert np.all(dec[0] == np.uint16(0x40E0))           # 7.0 in bf16, untouched


# ---- the pool forms: store = gather then encode, retrieve = decode then scatter ----

import oracle  # noqa: E402
from gpu_util import device_pool, host_bytes  # noqa: E402


def _oracle_gather(w, layers_dev, table, chunks):
    hp = oracle.HostPool([host_bytes(t) for t in layers_dev], w.block_size)
    out = [np.zeros((2, w.num_layers, n, w.row_bytes), np.uint8) for _, _, n in chunks]
    rc = oracle.gather(hp, table, w.starts, w.ends, w.chunk_size, w.save_unfull, out)
    return [o.view(np.uint16) for o in out], rc


@pytest.mark.parametrize("w", [
    wl.Workload("cg-small", 3, 2, 64, 16, 96, (300, 700), chunk_size=256),
    wl.Workload("cg-ragged", 2, 1, 32, 32, 80, (100, 64, 900), req_start=(0, 0, 256), chunk_size=128),
    wl.Workload("cg-no-tail", 2, 2, 64, 16, 64, (700,), chunk_size=256, save_unfull=False),
    # few regions of wide rows: each slice and region spread over several CTAs,
    # whose row ranges start inside pages
    wl.Workload("cg-wide-few", 2, 4, 128, 16, 96, (300, 200), chunk_size=256),
    wl.Workload("cg-wide-offset", 3, 8, 128, 16, 400, (1100, 1412), req_start=(0, 512), chunk_size=512),
], ids=lambda w: w.name)
def test_pool_store_and_retrieve_exact(w):
    """lmkv_cachegen_store_chunks gives the oracle's blobs of the oracle's
    gather; lmkv_cachegen_retrieve_chunks writes the oracle's decode of those
    blobs into exactly the chunks' rows (the other rows keep the sentinel)."""
    pool = device_pool(w, seed=3)
    table = wl.block_table(w, 5)
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, w.chunk_size, w.save_unfull)
    bins = cg.default_bins(w.num_layers)
    bins[1, 0] = 8
    codec = pkg.CachegenCodec(w.num_layers, w.row_elems, bins, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    blobs, sizes = codec.store(pool, bt, w.starts, w.ends, w.chunk_size, w.save_unfull, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    xs, rc = _oracle_gather(w, pool.layers, table, chunks)
    assert rc == 0
    expect = [cg.encode_chunk(x, bins) for x in xs]
    got = [b[:s].cpu().numpy().tobytes() for b, s in zip(blobs, sizes.cpu().tolist())]
    assert got == expect

    # retrieve into a sentinel pool under another table
    pool2 = device_pool(w, seed=None, fill="sentinel")
    table2 = wl.block_table(w, 6)
    bt2 = torch.from_numpy(table2).to(DEV)
    codec.retrieve(pool2, bt2, w.starts, w.ends, w.chunk_size, w.save_unfull, blobs, sizes, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    hp = oracle.HostPool([host_bytes(t) for t in wl.make_pool(w, "cpu", None, fill="sentinel")],
                         w.block_size)
    dec = [cg.decode_chunk(e, w.num_layers, n, w.row_elems, bins).view(np.uint8).reshape(2, w.num_layers, n, -1)
           for e, (_, _, n) in zip(expect, chunks)]
    assert oracle.scatter(hp, table2, w.starts, w.ends, w.chunk_size, w.save_unfull, dec) == 0
    for l in range(w.num_layers):
        assert np.array_equal(host_bytes(pool2.layers[l]), hp.layers[l]), f"layer {l}"


def test_pool_forms_equal_the_two_step_path_at_the_8b_shape():
    """The 8B batch (40 chunks): the fused store equals gather + encode and
    the fused retrieve equals decode + scatter, byte for byte; one chunk is
    also checked against the oracle."""
    w = wl.LLAMA8B.with_(num_blocks=1024)
    pool = device_pool(w, seed=0)
    table = wl.block_table(w, 1)
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, w.chunk_size, w.save_unfull)
    codec = pkg.CachegenCodec(w.num_layers, w.row_elems, device=DEV)
    blobs, sizes = codec.store(pool, bt, w.starts, w.ends, w.chunk_size, w.save_unfull)
    bufs = [torch.empty((2, w.num_layers, n, w.row_elems), dtype=torch.bfloat16, device=DEV) for _, _, n in chunks]
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, w.chunk_size, w.save_unfull,
                                pkg.pointer_array(bufs, DEV), None, None))
    blobs2, sizes2 = codec.encode(bufs)
    torch.cuda.synchronize()
    assert torch.equal(sizes, sizes2)
    for a, b, s in zip(blobs, blobs2, sizes.cpu().tolist()):
        assert torch.equal(a[:s], b[:s])
    g = 17
    assert blobs[g][:sizes[g]].cpu().numpy().tobytes() == cg.encode_chunk(bufs[g].cpu(), codec.bins)

    pool2 = device_pool(w, seed=None, fill="sentinel")
    pool3 = device_pool(w, seed=None, fill="sentinel")
    table2 = wl.block_table(w, 2)
    bt2 = torch.from_numpy(table2).to(DEV)
    codec.retrieve(pool2, bt2, w.starts, w.ends, w.chunk_size, w.save_unfull, blobs, sizes)
    outs = [torch.empty_like(b) for b in bufs]
    codec.decode(blobs, sizes, outs)
    pkg.check(pkg.scatter_chunks(pool3, bt2, w.starts, w.ends, w.chunk_size, w.save_unfull,
                                 pkg.pointer_array(outs, DEV), None, None))
    torch.cuda.synchronize()
    for a, b in zip(pool2.layers, pool3.layers):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_pool_store_bad_block_reads_zeros():
    """A block id outside the pool: its rows are coded as zeros (the oracle's
    gather leaves them zero too) and the call reports BAD_BLOCK; the retrieve
    leaves those rows unwritten."""
    w = wl.Workload("cg-bad", 2, 2, 64, 16, 64, (512,), chunk_size=256)
    pool = device_pool(w, seed=4)
    table = wl.block_table(w, 7)
    table[0, 3] = 1000
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, w.chunk_size, w.save_unfull)
    bins = cg.default_bins(w.num_layers)
    codec = pkg.CachegenCodec(w.num_layers, w.row_elems, bins, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    blobs, sizes = codec.store(pool, bt, w.starts, w.ends, w.chunk_size, w.save_unfull, status=status)
    torch.cuda.synchronize()
    assert status.item() == pkg.lmkv.ERR_BAD_BLOCK
    xs, rc = _oracle_gather(w, pool.layers, table, chunks)
    assert rc == oracle.BAD_BLOCK
    got = [b[:s].cpu().numpy().tobytes() for b, s in zip(blobs, sizes.cpu().tolist())]
    assert got == [cg.encode_chunk(x, bins) for x in xs]
    pool2 = device_pool(w, seed=None, fill="sentinel")
    status.zero_()
    codec.retrieve(pool2, bt, w.starts, w.ends, w.chunk_size, w.save_unfull, blobs, sizes, status=status)
    torch.cuda.synchronize()
    assert status.item() == pkg.lmkv.ERR_BAD_BLOCK
    assert int((pool2.layers[0].view(torch.uint8) != wl.SENTINEL_BYTE).any(dim=-1).sum()) == 2 * (512 - 16)


def test_codec_calls_capture_in_a_cuda_graph():
    """After a first call on the device, encode and decode can be captured in
    a CUDA graph; a replay reproduces the eager results."""
    L, H, ntoks = 4, 256, [256, 100]
    lib = pkg.lmkv
    codec = pkg.CachegenCodec(L, H, device=DEV)
    x = wl.cachegen_chunks(L, H, ntoks, seed=31, device=DEV)
    blobs, sizes = codec.encode(x)
    outs = [torch.empty_like(t) for t in x]
    codec.decode(blobs, sizes, outs)
    torch.cuda.synchronize()
    blobs2 = [torch.zeros_like(b) for b in blobs]
    sizes2 = torch.zeros_like(sizes)
    outs2 = [torch.zeros_like(t) for t in x]
    cptr, bptr, optr = (pkg.pointer_array(v, DEV) for v in (x, blobs2, outs2))
    ws = codec._workspace(ntoks)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pkg.check(lib.cachegen_encode(cptr, ntoks, L, H, codec.bins, bptr, sizes2, ws, None, None))
        pkg.check(lib.cachegen_decode(bptr, sizes2, ntoks, L, H, codec.bins, optr, ws, None, None))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(sizes, sizes2)
    for a, b, s in zip(blobs, blobs2, sizes.cpu().tolist()):
        assert torch.equal(a[:s], b[:s])
    for a, b in zip(outs, outs2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_codec_reuses_pointer_arrays():
    """Calls with the same buffers reuse one device pointer array each and give
    the same blobs; new buffers (another stream) get their own."""
    L, H, ntoks = 2, 512, [256, 77]
    codec = pkg.CachegenCodec(L, H, device=DEV)
    x = wl.cachegen_chunks(L, H, ntoks, seed=41, device=DEV)
    expect = [cg.encode_chunk(c.cpu(), codec.bins) for c in x]
    blobs, sizes = codec.encode(x)
    cached = len(codec._ptrs)
    for _ in range(3):
        codec.encode(x, blobs, sizes)
    assert len(codec._ptrs) == cached
    torch.cuda.synchronize()
    got = [b[:s].cpu().numpy().tobytes() for b, s in zip(blobs, sizes.cpu().tolist())]
    assert got == expect
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        x2 = [t.clone() for t in x]
        blobs2, sizes2 = codec.encode(x2)
        outs = [torch.empty_like(t) for t in x2]
        codec.decode(blobs2, sizes2, outs)
    torch.cuda.synchronize()
    assert len(codec._ptrs) == cached + 3
    got2 = [b[:s].cpu().numpy().tobytes() for b, s in zip(blobs2, sizes2.cpu().tolist())]
    assert got2 == expect
    for o, e, n in zip(outs, expect, ntoks):
        assert np.array_equal(host_u16(o), cg.decode_chunk(e, L, n, H, codec.bins))


def test_bad_pointers_skip_the_chunk():
    """A null or misaligned blob, a misaligned chunk buffer: that chunk is
    skipped by every kernel (size 0, nothing written) and the call reports
    BAD_POINTER; the other chunks are coded as usual."""
    L, H, ntoks = 2, 64, [256, 100, 300]
    bins = cg.default_bins(L)
    x = [t.to(DEV) for t in wl.cachegen_chunks(L, H, ntoks, seed=41)]
    codec = pkg.CachegenCodec(L, H, bins, device=DEV)
    lib = pkg.lmkv
    raw = torch.empty(codec.layout(300).max_bytes + 64, dtype=torch.uint8, device=DEV)
    odd = torch.empty(2 * L * 100 * H + 8, dtype=torch.bfloat16, device=DEV)[1:1 + 2 * L * 100 * H]
    odd = odd.view(2, L, 100, H)                                  # 2-byte aligned chunk buffer
    odd.copy_(x[1])
    blobs = [torch.full((codec.layout(n).max_bytes,), 0x5A, dtype=torch.uint8, device=DEV) for n in ntoks]
    cases = [
        ("null blob", [x[0], x[1], x[2]], [blobs[0].data_ptr(), 0, blobs[2].data_ptr()]),
        ("misaligned blob", [x[0], x[1], x[2]], [blobs[0].data_ptr(), raw.data_ptr() + 2, blobs[2].data_ptr()]),
        ("misaligned chunk", [x[0], odd, x[2]], [blobs[0].data_ptr(), blobs[1].data_ptr(), blobs[2].data_ptr()]),
    ]
    for what, chunks, bptrs in cases:
        for b in blobs:
            b.fill_(0x5A)
        sizes = torch.full((3,), 7, dtype=torch.int64, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        bptr = torch.tensor(bptrs, dtype=torch.int64, device=DEV)
        ws = codec._workspace(ntoks)
        pkg.check(lib.cachegen_encode(pkg.pointer_array(chunks, DEV), ntoks, L, H, bins, bptr, sizes, ws,
                                      status, None))
        torch.cuda.synchronize()
        assert status.item() == lib.ERR_BAD_POINTER, what
        assert sizes[1].item() == 0, what
        if what == "misaligned chunk":
            assert bool((blobs[1] == 0x5A).all()), what
        for g in (0, 2):
            s = int(sizes[g].item())
            assert blobs[g][:s].cpu().numpy().tobytes() == cg.encode_chunk(x[g].cpu(), bins), what


def test_seventy_b_layer_count_exact():
    """80 layers (the 70B shape): default bins K 10 x 32 + 70 x 16, V 2 x 32 +
    78 x 16; one full chunk and one partial chunk against the oracle."""
    L = 80
    bins = cg.default_bins(L)
    assert bins[0].tolist() == [32] * 10 + [16] * 70 and bins[1].tolist() == [32] * 2 + [16] * 78
    check_against_oracle(L, 1024, [256, 40], seed=80)


def test_pool_forms_with_more_chunks_than_one_launch():
    """A store / retrieve call of 250 chunks (four launch groups of at most
    64; full and partial chunks) through the pool equals gather + encode and
    decode + scatter."""
    w = wl.Workload("cg-many", 2, 1, 64, 16, 1024, (16, 32, 24) * 50, chunk_size=16)
    pool = device_pool(w, seed=8)
    table = wl.block_table(w, 9)
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, w.chunk_size, w.save_unfull)
    assert len(chunks) > 2 * 64
    codec = pkg.CachegenCodec(w.num_layers, w.row_elems, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    blobs, sizes = codec.store(pool, bt, w.starts, w.ends, w.chunk_size, w.save_unfull, status=status)
    bufs = [torch.empty((2, w.num_layers, n, w.row_elems), dtype=torch.bfloat16, device=DEV) for _, _, n in chunks]
    pkg.check(pkg.gather_chunks(pool, bt, w.starts, w.ends, w.chunk_size, w.save_unfull,
                                pkg.pointer_array(bufs, DEV), status, None))
    blobs2, sizes2 = codec.encode(bufs)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(sizes, sizes2)
    for a, b, s in zip(blobs, blobs2, sizes.cpu().tolist()):
        assert torch.equal(a[:s], b[:s])
    for g in (0, 77, len(chunks) - 1):
        assert blobs[g][:sizes[g]].cpu().numpy().tobytes() == cg.encode_chunk(bufs[g].cpu(), codec.bins)
    pool2 = device_pool(w, seed=None, fill="sentinel")
    pool3 = device_pool(w, seed=None, fill="sentinel")
    table2 = wl.block_table(w, 10)
    bt2 = torch.from_numpy(table2).to(DEV)
    codec.retrieve(pool2, bt2, w.starts, w.ends, w.chunk_size, w.save_unfull, blobs, sizes, status=status)
    outs = [torch.empty_like(b) for b in bufs]
    codec.decode(blobs, sizes, outs, status=status)
    pkg.check(pkg.scatter_chunks(pool3, bt2, w.starts, w.ends, w.chunk_size, w.save_unfull,
                                 pkg.pointer_array(outs, DEV), status, None))
    torch.cuda.synchronize()
    assert status.item() == 0
    for a, b in zip(pool2.layers, pool3.layers):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
