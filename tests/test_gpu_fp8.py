"""GPU parity of the fp8-e4m3 quantising gather and dequantising scatter.

Codes and scales must equal the oracle's bit for bit: the quantised code is
an integer decided by fp32 arithmetic, and both sides take that decision in
fp32 (absmax/448 by IEEE division, x/scale by IEEE division, round to nearest
even with saturation).  The LMCache fp8 serde casts to float8_e4m3fn at one
byte per element ("LMCache 分布式 KV Cache 序列化框架：Serde 双层接口设计与自定义扩展实战",
section 7.1); the per-(K/V, layer, chunk)
scale is the fused variant's definition.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_lmkv_gb300 as pkg
from paged_kv_cache_lmkv_gb300 import workloads as wl
from gpu_util import (DEV, alloc_chunks, compact_subbatch, device_pool, host_bytes, host_u16,
                      new_status, require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def gpu_quant(pool, w, table, flag):
    chunks = pkg.enumerate_chunks(w.starts, w.ends, w.chunk_size, flag)
    codes, cptrs = alloc_chunks(chunks, w, dtype=torch.uint8, fill=0xEE)
    scales = torch.full((len(chunks), 2, w.num_layers), -1.0, dtype=torch.float32, device=DEV)
    st = new_status()
    bt = torch.from_numpy(table).to(DEV)
    pkg.check(pkg.gather_chunks_fp8e4m3(pool, bt, w.starts, w.ends, w.chunk_size, flag, cptrs,
                                        scales, st))
    torch.cuda.synchronize()
    return chunks, codes, cptrs, scales, st


SMALL = [
    # L, H, D, B, nb, ends, starts, C, flag
    (3, 2, 64, 16, 64, (512,), (0,), 256, True),
    (2, 2, 64, 16, 96, (300, 1000, 17), (0, 256, 0), 256, True),
    (2, 2, 64, 16, 96, (300, 1000, 17), (0, 256, 0), 256, False),
    (2, 1, 16, 4, 300, (333, 64), (64, 0), 64, True),
    (2, 8, 128, 32, 64, (900,), (0,), 256, True),
    (2, 8, 128, 64, 32, (1100,), (256,), 256, True),
    (1, 1, 32, 8, 600, (2000,), (0,), 1024, True),     # chunk larger than the cluster's registers
    (2, 8, 128, 16, 96, (1100,), (0,), 512, True),     # 128 rows per quarter: one tile per cluster of 8
    (1, 8, 128, 16, 256, (2048 + 700,), (0,), 2048, True),  # slice beyond shared memory: register path
]


@pytest.mark.parametrize("shape", SMALL, ids=[str(i) for i in range(len(SMALL))])
def test_small_quant_dequant_vs_oracle(shape):
    L, H, D, B, nb, ends, starts, C, flag = shape
    w = wl.Workload("f", L, H, D, B, nb, ends, req_start=starts, chunk_size=C, outliers=True,
                    save_unfull=flag)
    table, table2 = wl.block_table(w, 1), wl.block_table(w, 2)
    pool = device_pool(w, 0)
    chunks, codes, cptrs, scales, st = gpu_quant(pool, w, table, flag)
    assert st.item() == 0
    host = [host_u16(t) for t in pool.layers]
    rc = [np.full((2, L, n, w.row_elems), 0xEE, np.uint8) for _, _, n in chunks]
    rs = np.full((len(chunks), 2, L), -1.0, np.float32)
    assert oracle.gather_fp8(oracle.HostPool(host, B), table, w.starts, w.ends, C, flag, rc, rs) == 0
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    for g, (a, b) in enumerate(zip(codes, rc)):
        np.testing.assert_array_equal(a.cpu().numpy(), b, err_msg=f"codes chunk {g}")
    # dequantising scatter into a sentinel pool
    pool2 = device_pool(w, None, fill="sentinel")
    st.zero_()
    pkg.check(pkg.scatter_chunks_fp8e4m3(pool2, torch.from_numpy(table2).to(DEV), w.starts,
                                         w.ends, C, flag, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    h2 = [np.full_like(a, wl.SENTINEL_BF16) for a in host]
    assert oracle.scatter_fp8(oracle.HostPool(h2, B), table2, w.starts, w.ends, C, flag, rc, rs) == 0
    for l, (t, h) in enumerate(zip(pool2.layers, h2)):
        np.testing.assert_array_equal(host_u16(t), h, err_msg=f"dequant layer {l}")


def test_exhaustive_bf16_against_many_scales():
    """Tile i holds every finite bf16 value whose magnitude is at most A_i
    (repeated to fill 256 x 1024 elements), so its scale is A_i / 448; 48
    tiles with A_i spread over the bf16 range cover all bf16 inputs under 48
    different scales."""
    all_bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (all_bits << 16).view(np.float32)
    finite = np.isfinite(vals)
    rng = np.random.default_rng(0)
    amaxes = np.concatenate([[448.0, 1.0, 2.0 ** -120, 3.0e38, 1.5e-5],
                             np.exp2(rng.uniform(-100, 100, 43))]).astype(np.float32)
    amax_bf16 = (amaxes.view(np.uint32) >> 16).astype(np.uint32)   # truncate to bf16
    L = len(amax_bf16)
    w = wl.Workload("x", L, 8, 128, 16, 16, (256,), chunk_size=256)
    layers = []
    for l, ab in enumerate(amax_bf16):
        a = (ab << 16).view(np.float32) if np.ndim(ab) else np.uint32(ab << 16).view(np.float32)
        pick = all_bits[finite & (np.abs(vals) <= a)].astype(np.uint16)
        tile = np.resize(rng.permutation(pick), 256 * 1024).reshape(16, 16, 1024)
        tile[0, 0, 0] = np.uint16(ab)                       # make sure +A_i is present
        lay = np.empty((2, 16, 16, 1024), np.uint16)
        lay[0] = tile
        lay[1] = tile[:, :, ::-1]
        layers.append(torch.from_numpy(lay.view(np.int16)).view(torch.bfloat16).to(DEV))
    pool = pkg.Pool(layers, 8, 128)
    table = np.arange(16, dtype=np.int32)[None, :]
    chunks, codes, cptrs, scales, st = gpu_quant(pool, w, table, True)
    assert st.item() == 0
    host = [host_u16(t) for t in layers]
    rc = [np.zeros((2, L, 256, 1024), np.uint8)]
    rs = np.zeros((1, 2, L), np.float32)
    assert oracle.gather_fp8(oracle.HostPool(host, 16), table, [0], [256], 256, True, rc, rs) == 0
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    np.testing.assert_array_equal(codes[0].cpu().numpy(), rc[0])


@pytest.mark.parametrize("block_size", [16, 32, 64])
def test_qwen32b_full_size_sampled(block_size):
    """Qwen2.5-32B shape, 16384 tokens, outlier channels; GPU run at full size,
    oracle on two sampled chunks (all layers, K and V)."""
    w = wl.qwen_with_block_size(block_size)
    table = wl.block_table(w, 1)
    table2 = wl.block_table(w, 2)
    pool = device_pool(w, 0)
    chunks, codes, cptrs, scales, st = gpu_quant(pool, w, table, True)
    assert st.item() == 0 and len(chunks) == 64
    sample = [0, 45]
    hp, tab, s, e, _ = compact_subbatch(pool.layers, table, chunks, sample)
    hp16 = oracle.HostPool([a.view(np.uint16) for a in hp.layers], block_size)
    rc = [np.zeros((2, 64, 256, 1024), np.uint8) for _ in sample]
    rs = np.zeros((len(sample), 2, 64), np.float32)
    assert oracle.gather_fp8(hp16, tab, s, e, 256, True, rc, rs) == 0
    for i, g in enumerate(sample):
        np.testing.assert_array_equal(scales[g].cpu().numpy().view(np.uint32), rs[i].view(np.uint32))
        np.testing.assert_array_equal(codes[g].cpu().numpy(), rc[i], err_msg=f"chunk {g}")
    pool2 = device_pool(w, None, fill="sentinel")
    pkg.check(pkg.scatter_chunks_fp8e4m3(pool2, torch.from_numpy(table2).to(DEV), w.starts,
                                         w.ends, 256, True, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    hq, tab2, s2, e2, _ = compact_subbatch(pool2.layers, table2, chunks, sample)
    h2 = [np.full(a.shape[:3] + (a.shape[3] // 2,), wl.SENTINEL_BF16, np.uint16) for a in hq.layers]
    assert oracle.scatter_fp8(oracle.HostPool(h2, block_size), tab2, s2, e2, 256, True, rc, rs) == 0
    for a, b in zip(hq.layers, h2):
        np.testing.assert_array_equal(a.view(np.uint16), b)


def test_quant_error_bound_full_8b_shape():
    """Closed-form bound on the round trip at the Llama-3.1-8B shape (a property
    that holds at any size): |deq - x| <= half an e4m3 step at the tile's scale
    plus one bf16 rounding."""
    w = wl.LLAMA8B.with_(outliers=True)
    pool = device_pool(w, 0)
    table = wl.block_table(w, 1)
    chunks, codes, cptrs, scales, st = gpu_quant(pool, w, table, True)
    pool2 = device_pool(w, None, fill="sentinel")
    pkg.check(pkg.scatter_chunks_fp8e4m3(pool2, torch.from_numpy(table).to(DEV), w.starts,
                                         w.ends, 256, True, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    ids = torch.as_tensor(table[0], dtype=torch.long, device=DEV)
    for l in range(0, w.num_layers, 7):
        x = pool.layers[l].index_select(1, ids).float().view(2, 40, 256, -1)
        y = pool2.layers[l].index_select(1, ids).float().view(2, 40, 256, -1)
        s = scales[:, :, l].t().reshape(2, 40, 1, 1)
        bound = torch.maximum(x.abs() * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -8) + \
            x.abs() * 2.0 ** -8
        assert bool(((y - x).abs() <= bound).all())


def bf16_nan_mask(a: np.ndarray) -> np.ndarray:
    return (a & 0x7FFF) > 0x7F80


@pytest.mark.parametrize("shape", [
    # L, H, D, B, nb, ends, C, rows per CTA.  The bench's launch shape (clusters
    # of 4: rows 0-7 of each CTA's 64 in registers, 8-63 staged in shared memory
    # by bulk copies); 512-token chunks (clusters of 8, the same split of 64
    # rows); 2048-token chunks (register-staged kernel, 256 rows per CTA,
    # re-reading what does not fit)
    (4, 8, 128, 16, 64, (512,), 256, 64),
    (4, 8, 128, 16, 96, (1024,), 512, 64),
    (2, 8, 128, 16, 256, (2048 + 700,), 2048, 256),
], ids=["cluster4", "cluster8", "register"])
def test_non_finite_values_vs_oracle(shape):
    """NaN and infinity in register-held and shared-memory-held rows: codes and
    scales bit for bit against the oracle (a NaN is left out of the absmax and
    codes as 0x7F; an infinite scale codes finite values as signed zeros); the
    dequantised pool against the oracle's, with NaN where the oracle has NaN."""
    L, H, D, B, nb, ends, C, rows_per_cta = shape
    w = wl.Workload("nf", L, H, D, B, nb, ends, chunk_size=C)
    table, table2 = wl.block_table(w, 1), wl.block_table(w, 2)
    layers = [t.view(torch.int16).numpy().view(np.uint16).copy() for t in wl.make_pool(w, "cpu", 0)]

    def put(l, kv, tok, col, bits):
        layers[l][kv, table[0, tok // B], tok % B, col] = bits

    put(0, 0, 3, 11, 0x7FC0)                          # NaN in a register-held row of CTA 0
    put(0, 1, rows_per_cta + 40, 5, 0xFF81)           # -NaN in a staged row of CTA 1
    put(1, 0, 2 * rows_per_cta + 1, 7, 0x7F80)        # +inf, register row
    put(1, 1, 3 * rows_per_cta + 50, 9, 0xFF80)       # -inf, staged row
    if L > 2:
        put(2, 0, 70, 1, 0x7F80)                      # inf and NaN in one tile
        put(2, 0, 200, 2, 0x7FFF)
        zero = table[0, :C // B]
        layers[3][1][zero] = 0                        # zeros and a single NaN: scale 0
        put(3, 1, 100, 0, 0xFFC0)
        put(3, 0, C + 10, 3, 0x7FC0)                  # a NaN in the second chunk
    pool = pkg.Pool([torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV) for a in layers],
                    H, D)
    chunks, codes, cptrs, scales, st = gpu_quant(pool, w, table, True)
    assert st.item() == 0
    rc = [np.full((2, L, n, w.row_elems), 0xEE, np.uint8) for _, _, n in chunks]
    rs = np.full((len(chunks), 2, L), -1.0, np.float32)
    assert oracle.gather_fp8(oracle.HostPool(layers, B), table, w.starts, w.ends, C, True, rc, rs) == 0
    assert np.isinf(rs).any() and (rs == 0).any() == (L > 2)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    for g, (a, b) in enumerate(zip(codes, rc)):
        np.testing.assert_array_equal(a.cpu().numpy(), b, err_msg=f"codes chunk {g}")
    pool2 = device_pool(w, None, fill="sentinel")
    st.zero_()
    pkg.check(pkg.scatter_chunks_fp8e4m3(pool2, torch.from_numpy(table2).to(DEV), w.starts,
                                         w.ends, C, True, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    h2 = [np.full_like(a, wl.SENTINEL_BF16) for a in layers]
    assert oracle.scatter_fp8(oracle.HostPool(h2, B), table2, w.starts, w.ends, C, True, rc, rs) == 0
    for l, (t, h) in enumerate(zip(pool2.layers, h2)):
        got = host_u16(t)
        nan = bf16_nan_mask(h)
        np.testing.assert_array_equal(bf16_nan_mask(got), nan, err_msg=f"NaN positions, layer {l}")
        np.testing.assert_array_equal(got[~nan], h[~nan], err_msg=f"dequant layer {l}")


def test_llama8b_fp8_bench_launch_sampled():
    """The fp8 pair exactly as `bench.py` times it (Llama-3.1-8B batch, N(0,1)
    values without outliers, tables of seeds 1 and 2): codes and scales of
    sampled chunks bit for bit against the oracle, and the dequantised pages
    of those chunks against the oracle's scatter."""
    w = wl.LLAMA8B
    table, table2 = wl.block_table(w, 1), wl.block_table(w, 2)
    pool = device_pool(w, 0)
    chunks, codes, cptrs, scales, st = gpu_quant(pool, w, table, True)
    assert st.item() == 0 and len(chunks) == 40
    sample = [0, 21, 39]
    hp, tab, s, e, _ = compact_subbatch(pool.layers, table, chunks, sample)
    hp16 = oracle.HostPool([a.view(np.uint16) for a in hp.layers], 16)
    rc = [np.zeros((2, 32, 256, 1024), np.uint8) for _ in sample]
    rs = np.zeros((len(sample), 2, 32), np.float32)
    assert oracle.gather_fp8(hp16, tab, s, e, 256, True, rc, rs) == 0
    for i, g in enumerate(sample):
        np.testing.assert_array_equal(scales[g].cpu().numpy().view(np.uint32), rs[i].view(np.uint32))
        np.testing.assert_array_equal(codes[g].cpu().numpy(), rc[i], err_msg=f"chunk {g}")
    del pool
    torch.cuda.empty_cache()
    pool2 = device_pool(w, None, fill="sentinel")
    pkg.check(pkg.scatter_chunks_fp8e4m3(pool2, torch.from_numpy(table2).to(DEV), w.starts,
                                         w.ends, 256, True, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    hq, tab2, s2, e2, _ = compact_subbatch(pool2.layers, table2, chunks, sample)
    h2 = [np.full(a.shape[:3] + (a.shape[3] // 2,), wl.SENTINEL_BF16, np.uint16) for a in hq.layers]
    assert oracle.scatter_fp8(oracle.HostPool(h2, 16), tab2, s2, e2, 256, True, rc, rs) == 0
    for a, b in zip(hq.layers, h2):
        np.testing.assert_array_equal(a.view(np.uint16), b)


def fp8_gather_call(pool, bt, w, flag, cptrs, scales, st):
    return pkg.gather_chunks_fp8e4m3(pool, bt, w.starts, w.ends, w.chunk_size, flag, cptrs, scales, st)


def test_bad_block_ids_vs_oracle():
    """Out-of-range block ids: those rows take no part in the absmax and get
    no codes (the buffers keep their fill), the status says LMKV_ERR_BAD_BLOCK,
    and everything else equals the oracle's codes and scales."""
    w = wl.Workload("bad8", 2, 2, 64, 4, 64, (90, 40), req_start=(0, 0), chunk_size=32)
    table = wl.block_table(w, 1)
    table[0, 2] = 64
    table[0, 9] = -7
    table[1, 0] = 1 << 30
    pool = device_pool(w, 0)
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, w.chunk_size, True)
    codes, cptrs = alloc_chunks(chunks, w, dtype=torch.uint8, fill=0xEE)
    scales = torch.full((len(chunks), 2, w.num_layers), -1.0, dtype=torch.float32, device=DEV)
    st = new_status()
    pkg.check(fp8_gather_call(pool, bt, w, True, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == pkg.lmkv.ERR_BAD_BLOCK
    host = [host_u16(t) for t in pool.layers]
    rc = [np.full((2, w.num_layers, n, w.row_elems), 0xEE, np.uint8) for _, _, n in chunks]
    rs = np.full((len(chunks), 2, w.num_layers), -1.0, np.float32)
    assert oracle.gather_fp8(oracle.HostPool(host, 4), table, w.starts, w.ends, w.chunk_size, True,
                             rc, rs) == oracle.BAD_BLOCK
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    for g, (a, b) in enumerate(zip(codes, rc)):
        np.testing.assert_array_equal(a.cpu().numpy(), b, err_msg=f"codes chunk {g}")


def test_null_code_pointer_reported():
    """A null code pointer: LMKV_ERR_BAD_POINTER; that chunk gets no codes and
    its tiles' scales are 0 (nothing of the tile is read); the other chunk
    equals the oracle."""
    w = wl.TINY
    pool = device_pool(w, 0)
    table = wl.block_table(w, 0)
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 256, True)
    codes, cptrs = alloc_chunks(chunks, w, dtype=torch.uint8, fill=0xEE)
    cptrs[1] = 0
    scales = torch.full((len(chunks), 2, w.num_layers), -1.0, dtype=torch.float32, device=DEV)
    st = new_status()
    pkg.check(fp8_gather_call(pool, bt, w, True, cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == pkg.lmkv.ERR_BAD_POINTER
    assert (codes[1] == 0xEE).all()
    assert (scales[1] == 0).all()
    host = [host_u16(t) for t in pool.layers]
    rc = [np.zeros((2, w.num_layers, 256, w.row_elems), np.uint8)]
    rs = np.zeros((1, 2, w.num_layers), np.float32)
    assert oracle.gather_fp8(oracle.HostPool(host, w.block_size), table, [0], [256], 256, True, rc, rs) == 0
    np.testing.assert_array_equal(scales[0].cpu().numpy().view(np.uint32), rs[0].view(np.uint32))
    np.testing.assert_array_equal(codes[0].cpu().numpy(), rc[0])


def test_many_requests_split_over_launches():
    """300 requests: more than one launch's parameter block holds (256), so
    the quantising gather and the dequantising scatter each take two
    launches; codes, scales and the dequantised pool equal the oracle's."""
    rng = np.random.default_rng(9)
    ends = tuple(int(x) for x in rng.integers(0, 70, 300))
    w = wl.Workload("many8", 2, 1, 16, 4, 6000, ends, chunk_size=16, outliers=True)
    table, table2 = wl.block_table(w, 5), wl.block_table(w, 6)
    pool = device_pool(w, 0)
    bt = torch.from_numpy(table).to(DEV)
    chunks = pkg.enumerate_chunks(w.starts, w.ends, 16, True)
    codes, cptrs = alloc_chunks(chunks, w, dtype=torch.uint8, fill=0xEE)
    scales = torch.full((len(chunks), 2, w.num_layers), -1.0, dtype=torch.float32, device=DEV)
    st = new_status()
    before = pkg.lmkv.launch_count()
    pkg.check(fp8_gather_call(pool, bt, w, True, cptrs, scales, st))
    assert pkg.lmkv.launch_count() - before == 2
    torch.cuda.synchronize()
    assert st.item() == 0
    host = [host_u16(t) for t in pool.layers]
    rc = [np.full((2, w.num_layers, n, w.row_elems), 0xEE, np.uint8) for _, _, n in chunks]
    rs = np.full((len(chunks), 2, w.num_layers), -1.0, np.float32)
    assert oracle.gather_fp8(oracle.HostPool(host, 4), table, w.starts, w.ends, 16, True, rc, rs) == 0
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    for g, (a, b) in enumerate(zip(codes, rc)):
        np.testing.assert_array_equal(a.cpu().numpy(), b, err_msg=f"codes chunk {g}")
    pool2 = device_pool(w, None, fill="sentinel")
    pkg.check(pkg.scatter_chunks_fp8e4m3(pool2, torch.from_numpy(table2).to(DEV), w.starts, w.ends, 16, True,
                                         cptrs, scales, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    h2 = [np.full_like(a, wl.SENTINEL_BF16) for a in host]
    assert oracle.scatter_fp8(oracle.HostPool(h2, 4), table2, w.starts, w.ends, 16, True, rc, rs) == 0
    for l, (t, h) in enumerate(zip(pool2.layers, h2)):
        np.testing.assert_array_equal(host_u16(t), h, err_msg=f"dequant layer {l}")
