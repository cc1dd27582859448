"""Pins for the oracle's number formats and fp8 quantising gather (CPU only).

The fp8 serde of LMCache casts each element to torch.float8_e4m3fn
("LMCache 分布式 KV Cache 序列化框架", section 7.1).  The fused variant adds one
fp32 absmax/448 scale per (K/V, layer, chunk).  Pins: the OCP E4M3 table (golden file), torch's own
float8_e4m3fn and bfloat16 conversions (independent implementations of the
same formats), numpy's fp32 division, the unscaled special case that is
exactly the serde's cast, closed-form error bounds.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_lmkv_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ocp.txt")


def all_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


def torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_golden_ocp_table():
    codes, vals = [], []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                codes.append(int(c, 16))
                vals.append(v)
    got = oracle.e4m3_to_f32(np.array(codes, np.uint8))
    for c, v, g in zip(codes, vals, got):
        if v == "nan":
            assert np.isnan(g), hex(c)
        else:
            assert g == float(v) and np.signbit(g) == v.startswith("-"), hex(c)
            if v not in ("0", "-0"):
                # encoding the exact value gives the code back
                assert oracle.f32_to_e4m3(np.array([g], np.float32))[0] == c


def test_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and nan.sum() == 2
    np.testing.assert_array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_encode_all_bf16_values_vs_torch():
    """Every finite bf16 value with |v| < 464 rounds the same way in torch's
    (non-saturating) cast; above that the oracle saturates to +-448."""
    v = all_bf16_as_f32()
    inr = np.abs(v) < 464
    np.testing.assert_array_equal(oracle.f32_to_e4m3(v[inr]), torch_e4m3(v[inr]))
    big = oracle.f32_to_e4m3(v[~inr])
    assert ((big == 0x7E) | (big == 0xFE)).all()
    assert (big[v[~inr] > 0] == 0x7E).all() and (big[v[~inr] < 0] == 0xFE).all()


def test_encode_random_f32_and_ties_vs_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp2(rng.uniform(-14, 9, 200000))).astype(np.float32)
    x = x[np.abs(x) < 464]
    np.testing.assert_array_equal(oracle.f32_to_e4m3(x), torch_e4m3(x))
    # exact midpoints between adjacent finite e4m3 values: ties go to the even code
    pos = oracle.e4m3_to_f32(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert (mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2).all()
    codes = oracle.f32_to_e4m3(mids)
    assert (codes % 2 == 0).all()
    np.testing.assert_array_equal(codes, torch_e4m3(mids))
    np.testing.assert_array_equal(oracle.f32_to_e4m3(-mids), torch_e4m3(-mids))


def test_encode_special_values():
    v = np.array([0.0, -0.0, np.inf, -np.inf, 1e30, -1e30, 448.0, 449.0, 1e-30, -1e-30],
                 np.float32)
    got = oracle.f32_to_e4m3(v)
    assert list(got) == [0x00, 0x80, 0x7E, 0xFE, 0x7E, 0xFE, 0x7E, 0x7E, 0x00, 0x80]
    assert oracle.f32_to_e4m3(np.array([np.nan], np.float32))[0] == 0x7F


def test_every_e4m3_value_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    np.testing.assert_array_equal(oracle.f32_to_e4m3(oracle.e4m3_to_f32(codes)), codes)


def test_bf16_rounding_vs_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 32, 400000, dtype=np.uint64).astype(np.uint32)
    # force a share of exact ties (low 16 bits = 0x8000) and near ties
    bits[:50000] = (bits[:50000] & 0xFFFF0000) | 0x8000
    bits[50000:60000] = (bits[50000:60000] & 0xFFFF0000) | 0x7FFF
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    ours = oracle.f32_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_div_is_ieee_f32():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(100000).astype(np.float32)
    for s in (np.float32(1.0), np.float32(0.1), np.float32(3.0) / np.float32(448.0),
              np.float32(7.3e-3)):
        np.testing.assert_array_equal(oracle.div_f32(x, float(s)), x / s)


# ---------------------------------------------------------------------------
# The quantising gather / dequantising scatter on small pools.

def bf16_pool(w, seed):
    layers = [t.view(torch.int16).numpy().view(np.uint16).copy()
              for t in wl.make_pool(w, "cpu", seed)]
    return layers


def torch_reference_quant(layers, table, chunks, w):
    """codes / scales by torch composition: amax, fp32 divide, float8 cast."""
    codes, scales = [], np.zeros((len(chunks), 2, w.num_layers), np.float32)
    for g, (r, t0, n) in enumerate(chunks):
        c = np.zeros((2, w.num_layers, n, w.row_elems), np.uint8)
        for kv in range(2):
            for l in range(w.num_layers):
                rows = np.stack([layers[l][kv, table[r, tok // w.block_size], tok % w.block_size]
                                 for tok in range(t0, t0 + n)])
                x = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).float()
                amax = x.abs().max()
                s = amax / 448.0
                scales[g, kv, l] = s.item()
                if amax.item() == 0:
                    continue
                c[kv, l] = (x / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        codes.append(c)
    return codes, scales


@pytest.mark.parametrize("B,ends,flag", [(16, (512,), True), (4, (100, 37), True),
                                          (8, (300,), False), (32, (70,), True)])
def test_quant_gather_vs_torch_composition(B, ends, flag):
    w = wl.Workload("q", 3, 2, 32, B, 64 * 16 // B, ends, outliers=True, save_unfull=flag)
    layers = bf16_pool(w, 0)
    table = wl.block_table(w, seed=1)
    chunks = oracle.enumerate_chunks(w.starts, w.ends, w.chunk_size, flag)
    codes = [np.zeros((2, w.num_layers, n, w.row_elems), np.uint8) for _, _, n in chunks]
    scales = np.zeros((len(chunks), 2, w.num_layers), np.float32)
    pool = oracle.HostPool(layers, B)
    assert oracle.gather_fp8(pool, table, w.starts, w.ends, w.chunk_size, flag, codes, scales) == 0
    rc, rs = torch_reference_quant(layers, table, chunks, w)
    np.testing.assert_array_equal(scales, rs)
    for a, b in zip(codes, rc):
        np.testing.assert_array_equal(a, b)
    # the element(s) equal to amax map to +-448
    for g, c in enumerate(codes):
        assert ((c == 0x7E) | (c == 0xFE)).reshape(2, w.num_layers, -1).any(axis=-1).all()
    # dequantising scatter == torch composition, into a sentinel pool
    p2 = [np.full_like(a, wl.SENTINEL_BF16) for a in layers]
    t2 = wl.block_table(w, seed=2)
    assert oracle.scatter_fp8(oracle.HostPool(p2, B), t2, w.starts, w.ends, w.chunk_size, flag,
                              codes, scales) == 0
    for g, (r, t0, n) in enumerate(chunks):
        for kv in range(2):
            for l in range(w.num_layers):
                q = torch.from_numpy(codes[g][kv, l]).view(torch.float8_e4m3fn).float()
                y = (q * float(scales[g, kv, l])).to(torch.bfloat16).view(torch.int16).numpy()
                for t in range(n):
                    tok = t0 + t
                    got = p2[l][kv, t2[r, tok // B], tok % B]
                    np.testing.assert_array_equal(got, y[t].view(np.uint16))


def test_quant_error_bound_and_unscaled_special_case():
    """|deq - x| within half an e4m3 step (relative 2^-4, or 2^-10 * scale in the
    subnormal range) plus one bf16 rounding; and a tile whose absmax is 448 has
    scale 1, where the codes are exactly the serde's plain float8 cast."""
    w = wl.Workload("e", 2, 1, 64, 16, 32, (256,))
    layers = bf16_pool(w, 5)
    # make layer 1 / kv 0 have absmax exactly 448 (bf16 448 = 0x43E0)
    table = wl.block_table(w, seed=1)
    layers[1][0, table[0, 3], 5, 7] = 0x43E0
    chunks = oracle.enumerate_chunks(w.starts, w.ends, w.chunk_size, True)
    codes = [np.zeros((2, 2, 256, 64), np.uint8)]
    scales = np.zeros((1, 2, 2), np.float32)
    pool = oracle.HostPool(layers, 16)
    oracle.gather_fp8(pool, table, w.starts, w.ends, 256, True, codes, scales)
    assert scales[0, 0, 1] == 1.0
    rows = np.stack([layers[1][0, table[0, t // 16], t % 16] for t in range(256)])
    x = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16)
    np.testing.assert_array_equal(codes[0][0, 1], x.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # error bound on every tile
    p2 = [np.zeros_like(a) for a in layers]
    oracle.scatter_fp8(oracle.HostPool(p2, 16), table, w.starts, w.ends, 256, True, codes, scales)
    for l in range(2):
        for kv in range(2):
            s = float(scales[0, kv, l])
            xs = np.stack([layers[l][kv, table[0, t // 16], t % 16] for t in range(256)])
            ys = np.stack([p2[l][kv, table[0, t // 16], t % 16] for t in range(256)])
            xf = (xs.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            yf = (ys.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            bound = np.maximum(np.abs(xf) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -8) \
                + np.abs(xf) * 2.0 ** -8
            assert (np.abs(yf - xf) <= bound).all()


def test_zero_tile():
    w = wl.Workload("z", 1, 1, 16, 4, 8, (8,), chunk_size=8)
    layers = [np.zeros((2, 8, 4, 16), np.uint16)]
    layers[0][0, :, :, 3] = 0x8000     # -0 in the K half
    table = np.arange(8, dtype=np.int32)[None, :]
    codes = [np.full((2, 1, 8, 16), 0x55, np.uint8)]
    scales = np.full((1, 2, 1), 9.0, np.float32)
    oracle.gather_fp8(oracle.HostPool(layers, 4), table, [0], [8], 8, True, codes, scales)
    assert (scales == 0).all() and (codes[0] == 0).all()
    p2 = [np.full((2, 8, 4, 16), 0x1234, np.uint16)]
    oracle.scatter_fp8(oracle.HostPool(p2, 4), table, [0], [8], 8, True, codes, scales)
    assert (p2[0][:, :2] == 0).all()


def test_non_finite_values():
    """Tiles holding NaN or infinity, against the formulas evaluated with
    numpy's IEEE float32 arithmetic: a NaN takes no part in the absmax
    (numpy's nanmax) and codes as the canonical e4m3fn NaN 0x7F; an infinity
    makes the scale infinite, so finite values code as signed zeros (x / inf)
    and the infinities as NaN (inf / inf); a tile whose only non-zero value is
    a NaN has scale 0 and all codes 0."""
    w = wl.Workload("nf", 4, 1, 32, 16, 32, (64,), chunk_size=64)
    layers = bf16_pool(w, 7)
    table = wl.block_table(w, seed=1)

    def put(l, kv, tok, col, bits):
        layers[l][kv, table[0, tok // 16], tok % 16, col] = bits

    put(0, 0, 5, 3, 0x7FC0)            # +NaN
    put(0, 0, 40, 9, 0xFF81)           # -NaN with a payload
    put(1, 1, 17, 0, 0x7F80)           # +inf
    put(1, 1, 18, 1, 0xFF80)           # -inf
    put(2, 0, 3, 4, 0x7F80)            # inf and NaN in one tile
    put(2, 0, 60, 5, 0x7FC1)
    layers[3][1][table[0, :4]] = 0     # layer 3 V: zeros and one NaN
    put(3, 1, 30, 2, 0xFFC0)
    codes = [np.zeros((2, 4, 64, 32), np.uint8)]
    scales = np.zeros((1, 2, 4), np.float32)
    assert oracle.gather_fp8(oracle.HostPool(layers, 16), table, [0], [64], 64, True, codes, scales) == 0
    for l in range(4):
        for kv in range(2):
            rows = np.stack([layers[l][kv, table[0, t // 16], t % 16] for t in range(64)])
            x = (rows.astype(np.uint32) << 16).view(np.float32)
            nan = np.isnan(x)
            s = np.float32(np.nanmax(np.abs(x))) / np.float32(448.0)
            assert scales[0, kv, l].tobytes() == np.float32(s).tobytes(), (l, kv)
            c = codes[0][kv, l]
            if s == 0:
                assert (c == 0).all()
                continue
            with np.errstate(invalid="ignore", divide="ignore"):
                y = x / s
            ok = ~np.isnan(y)
            ref = torch.from_numpy(y[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(c[ok], ref)
            assert (c[~ok] == 0x7F).all()
            assert (c[nan] == 0x7F).all()
            if np.isinf(s):
                assert set(np.unique(c[ok]).tolist()) <= {0x00, 0x80}
                np.testing.assert_array_equal(c[ok] == 0x80, np.signbit(x[ok]))
    # the round trip: NaN codes and 0 * inf give NaN, the rest is the plain formula
    p2 = [np.zeros_like(a) for a in layers]
    assert oracle.scatter_fp8(oracle.HostPool(p2, 16), table, [0], [64], 64, True, codes, scales) == 0
    y = (p2[2][0, table[0, 0]].astype(np.uint32) << 16).view(np.float32)
    assert np.isnan(y).all()                       # every value of the inf tile: 0 * inf or NaN
    y = (p2[0][0, table[0, 0], 5, 3].astype(np.uint32) << 16).view(np.float32)
    assert np.isnan(y)
