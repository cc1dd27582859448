"""Pins for the CacheGen codec oracle (CPU only).

The oracle follows "LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与
源码解析", sections 1-5.  Nothing here re-runs the oracle's own formulas:
the checks are hand-worked fixtures (tests/golden/cachegen.txt), exact
rational arithmetic through Python's fractions, closed forms of the coder on
dyadic CDFs, the information-theoretic bounds on the code length, round trips
and the quantisation error bound.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import cachegen as cg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "cachegen.txt")


def _golden(kind):
    out = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line.startswith(kind + " "):
            out.append(line[len(kind) + 1:])
    assert out, kind
    return out


def _bf16(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


# ---- bins (section 1) ----

@pytest.mark.parametrize("case", _golden("bins"))
def test_golden_bins(case):
    lhs, rhs = case.split("->")
    L = int(lhs)
    k_part, v_part = rhs.split("V:")
    expect = []
    for part in (k_part.replace("K:", ""), v_part):
        row = []
        for run in part.split():
            cnt, b = run.split("x")
            row += [int(b)] * int(cnt)
        expect.append(row)
    assert cg.default_bins(L).tolist() == expect


# ---- CDF (section 3) ----

@pytest.mark.parametrize("case", _golden("cdf"))
def test_golden_cdf(case):
    lhs, rhs = case.split("->")
    bins, *syms = [int(v) for v in lhs.split()]
    assert cg.cdf(np.array(syms, np.uint8), cg.nsym(bins)).tolist() == [int(v) for v in rhs.split()]


def _cdf_exact(syms, nsym):
    """C[k] = round(cum[k] * (2^16 - nsym) / n) + k with exact rationals;
    Python's round() of a Fraction sends halves to the even neighbour."""
    n = len(syms)
    counts = np.bincount(syms, minlength=nsym)
    cum = np.concatenate([[0], np.cumsum(counts)])
    return [round(Fraction(int(c) * (65536 - nsym), n)) + k for k, c in enumerate(cum)]


@pytest.mark.parametrize("bins", [4, 8, 16, 32])
@pytest.mark.parametrize("n", [1, 2, 3, 7, 256, 768])
def test_cdf_matches_exact_rational(bins, n):
    rng = np.random.default_rng(bins * 1000 + n)
    nsym = cg.nsym(bins)
    for trial in range(20):
        if trial % 3 == 0:
            syms = rng.integers(0, nsym, n)
        else:    # peaked, like quantised KV: mass near MAX
            syms = np.clip(np.rint(rng.normal(nsym // 2, 1 + trial % 4, n)), 0, nsym - 1).astype(int)
        C = cg.cdf(syms.astype(np.uint8), nsym)
        assert C.tolist() == _cdf_exact(syms, nsym)
        assert C[0] == 0 and C[-1] == 65536
        assert np.all(np.diff(C.astype(np.int64)) >= 1)


# ---- the arithmetic coder (section 4) ----

def _hex(s):
    return bytes(int(v, 16) for v in s.split())


@pytest.mark.parametrize("case", _golden("code"))
def test_golden_code(case):
    lhs, rhs = case.split("->")
    cdf_part, sym_part = lhs.split(":")
    C = np.array([int(v) for v in cdf_part.split()], np.uint32)
    syms = np.array([int(v) for v in sym_part.split()], np.uint8)
    code = cg.encode(syms, C)
    assert code == _hex(rhs)
    assert np.array_equal(cg.decode(code, len(syms), C), syms)


def _bits_to_bytes(bits):
    bits = bits + "0" * (-len(bits) % 8)
    return bytes(int(bits[i:i + 8], 2) for i in range(0, len(bits), 8))


@pytest.mark.parametrize("j", [1, 2, 3, 4, 5])
def test_uniform_dyadic_cdf_is_fixed_width(j):
    """2^j equal symbols: every symbol costs exactly its j-bit index, and the
    two final bits are 01 (the interval is [0, 1) again after each symbol)."""
    rng = np.random.default_rng(j)
    C = np.arange(0, 65537, 65536 >> j, dtype=np.uint32)
    syms = rng.integers(0, 1 << j, 200).astype(np.uint8)
    expect = "".join(format(int(s), f"0{j}b") for s in syms) + "01"
    assert cg.encode(syms, C) == _bits_to_bytes(expect)


def test_prefix_code_cdf():
    """Intervals 1/2, 1/4, 1/8, 1/16, 1/16: the output is the prefix code."""
    C = np.array([0, 32768, 49152, 57344, 61440, 65536], np.uint32)
    codes = ["0", "10", "110", "1110", "1111"]
    rng = np.random.default_rng(5)
    syms = rng.integers(0, 5, 300).astype(np.uint8)
    assert cg.encode(syms, C) == _bits_to_bytes("".join(codes[s] for s in syms) + "01")


def _ideal_bits(syms, C):
    f = (C[1:].astype(np.int64) - C[:-1])[syms]
    return float(np.sum(16 - np.log2(f)))


def _random_cdf(rng, nsym, peaked):
    if peaked:
        p = np.exp(-0.5 * ((np.arange(nsym) - nsym // 2) / rng.uniform(0.5, 3)) ** 2)
    else:
        p = rng.uniform(0, 1, nsym)
    w = np.floor(p / p.sum() * (65536 - nsym)).astype(np.int64) + 1
    w[np.argmax(w)] += 65536 - w.sum()
    return np.concatenate([[0], np.cumsum(w)]).astype(np.uint32)


@pytest.mark.parametrize("nsym", [3, 15, 31])
def test_round_trip_and_length_bounds(nsym):
    """Decoding gives the symbols back, and the length sits between the ideal
    code length sum(-log2 p) and that plus the two final bits, the byte
    padding and the truncation loss (at most -log2(1 - 2^-14) per symbol)."""
    rng = np.random.default_rng(nsym)
    for trial in range(40):
        C = _random_cdf(rng, nsym, trial % 2 == 0)
        p = (C[1:].astype(np.float64) - C[:-1]) / 65536
        n = int(rng.integers(1, 300))
        syms = rng.choice(nsym, n, p=p).astype(np.uint8) if trial % 4 else rng.integers(0, nsym, n).astype(np.uint8)
        code = cg.encode(syms, C)
        assert np.array_equal(cg.decode(code, n, C), syms)
        ideal = _ideal_bits(syms, C)
        bits = 8 * len(code)
        assert bits >= ideal - 1e-6
        assert bits <= ideal + 2 + 7 + n * -math.log2(1 - 2.0 ** -14) + 1e-6


def test_rarest_symbols_reach_the_18_bit_bound():
    """Symbols of frequency 1/65536 cost about 16 bits each; no stream may
    pass 18 bits per symbol plus 2 (the bound the blob layout reserves)."""
    C = np.array([0, 1, 65535, 65536], np.uint32)
    for pattern in ([0], [2], [0, 2], [2, 0], [0, 1, 2]):
        syms = np.array((pattern * 256)[:256], np.uint8)
        code = cg.encode(syms, C)
        assert np.array_equal(cg.decode(code, 256, C), syms)
        assert 8 * len(code) <= 18 * 256 + 2 + 7


def test_decoder_reads_zeros_past_the_end():
    """The last bytes of a stream are not needed when they are zero: the
    decoder supplies zero bits past the stream."""
    C = np.array([0, 16384, 49152, 65536], np.uint32)
    syms = np.array([1, 1, 1, 1], np.uint8)
    code = cg.encode(syms, C)
    assert np.array_equal(cg.decode(code.rstrip(b"\0"), 4, C), syms)


# ---- quantisation and dequantisation (sections 2 and 5) ----

@pytest.mark.parametrize("case", _golden("quant"))
def test_golden_quant(case):
    lhs, rhs = case.split("->")
    bins, *vals = lhs.split()
    sym_part, deq_part = rhs.split("|")
    row = _bf16([float(v) for v in vals])[None, :]
    sym, max1 = cg.quantize(row, int(bins))
    assert sym[0].tolist() == [int(v) for v in sym_part.split()]
    assert max1[0] == np.max(np.abs(_bf16_to_f32(row[0])))
    back = cg.dequantize(sym, max1, int(bins))
    assert [f"{v:04x}" for v in back[0]] == deq_part.split()


@pytest.mark.parametrize("bins", [4, 16, 32])
def test_quantisation_error_bound(bins):
    """|dequantised - x| stays within half a quantisation step max1/MAX (plus
    the final bf16 rounding), the row's largest |x| lands on an end symbol,
    and max1 is the row's largest |x|."""
    rng = np.random.default_rng(bins)
    MAX = bins // 2 - 1
    x = rng.standard_normal((64, 96)).astype(np.float32)
    x[::7] *= 50
    x[3, 5] = 0
    bits = _bf16(x)
    xf = _bf16_to_f32(bits)
    sym, max1 = cg.quantize(bits, bins)
    assert np.array_equal(max1, np.abs(xf).max(axis=1))
    assert sym.max() <= 2 * MAX
    arg = np.abs(xf).argmax(axis=1)
    ends = sym[np.arange(64), arg]
    assert np.all((ends == 0) | (ends == 2 * MAX))
    y = _bf16_to_f32(cg.dequantize(sym, max1, bins))
    bound = max1[:, None] * (0.5 / MAX * (1 + 1e-5) + 2.0 ** -8)
    assert np.all(np.abs(y - xf) <= bound)


@pytest.mark.parametrize("bins", [4, 16, 32])
def test_dequantise_closed_forms(bins):
    """Symbol MAX gives +0, symbol 0 gives -max1, symbol 2*MAX gives +max1."""
    MAX = bins // 2 - 1
    max1 = _bf16_to_f32(_bf16([0.5, 3.0, 1e-3, 7.25]))
    sym = np.array([[MAX, 0, 2 * MAX]] * 4, np.uint8)
    y = cg.dequantize(sym, max1, bins)
    assert np.all(y[:, 0] == 0)
    assert np.array_equal(_bf16_to_f32(y[:, 1]), -max1)
    assert np.array_equal(_bf16_to_f32(y[:, 2]), max1)


# ---- the whole chunk ----

def _chunk(L, n, H, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((2, L, n, H), generator=g)
    x[:, :, :, ::17] *= 8
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("n", [1, 5, 256, 300, 513])
def test_chunk_round_trip(n):
    """decode(encode(x)) equals dequantise(quantise(x)) slice by slice, every
    stream decodes from its prefix-sum offset with its channel's CDF, the
    CDF entries are the ones of the chunk's symbols, and the size respects
    the layout bound."""
    L, H = 3, 40
    bins = cg.default_bins(L)
    bins[0, 1] = 8
    x = _chunk(L, n, H, n)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    blob = cg.encode_chunk(x, bins)
    parts = cg.parse(blob, L, n, H, bins)
    assert len(blob) == parts["layout"]["bytes"] + int(parts["lengths"].sum())
    assert len(blob) <= parts["layout"]["bound"]
    got = cg.decode_chunk(blob, L, n, H, bins)
    offs = np.concatenate([[0], np.cumsum(parts["lengths"].reshape(-1), dtype=np.int64)])
    nb = (n + 255) // 256
    for kv in range(2):
        for l in range(L):
            b = int(bins[kv, l])
            sym, max1 = cg.quantize(xb[kv, l], b)
            assert np.array_equal(parts["max1"][kv, l], max1)
            assert np.array_equal(got[kv, l], cg.dequantize(sym, max1, b))
            s = kv * L + l
            for c in range(H):
                C = cg.cdf(sym[:, c], cg.nsym(b))
                assert np.array_equal(parts["cdf"][s][c], C[1:-1])
                for bi in range(nb):
                    i = (bi * 2 * L + s) * H + c
                    stream = parts["bytes"][offs[i]:offs[i + 1]].tobytes()
                    t0, t1 = 256 * bi, min(n, 256 * (bi + 1))
                    assert np.array_equal(cg.decode(stream, t1 - t0, C), sym[t0:t1, c])


def test_compression_on_gaussian_kv():
    """Quantised N(0,1) rows take about 3-4 bits per element once coded, so a
    256-token chunk compresses by well over 3x."""
    L, n, H = 4, 256, 256
    x = _chunk(L, n, H, 7)
    blob = cg.encode_chunk(x, cg.default_bins(L))
    assert x.numel() * 2 / len(blob) > 3.0


def test_invalid_layout_is_rejected():
    with pytest.raises(ValueError):
        cg.layout(2, 4, 8, [2, 16, 16, 16])
    with pytest.raises(ValueError):
        cg.layout(2, 0, 8, [16] * 4)
