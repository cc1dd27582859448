"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of the oracle's C source, builds it
into a temporary library and runs a compact battery of the same pins the
other oracle tests use (golden chunk counts, the per-token dictionary model,
torch's float8 / bfloat16 conversions and the torch composition of the fp8
definition).  Every planted mistake must fail at least one pin, and the
unmodified source must pass them all.
"""
import importlib.util
import os

import numpy as np
import pytest
import torch

import brute
from paged_kv_cache_lmkv_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lmkv_oracle.c")

MUTANTS = {
    "kv_layer_order_swapped": ("int64_t row_index = ((int64_t)kv * num_layers + l) * n_g + t;",
                               "int64_t row_index = ((int64_t)l * 2 + kv) * n_g + t;"),
    "slot_off_by_one": ("uint8_t* p = pool_row(layer_base, l, kv, num_blocks, block_size,\n"
                        "                                              row_bytes, blk, slot);",
                        "uint8_t* p = pool_row(layer_base, l, kv, num_blocks, block_size,\n"
                        "                                              row_bytes, blk, (slot + 1) % block_size);"),
    "tail_always_dropped": ("if (!save_unfull) break;", "break;", "all"),
    "ties_away_from_zero": ("else if (frac == 0.5 && fmod(n, 2.0) != 0.0) n += 1.0;",
                            "else if (frac == 0.5) n += 1.0;"),
    "no_saturation": ("double r = (a >= 448.0) ? 448.0 : round_to_grid_rne(a, 3, -6);\n    if (r > 448.0) r = 448.0;",
                      "double r = round_to_grid_rne(a, 3, -6);"),
    "e4m3_subnormal_quantum": ("code = (uint8_t)(r / ldexp(1.0, -9));",
                               "code = (uint8_t)(r / ldexp(1.0, -10));"),
    "bf16_six_bits": ("round_to_grid_rne(a, 7, -126)", "round_to_grid_rne(a, 6, -126)"),
    "scale_480": ("volatile float scale = amax / 448.0f;", "volatile float scale = amax / 480.0f;"),
    "absmax_skips_first_row": ("                    float amax = 0.0f;\n                    for (int32_t t = 0; t < n_g; ++t) {",
                               "                    float amax = 0.0f;\n                    for (int32_t t = 1; t < n_g; ++t) {"),
    "dequant_without_scale": ("volatile float y = lmkvo_e4m3_to_f32(q[i]) * scale;",
                              "volatile float y = lmkvo_e4m3_to_f32(q[i]);"),
    "negative_zero_lost": ("uint8_t sign = signbit(v) ? 0x80 : 0x00;", "uint8_t sign = v < 0 ? 0x80 : 0x00;"),
}


def load_oracle(tmp_path, name, mutation=None):
    src = open(SRC).read()
    if mutation is not None:
        old, new = mutation[:2]
        assert src.count(old) >= 1, f"mutation site not found: {name}"
        src = src.replace(old, new, -1 if mutation[2:] == ("all",) else 1)
    d = tmp_path / name
    d.mkdir()
    (d / "lmkv_oracle.c").write_text(src)
    spec = importlib.util.spec_from_file_location(f"oracle_{name}", os.path.join(ROOT, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "lmkv_oracle.c")
    mod._LIB = str(d / "liblmkv_oracle.so")
    mod._lib = None
    return mod


def torch_e4m3(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pins(o):
    """Names of the pins that fail for oracle module `o`."""
    failed = []
    # golden chunk counts
    if len(o.enumerate_chunks([0] * 4, [4096, 9000, 20000, 32768], 256, True) or []) != 259:
        failed.append("chunk_counts")
    # gather / scatter vs the dictionary model
    rng = np.random.default_rng(0)
    L, nb, B, row, C = 3, 40, 4, 8, 16
    layers = [rng.integers(0, 65535, (2, nb, B, row), dtype=np.uint16) for _ in range(L)]
    starts, ends = np.array([0, 16]), np.array([37, 50])
    table = np.stack([rng.permutation(nb)[:13], rng.permutation(nb)[:13]]).astype(np.int32)
    table[1] = np.setdiff1d(np.arange(nb), table[0])[:13]
    ch = o.enumerate_chunks(starts, ends, C, True) or []
    ch_ref = [(r, toks[0], len(toks)) for r, toks in brute.chunk_token_lists(starts, ends, C, True)]
    if ch != ch_ref:
        failed.append("enumerate_vs_dict")
    else:
        got = [np.zeros((2, L, n, row), np.uint16) for _, _, n in ch]
        ref = [np.zeros((2, L, n, row), np.uint16) for _, _, n in ch]
        o.gather(o.HostPool(layers, B), table, starts, ends, C, True, got)
        brute.gather(layers, table, starts, ends, C, True, ref)
        if any(not np.array_equal(a, b) for a, b in zip(got, ref)):
            failed.append("gather_vs_dict")
    # e4m3 encode / decode vs torch, bf16 vs torch
    bits = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    v = bits[np.isfinite(bits) & (np.abs(bits) < 464)]
    if not np.array_equal(o.f32_to_e4m3(v), torch_e4m3(v)):
        failed.append("e4m3_encode")
    if not np.array_equal(o.f32_to_e4m3(np.array([1e9, -1e9], np.float32)), np.array([0x7E, 0xFE], np.uint8)):
        failed.append("e4m3_saturation")
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    if not np.array_equal(o.e4m3_to_f32(codes), torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()):
        failed.append("e4m3_decode")
    x = rng.standard_normal(20000).astype(np.float32) * 3
    if not np.array_equal(o.f32_to_bf16(x), torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)):
        failed.append("bf16")
    # fp8 gather / scatter vs the torch composition of the definition
    w = wl.Workload("m", 2, 1, 32, 4, 32, (40,), chunk_size=16, outliers=True)
    pool = [t.view(torch.int16).numpy().view(np.uint16).copy() for t in wl.make_pool(w, "cpu", 0)]
    pool[0][0, 0, 0, 0] = 0x8000                      # a -0 in the first row
    tab = np.arange(10, dtype=np.int32)[None, :]
    ch = o.enumerate_chunks(w.starts, w.ends, 16, True) or []
    q = [np.zeros((2, 2, n, 32), np.uint8) for _, _, n in ch]
    sc = np.zeros((len(ch), 2, 2), np.float32)
    o.gather_fp8(o.HostPool(pool, 4), tab, w.starts, w.ends, 16, True, q, sc)
    ok = len(ch) == 3
    for g, (r, t0, n) in enumerate(ch if ok else []):
        for kv in range(2):
            for l in range(2):
                rows = np.stack([pool[l][kv, (t0 + t) // 4, (t0 + t) % 4] for t in range(n)])
                xt = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).float()
                s = xt.abs().max() / 448.0
                ok &= sc[g, kv, l] == s.item()
                ok &= np.array_equal(q[g][kv, l], (xt / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
                y = (torch.from_numpy(q[g][kv, l]).view(torch.float8_e4m3fn).float() * s).to(torch.bfloat16)
                p2 = [np.zeros_like(a) for a in pool]
                o.scatter_fp8(o.HostPool(p2, 4), tab, w.starts, w.ends, 16, True, q, sc)
                back = np.stack([p2[l][kv, (t0 + t) // 4, (t0 + t) % 4] for t in range(n)])
                ok &= np.array_equal(back, y.view(torch.int16).numpy().view(np.uint16))
    if not ok:
        failed.append("fp8_vs_torch")
    return failed


def test_unmodified_oracle_passes_every_pin(tmp_path):
    assert pins(load_oracle(tmp_path, "clean")) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    failed = pins(load_oracle(tmp_path, name, MUTANTS[name]))
    assert failed, f"mutant {name} passed every pin"


# ---- the CacheGen codec oracle ----

CG_SRC = os.path.join(ROOT, "oracle", "cachegen_oracle.c")

CG_MUTANTS = {
    "max_is_half_bins": ("int32_t MAX = bins / 2 - 1;", "int32_t MAX = bins / 2;", "all"),
    "cdf_floor": ("        if (2 * r > (uint64_t)n || (2 * r == (uint64_t)n && (q & 1))) q += 1;\n", ""),
    "cdf_ties_up": ("(2 * r == (uint64_t)n && (q & 1))", "(2 * r == (uint64_t)n)"),
    "cdf_no_ramp": ("C[k] = (uint32_t)(q + (uint64_t)k);", "C[k] = (uint32_t)q;"),
    "cdf_inclusive_cumsum": ("uint64_t num = cum * M;", "uint64_t num = (cum + (uint64_t)count[k]) * M;"),
    "follow_bits_same_value": ("write_bit(w, !bit);", "write_bit(w, bit);"),
    "final_bits_flipped": ("low < CG_QUARTER ? 0 : 1", "low < CG_QUARTER ? 1 : 0"),
    "decoder_keeps_top_half": ("                value -= CG_HALF;\n", ""),
    "batch_of_128": ("#define CG_BATCH 256", "#define CG_BATCH 128"),
    "v_bins_like_k": ("bins[num_layers + l] = (all32 || l < 2)", "bins[num_layers + l] = (all32 || l < 10)"),
    "max1_skips_first_channel": ("        for (int32_t c = 0; c < H; ++c) {\n            float a",
                                 "        for (int32_t c = 1; c < H; ++c) {\n            float a"),
    "dequant_without_offset": ("(float)((int32_t)sym[(int64_t)t * H + c] - MAX) / (float)MAX",
                               "(float)((int32_t)sym[(int64_t)t * H + c]) / (float)MAX"),
    "quant_truncates": ("q = (int32_t)nearbyintf(zc);", "q = (int32_t)zc;"),
    "nan_clamps_high": ("fminf(fmaxf(z, 0.0f), (float)(2 * MAX))", "fmaxf(fminf(z, (float)(2 * MAX)), 0.0f)"),
}


def load_cachegen(tmp_path, name, mutation=None):
    src = open(CG_SRC).read()
    if mutation is not None:
        old, new = mutation[:2]
        assert src.count(old) >= 1, f"mutation site not found: {name}"
        src = src.replace(old, new, -1 if mutation[2:] == ("all",) else 1)
    d = tmp_path / ("cg_" + name)
    d.mkdir()
    (d / "cachegen_oracle.c").write_text(src)
    spec = importlib.util.spec_from_file_location(f"cachegen_{name}", os.path.join(ROOT, "oracle", "cachegen.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "cachegen_oracle.c")
    mod._LIB = str(d / "libcachegen_oracle.so")
    mod._lib = None
    return mod


def cachegen_pins(o):
    """Names of the CacheGen pins that fail for oracle module `o` (the same
    kinds of check as tests/test_oracle_cachegen.py, compacted)."""
    import test_oracle_cachegen as t
    failed = []

    def run(name, fn):
        try:
            if fn() is False:
                failed.append(name)
        except Exception:       # a crash or a rejected call fails the pin too
            failed.append(name)

    def golden_bins():
        for case in t._golden("bins"):
            lhs, rhs = case.split("->")
            L = int(lhs)
            k_part, v_part = rhs.split("V:")
            expect = [[int(b) for run in part.split() for b in [run.split("x")[1]] * int(run.split("x")[0])]
                      for part in (k_part.replace("K:", ""), v_part)]
            if o.default_bins(L).tolist() != expect:
                return False

    def golden_cdf():
        for case in t._golden("cdf"):
            lhs, rhs = case.split("->")
            bins, *syms = [int(v) for v in lhs.split()]
            if o.cdf(np.array(syms, np.uint8), o.nsym(bins)).tolist() != [int(v) for v in rhs.split()]:
                return False
        rng = np.random.default_rng(1)
        for n in (3, 256):
            syms = rng.integers(0, 15, n)
            if o.cdf(syms.astype(np.uint8), 15).tolist() != t._cdf_exact(syms, 15):
                return False

    def golden_code():
        for case in t._golden("code"):
            lhs, rhs = case.split("->")
            cdf_part, sym_part = lhs.split(":")
            C = np.array([int(v) for v in cdf_part.split()], np.uint32)
            syms = np.array([int(v) for v in sym_part.split()], np.uint8)
            code = o.encode(syms, C)
            if code != t._hex(rhs) or not np.array_equal(o.decode(code, len(syms), C), syms):
                return False

    def round_trip():
        rng = np.random.default_rng(2)
        for trial in range(12):
            C = t._random_cdf(rng, 15, trial % 2 == 0)
            syms = rng.integers(0, 15, 200).astype(np.uint8)
            code = o.encode(syms, C)
            ideal = t._ideal_bits(syms, C)
            if not np.array_equal(o.decode(code, 200, C), syms) or not ideal <= 8 * len(code) <= ideal + 10:
                return False

    def golden_quant():
        for case in t._golden("quant"):
            lhs, rhs = case.split("->")
            bins, *vals = lhs.split()
            sym_part, deq_part = rhs.split("|")
            row = t._bf16([float(v) for v in vals])[None, :]
            sym, max1 = o.quantize(row, int(bins))
            if sym[0].tolist() != [int(v) for v in sym_part.split()]:
                return False
            if [f"{v:04x}" for v in o.dequantize(sym, max1, int(bins))[0]] != deq_part.split():
                return False

    def chunk():
        L, n, H = 2, 300, 16
        bins = o.default_bins(L)
        x = t._chunk(L, n, H, 3)
        blob = o.encode_chunk(x, bins)
        parts = o.parse(blob, L, n, H, bins)
        if parts["lengths"].shape[0] != 2 or len(blob) != parts["layout"]["bytes"] + int(parts["lengths"].sum()):
            return False
        xb = x.view(torch.int16).numpy().view(np.uint16)
        got = o.decode_chunk(blob, L, n, H, bins)
        xf = (xb.astype(np.uint32) << 16).view(np.float32)
        yf = (got.astype(np.uint32) << 16).view(np.float32)
        max1 = np.abs(xf).max(axis=3, keepdims=True)
        MAX = (bins // 2 - 1)[:, :, None, None]
        return bool(np.all(np.abs(yf - xf) <= max1 * (0.5 / MAX * (1 + 1e-5) + 2.0 ** -8)))

    for name, fn in [("bins", golden_bins), ("cdf", golden_cdf), ("code", golden_code),
                     ("round_trip", round_trip), ("quant", golden_quant), ("chunk", chunk)]:
        run(name, fn)
    return failed


def test_unmodified_cachegen_oracle_passes_every_pin(tmp_path):
    assert cachegen_pins(load_cachegen(tmp_path, "clean")) == []


@pytest.mark.parametrize("name", sorted(CG_MUTANTS))
def test_planted_cachegen_mistake_is_caught(tmp_path, name):
    failed = cachegen_pins(load_cachegen(tmp_path, name, CG_MUTANTS[name]))
    assert failed, f"mutant {name} passed every pin"
