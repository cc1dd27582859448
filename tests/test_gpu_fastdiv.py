"""Exhaustive GPU check of the quantiser's division by the per-tile scale.

The quantising gather divides by the tile's scale with a correctly rounded
reciprocal and one remainder-correction step (Markstein's method) on the
packed fp32 pipe instead of the IEEE division routine.  Over every scale a bf16 absmax can produce and
every bf16 input that can share a tile with it, the resulting e4m3 codes
must equal those from IEEE division (which the oracle uses; its division is
pinned to numpy's IEEE fp32 division in test_oracle_fp8.py).
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_fast_division_codes_equal_ieee(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    so = str(tmp_path / "libfastdiv.so")
    subprocess.run(["nvcc", "-gencode=arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC",
                    "-I", os.path.join(ROOT, "paged_kv_cache_lmkv_gb300", "csrc"),
                    "-o", so, os.path.join(HERE, "csrc", "fastdiv_check.cu")], check=True)
    lib = ctypes.CDLL(so)
    out = (ctypes.c_ulonglong * 4)()
    assert lib.lmkv_test_fastdiv_exhaustive(out) == 0
    checked, code_mismatch, first = out[0], out[1], out[3]
    assert checked > 1_000_000_000
    assert code_mismatch == 0, f"first mismatch amax/x bits {first:#010x}"
    print(f"checked {checked} (x, scale) pairs")
