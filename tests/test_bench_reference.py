"""The bench's reference arm is the CPU oracle alone: it runs without a GPU,
loads no part of the CUDA library, and prints one JSON line whose step time is
the sample's own (not an extrapolation)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SNIPPET = r"""
import contextlib, io, json, sys
sys.argv = ["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1", "--ref-seconds", "3"]
import bench
buf = io.StringIO()
with contextlib.redirect_stdout(buf):
    bench.main()
maps = open("/proc/self/maps").read()
print(json.dumps({"line": buf.getvalue().strip(), "liblmkv": "liblmkv.so" in maps,
                  "oracle": "liblmkv_oracle.so" in maps}))
"""


def test_reference_arm_runs_the_oracle_only():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", SNIPPET], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert not res["liblmkv"] and res["oracle"]
    line = json.loads(res["line"])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the step time is the sample's own; the full-batch figure is reported beside it
    assert line["ms_per_step"] < line["ms_per_step_full_batch_extrapolated"]
    assert line["ms_per_step"] < 10_000
