"""bench.py's JSON line on a GPU: every key the benchmark contract names, with sane values, for
the headline-style path and for the other workload families (small runs)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def check_line(d, e2e=True):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["n_gpus"] == 1 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert "workload" in d["config"]
    r = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] in ("tensor", "hbm") and 0 < r["frac"] < 1.5
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    if e2e:
        e = d["e2e"]
        assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
        # the end-to-end step time is the median of its repeats too
        er = sorted(e["repeat_ms_per_step"])
        assert len(er) == d["repeats"] and abs(e["ms_per_step"] - er[len(er) // 2]) <= 1e-9 * max(1.0, e["ms_per_step"])
    assert d["gpu_launches"] >= d["steps"] * d["repeats"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    # the reported step time is the median of the repeats' step times
    reps = sorted(d["repeat_ms_per_step"])
    assert len(reps) == d["repeats"] >= 1
    assert abs(d["ms_per_step"] - reps[len(reps) // 2]) <= 1e-9 * max(1.0, d["ms_per_step"])


def test_forward_line():
    check_line(run("--workload", "causal_bf16_n2048_d128", "--steps", "5", "--warmup", "3", "--cpu-seconds", "1"))


@pytest.mark.parametrize("workload,e2e", [("decode_gqa_bf16_nq16_nk8192_d128", False),
                                          ("varlen_causal_gqa_bf16_16seq_d128", True),
                                          ("bwd_causal_gqa_bf16_n8192_d128", True),
                                          ("fp8_block_hadamard_noncausal_n8192_d128", True)])
def test_other_families(workload, e2e):
    args = ["--workload", workload, "--steps", "3", "--warmup", "3", "--cpu-seconds", "1"]
    if workload.startswith("bwd"):
        args += ["--batch", "1"]
    check_line(run(*args), e2e=e2e)
