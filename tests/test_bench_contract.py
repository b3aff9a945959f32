"""The benchmark's JSON contract on the CPU: the reference arm (the oracle,
timed on the host) prints one line with the keys the contract names, and
every workload has a byte count (no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mhc_residual_seam_gb300 import accounting as ACC  # noqa: E402


def test_every_workload_has_algorithmic_bytes():
    for name, w in bench.WORKLOADS.items():
        b = ACC.seam_bytes(w["T"], w["H"], post=w["post"], out=w["out"], ident=w.get("ident", False))
        per_token = b // w["T"]
        assert per_token in {20 * w["H"], 18 * w["H"], 10 * w["H"], 22 * w["H"],
                             20 * w["H"] + w["H"] + w["H"] // 32}, name
    assert bench.DEFAULT == "seam_T16384_H5120_post_bf16"


@pytest.mark.parametrize("workload", ["seam_T4_H5120_post_bf16", "seam_T32_H5120_post_unshifted"])
def test_reference_arm_prints_the_contract_line(workload):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "TB/s" and d["value"] > 0
    assert d["config"]["workload"] == workload
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr
