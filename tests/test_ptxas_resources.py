"""Resource check of the streaming kernel from the assembler's own report
(nvcc -Xptxas -v, no GPU): every variant fits the 128 registers a thread has
with 13-16 warps per SM, and the tcgen05 variants with the static or the
ticket schedule spill nothing (the warp-MMA variants, for widths above 5120,
and the variants that split the partial last round spill a few bytes at
most)."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mhc_residual_seam_gb300", "csrc")


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_stream_kernel_registers_and_spills(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    kernels = {}
    for src in ("mhc_stream.cu", "mhc_stream_split.cu"):
        r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler",
                            "-fPIC", "-I", os.path.join(ROOT, "include"), "-Xptxas", "-v", "-c",
                            os.path.join(CSRC, src), "-o", str(tmp_path / (src + ".o"))],
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        current = None
        for line in r.stderr.splitlines():
            m = re.search(r"Compiling entry function '(_ZN3mhc18stream_seam_kernel\w+)'", line)
            if m:
                current = m.group(1)
                kernels[current] = {}
                continue
            if current is None:
                continue
            m = re.search(r"(\d+) bytes spill stores", line)
            if m:
                kernels[current]["spill"] = int(m.group(1))
            m = re.search(r"Used (\d+) registers", line)
            if m:
                kernels[current]["regs"] = int(m.group(1))
    scheds = [re.search(r"ELi(\d)EEEv", n).group(1) for n in kernels]
    # 3 forms x 3 outputs x 3 projection / cluster forms, static and split;
    # tickets for the bf16 post and no_post forms on clusters of 4 (tcgen05)
    assert scheds.count("0") == 27 and scheds.count("2") == 27 and scheds.count("1") == 2, scheds
    for name, k in kernels.items():
        form, out, ms, kcl, sched = re.search(r"ILi(\d)ELi(\d)ELb(\d)ELi(\d+)ELi(\d)E", name).groups()
        assert k["regs"] <= 128, (name, k)
        if ms == "0" and sched != "2":
            assert k.get("spill", 0) == 0, (name, k)
        else:
            assert k.get("spill", 0) <= 64, (name, k)
