"""The byte accounting that bench.py's TB/s and roofline use, pinned to the
byte counts and rates the pages print (tests/golden/seam_bytes.txt)."""
import os

from mhc_residual_seam_gb300.accounting import seam_bytes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "seam_bytes.txt")
UNIT = {"GB": 1e9, "MB": 1e6}


def _rows():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            yield line.split()


def test_bytes_match_pages():
    n = 0
    for r in _rows():
        if r[0] == "rate":
            continue
        form, T, H, val, unit = r[0], int(r[1]), int(r[2]), float(r[3]), r[4]
        out = "fp8_grid" if form == "fp8_grid" else "bf16"
        got = seam_bytes(T, H, post=True, out=out) / UNIT[unit]
        digits = len(r[3].split(".")[1]) if "." in r[3] else 0
        assert round(got, digits) == val, (form, T, got)
        n += 1
    assert n == 3


def test_rates_match_pages():
    n = 0
    for r in _rows():
        if r[0] != "rate":
            continue
        T, us, tbs = int(r[1]), float(r[2]), float(r[3])
        assert round(seam_bytes(T, 5120) / (us * 1e-6) / 1e12, 2) == tbs
        n += 1
    assert n == 2
