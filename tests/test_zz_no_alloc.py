"""mhc_seam_noalloc, the entry point for callers that cannot allocate device
memory (a plug-in inside a host program that owns every allocation, code in an
allocator callback, a loop that must never block in the allocator): its
output must match mhc_seam's (the caller-provided-workspace entry point) within
the parity tolerance, on two calls in a row that share the static scratch.

Collected last on purpose; it must pass alone in a fresh process and after the
other tests."""
import numpy as np
import pytest
import torch

from mhc_residual_seam_gb300 import binding as B

from seam_case import make_case, run_gpu, to_dev, to_host, ulp_diff

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


def _noalloc(d, g, out, cfg=None):
    B.mhc_seam_noalloc(g["R"], g["Y"], g["post_prev"], g["comb_prev"], g["pre_prev"], g["fn"], g["bias"],
                       g["alpha"], g["gamma"], d["eps"], d["out_mode"], out["residual_out"], out["norm"],
                       out["fp8_codes"], out["e8m0_scales"], out["pre_out"], out["post_out"], out["comb_out"],
                       cfg=cfg)


def _close(a, b):
    for k in ("residual_out", "norm"):
        assert np.mean(ulp_diff(a[k], b[k]) <= 1) >= 0.9999, k
    for k in ("pre_out", "post_out", "comb_out"):
        assert np.max(np.abs(a[k].astype(np.float64) - b[k])) <= 1e-3, k
    if "fp8_codes" in a:
        assert np.array_equal(a["fp8_codes"], b["fp8_codes"]) and np.array_equal(a["e8m0_scales"], b["e8m0_scales"])


@pytest.mark.parametrize("T,mx,post", [(4, False, True), (64, True, True), (480, False, False)])
def test_noalloc_matches_workspace_entry_two_calls_in_a_row(T, mx, post):
    d = make_case(T, 5120, 9100 + T, post=post, mxfp8=mx)
    g = to_dev(d)
    ref = to_host(run_gpu(d, g=g, cfg=B.MhcConfig(path=1)))
    out = B.alloc_outputs(T, 5120, d["out_mode"], "cuda")
    _noalloc(d, g, out)  # the first call on the device resolves the scratch address
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        for v in out.values():
            if v is not None and v is not out["workspace"]:
                v.zero_()
        _noalloc(d, g, out)
        B.mhc_noalloc_check_status()
        _close(to_host(out), ref)
    # the calls took no device memory (cudaMalloc works in 2 MiB pages, so one would show)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_refuses_calls_beyond_its_scratch():
    d = make_case(481, 5120, 9200)
    g = to_dev(d)
    out = B.alloc_outputs(481, 5120, d["out_mode"], "cuda")
    with pytest.raises(B.MhcError) as e:
        _noalloc(d, g, out)
    assert e.value.code == -5 and "scratch" in str(e.value)
    with pytest.raises(B.MhcError) as e:
        _noalloc(d, g, out, cfg=B.MhcConfig(path=2))
    assert e.value.code == -10


def test_noalloc_reports_a_wait_that_ran_out():
    # A spin limit of one makes the split path's non-finishing CTAs give up
    # waiting: the status word in the static scratch keeps that until
    # mhc_noalloc_check_status() reads it (later calls do not clear it), and a
    # normal call afterwards is correct again.
    d = make_case(8, 5120, 9300)
    g = to_dev(d)
    out = B.alloc_outputs(8, 5120, d["out_mode"], "cuda")
    B.mhc_noalloc_check_status()  # start from a clear status word
    hit = False
    for _ in range(5):
        _noalloc(d, g, out, cfg=B.MhcConfig(path=1, spin_limit=1))
        _noalloc(d, g, out)       # a normal call in between leaves the record alone
        try:
            B.mhc_noalloc_check_status()
        except B.MhcError as e:
            assert e.code == -7
            hit = True
            break
    assert hit
    ref = to_host(run_gpu(d, g=g, cfg=B.MhcConfig(path=1)))
    _noalloc(d, g, out)
    B.mhc_noalloc_check_status()
    _close(to_host(out), ref)


def test_noalloc_identity_form():
    # no comb, Y or post: R' = R, the residual buffer is left alone
    d = make_case(64, 5120, 9400, ident=True)
    g = to_dev(d)
    ref = to_host(run_gpu(d, g=g, cfg=B.MhcConfig(path=1)))
    out = B.alloc_outputs(64, 5120, d["out_mode"], "cuda")
    out["residual_out"].fill_(5.0)
    _noalloc(d, g, out)
    torch.cuda.synchronize()
    assert bool((out["residual_out"] == 5.0).all())
    h = to_host(out)
    assert np.mean(ulp_diff(h["norm"], ref["norm"]) <= 1) >= 0.9999
    for k in ("pre_out", "post_out", "comb_out"):
        assert np.max(np.abs(h[k].astype(np.float64) - ref[k])) <= 1e-3, k

