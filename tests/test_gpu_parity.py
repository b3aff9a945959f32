"""GPU parity of the seam against the oracle, through the C ABI.

Workloads are the pages' configurations at H = 5120 (T = 4, 64, 1024 mxfp8
with crafted quantiser groups, 4160, 16384; post and no_post), tails and odd
widths, and every launch-policy branch.  Every element of every output is
compared with the oracle: the full-size cases draw 1024 or 2048 distinct tokens
repeated along T, the oracle runs on the distinct ones, and each GPU row is
checked against the oracle row of its token class.
"""
import numpy as np
import pytest
import torch

from mhc_residual_seam_gb300 import binding as B
from mhc_residual_seam_gb300 import inputs as I

import oracle as O
from seam_case import GATE_TOL, compare, compare_all_tokens, make_case, run_gpu, to_dev, to_host, ulp_diff

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


# ------------------------------------------------------ the pages' configs --
def test_config0_T4_post_bf16():
    d = make_case(4, 5120, 1000)
    compare(d, to_host(run_gpu(d)))


@pytest.mark.parametrize("post", [True, False])
def test_config1_T64(post):
    d = make_case(64, 5120, 1001, post=post)
    compare(d, to_host(run_gpu(d)))


def test_config2_T1024_mxfp8_crafted():
    d = make_case(1024, 5120, 1002, mxfp8=True, craft=True)
    h = to_host(run_gpu(d))
    rep = compare(d, h)
    # the crafted tokens really carry the crafted groups: their norm is gamma
    g = I.bf16_bits(d["gamma"])
    for t in d["crafted_rows"]:
        for grp in d["crafted_groups"]:
            sl = slice(32 * grp, 32 * grp + 32)
            assert np.array_equal(h["norm"][t, sl], g[sl]), (t, grp)
    assert rep["codes_mismatch"] == 0


@pytest.mark.parametrize("T", [4159, 4160, 4161])
def test_config3_wave_edge(T):
    d = make_case(T, 5120, 1003, unique_tokens=1024)
    h = to_host(run_gpu(d))
    rep = compare_all_tokens(d, h, 1024)
    assert rep["norm_elements"] == T * 5120


@pytest.mark.parametrize("post", [True, False])
def test_config4_T16384(post):
    d = make_case(16384, 5120, 1004, post=post, unique_tokens=2048)
    h = to_host(run_gpu(d))
    rep = compare_all_tokens(d, h, 2048)
    assert rep["residual_out_elements"] == 16384 * 4 * 5120


# ----------------------------------------------------------- tails, widths --
@pytest.mark.parametrize("T", [1, 2, 3, 5, 9, 17, 33, 129, 257])
def test_ragged_token_counts(T):
    d = make_case(T, 5120, 2000 + T)
    compare(d, to_host(run_gpu(d)))


@pytest.mark.parametrize("H,mx", [(8, False), (40, False), (64, False), (136, False), (1024, False),
                                  (7168, False), (32, True), (96, True), (4096, True)])
def test_widths(H, mx):
    d = make_case(37, H, 3000 + H, mxfp8=mx)
    compare(d, to_host(run_gpu(d)))


@pytest.mark.parametrize("bm,cols", [(1, 64), (2, 64), (4, 96), (8, 128), (16, 640), (32, 1024), (2, 5120)])
def test_policy_overrides(bm, cols):
    d = make_case(45, 5120, 4000 + bm)
    cfg = B.MhcConfig(path=1, block_m=bm, cols_per_cta=cols)
    compare(d, to_host(run_gpu(d, cfg=cfg)))


def test_policy_rejects_oversized_tile():
    d = make_case(4, 5120, 4050)
    with pytest.raises(B.MhcError) as e:
        run_gpu(d, cfg=B.MhcConfig(path=1, block_m=32, cols_per_cta=4096))
    assert e.value.code == -10


def test_multi_wave_launch():
    # more token groups than fit on the GPU at once: several cooperative waves
    d = make_case(3000, 1024, 4100)
    cfg = B.MhcConfig(path=1, block_m=1, cols_per_cta=32)
    out = run_gpu(d, cfg=cfg)
    assert B.mhc_last_launch_count() >= 2
    compare(d, to_host(out))


# ------------------------------------------------------------ behaviours ----
def test_in_place_residual():
    d = make_case(33, 5120, 5000)
    compare(d, to_host(run_gpu(d, inplace=True)))


def test_repeat_calls_are_deterministic_and_self_resetting():
    d = make_case(64, 5120, 5001, mxfp8=True)
    g = to_dev(d)
    out = B.alloc_outputs(64, 5120, d["out_mode"], "cuda")
    a = to_host(run_gpu(d, g=g, out=out))
    b = to_host(run_gpu(d, g=g, out=out))
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    compare(d, b)
    B.mhc_check_status(out["workspace"])


def test_cuda_graph_capture_and_replay():
    d = make_case(64, 5120, 5002)
    g = to_dev(d)
    out = B.alloc_outputs(64, 5120, d["out_mode"], "cuda")
    run_gpu(d, g=g, out=out)  # eager first call (per-device set-up)
    torch.cuda.synchronize()
    for v in out.values():
        if v is not None and v is not out["workspace"]:
            v.zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run_gpu(d, g=g, out=out, stream=s)
    for _ in range(3):
        graph.replay()
    compare(d, to_host(out))


def test_two_streams_separate_workspaces():
    d1, d2 = make_case(16, 5120, 5003), make_case(40, 5120, 5004, post=False)
    g1, g2 = to_dev(d1), to_dev(d2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1 = B.alloc_outputs(16, 5120, 0, "cuda")
    o2 = B.alloc_outputs(40, 5120, 0, "cuda")
    torch.cuda.synchronize()
    for _ in range(4):
        run_gpu(d1, g=g1, out=o1, stream=s1)
        run_gpu(d2, g=g2, out=o2, stream=s2)
    compare(d1, to_host(o1))
    compare(d2, to_host(o2))


def test_bounded_wait_runs_out_and_reports():
    # A spin limit of one iteration makes the non-finishing CTAs give up
    # waiting for rstd: the kernel still returns, the status word reports it,
    # and the next call on the same workspace is correct again.
    d = make_case(8, 5120, 5005)
    g = to_dev(d)
    out = B.alloc_outputs(8, 5120, 0, "cuda")
    cfg = B.MhcConfig(path=1, spin_limit=1)
    hit = False
    for _ in range(5):
        run_gpu(d, g=g, out=out, cfg=cfg)
        try:
            B.mhc_check_status(out["workspace"])
        except B.MhcError as e:
            assert e.code == -7
            hit = True
            break
    assert hit
    run_gpu(d, g=g, out=out)
    B.mhc_check_status(out["workspace"])
    compare(d, to_host(out))


@pytest.mark.parametrize("path,T", [(2, 1100), (3, 64)])
def test_stream_bounded_wait_reports_and_next_call_is_correct(path, T):
    # A spin limit of one (about 100 ns) puts every wait that is not already
    # done past the report threshold on the streaming paths: the status word
    # reports it, the call still completes (a wait is abandoned only a second
    # past the threshold, which no wait here comes near), and the next call on
    # the same workspace is correct and clean.
    d = make_case(T, 5120, 9600 + T)
    g = to_dev(d)
    cfg = B.MhcConfig(path=path)
    out = B.alloc_outputs(T, 5120, d["out_mode"], "cuda", cfg)
    run_gpu(d, g=g, out=out, cfg=B.MhcConfig(path=path, spin_limit=1))
    with pytest.raises(B.MhcError) as e:
        B.mhc_check_status(out["workspace"])
    assert e.value.code == -7
    compare(d, to_host(out))
    for k in ("residual_out", "norm", "pre_out", "post_out", "comb_out"):
        out[k].zero_()
    run_gpu(d, g=g, out=out, cfg=cfg)
    B.mhc_check_status(out["workspace"])
    compare(d, to_host(out))


@pytest.mark.parametrize("path,T", [(2, 1100), (3, 64)])
def test_out_mode_switch_on_shared_buffers(path, T):
    # fp8_grid, then mxfp8, then fp8_grid again on the same buffers (one
    # quantised-output buffer of 2 T H bytes serves both modes, as when a
    # model's attention seams emit the grid and its FFN seams mxfp8): the
    # tensor maps the library keeps per buffer set must follow the mode.
    H = 5120
    d = make_case(T, H, 9700 + T, grid=True)
    g = to_dev(d)
    cfg = B.MhcConfig(path=path)
    out = B.alloc_outputs(T, H, B.MHC_OUT_FP8_GRID, "cuda", cfg)
    grid = out["fp8_codes"]                                   # [T, H] bf16: 2 T H bytes
    codes = grid.view(torch.uint8).reshape(-1)[:T * H].view(T, H)  # the same base address, [T, H] u8
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    for mode in (B.MHC_OUT_FP8_GRID, B.MHC_OUT_MXFP8, B.MHC_OUT_FP8_GRID):
        dm = dict(d, out_mode=mode)
        o = dict(out, fp8_codes=grid if mode == B.MHC_OUT_FP8_GRID else codes,
                 e8m0_scales=scales if mode == B.MHC_OUT_MXFP8 else None)
        for k in ("residual_out", "norm", "pre_out", "post_out", "comb_out"):
            o[k].zero_()
        grid.zero_()
        scales.zero_()
        h = to_host(run_gpu(dm, g=g, out=o, cfg=cfg))
        rep = compare(dm, h)
        assert rep.get("grid_mismatch", 0) == 0 and rep.get("codes_mismatch", 0) == 0


def test_empty_input_launches_nothing():
    d = make_case(0, 5120, 5006)
    out = B.alloc_outputs(0, 5120, 0, "cuda")
    run_gpu(d, out=out)
    assert B.mhc_last_launch_count() == 0


# ------------------------------------------------------- standalone kernels --
def test_standalone_quantiser_crafted_groups():
    import oracle as O
    x, picked = I.crafted_quant_tensor(1024, 5120, seed=1002)
    xd = x.cuda()
    codes = torch.empty((1024, 5120), dtype=torch.uint8, device="cuda")
    scales = torch.empty((1024, 160), dtype=torch.uint8, device="cuda")
    B.mhc_quant_ue8m0(xd, codes, scales)
    c_ref, s_ref = O.quant_ue8m0(x)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(scales.cpu().numpy(), s_ref)


def test_standalone_quantiser_every_bf16_value():
    # every finite bf16 bit pattern, in groups whose amax sets every exponent
    import oracle as O
    bits = np.arange(0, 0x10000, dtype=np.uint32)
    bits = bits[((bits & 0x7F80) != 0x7F80)].astype(np.uint16)
    n = (len(bits) + 31) // 32 * 32
    bits = np.concatenate([bits, np.zeros(n - len(bits), np.uint16)]).reshape(-1, 32)
    x = I.from_bf16_bits(bits)
    xd = x.cuda()
    rows, H = x.shape
    codes = torch.empty((rows, H), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, H // 32), dtype=torch.uint8, device="cuda")
    B.mhc_quant_ue8m0(xd, codes, scales)
    c_ref, s_ref = O.quant_ue8m0(x)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(scales.cpu().numpy(), s_ref)


def test_pack_fn_hi_lo():
    d = make_case(1, 256, 6000)
    fn = d["fn"].cuda()
    pk = torch.empty(B.mhc_packed_fn_bytes(256) // 2, dtype=torch.bfloat16, device="cuda")
    B.mhc_pack_fn(fn, pk)
    p = pk.view(48, 1024).cpu().to(torch.float64)
    f = d["fn"].to(torch.float64).t()
    hi, lo = p[:24], p[24:]
    assert torch.equal(hi, f.to(torch.bfloat16).to(torch.float64))
    assert torch.max(torch.abs(hi + lo - f) / torch.abs(f).clamp_min(1e-30)).item() < 2.0 ** -15


def test_copy_kernel():
    src = torch.randint(0, 255, (1 << 24,), dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    B.mhc_copy(src, dst)
    assert torch.equal(src, dst)


# ------------------------------------------------- streaming path (path 2) --
STREAM = dict(path=2)


@pytest.mark.parametrize("T", [1184, 1380, 1600])
def test_stream_partial_last_round(T):
    # 37, 44 and 50 blocks over the 36 clusters of 4 a GB300 holds: a last
    # round that only some clusters take
    d = make_case(T, 5120, 7050 + T, unique_tokens=512)
    h = to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM)))
    compare_all_tokens(d, h, 512)


@pytest.mark.parametrize("T", [1, 31, 32, 33, 257, 1000])
def test_stream_ragged_tokens(T):
    d = make_case(T, 5120, 7000 + T)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM))))


@pytest.mark.parametrize("H", [512, 576, 1024, 4096, 7168])
@pytest.mark.parametrize("mx", [False, True])
def test_stream_widths(H, mx):
    d = make_case(70, H, 7100 + H, mxfp8=mx)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM))))


def test_stream_no_post_and_in_place():
    d = make_case(300, 5120, 7200, post=False)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM), inplace=True)))


def test_stream_mxfp8_crafted():
    d = make_case(256, 5120, 7300, mxfp8=True, craft=True)
    h = to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM)))
    compare(d, h)
    g = I.bf16_bits(d["gamma"])
    for t in d["crafted_rows"]:
        for grp in d["crafted_groups"]:
            sl = slice(32 * grp, 32 * grp + 32)
            assert np.array_equal(h["norm"][t, sl], g[sl]), (t, grp)


def test_stream_matches_split_path_closely():
    d = make_case(200, 5120, 7400)
    a = to_host(run_gpu(d, cfg=B.MhcConfig(path=1)))
    b = to_host(run_gpu(d, cfg=B.MhcConfig(path=2)))
    from seam_case import ulp_diff
    assert np.mean(ulp_diff(a["residual_out"], b["residual_out"]) <= 1) >= 0.9999
    assert np.max(np.abs(a["comb_out"] - b["comb_out"])) < 1e-3


def test_stream_repeat_deterministic_and_graph():
    d = make_case(1024, 5120, 7500, mxfp8=True)
    g = to_dev(d)
    out = B.alloc_outputs(1024, 5120, d["out_mode"], "cuda")
    a = to_host(run_gpu(d, g=g, out=out))
    assert B.mhc_last_launch_count() == 1
    b = to_host(run_gpu(d, g=g, out=out))
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    out["norm"].zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run_gpu(d, g=g, out=out, stream=s)
    graph.replay()
    c = to_host(out)
    assert np.array_equal(a["norm"], c["norm"])
    compare(d, c)
    B.mhc_check_status(out["workspace"])


def test_stream_requires_packed_fn_and_supported_width():
    d = make_case(40, 5120, 7600)
    with pytest.raises(B.MhcError) as e:
        run_gpu(d, cfg=B.MhcConfig(**STREAM), packed=False)
    assert e.value.code == -1
    d = make_case(40, 520, 7601)
    with pytest.raises(B.MhcError) as e:
        run_gpu(d, cfg=B.MhcConfig(**STREAM))
    assert e.value.code == -2


# ------------------------------------- streaming path, clusters of 16 (path 3) --
STREAM16 = dict(path=3)


@pytest.mark.parametrize("T", [1, 31, 32, 33, 257, 1000, 1100])
def test_stream16_ragged_tokens(T):
    d = make_case(T, 5120, 7800 + T)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM16))))


@pytest.mark.parametrize("H", [512, 576, 1024, 4096, 7168, 8192])
@pytest.mark.parametrize("mx", [False, True])
def test_stream16_widths(H, mx):
    # H = 512 and 576 leave CTAs of the cluster without a chunk
    d = make_case(45, H, 7900 + H, mxfp8=mx)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM16))))


def test_stream16_no_post_in_place_and_crafted():
    d = make_case(100, 5120, 8000, post=False)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM16), inplace=True)))
    d = make_case(128, 5120, 8001, mxfp8=True, craft=True)
    h = to_host(run_gpu(d, cfg=B.MhcConfig(**STREAM16)))
    compare(d, h)
    g = I.bf16_bits(d["gamma"])
    for t in d["crafted_rows"]:
        for grp in d["crafted_groups"]:
            sl = slice(32 * grp, 32 * grp + 32)
            assert np.array_equal(h["norm"][t, sl], g[sl]), (t, grp)


def test_stream16_refuses_warp_mma():
    d = make_case(8, 5120, 8002)
    with pytest.raises(B.MhcError) as e:
        run_gpu(d, cfg=B.MhcConfig(path=3, projection=1))
    assert e.value.code == -10


@pytest.mark.parametrize("T,post", [(4, True), (64, True), (64, False)])
def test_split_path_on_the_decode_configs(T, post):
    d = make_case(T, 5120, 8100 + T, post=post)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(path=1))))


@pytest.mark.parametrize("proj", [1, 2])
@pytest.mark.parametrize("T,H,mx,post", [(300, 5120, False, True), (97, 4096, True, True), (64, 7168, False, False)])
def test_stream_projection_variants(proj, T, H, mx, post):
    # 1 = warp-level tensor-core MMA in the compute warps, 2 = tcgen05 MMA into tensor memory
    d = make_case(T, H, 7700 + T + proj, mxfp8=mx, post=post)
    cfg = B.MhcConfig(path=2, projection=proj)
    if proj == 2 and H > 5120:  # x and the tcgen05 accumulator do not both fit in tensor memory
        with pytest.raises(B.MhcError) as e:
            run_gpu(d, cfg=cfg)
        assert e.value.code == -10
        return
    compare(d, to_host(run_gpu(d, cfg=cfg)))


# ------------------------------------------------------ chained seams (f3) --
@pytest.mark.parametrize("T,path,post,first", [(64, 3, True, False), (1100, 2, True, False), (40, 1, True, False),
                                               (300, 2, False, False), (64, 3, True, True), (1100, 2, True, True),
                                               (40, 1, True, True)])
def test_three_seams_chained(T, path, post, first):
    """Three seams in a row, each fed the previous seam's residual and gates
    (a fresh sub-layer output Y per seam).  The oracle chain runs on its own
    outputs and the GPU chain on its own; they must agree at every seam (the
    bar is 1 ulp on >= 99.9% of the bf16 elements: a 1-ulp difference in one
    seam's residual is an input difference to the next).  With ``first`` the
    chain opens with the identity (first-block) seam: no Y, no post, no comb,
    the residual passes through unwritten."""
    H = 5120
    d = make_case(T, H, 8200 + T, post=post)
    g = to_dev(d)
    cfg = B.MhcConfig(path=path)
    o_state = {"R": d["R"], "pre_prev": d["pre_prev"], "post_prev": d["post_prev"], "comb_prev": d["comb_prev"]}
    g_state = {"R": g["R"], "pre_prev": g["pre_prev"], "post_prev": g["post_prev"], "comb_prev": g["comb_prev"]}
    if first:
        o_state.update(post_prev=None, comb_prev=None)
        g_state.update(post_prev=None, comb_prev=None)
    for step in range(3):
        ident = first and step == 0
        Y = I.seam_draws(T, H, 8300 + 10 * T + step, post=post)["Y"] if post and not ident else None
        o = O.seam(o_state["R"], Y, o_state["post_prev"], o_state["comb_prev"], o_state["pre_prev"], d["fn"],
                   d["bias"], d["alpha"], d["gamma"], d["eps"])
        out = B.alloc_outputs(T, H, B.MHC_OUT_BF16, "cuda", cfg)
        if ident:  # a sentinel residual_out: the identity form must leave it alone
            out["residual_out"].fill_(7.0)
        B.mhc_seam(g_state["R"], None if Y is None else Y.to("cuda"), g_state["post_prev"], g_state["comb_prev"],
                   g_state["pre_prev"], g["fn"], g["fn_packed"], g["bias"], g["alpha"], g["gamma"], d["eps"],
                   B.MHC_OUT_BF16, out["residual_out"], out["norm"], None, None, out["pre_out"], out["post_out"],
                   out["comb_out"], out["workspace"], cfg=cfg)
        h = to_host(out)
        if ident:
            assert bool((out["residual_out"] == 7.0).all())
            h.pop("residual_out")
            assert np.array_equal(o["residual_out"], I.bf16_bits(d["R"]))
        for k in ("residual_out", "norm"):
            if k not in h:
                continue
            # from the second seam on the inputs differ by the earlier seams'
            # roundings (and the difference grows along the chain), so a
            # near-cancelling sum may land on either side of zero: an element
            # passes within 2 ulp or within 1e-4 absolute
            u = ulp_diff(h[k], o[k])
            ad = np.abs(I.from_bf16_bits(h[k]).float().numpy() - I.from_bf16_bits(o[k]).float().numpy())
            ok = (u <= 2) | (ad <= 1e-4)
            assert np.mean(ok) >= 0.999 and ad.max() <= 0.05, (step, k, float(np.mean(ok)), float(ad.max()))
            if step == 0:
                assert np.mean(u <= 1) >= 0.9999, (k, float(np.mean(u <= 1)))
        for gk, ok in (("pre_out", "pre"), ("post_out", "post"), ("comb_out", "comb")):
            assert np.abs(h[gk].astype(np.float64) - o[ok].reshape(h[gk].shape)).max() <= GATE_TOL, (step, ok)
        # the next seam's inputs: each chain feeds itself (after the identity
        # seam the residual is its input, unchanged)
        o_state = {"R": o["residual_out"], "pre_prev": o["pre"].astype(np.float32),
                   "post_prev": o["post"].astype(np.float32) if post else None,
                   "comb_prev": o["comb"].astype(np.float32)}
        g_state = {"R": g_state["R"] if ident else out["residual_out"], "pre_prev": out["pre_out"],
                   "post_prev": out["post_out"] if post else None, "comb_prev": out["comb_out"]}


# ------------------------------------------------------ fp8_grid out (f1) --
@pytest.mark.parametrize("T,path,craft", [(1024, 2, True), (300, 2, False), (64, 3, True), (5, 3, False)])
def test_fp8_grid(T, path, craft):
    d = make_case(T, 5120, 8400 + T, grid=True, craft=craft)
    h = to_host(run_gpu(d, cfg=B.MhcConfig(path=path)))
    rep = compare(d, h)
    assert rep["grid_mismatch"] == 0
    if craft:  # crafted gamma groups: the grid of a 448 * 2^k group is the group itself
        g = I.bf16_bits(d["gamma"])
        for t in d["crafted_rows"]:
            for grp in d["crafted_groups"]:
                sl = slice(32 * grp, 32 * grp + 32)
                assert np.array_equal(h["norm"][t, sl], g[sl]), (t, grp)


@pytest.mark.parametrize("H", [512, 4096, 7168])
def test_fp8_grid_widths(H):
    d = make_case(40, H, 8500 + H, grid=True)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(path=2))))


def test_fp8_grid_no_post_and_split_path_refused():
    d = make_case(70, 5120, 8600, grid=True, post=False)
    compare(d, to_host(run_gpu(d, cfg=B.MhcConfig(path=2))))
    with pytest.raises(B.MhcError) as e:
        run_gpu(d, cfg=B.MhcConfig(path=1))
    assert e.value.code == -10


# ------------------------------------------- identity (first-block) form (f3) --
@pytest.mark.parametrize("T,H,path,mode", [(64, 5120, 3, B.MHC_OUT_BF16), (5, 5120, 3, B.MHC_OUT_FP8_GRID),
                                           (1100, 5120, 2, B.MHC_OUT_MXFP8), (300, 5120, 2, B.MHC_OUT_FP8_GRID),
                                           (2050, 5120, 2, B.MHC_OUT_BF16), (97, 7168, 2, B.MHC_OUT_BF16),
                                           (40, 5120, 1, B.MHC_OUT_BF16), (33, 160, 1, B.MHC_OUT_MXFP8)])
def test_identity_form(T, H, path, mode):
    d = make_case(T, H, 8600 + T + H, ident=True, mxfp8=mode == B.MHC_OUT_MXFP8, grid=mode == B.MHC_OUT_FP8_GRID)
    cfg = B.MhcConfig(path=path)
    out = B.alloc_outputs(T, H, d["out_mode"], "cuda", cfg)
    out["residual_out"].fill_(-3.0)  # must stay untouched
    sentinel = out["residual_out"]
    out["residual_out"] = None
    h = to_host(run_gpu(d, cfg=cfg, out=out))
    assert bool((sentinel == -3.0).all())
    compare(d, h)


@pytest.mark.parametrize("mode", [B.MHC_OUT_BF16, B.MHC_OUT_MXFP8])
def test_identity_form_warp_mma_projection(mode):
    # with the tcgen05 projection the identity form's MMAs read R from the
    # input stage (its own shared-memory layout); with the warp-level
    # projection the compute warps still copy R into the output stage: both
    # layouts at the same width
    T, H = 300, 5120
    d = make_case(T, H, 8650, ident=True, mxfp8=mode == B.MHC_OUT_MXFP8)
    for proj in (1, 2):
        cfg = B.MhcConfig(path=2, projection=proj)
        out = B.alloc_outputs(T, H, d["out_mode"], "cuda", cfg)
        out["residual_out"] = None
        compare(d, to_host(run_gpu(d, cfg=cfg, out=out)))


def test_identity_form_matches_identity_comb_and_rejects_y():
    # away from signed zeros (none in these draws) the identity form equals the
    # no_post seam with comb = I on the same inputs
    T, H = 300, 5120
    d = make_case(T, H, 8700, ident=True)
    g = to_dev(d)
    a = to_host(run_gpu(d, cfg=B.MhcConfig(path=2), g=g))
    eye = torch.eye(4, dtype=torch.float32).expand(T, 4, 4).contiguous()
    d2 = dict(d, comb_prev=eye)
    g2 = dict(g, comb_prev=eye.cuda())
    b = to_host(run_gpu(d2, cfg=B.MhcConfig(path=2), g=g2))
    assert np.array_equal(b["residual_out"], I.bf16_bits(d["R"]))
    assert np.array_equal(a["norm"], b["norm"])
    for k in ("pre_out", "post_out", "comb_out"):
        assert np.array_equal(a[k], b[k]), k
    out = B.alloc_outputs(T, H, B.MHC_OUT_BF16, "cuda")
    Y = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    post = torch.ones(T, 4, device="cuda")
    with pytest.raises(RuntimeError, match="identity form"):
        B.mhc_seam(g["R"], Y, post, None, g["pre_prev"], g["fn"], g["fn_packed"], g["bias"], g["alpha"],
                   g["gamma"], d["eps"], B.MHC_OUT_BF16, out["residual_out"], out["norm"], None, None,
                   out["pre_out"], out["post_out"], out["comb_out"], out["workspace"])


# ------------------------------------------------------ unshifted ordering (f4) --
def _run_unshifted(d, cfg=None):
    T, H = d["T"], d["H"]
    g = to_dev(d)
    out = B.alloc_outputs(T, H, B.MHC_OUT_BF16, "cuda", cfg, unshifted=True)
    if d["comb_prev"] is None:
        out["residual_out"] = None
    B.mhc_seam_unshifted(g["R"], g["Y"], g["post_prev"], g["comb_prev"], g["fn"], g["fn_packed"], g["bias"],
                         g["alpha"], d["eps"], out["residual_out"], out["norm"], out["pre_out"], out["post_out"],
                         out["comb_out"], out["workspace"], cfg=cfg)
    h = to_host(out)
    h["launches"] = B.mhc_last_launch_count()
    return h


def check_unshifted_x(xg: np.ndarray, pre_g: np.ndarray, o: dict, rp_g: np.ndarray | None = None) -> None:
    """The unshifted x against the oracle.  x = sum_i pre[i] R'[i] takes the
    FRESH pre, which the kernel computes in fp32 (within the 1e-3 gate bar,
    in practice about 1e-6) and the oracle in double, and the kernel's R' may
    differ from the oracle's by the 1 ulp the residual bar allows; where the
    four terms nearly cancel, those differences are many ulps of x.  So every
    element must be within 1 ulp of the oracle or within the difference the
    inputs explain, sum_i |dpre_i| |R'_i| + sum_i |pre_i| |dR'_i| + 2^-20
    sum_i |pre_i R'_i| (fp32 accumulation) + 1 ulp; and 99.9 % of them within
    1 ulp.  rp_g: the kernel's R' bits (None where R' = R on both sides)."""
    u = ulp_diff(xg, o["x"])
    rp = I.from_bf16_bits(o["residual_out"]).double().numpy()             # [n, 4, H]
    dpre = np.abs(pre_g.astype(np.float64) - o["pre"])                      # [n, 4]
    bound = (np.einsum("ni,nih->nh", dpre, np.abs(rp)) +
             2.0 ** -20 * np.einsum("ni,nih->nh", np.abs(o["pre"]), np.abs(rp)))
    if rp_g is not None:
        drp = np.abs(I.from_bf16_bits(rp_g).double().numpy() - rp)
        bound += np.einsum("ni,nih->nh", np.abs(o["pre"]), drp)
    xo = I.from_bf16_bits(o["x"]).double().numpy()
    ulp_o = np.maximum(np.abs(xo), 2.0 ** -126) * 2.0 ** -7
    ad = np.abs(I.from_bf16_bits(xg).double().numpy() - xo)
    ok = (u <= 1) | (ad <= bound + ulp_o)
    assert ok.all(), ("x", int((~ok).sum()), float(ad[~ok].max()))
    assert np.mean(u <= 1) >= 0.999, ("x", float(np.mean(u <= 1)))


@pytest.mark.parametrize("T,H,post,ident,path", [
    (4, 5120, True, False, 0), (64, 5120, False, False, 0), (300, 5120, True, False, 1), (1100, 5120, True, False, 0),
    (1100, 5120, True, False, 1), (33, 160, True, False, 0), (40, 5120, False, True, 0), (40, 5120, False, True, 1),
    (2050, 4096, True, False, 2), (17, 7168, True, False, 0), (1500, 7168, False, False, 2), (300, 5120, True, True, 3),
    (97, 1024, True, False, 3)])
def test_unshifted(T, H, post, ident, path):
    d = make_case(T, H, 8800 + T + H, post=post, ident=ident)
    h = _run_unshifted(d, cfg=B.MhcConfig(path=path))
    take = lambda x: x  # noqa: E731  (every token)
    o = O.seam_unshifted(d["R"], d["Y"], d["post_prev"], d["comb_prev"], d["fn"], d["bias"], d["alpha"], d["eps"])
    if not ident:
        u = ulp_diff(take(h["residual_out"]), o["residual_out"])
        assert np.mean(u <= 1) >= 0.9999, ("residual_out", float(np.mean(u <= 1)), int(u.max()))
    check_unshifted_x(take(h["norm"]), take(h["pre_out"]), o, None if ident else take(h["residual_out"]))
    for gk, ok in (("pre_out", "pre"), ("post_out", "post"), ("comb_out", "comb")):
        err = np.abs(take(h[gk]).astype(np.float64) - o[ok].reshape(take(h[gk]).shape))
        assert err.max() <= GATE_TOL, (ok, float(err.max()))


def test_unshifted_paths_agree_and_launch_counts():
    d = make_case(300, 5120, 8900)
    o = O.seam_unshifted(d["R"], d["Y"], d["post_prev"], d["comb_prev"], d["fn"], d["bias"], d["alpha"], d["eps"])
    a = _run_unshifted(d, cfg=B.MhcConfig(block_m=8, cols_per_cta=128))   # split path, another tiling
    b = _run_unshifted(d, cfg=B.MhcConfig(path=2))                        # streaming: two launches
    c = _run_unshifted(d, cfg=B.MhcConfig(path=3))
    assert a["launches"] >= 1 and b["launches"] == 2 and c["launches"] == 2
    for h in (a, b, c):
        check_unshifted_x(h["norm"], h["pre_out"], o, h["residual_out"])
        assert np.mean(ulp_diff(h["residual_out"], o["residual_out"]) <= 1) >= 0.9999
    big = B.MhcConfig(block_m=32, cols_per_cta=640)   # the split path's R' tile does not fit
    with pytest.raises(RuntimeError, match="shared memory"):
        _run_unshifted(d, cfg=big)


# ------------------------------------------------ robustness of the new forms --
@pytest.mark.parametrize("path", [1, 2])
def test_unshifted_in_place_and_empty(path):
    d = make_case(300, 5120, 9300 + path)
    o = O.seam_unshifted(d["R"], d["Y"], d["post_prev"], d["comb_prev"], d["fn"], d["bias"], d["alpha"], d["eps"])
    g = to_dev(d)
    cfg = B.MhcConfig(path=path)
    out = B.alloc_outputs(300, 5120, B.MHC_OUT_BF16, "cuda", cfg, unshifted=True)
    # residual_out == R: R' overwrites R in place, and the second pass reads it back
    B.mhc_seam_unshifted(g["R"], g["Y"], g["post_prev"], g["comb_prev"], g["fn"], g["fn_packed"], g["bias"],
                         g["alpha"], d["eps"], g["R"], out["norm"], out["pre_out"], out["post_out"], out["comb_out"],
                         out["workspace"], cfg=cfg)
    torch.cuda.synchronize()
    rp = I.bf16_bits(g["R"].cpu())
    assert np.mean(ulp_diff(rp, o["residual_out"]) <= 1) >= 0.9999
    h = to_host(out)
    check_unshifted_x(h["norm"], h["pre_out"], o, rp)
    # T = 0: nothing launched
    B.mhc_seam_unshifted(g["R"], g["Y"], g["post_prev"], g["comb_prev"], g["fn"], g["fn_packed"], g["bias"],
                         g["alpha"], d["eps"], out["residual_out"], out["norm"], out["pre_out"], out["post_out"],
                         out["comb_out"], out["workspace"], cfg=cfg, T=0)
    assert B.mhc_last_launch_count() == 0


def test_unshifted_graph_capture_matches_eager():
    d = make_case(1100, 5120, 9310)
    g = to_dev(d)
    cfg = B.MhcConfig(path=2)
    out = B.alloc_outputs(1100, 5120, B.MHC_OUT_BF16, "cuda", cfg, unshifted=True)

    def call(s=None):
        B.mhc_seam_unshifted(g["R"], g["Y"], g["post_prev"], g["comb_prev"], g["fn"], g["fn_packed"], g["bias"],
                             g["alpha"], d["eps"], out["residual_out"], out["norm"], out["pre_out"], out["post_out"],
                             out["comb_out"], out["workspace"], cfg=cfg, stream=s)

    call()
    eager = to_host(out)
    for k in ("residual_out", "norm", "pre_out", "post_out", "comb_out"):
        out[k].zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            call(s)                     # both launches captured
    for _ in range(3):
        graph.replay()
    rep = to_host(out)
    for k in ("residual_out", "norm", "pre_out", "post_out", "comb_out"):
        assert np.array_equal(rep[k], eager[k]), k


def test_fp8_grid_graph_replay_is_deterministic():
    d = make_case(1024, 5120, 9320, grid=True)
    g = to_dev(d)
    out = run_gpu(d, g=g, cfg=B.MhcConfig(path=2))
    eager = to_host(out)
    out["fp8_codes"].zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run_gpu(d, g=g, out=out, cfg=B.MhcConfig(path=2), stream=s)
    for _ in range(2):
        graph.replay()
    rep = to_host(out)
    assert np.array_equal(rep["fp8_codes"], eager["fp8_codes"]) and np.array_equal(rep["norm"], eager["norm"])


# ------------------------------------------- the NEXT rows at the full size --
def test_full_size_fp8_grid_and_identity():
    # T = 16384, in the launch configuration the benchmark times: every token
    # against the oracle, the whole grid against the oracle's grid of the
    # kernel's own norm
    d = make_case(16384, 5120, 1004, grid=True, unique_tokens=2048)
    h = to_host(run_gpu(d))
    rep = compare_all_tokens(d, h, 2048)
    assert rep["grid_mismatch"] == 0
    d = make_case(16384, 5120, 1004, ident=True, unique_tokens=2048)
    h = to_host(run_gpu(d))
    rep = compare_all_tokens(d, h, 2048)
    assert rep["norm_elements"] == 16384 * 5120


def test_full_size_unshifted():
    # every token: the oracle on the 2048 distinct tokens, each GPU row against
    # the oracle row of its token class (checked in slices of one class period)
    U = 2048
    d = make_case(16384, 5120, 1004, unique_tokens=U)
    h = _run_unshifted(d)
    assert h["launches"] == 2
    t = torch.arange(U)
    o = O.seam_unshifted(d["R"][t], d["Y"][t], d["post_prev"][t], d["comb_prev"][t], d["fn"], d["bias"],
                         d["alpha"], d["eps"])
    for t0 in range(0, 16384, 256):
        sl = slice(t0, t0 + 256)
        cls = np.arange(t0, t0 + 256) % U
        oc = {k: o[k][cls] for k in ("residual_out", "x", "pre")}
        assert np.mean(ulp_diff(h["residual_out"][sl], oc["residual_out"]) <= 1) >= 0.9999
        check_unshifted_x(h["norm"][sl], h["pre_out"][sl], oc, h["residual_out"][sl])
    for gk, ok in (("pre_out", "pre"), ("post_out", "post"), ("comb_out", "comb")):
        ref = o[ok][np.arange(16384) % U].reshape(h[gk].shape)
        assert np.abs(h[gk].astype(np.float64) - ref).max() <= GATE_TOL


# -------------------------------------- split partial round (the wave edge) --
# A GB300 holds 36 clusters of 4 (9 of 16) of the streaming kernel at once, so
# token blocks beyond a whole number of rounds leave a partial last round; its
# blocks may be cut into column parts whose sums meet in the workspace (on
# request: the default policy does not split at H = 5120).
@pytest.mark.parametrize("T,k", [(1184, 0), (1184, 2), (1184, 7), (1184, 20), (1600, 4), (2336, 3), (4160, 3),
                                 (4161, 3), (4161, 2)])
def test_wave_split_partial_round(T, k):
    d = make_case(T, 5120, 9800 + T + k, unique_tokens=512)
    g = to_dev(d)
    h = to_host(run_gpu(d, g=g, cfg=B.MhcConfig(path=2, wave_split=k)))
    parts = B.mhc_last_wave_parts()
    assert parts == (k if k else 1), parts
    compare_all_tokens(d, h, 512)
    # the same call without the split: R' does not depend on it (bit for bit),
    # the gates and norm agree within the parity bar
    n = to_host(run_gpu(d, g=g, cfg=B.MhcConfig(path=2, wave_split=1)))
    assert B.mhc_last_wave_parts() == 1
    assert np.array_equal(h["residual_out"], n["residual_out"])
    assert np.mean(ulp_diff(h["norm"], n["norm"]) <= 1) >= 0.9999
    for gk in ("pre_out", "post_out", "comb_out"):
        assert np.abs(h[gk] - n[gk]).max() <= GATE_TOL, gk


@pytest.mark.parametrize("form", ["no_post", "identity", "mxfp8", "fp8_grid", "in_place"])
def test_wave_split_forms_and_outputs(form):
    T = 1184
    d = make_case(T, 5120, 9900, post=form != "no_post", ident=form == "identity", mxfp8=form == "mxfp8",
                  grid=form == "fp8_grid", craft=form == "mxfp8", unique_tokens=512)
    cfg = B.MhcConfig(path=2, wave_split=5)
    out = None
    if form == "identity":
        out = B.alloc_outputs(T, 5120, d["out_mode"], "cuda", cfg)
        out["residual_out"] = None
    h = to_host(run_gpu(d, cfg=cfg, out=out, inplace=form == "in_place"))
    assert B.mhc_last_wave_parts() == 5
    rep = compare_all_tokens(d, h, 512)
    assert rep.get("codes_mismatch", 0) == 0 and rep.get("grid_mismatch", 0) == 0


@pytest.mark.parametrize("T,k", [(300, 0), (352, 5), (352, 2), (1000, 2)])
def test_wave_split_clusters_of_16(T, k):
    # 7 to 10 clusters of 16 fit (by variant): T = 352 (11 blocks) and
    # T = 1000 (32 blocks) leave a partial last round, cut into at most k parts
    # (fewer where two parts per cluster would not cover them); the policy's
    # own choice (k = 0, no split) is checked for parity only
    d = make_case(T, 5120, 9950 + T + k, unique_tokens=256)
    h = to_host(run_gpu(d, cfg=B.MhcConfig(path=3, wave_split=k)))
    parts = B.mhc_last_wave_parts()
    if k:
        assert 2 <= parts <= k, parts
    compare_all_tokens(d, h, 256)


def test_wave_split_warp_mma_projection_and_unshifted():
    # H = 7168 runs the warp-level projection (x alone fills tensor memory)
    d = make_case(1184, 7168, 9970, unique_tokens=256)
    h = to_host(run_gpu(d, cfg=B.MhcConfig(path=2, wave_split=4)))
    assert B.mhc_last_wave_parts() == 4
    compare_all_tokens(d, h, 256)
    # the unshifted ordering's first launch takes the split too
    d = make_case(1184, 5120, 9971)
    hu = _run_unshifted(d, cfg=B.MhcConfig(path=2, wave_split=6))
    o = O.seam_unshifted(d["R"], d["Y"], d["post_prev"], d["comb_prev"], d["fn"], d["bias"], d["alpha"], d["eps"])
    assert np.mean(ulp_diff(hu["residual_out"], o["residual_out"]) <= 1) >= 0.9999
    check_unshifted_x(hu["norm"], hu["pre_out"], o, hu["residual_out"])
    for gk, ok in (("pre_out", "pre"), ("post_out", "post"), ("comb_out", "comb")):
        assert np.abs(hu[gk].astype(np.float64) - o[ok].reshape(hu[gk].shape)).max() <= GATE_TOL


def test_wave_split_repeat_graph_and_report():
    # the split's workspace counters reset themselves: repeated calls and graph
    # replays give the same bits; a forced report on a split call is flagged and
    # the next call is clean
    T = 2336
    d = make_case(T, 5120, 9980, unique_tokens=512)
    g = to_dev(d)
    cfg = B.MhcConfig(path=2, wave_split=10)
    out = B.alloc_outputs(T, 5120, d["out_mode"], "cuda", cfg)
    a = to_host(run_gpu(d, g=g, out=out, cfg=cfg))
    assert B.mhc_last_wave_parts() == 10
    b = to_host(run_gpu(d, g=g, out=out, cfg=cfg))
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    for k in ("norm", "pre_out", "comb_out"):
        out[k].zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run_gpu(d, g=g, out=out, cfg=cfg, stream=s)
    for _ in range(3):
        graph.replay()
    c = to_host(out)
    for k in a:
        assert np.array_equal(a[k], c[k]), k
    B.mhc_check_status(out["workspace"])
    compare_all_tokens(d, c, 512)
    run_gpu(d, g=g, out=out, cfg=B.MhcConfig(path=2, wave_split=10, spin_limit=1))
    with pytest.raises(B.MhcError) as e:
        B.mhc_check_status(out["workspace"])
    assert e.value.code == -7
    compare_all_tokens(d, to_host(out), 512)
    run_gpu(d, g=g, out=out, cfg=cfg)
    B.mhc_check_status(out["workspace"])
    assert np.array_equal(to_host(out)["norm"], a["norm"])
