"""Pins of the seam oracle against facts fixed outside it (CPU only).

Each test checks one function of the oracle against something the oracle did
not compute: closed forms, invariants, an independent exact-arithmetic brute
force, exhaustive sweeps against the format definitions, or a library routine
of a different implementation.  A plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a wrong rounding rule)
fails at least one of them.
"""
import math
import os
import struct
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

from mhc_residual_seam_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers --
def bf16_rne_exact(v: Fraction) -> int:
    """bf16 bits of an exact rational, rounded to nearest even (test-side,
    integer arithmetic; independent of the oracle's double-based rounding)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    elif Fraction(2) ** (E + 1) <= a:
        E += 1
    E = max(E, -126)
    spacing = Fraction(2) ** (E - 7)
    r = round(a / spacing) * spacing          # Fraction round(): half to even
    if r >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = struct.unpack("<I", struct.pack("<f", float(r)))[0]
    return sign | (bits >> 16)


def bf16_val(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def e4m3_table():
    """Values of the 254 finite e4m3fn codes from the format definition."""
    vals = {}
    for code in range(256):
        s, ex, m = code >> 7, (code >> 3) & 0xF, code & 7
        if ex == 15 and m == 7:
            continue  # NaN
        mag = m * 2.0 ** -9 if ex == 0 else (1 + m / 8.0) * 2.0 ** (ex - 7)
        vals[code] = -mag if s else mag
    return vals


def e4m3_by_table(v: float) -> int:
    """Nearest e4m3fn code by search over the table, ties to the even code,
    finite overflow saturates to +-448 (independent of the oracle)."""
    table = e4m3_table()
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a >= 448.0:
        return sign | 0x7E
    best = None
    for code in range(0x7F):
        mag = table[code]
        d = abs(mag - a)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return sign | best[1]


def seam_inputs(T, H, seed, post=True, oracle=None):
    d = I.seam_draws(T, H, seed, post=post)
    pre, post_g, comb = oracle.carried_gates(d["pre_logits"], d["post_logits"], d["comb_logits"])
    d["pre_prev"], d["post_prev"], d["comb_prev"] = pre, (post_g if post else None), comb
    return d


def run(oracle, d, **kw):
    return oracle.seam(d["R"], d["Y"], d["post_prev"], d["comb_prev"], d["pre_prev"], d["fn"],
                       d["bias"], d["alpha"], d["gamma"], d["eps"], **kw)


# ------------------------------------------------------------------- bf16 ---
def test_bf16_rne_matches_torch_cast_on_float32_inputs(oracle):
    # float32 inputs make torch's cast a single rounding; include exact ties,
    # subnormals, the overflow edge and random patterns.
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits[:2000] = (bits[:2000] & 0xFFFF0000) | 0x8000          # exact ties
    bits[2000:3000] = bits[2000:3000] & 0x807FFFFF            # subnormals
    bits[3000:3100] = 0x7F7F0000 | (bits[3000:3100] & 0xFFFF)  # near the top
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rne_matches_exact_rational_rounding(oracle):
    rng = np.random.default_rng(8)
    for _ in range(3000):
        num = int(rng.integers(-2**40, 2**40))
        den = int(rng.integers(1, 2**20))
        sc = int(rng.integers(-140, 120))
        v = Fraction(num, den) * Fraction(2) ** sc
        dv = float(v)
        if Fraction(dv) != v:
            continue  # only doubles are oracle inputs
        assert oracle.bf16_rne(dv) == bf16_rne_exact(v), v


# ------------------------------------------------------------------- e4m3 ---
def test_e4m3_golden_codes_from_ocp_spec(oracle):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e4m3fn_ocp.txt")) if l.strip() and not l.startswith("#")]
    for v, code in rows:
        assert oracle.e4m3(float(v)) == int(code, 16), (v, code)


def test_e4m3_exhaustive_over_significands_and_exponents(oracle):
    # Every 8-significant-bit magnitude (what a bf16 times a power of two can
    # be) at every exponent from total underflow to saturation, both signs.
    vals = [0.0, -0.0]
    for sig in range(128, 256):
        for E in range(-22, 12):
            v = sig * 2.0 ** (E - 7)
            vals += [v, -v]
    for v in vals:
        assert oracle.e4m3(v) == e4m3_by_table(v), v


# ------------------------------------------------------------------ ue8m0 ---
def test_ue8m0_exponent_exhaustive_over_bf16_amax(oracle):
    # All 32640 non-negative finite bf16 values: e must be the smallest
    # integer with amax <= 448 * 2^e (exact rationals), after the 1e-10 floor,
    # clamped to [-127, 127].
    floor = 1e-10
    for b in range(0, 0x7F80):
        a = bf16_val(b)
        aa = Fraction(max(a, floor))
        e = math.floor(math.log2(float(aa) / 448.0)) - 2
        while Fraction(448) * Fraction(2) ** e < aa:
            e += 1
        e = min(max(e, -127), 127)
        assert oracle.ue8m0_exponent(a, floor) == e, (hex(b), a)


def test_ue8m0_exponent_equals_float_ceil_log2_where_quotient_is_normal(oracle):
    for b in range(0x0080, 0x7F80, 7):
        a = bf16_val(b)
        q = a / 448.0
        if q < 2.0 ** -126 or a < 1e-10:
            continue
        assert oracle.ue8m0_exponent(a) == min(127, math.ceil(math.log2(q)))


def test_crafted_groups_448_times_power_of_two(oracle):
    for k in range(-20, 21):
        g = np.full(32, 3.0 * 2.0 ** k, np.float32)
        g[5] = 448.0 * 2.0 ** k
        g[9] = -448.0 * 2.0 ** k
        codes, scales = oracle.quant_ue8m0(I.to_bf16(g.astype(np.float64)).reshape(1, 32))
        assert scales[0, 0] == k + 127
        assert codes[0, 5] == 0x7E and codes[0, 9] == 0xFE
        assert codes[0, 0] == e4m3_by_table(3.0)  # 3 * 2^k / 2^k
        # the scale is a power of two and the codes round-trip to the inputs
        dec = np.array([e4m3_table()[c] for c in codes[0]]) * 2.0 ** (int(scales[0, 0]) - 127)
        assert np.array_equal(dec, g.astype(np.float64))


def test_crafted_groups_zero_subnormal_nearmax(oracle):
    z = I.to_bf16(np.array([0.0, -0.0] * 16))
    codes, scales = oracle.quant_ue8m0(z.reshape(1, 32))
    assert list(codes[0]) == [0x00, 0x80] * 16
    assert scales[0, 0] == -42 + 127          # amax floored at 1e-10
    sub = I.to_bf16(np.arange(1, 33) * 2.0 ** -133)
    codes, scales = oracle.quant_ue8m0(sub.reshape(1, 32))
    assert scales[0, 0] == 85 and np.all(codes == 0)
    near = np.full(32, 1.0)
    near[0] = 446.0 * 2.0 ** 3                # bf16 neighbour below 448 * 2^3
    codes, scales = oracle.quant_ue8m0(I.to_bf16(near).reshape(1, 32))
    assert scales[0, 0] == 3 + 127 and codes[0, 0] == e4m3_by_table(446.0)


def test_quant_matches_table_reimplementation_on_crafted_tensor(oracle):
    x, picked = I.crafted_quant_tensor(16, 512, seed=1002, frac=0.2)
    codes, scales = oracle.quant_ue8m0(x)
    xv = x.to(torch.float64).numpy()
    table = e4m3_table()
    vals = np.array(sorted(set(abs(v) for v in table.values())))
    for r in range(16):
        for g in range(512 // 32):
            grp = xv[r, 32 * g:32 * g + 32]
            amax = max(np.max(np.abs(grp)), 1e-10)
            e = math.ceil(math.log2(amax / 448.0))
            while 448.0 * 2.0 ** (e - 1) >= amax:
                e -= 1
            while 448.0 * 2.0 ** e < amax:
                e += 1
            e = min(max(e, -127), 127)
            assert scales[r, g] == e + 127
            for j in range(32):
                v = grp[j] * 2.0 ** -e
                a = min(abs(v), 448.0)
                i = np.searchsorted(vals, a)
                cand = [vals[max(i - 1, 0)], vals[min(i, len(vals) - 1)]]
                want = min(cand, key=lambda c: (abs(c - a), [k for k, tv in table.items() if tv == c][0] % 2))
                got = abs(table[int(codes[r, 32 * g + j])])
                assert got == want, (r, g, j, v)
                assert (codes[r, 32 * g + j] >> 7) == (1 if math.copysign(1, grp[j]) < 0 else 0)


# --------------------------------------------------------------- Sinkhorn ---
def test_sinkhorn_rank_one_logits_give_uniform(oracle):
    a = np.array([0.3, -1.0, 2.0, 0.5])
    b = np.array([1.5, 0.0, -0.7, 0.2])
    M = oracle.sinkhorn(np.exp(a[:, None] + b[None, :]), 20)
    assert np.allclose(M, 0.25, atol=1e-15, rtol=0)


def test_sinkhorn_2x2_closed_form(oracle):
    # The doubly stochastic scaling of [[a, b], [c, d]] is [[p, 1-p], [1-p, p]]
    # with p = sqrt(ad) / (sqrt(ad) + sqrt(bc)).
    rng = np.random.default_rng(3)
    for _ in range(50):
        A = np.exp(rng.uniform(-1, 1, size=(2, 2)))
        p = math.sqrt(A[0, 0] * A[1, 1]) / (math.sqrt(A[0, 0] * A[1, 1]) + math.sqrt(A[0, 1] * A[1, 0]))
        want = [[p, 1 - p], [1 - p, p]]
        # the rounds converge geometrically to the closed form
        assert np.allclose(oracle.sinkhorn(A, 20), want, atol=1e-10, rtol=0)
        assert np.allclose(oracle.sinkhorn(A, 40), want, atol=1e-14, rtol=0)


def test_sinkhorn_one_round_is_row_then_column(oracle):
    # After exactly one round the columns sum to one but the rows do not: this
    # fixes the order of the two normalisations inside a round.
    A = np.exp(np.array([[0.0, 1.0, 0.0, 0.0], [0.0, 0.0, 2.0, 0.0], [1.0, 0.0, 0.0, 0.0], [0.0, 0.5, 0.0, 3.0]]))
    M = oracle.sinkhorn(A, 1)
    assert np.allclose(M.sum(0), 1.0, atol=1e-15)
    assert not np.allclose(M.sum(1), 1.0, atol=1e-3)
    R = A / A.sum(1, keepdims=True)
    assert np.allclose(M, R / R.sum(0, keepdims=True), atol=1e-15)


# ------------------------------------------------------------------- seam ---
def test_identity_comb_zero_post_reproduces_R(oracle):
    d = seam_inputs(3, 64, 11, oracle=oracle)
    d["comb_prev"] = np.tile(np.eye(4, dtype=np.float32), (3, 1, 1))
    d["post_prev"] = np.zeros((3, 4), np.float32)
    o = run(oracle, d)
    assert np.array_equal(o["residual_out"], I.bf16_bits(d["R"]))


def test_permutation_comb_permutes_streams(oracle):
    d = seam_inputs(2, 64, 12, oracle=oracle)
    perm = [2, 0, 3, 1]
    P = np.zeros((4, 4), np.float32)
    for i, j in enumerate(perm):
        P[i, j] = 1.0
    d["comb_prev"] = np.tile(P, (2, 1, 1))
    d["post_prev"] = np.zeros((2, 4), np.float32)
    o = run(oracle, d)
    Rb = I.bf16_bits(d["R"])
    for i, j in enumerate(perm):
        assert np.array_equal(o["residual_out"][:, i], Rb[:, j])


def test_uniform_comb_gives_mean_stream(oracle):
    d = seam_inputs(2, 32, 13, oracle=oracle)
    d["comb_prev"] = np.full((2, 4, 4), 0.25, np.float32)
    d["post_prev"] = np.zeros((2, 4), np.float32)
    o = run(oracle, d)
    Rv = d["R"].to(torch.float64).numpy()
    for t in range(2):
        for h in range(32):
            m = sum(Fraction(float(Rv[t, j, h])) for j in range(4)) / 4
            for i in range(4):
                assert o["residual_out"][t, i, h] == bf16_rne_exact(m)


def test_post_term_adds_post_times_Y(oracle):
    # comb = 0: R' = post (x) Y exactly (a product of an fp32 and a bf16 value,
    # rounded once to bf16).
    d = seam_inputs(2, 32, 14, oracle=oracle)
    d["comb_prev"] = np.zeros((2, 4, 4), np.float32)
    o = run(oracle, d)
    Yv = d["Y"].to(torch.float64).numpy()
    for t in range(2):
        for i in range(4):
            for h in range(32):
                want = bf16_rne_exact(Fraction(float(d["post_prev"][t, i])) * Fraction(float(Yv[t, h])))
                assert o["residual_out"][t, i, h] == want


def test_no_post_equals_post_form_with_zero_post(oracle):
    d = seam_inputs(3, 64, 15, oracle=oracle)
    a = run(oracle, dict(d, Y=None, post_prev=None))
    b = run(oracle, dict(d, post_prev=np.zeros((3, 4), np.float32)))
    for k in ("residual_out", "norm", "pre", "post", "comb"):
        assert np.array_equal(a[k], b[k])


def test_collapse_uses_carried_pre(oracle):
    d = seam_inputs(2, 64, 16, oracle=oracle)
    d["pre_prev"] = np.full((2, 4), 0.25, np.float32)
    o = run(oracle, d, want_x=True)
    rp = np.vectorize(bf16_val)(o["residual_out"]).astype(np.float64)
    assert np.array_equal(o["x"], rp.sum(1) / 4)      # exact: sum of 4 bf16 / 4
    for i in range(4):
        e = np.zeros((2, 4), np.float32)
        e[:, i] = 1.0
        o = run(oracle, dict(d, pre_prev=e), want_x=True)
        assert np.array_equal(o["x"], rp[:, i])


@pytest.mark.parametrize("perm", [(1, 0, 2, 3), (3, 2, 1, 0), (2, 3, 0, 1), (1, 2, 3, 0)])
def test_stream_permutation_equivariance(oracle, perm):
    # Relabel the four streams: R, the rows and columns of comb, post, pre and
    # the fn row blocks all move together.  R' moves with them; the logits are
    # sums over every (stream, column) pair, so the gates are unchanged, and
    # so are x and the norm (the same terms, summed in another order: within
    # rounding, and bit-identical here).
    T, H = 3, 32
    d = seam_inputs(T, H, 44, oracle=oracle)
    d["comb_prev"] = d["comb_prev"] + np.float32(0.05) * np.arange(16, dtype=np.float32).reshape(1, 4, 4)
    p = list(perm)
    e = dict(d)
    e["R"] = d["R"][:, p, :]
    e["comb_prev"] = np.ascontiguousarray(d["comb_prev"][:, p, :][:, :, p])
    e["post_prev"] = np.ascontiguousarray(d["post_prev"][:, p])
    e["pre_prev"] = np.ascontiguousarray(d["pre_prev"][:, p])
    e["fn"] = d["fn"].reshape(4, H, 24)[p].reshape(4 * H, 24)
    a, b = run(oracle, d), run(oracle, e)
    assert np.array_equal(b["residual_out"], a["residual_out"][:, p, :])
    assert np.max(np.abs(b["pre"] - a["pre"])) < 1e-12
    assert np.max(np.abs(b["post"] - a["post"])) < 1e-12
    assert np.max(np.abs(b["comb"] - a["comb"])) < 1e-12
    ulp = np.abs(b["norm"].astype(np.int64) - a["norm"].astype(np.int64))
    assert ulp.max() <= 1 and np.mean(ulp == 0) > 0.99


def test_zero_fn_gives_bias_gates(oracle):
    d = seam_inputs(2, 64, 17, oracle=oracle)
    d["fn"] = torch.zeros_like(d["fn"])
    o = run(oracle, d)
    assert np.all(o["pre"] == 0.5) and np.all(o["post"] == 1.0)
    assert np.allclose(o["comb"], 0.25, atol=1e-15, rtol=0)
    bias = np.zeros(24, np.float32)
    bias[0:4] = math.log(3.0)
    bias[4:8] = -math.log(3.0)
    a = np.array([0.5, -0.25, 1.0, 0.0])
    b = np.array([-1.0, 0.75, 0.0, 0.5])
    bias[8:] = (a[:, None] + b[None, :]).reshape(16)
    o = run(oracle, dict(d, bias=torch.from_numpy(bias)))
    assert np.allclose(o["pre"], 0.75, atol=1e-7) and np.allclose(o["post"], 0.5, atol=1e-7)
    assert np.allclose(o["comb"], 0.25, atol=1e-12, rtol=0)


def test_one_hot_fn_picks_stream_signs(oracle):
    # Streams held at +-2^k (comb = I, post = 0, eps = 0): rstd_R = 2^-k, so a
    # one-hot fn column on stream i gives logit alpha * sign(c_i).  With
    # alpha = ln 3 the gates are exactly 3/4 or 1/4 (pre) and 3/2 or 1/2 (post):
    # a wrong stream index or an orientation slip flips a sign.
    T, H = 1, 16
    d = seam_inputs(T, H, 18, oracle=oracle)
    c = np.array([1.0, -1.0, 1.0, -1.0]) * 4.0
    d["R"] = I.to_bf16(np.broadcast_to(c[None, :, None], (T, 4, H)).copy())
    d["comb_prev"] = np.tile(np.eye(4, dtype=np.float32), (T, 1, 1))
    d["post_prev"] = np.zeros((T, 4), np.float32)
    d["eps"] = 0.0
    fn = np.zeros((4 * H, 24), np.float32)
    streams = [1, 0, 3, 2, 0, 1, 2, 3]
    for k, i in enumerate(streams):
        fn[i * H + (5 + k) % H, k] = 1.0
    d["fn"] = torch.from_numpy(fn)
    d["alpha"] = torch.tensor([math.log(3.0), math.log(3.0), 1.0])
    o = run(oracle, d)
    sgn = c[streams] / 4.0
    assert np.allclose(o["pre"][0], np.where(sgn[:4] > 0, 0.75, 0.25), atol=1e-7)
    assert np.allclose(o["post"][0], np.where(sgn[4:] > 0, 1.5, 0.5), atol=1e-7)


def test_power_of_two_scale_invariance(oracle):
    d = seam_inputs(2, 128, 19, oracle=oracle)
    d["eps"] = 0.0
    a = run(oracle, d)
    s = 2.0 ** 5
    d2 = dict(d, R=(d["R"].to(torch.float64) * s).to(torch.bfloat16), Y=(d["Y"].to(torch.float64) * s).to(torch.bfloat16))
    b = run(oracle, d2)
    for k in ("norm", "pre", "post", "comb"):
        assert np.array_equal(a[k], b[k]), k
    ra = np.vectorize(bf16_val)(a["residual_out"])
    rb = np.vectorize(bf16_val)(b["residual_out"])
    assert np.array_equal(ra * s, rb)


def test_constant_row_norm_closed_form(oracle):
    # x == c along H and eps = 0: norm = bf16(gamma * sign(c)) = gamma * sign(c).
    T, H = 2, 64
    d = seam_inputs(T, H, 20, oracle=oracle)
    d["R"] = I.to_bf16(np.full((T, 4, H), -3.0))
    d["Y"] = I.to_bf16(np.zeros((T, H)))
    d["eps"] = 0.0
    o = run(oracle, d)
    g = I.bf16_bits(d["gamma"])
    # x = sum_i pre_i * sum_j comb_ij * (-3) < 0
    assert np.array_equal(o["norm"], np.broadcast_to(g ^ 0x8000, (T, H)))


def test_unit_gamma_zero_eps_norm_has_unit_rms(oracle):
    # gamma = 1 and eps = 0: norm = x / rms(x), so each row's mean square is 1
    # up to the bf16 rounding of every element (relative 2^-9 each)
    T, H = 4, 512
    d = seam_inputs(T, H, 21, oracle=oracle)
    d["gamma"] = I.to_bf16(np.ones(H))
    d["eps"] = 0.0
    o = run(oracle, d, want_x=True)
    nv = np.array([[bf16_val(b) for b in row] for row in o["norm"]])
    ms = np.mean(nv * nv, axis=1)
    assert np.all(np.abs(ms - 1.0) < 2 * 2.0 ** -8), ms
    # and each element is the RNE of x / rms(x) computed exactly from x
    x = o["x"]
    for t in range(T):
        rms = math.sqrt(float(np.mean(x[t] * x[t])))
        for h in range(0, H, 37):
            assert o["norm"][t, h] == bf16_rne_exact(Fraction(x[t, h] / rms)), (t, h)


def test_gate_ranges_and_doubly_stochastic_on_config_inputs(oracle):
    d = seam_inputs(16, 256, 1000, oracle=oracle)
    o = run(oracle, d)
    assert np.all((o["pre"] > 0) & (o["pre"] < 1))
    assert np.all((o["post"] > 0) & (o["post"] < 2))
    assert np.all(o["comb"] > 0)
    assert np.max(np.abs(o["comb"].sum(-1) - 1)) < 1e-5
    assert np.max(np.abs(o["comb"].sum(-2) - 1)) < 1e-12


def test_rounded_vs_unrounded_rprime_reading_is_small(oracle):
    # Documents the size of the "stored bf16 R' feeds the sums" reading.
    d = seam_inputs(4, 512, 21, oracle=oracle)
    a = run(oracle, d)
    b = run(oracle, d, rprime_unrounded=True)
    assert np.array_equal(a["residual_out"], b["residual_out"])
    assert np.max(np.abs(a["pre"] - b["pre"])) < 1e-3
    assert np.max(np.abs(a["comb"] - b["comb"])) < 1e-3


# ------------------------------------------------- high-precision brute force
def _brute_force_seam(d, t=0, unshifted=False):
    """The seam at one token in exact rationals (sums, products, roundings) and
    60-digit decimals (sqrt, exp, Sinkhorn divisions), straight from the
    definition; independent of the oracle's code.  With ``unshifted`` it also
    returns the unshifted layer input bf16(sum_i pre[i] R'[i]) with the fresh
    pre, no norm."""
    getcontext().prec = 60
    H = d["H"]
    Rv = d["R"].to(torch.float64).numpy()[t]
    Yv = None if d["Y"] is None else d["Y"].to(torch.float64).numpy()[t]
    comb = None if d["comb_prev"] is None else d["comb_prev"][t].astype(np.float64)
    post = None if d["post_prev"] is None else d["post_prev"][t].astype(np.float64)
    pre = d["pre_prev"][t].astype(np.float64)
    fn = d["fn"].to(torch.float64).numpy()
    gam = d["gamma"].to(torch.float64).numpy()
    eps = Fraction(d["eps"])
    res = np.zeros((4, H), np.uint16)
    rp = [[None] * H for _ in range(4)]
    for i in range(4):
        for h in range(H):
            if comb is None:  # the identity form: R' = R, no rounding
                b = int(I.bf16_bits(d["R"][t])[i, h])
            else:
                v = sum(Fraction(comb[i, j]) * Fraction(Rv[j, h]) for j in range(4))
                if Yv is not None:
                    v += Fraction(post[i]) * Fraction(Yv[h])
                b = bf16_rne_exact(v)
            res[i, h] = b
            rp[i][h] = Fraction(bf16_val(b))
    K = 4 * H
    sR = sum(rp[i][h] ** 2 for i in range(4) for h in range(H))
    dk = [sum(rp[i][h] * Fraction(fn[i * H + h, k]) for i in range(4) for h in range(H)) for k in range(24)]
    D = lambda f: Decimal(f.numerator) / Decimal(f.denominator)
    rstdR = 1 / (D(sR / K + eps)).sqrt()
    alpha = d["alpha"].to(torch.float64).numpy()
    bias = d["bias"].to(torch.float64).numpy()
    logit = [D(Fraction(alpha[0 if k < 4 else (1 if k < 8 else 2)])) * rstdR * D(dk[k]) + D(Fraction(bias[k])) for k in range(24)]
    sig = lambda z: 1 / (1 + (-z).exp())
    g_pre = [sig(logit[i]) for i in range(4)]
    g_post = [2 * sig(logit[4 + i]) for i in range(4)]
    M = [[logit[8 + 4 * i + j].exp() for j in range(4)] for i in range(4)]
    for _ in range(20):
        for i in range(4):
            s = sum(M[i])
            M[i] = [m / s for m in M[i]]
        for j in range(4):
            s = sum(M[i][j] for i in range(4))
            for i in range(4):
                M[i][j] = M[i][j] / s
    x = [sum(Fraction(pre[i]) * rp[i][h] for i in range(4)) for h in range(H)]
    sx = sum(v * v for v in x)
    rstdx = 1 / (D(sx / H + eps)).sqrt()
    norm = np.zeros(H, np.uint16)
    for h in range(H):
        y = D(x[h]) * rstdx * D(Fraction(gam[h]))
        norm[h] = bf16_rne_exact(Fraction(y))
    out = (res, norm, np.array([float(v) for v in g_pre]), np.array([float(v) for v in g_post]),
           np.array([[float(v) for v in r] for r in M]))
    if unshifted:
        xu = np.zeros(H, np.uint16)
        for h in range(H):
            v = sum(g_pre[i] * D(rp[i][h]) for i in range(4))
            xu[h] = bf16_rne_exact(Fraction(v))
        out = out + (xu,)
    return out


@pytest.mark.parametrize("seed", [31, 32, 33])
def test_brute_force_T1_H8_asymmetric_comb(oracle, seed):
    d = seam_inputs(1, 8, seed, oracle=oracle)
    # a deliberately non-symmetric, non-stochastic comb pins its orientation
    d["comb_prev"] = np.array([[[0.9, 0.05, 0.3, -0.2], [0.1, 0.7, 0.0, 0.4], [-0.3, 0.2, 1.1, 0.05], [0.25, -0.1, 0.15, 0.6]]], np.float32)
    d["bias"] = torch.linspace(-0.5, 0.5, 24)
    d["alpha"] = torch.tensor([0.8, 1.3, 0.6])
    o = run(oracle, d)
    res, norm, g_pre, g_post, comb = _brute_force_seam(d)
    assert np.array_equal(o["residual_out"][0], res)
    assert np.array_equal(o["norm"][0], norm)
    assert np.allclose(o["pre"][0], g_pre, atol=1e-13, rtol=0)
    assert np.allclose(o["post"][0], g_post, atol=1e-13, rtol=0)
    assert np.allclose(o["comb"][0], comb, atol=1e-13, rtol=0)


@pytest.mark.parametrize("seed", [34, 35])
def test_brute_force_T1_H8_identity_form(oracle, seed):
    # the first-block form: nothing mixed in, R' = R; gates and norm from R
    d = seam_inputs(1, 8, seed, post=False, oracle=oracle)
    d["comb_prev"] = None
    d["bias"] = torch.linspace(-0.4, 0.6, 24)
    d["alpha"] = torch.tensor([1.1, 0.7, 0.9])
    o = run(oracle, d)
    res, norm, g_pre, g_post, comb = _brute_force_seam(d)
    assert np.array_equal(o["residual_out"][0], res)
    assert np.array_equal(o["residual_out"][0], I.bf16_bits(d["R"][0]))
    assert np.array_equal(o["norm"][0], norm)
    assert np.allclose(o["pre"][0], g_pre, atol=1e-13, rtol=0)
    assert np.allclose(o["post"][0], g_post, atol=1e-13, rtol=0)
    assert np.allclose(o["comb"][0], comb, atol=1e-13, rtol=0)


def test_identity_form_keeps_signed_zeros_and_subnormals(oracle):
    # R' = R bit for bit, where comb = I would turn -0 into +0 (1 * -0 + 0 * r)
    d = seam_inputs(2, 64, 36, post=False, oracle=oracle)
    bits = I.bf16_bits(d["R"]).copy()
    bits[0, 0, :8] = 0x8000                     # -0
    bits[0, 1, :8] = 0x0001                     # smallest subnormal
    bits[1, 2, 5] = 0x8001
    d["R"] = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    ident = run(oracle, dict(d, comb_prev=None))
    assert np.array_equal(ident["residual_out"], bits)
    eye = run(oracle, dict(d, comb_prev=np.tile(np.eye(4, dtype=np.float32), (2, 1, 1))))
    assert not np.array_equal(eye["residual_out"], bits)  # the -0 entries differ
    # away from the signed zeros the two forms agree
    assert np.array_equal(ident["norm"][1], eye["norm"][1])


# ------------------------------------------------------ unshifted seam ----
def run_unshifted(oracle, d):
    return oracle.seam_unshifted(d["R"], d["Y"], d["post_prev"], d["comb_prev"], d["fn"], d["bias"], d["alpha"],
                                 d["eps"])


@pytest.mark.parametrize("seed,post,ident", [(37, True, False), (38, False, False), (39, False, True)])
def test_brute_force_T1_H8_unshifted(oracle, seed, post, ident):
    d = seam_inputs(1, 8, seed, post=post, oracle=oracle)
    d["comb_prev"] = None if ident else np.array(
        [[[0.9, 0.05, 0.3, -0.2], [0.1, 0.7, 0.0, 0.4], [-0.3, 0.2, 1.1, 0.05], [0.25, -0.1, 0.15, 0.6]]], np.float32)
    d["bias"] = torch.linspace(-0.7, 0.3, 24)
    d["alpha"] = torch.tensor([1.2, 0.9, 0.7])
    o = run_unshifted(oracle, d)
    res, _, g_pre, g_post, comb, xu = _brute_force_seam(d, unshifted=True)
    assert np.array_equal(o["residual_out"][0], res)
    assert np.array_equal(o["x"][0], xu)
    assert np.allclose(o["pre"][0], g_pre, atol=1e-13, rtol=0)
    assert np.allclose(o["post"][0], g_post, atol=1e-13, rtol=0)
    assert np.allclose(o["comb"][0], comb, atol=1e-13, rtol=0)


def test_unshifted_zero_fn_gives_half_sum_of_streams(oracle):
    # zero fn and bias: every logit is 0, so the fresh pre is sigma(0) = 1/2 and
    # x = bf16(sum_i R'[i] / 2) exactly (the carried pre of the draws is not 1/2)
    d = seam_inputs(3, 64, 42, oracle=oracle)
    d["fn"] = torch.zeros_like(d["fn"])
    d["bias"] = torch.zeros(24)
    o = run_unshifted(oracle, d)
    assert np.all(o["pre"] == 0.5) and np.all(o["post"] == 1.0) and np.allclose(o["comb"], 0.25, atol=1e-15)
    rp = o["residual_out"]
    for t in range(3):
        for h in range(64):
            v = Fraction(1, 2) * sum(Fraction(bf16_val(rp[t, i, h])) for i in range(4))
            assert o["x"][t, h] == bf16_rne_exact(v), (t, h)


def test_unshifted_shares_the_delayed_seams_residual_and_gates(oracle):
    d = seam_inputs(4, 128, 43, oracle=oracle)
    a = run_unshifted(oracle, d)
    b = run(oracle, d)
    assert np.array_equal(a["residual_out"], b["residual_out"])
    for k in ("pre", "post", "comb"):
        assert np.array_equal(a[k], b[k]), k


def test_oracle_rejects_y_without_comb(oracle):
    d = seam_inputs(1, 8, 41, oracle=oracle)
    with pytest.raises(ValueError):
        run(oracle, dict(d, comb_prev=None))


def test_oracle_rejects_half_present_post(oracle):
    d = seam_inputs(1, 8, 40, oracle=oracle)
    with pytest.raises(ValueError):
        run(oracle, dict(d, post_prev=None))


# ------------------------------------------------------------ fp8_grid ----
def test_e4m3_decode_matches_format_definition(oracle):
    # every finite code decodes to its value in the OCP definition (the golden
    # file's listed code points and the table built from the bit fields)
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e4m3fn_ocp.txt")) if l.strip() and not l.startswith("#")]
    for v, code in rows:
        assert oracle.e4m3_decode(int(code, 16)) == float(v), (v, code)
    for code, v in e4m3_table().items():
        assert oracle.e4m3_decode(code) == v, code
        assert oracle.e4m3(v) == code or (v == 0.0 and code in (0x00, 0x80)), code
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_grid_exact_on_the_e4m3_lattice(oracle):
    # a group whose amax is 448 * 2^k and whose values are e4m3 values times
    # 2^k reconstructs exactly (the grid is the identity on its own lattice)
    table = e4m3_table()
    codes = sorted(c for c in table if c not in (0x7F, 0xFF))
    rng = np.random.default_rng(7)
    for k in (-30, -5, 0, 3, 20):
        vals = np.array([table[c] for c in rng.choice(codes, 32)]) * 2.0 ** k
        vals[0] = 448.0 * 2.0 ** k
        x = I.to_bf16(vals).reshape(1, 32)
        grid = oracle.grid_ue8m0(x)
        assert np.array_equal(grid, I.bf16_bits(x)), k


def test_grid_is_the_dequantised_mxfp8_output(oracle):
    # grid = decode(code) * 2^(scale - 127) from the quantiser's own outputs,
    # decoded by the table above, within the e4m3 rounding bound of the input
    x, _ = I.crafted_quant_tensor(8, 256, seed=1005, frac=0.2)
    grid = oracle.grid_ue8m0(x)
    codes, scales = oracle.quant_ue8m0(x)
    table = e4m3_table()
    xv = x.to(torch.float64).numpy()
    for r in range(8):
        for h in range(256):
            e = int(scales[r, h // 32]) - 127
            want = I.bf16_bits(I.to_bf16(np.array([table[int(codes[r, h])] * 2.0 ** e])))[0]
            assert grid[r, h] == want, (r, h)
            g = bf16_val(grid[r, h])
            assert abs(g - xv[r, h]) <= max(abs(xv[r, h]) * 2.0 ** -4, 2.0 ** (e - 10)), (r, h)
