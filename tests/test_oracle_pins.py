"""Pins for the CPU oracle: every oracle function is checked here against
something other than itself -- hand-derived fixtures under tests/golden/,
closed forms, exact rational arithmetic, invariants that follow from the
definitions, or brute force on tiny inputs.  CPU only.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc
from tests.exact import round_to_f32, ulp_f32
from w8a8_quantized_speculative_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def bf16(values):
    """Exact BF16 bits of values that are representable in BF16."""
    a = np.asarray(values, dtype=np.float32)
    bits = a.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "fixture value not representable in BF16"
    return (bits >> 16).astype(np.uint16)


# ---------------------------------------------------------------- BF16 rounding

def test_bf16_rne_fixture():
    for c in load("bf16_rne.json")["cases"]:
        got = int(orc.f32_to_bf16(np.array([c["x"]], np.float32))[0])
        assert got == int(c["bf16"], 16), c


def test_bf16_roundtrip_exact():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 0x7F80, size=5000).astype(np.uint16)   # finite positives
    bits = np.concatenate([bits, bits | 0x8000])
    assert np.array_equal(orc.f32_to_bf16(orc.bf16_to_f32(bits)), bits)


def test_bf16_rounding_is_nearest():
    # Against exact rationals: the chosen BF16 is at most half a BF16 ulp away.
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(2000) * 100).astype(np.float32)
    y = orc.bf16_to_f32(orc.f32_to_bf16(x))
    for xi, yi in zip(x[:400], y[:400]):
        q = Fraction(float(xi))
        half_ulp = ulp_f32(q) * 2 ** 16 / 2
        assert abs(Fraction(float(yi)) - q) <= half_ulp


# ---------------------------------------------------------------- quantizer

@pytest.mark.parametrize("kind", ["activation_cases", "weight_cases"])
def test_quantizer_fixture(kind):
    for c in load("quantizer_rows.json")[kind]:
        smooth = np.asarray(c["smooth"], np.float32)
        if kind == "activation_cases":
            codes, scale = orc.smooth_quant_act(bf16([c["x"]]), smooth)
        else:
            codes, scale = orc.pack_weights(bf16([c["w"]]), smooth)
        assert codes.tolist() == [c["codes"]], c["why"]
        num, den = c["scale_exact"]
        exact = Fraction(num, den)
        # the scale is the correctly rounded fp32 value of absmax/127
        assert Fraction(float(scale[0])) == round_to_f32(exact), c["why"]


def test_quantizer_invariants_random():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((64, 300)) * np.exp(rng.uniform(-6, 6, size=(64, 1)))).astype(np.float32)
    v[5] = 0.0
    codes, scale = orc.quantize_rows(v)
    assert codes.dtype == np.int8
    assert codes.min() >= -127 and codes.max() <= 127
    assert scale[5] == 0 and not codes[5].any()
    nz = np.abs(v).max(axis=1) > 0
    # every nonzero row uses the full range once (its absmax maps to +-127)
    assert np.all(np.abs(codes[nz]).max(axis=1) == 127)
    # reconstruction error at most half a step (plus fp32 rounding of the scales)
    amax = np.abs(v).max(axis=1).astype(np.float64)
    err = np.abs(codes.astype(np.float64) * scale[:, None].astype(np.float64) - v.astype(np.float64))
    bound = scale[:, None].astype(np.float64) * 0.5 + amax[:, None] * 2.0 ** -20
    assert np.all(err <= bound)


def test_quantizer_is_nearest_code():
    # brute force: for each element, no other code is strictly closer to v/scale
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((8, 40)) * 3).astype(np.float32)
    codes, scale = orc.quantize_rows(v)
    for i in range(v.shape[0]):
        t = v[i].astype(np.float64) * 127.0 / np.abs(v[i]).max()
        for j in range(v.shape[1]):
            best = np.abs(np.arange(-127, 128) - t[j]).min()
            assert abs(int(codes[i, j]) - t[j]) <= best + 1e-5


def test_smoothing_direction():
    """Activations are multiplied by smooth and weights divided (the pages'
    identity): the dequantized operands must approximate X*s and W/s."""
    rng = np.random.default_rng(4)
    K = 96
    s = np.exp(rng.uniform(-2.5, 2.5, K)).astype(np.float32)
    x = synth.f32_to_bf16_bits(rng.standard_normal((6, K)).astype(np.float32))
    w = synth.f32_to_bf16_bits((rng.standard_normal((10, K)) * 0.02).astype(np.float32))
    xq, sa = orc.smooth_quant_act(x, s)
    wq, sw = orc.pack_weights(w, s)
    xs = synth.bf16_bits_to_f32(x).astype(np.float64) * s
    ws = synth.bf16_bits_to_f32(w).astype(np.float64) / s
    assert np.all(np.abs(xq * sa[:, None].astype(np.float64) - xs) <= sa[:, None] * 0.5000001)
    assert np.all(np.abs(wq * sw[:, None].astype(np.float64) - ws) <= sw[:, None] * 0.5000001)


# ---------------------------------------------------------------- calibration

def test_calibrate_fixture():
    g = load("calibrate.json")
    x = bf16(g["x_cal"])
    w = bf16(g["w"])
    s = orc.calibrate_smooth(x, w, 0.5)
    assert s.dtype == np.float32
    assert s.tolist() == g["alpha_0.5"]
    s2 = orc.calibrate_smooth(x, w, 0.25)
    for got, want in zip(s2.tolist(), g["alpha_0.25"]):
        if want is not None:
            assert got == want


def test_calibrate_shrinks_outliers():
    case = synth.small_case()
    s = orc.calibrate_smooth(case.x_cal(), case.w())
    out = case.outliers()
    rest = np.setdiff1d(np.arange(case.K), out)
    # outlier channels get a much smaller factor than the others
    assert s[out].max() < 0.5 * np.median(s[rest])


# ---------------------------------------------------------------- integer GEMM

def brute_gemm(xq, wq):
    M, K = xq.shape
    N = wq.shape[0]
    out = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            t = 0
            for k in range(K):
                t += int(xq[m, k]) * int(wq[n, k])
            out[m][n] = t
    return np.array(out, dtype=np.int64)


def test_int_gemm_brute_force():
    rng = np.random.default_rng(5)
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (4, 8, 32), (2, 3, 64)]:
        xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        wq = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
        xq[0, 0] = -127
        wq[0, 0] = -127
        assert np.array_equal(orc.int_gemm(xq, wq), brute_gemm(xq, wq))


def test_int_gemm_closed_forms():
    K = 1024
    ones = np.full((1, K), 127, np.int8)
    assert orc.int_gemm(ones, ones)[0, 0] == 127 * 127 * K == 16516096
    alt = np.tile(np.array([127, -127], np.int8), K // 2)[None, :]
    assert orc.int_gemm(alt, ones)[0, 0] == 0
    assert orc.int_gemm(alt, alt)[0, 0] == 16516096
    neg = np.full((1, K), -127, np.int8)
    assert orc.int_gemm(neg, ones)[0, 0] == -16516096
    # beyond 2^24 the integer result is still exact
    K2 = 131072
    big = np.full((1, K2), 127, np.int8)
    assert orc.int_gemm(big, big)[0, 0] == 127 * 127 * K2


def test_int_gemm_matches_int64_matmul():
    rng = np.random.default_rng(6)
    xq = rng.integers(-127, 128, size=(9, 700)).astype(np.int8)
    wq = rng.integers(-127, 128, size=(13, 700)).astype(np.int8)
    assert np.array_equal(orc.int_gemm(xq, wq), xq.astype(np.int64) @ wq.astype(np.int64).T)


# ---------------------------------------------------------------- dequant

def test_dequant_fixture():
    g = load("dequant.json")
    y = orc.dequant(np.array(g["acc"], np.int64), np.array(g["sa"], np.float32), np.array(g["sw"], np.float32))
    want = np.array([[int(h, 16) for h in row] for row in g["bf16"]], np.uint16)
    assert np.array_equal(y, want)


def test_dequant_int_to_f32_rounding():
    # 2^24 + 1 is a tie between 2^24 and 2^24 + 2 -> even -> 2^24; then x1 x1 -> bf16(2^24)
    acc = np.array([[16777217, 16777219, -16777217]], np.int64)
    one = np.array([1.0], np.float32)
    f = orc.dequant_f32(acc, one, np.ones(3, np.float32))
    assert f.tolist() == [[16777216.0, 16777220.0, -16777216.0]]


def test_dequant_is_correctly_rounded_steps():
    # each fp32 multiply is a single correct rounding (exact rational model)
    rng = np.random.default_rng(7)
    M, N = 16, 40
    acc = rng.integers(-2 ** 26, 2 ** 26, size=(M, N)).astype(np.int64)
    sa = (rng.uniform(0.001, 0.2, M)).astype(np.float32)
    sw = (rng.uniform(1e-5, 1e-3, N)).astype(np.float32)
    f = orc.dequant_f32(acc, sa, sw)
    for m in range(M):
        for n in range(N):
            a = round_to_f32(Fraction(int(acc[m, n])))
            t = round_to_f32(a * Fraction(float(sa[m])))
            y = round_to_f32(t * Fraction(float(sw[n])))
            assert Fraction(float(f[m, n])) == y


# ---------------------------------------------------------------- whole linear

def test_fp64_identity():
    """(W diag(s)^-1)(diag(s) X) == W X (zh §2) for arbitrary positive s."""
    rng = np.random.default_rng(8)
    x = synth.activations(11, 7, 64)
    w = synth.weights(12, 9, 64)
    s = np.exp(rng.uniform(-3, 3, 64)).astype(np.float32)
    a = orc.smoothed_linear_f64(x, w, s)
    b = orc.reference_linear_f64(x, w)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_scaled_identity_weight_closed_form():
    """W = c*I, smooth = 1: each weight row quantizes to a single 127 with
    sw = c/127, so acc = 127 * Xq exactly."""
    K = 48
    c = 0.5
    w = bf16(np.eye(K) * c)
    x = synth.activations(13, 5, K)
    wq, sw = orc.pack_weights(w, np.ones(K, np.float32))
    assert np.array_equal(wq, (np.eye(K) * 127).astype(np.int8))
    assert np.all(Fraction(float(sw[0])) == round_to_f32(Fraction(1, 2) / 127))
    xq, sa = orc.smooth_quant_act(x, np.ones(K, np.float32))
    acc = orc.int_gemm(xq, wq)
    assert np.array_equal(acc, 127 * xq.astype(np.int64))
    y = synth.bf16_bits_to_f32(orc.dequant(acc, sa, sw)).astype(np.float64)
    xv = synth.bf16_bits_to_f32(x).astype(np.float64)
    assert np.all(np.abs(y - c * xv) <= c * sa[:, None] * 0.5 + np.abs(c * xv) * 2 ** -7 + 1e-6)


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_small_case_accuracy_and_reading():
    """Calibrated smoothing keeps the W8A8 output within 2e-2 relative
    Frobenius error of the unquantized product; the literal inverse reading
    of s (outlier channels multiplied up) is clearly worse."""
    case = synth.small_case()
    x, w, xc = case.x(), case.w(), case.x_cal()
    s = orc.calibrate_smooth(xc, w)
    ref = orc.reference_linear_f64(x, w)

    def run(smooth):
        xq, sa = orc.smooth_quant_act(x, smooth)
        wq, sw = orc.pack_weights(w, smooth)
        return synth.bf16_bits_to_f32(orc.w8a8_linear(xq, sa, wq, sw)).astype(np.float64)

    e_good = rel_fro(run(s), ref)
    e_lit = rel_fro(run((1.0 / s.astype(np.float64)).astype(np.float32)), ref)
    e_none = rel_fro(run(np.ones(case.K, np.float32)), ref)
    assert e_good <= 2e-2, e_good
    assert e_lit > 2 * e_good
    assert e_none > e_good


def test_smooth_one_reduces_to_plain_w8a8():
    case = synth.small_case()
    x, w = case.x(), case.w()
    one = np.ones(case.K, np.float32)
    xq, sa = orc.smooth_quant_act(x, one)
    xq2, sa2 = orc.quantize_rows(synth.bf16_bits_to_f32(x))
    assert np.array_equal(xq, xq2) and np.array_equal(sa, sa2)
    wq, sw = orc.pack_weights(w, one)
    wq2, sw2 = orc.quantize_rows(synth.bf16_bits_to_f32(w))
    assert np.array_equal(wq, wq2) and np.array_equal(sw, sw2)


# ---------------------------------------------------------------- verification

def test_verify_greedy_fixture():
    g = load("verify_cases.json")
    lg = bf16(g["logits"])
    for row, am in zip(g["logits"], g["argmax_by_row"]):
        assert int(np.argmax(row)) == am
    for c in g["cases"]:
        n_acc, nxt = orc.verify_accept(lg[None], np.array([c["draft"]], np.int32), 0.0)
        assert int(n_acc[0]) == c["n_acc"], c["why"]
        assert int(nxt[0]) == c["next"], c["why"]


def test_verify_no_drafts():
    g = load("verify_cases.json")
    lg = bf16(g["logits"])[:1][None]
    n_acc, nxt = orc.verify_accept(lg, np.zeros((1, 0), np.int32), 0.0)
    assert n_acc.tolist() == [0] and nxt.tolist() == [2]


@pytest.mark.parametrize("T", [1.0, 0.5, 2.0])
def test_verify_two_level_closed_form(T):
    """Logits: one entry L, the rest 0 -> p = e^(L/T) / (e^(L/T) + V - 1)."""
    V, L, hot = 1000, 2.0, 17
    row = np.zeros(V, np.float32)
    row[hot] = L
    lg = np.stack([row, row, row])[None]          # D = 2
    bits = bf16(lg)
    c = math.exp(L / T)
    p_hot = c / (c + V - 1)
    p_cold = 1.0 / (c + V - 1)
    p = orc.acceptance_probabilities(bits, np.array([[hot, 3]], np.int32), T)
    assert abs(p[0, 0] - p_hot) < 1e-12 and abs(p[0, 1] - p_cold) < 1e-12
    cases = [
        ([hot, hot], [p_hot / 2, p_hot / 2], 2),
        ([hot, hot], [(1 + p_hot) / 2, 0.0], 0),
        ([hot, 5], [p_hot / 2, p_cold / 2], 2),
        ([hot, 5], [p_hot / 2, (p_cold + 1) / 2], 1),
    ]
    for draft, u, want in cases:
        n_acc, nxt = orc.verify_accept(bits, np.array([draft], np.int32), T, np.array([u], np.float32))
        assert int(n_acc[0]) == want
        assert int(nxt[0]) == -1


def test_verify_forced_mask_invariant():
    """Drafts forced to the argmax on a seeded mask: n_acc is the first
    unforced position unless a random draft happens to match."""
    B, D, V = 6, 5, 257
    lg, draft, mask, _ = synth.verify_inputs(B, D, V, 11, 12, 13, 14)
    am = np.argmax(orc.bf16_to_f32(lg), axis=2)
    d = np.where(mask, am[:, :D], draft).astype(np.int32)
    n_acc, nxt = orc.verify_accept(lg, d, 0.0)
    for b in range(B):
        ok = d[b] == am[b, :D]
        want = D if ok.all() else int(np.argmin(ok))
        assert n_acc[b] == want
        assert nxt[b] == am[b, want]


# ---------------------------------------------------------------- lossless next token (R7)

@pytest.mark.parametrize("T", [1.0, 0.5])
def test_sample_residual_two_level_closed_form(T):
    """Reject the hot draft of a two-level row: the residual is uniform over
    the V - 1 other tokens, so u_next = (k + 1/2) / (V - 1) must give the
    k-th token that is not the hot one."""
    V, L, hot = 64, 3.0, 17
    row = np.zeros(V, np.float32)
    row[hot] = L
    bits = bf16(np.stack([row, row])[None])        # D = 1
    c = math.exp(L / T)
    p_hot = c / (c + V - 1)
    others = [v for v in range(V) if v != hot]
    for k in (0, 1, 16, 17, 40, V - 2):
        u = np.array([[(1 + p_hot) / 2]], np.float32)                 # rejects the hot draft
        n_acc, nxt = orc.verify_sample(bits, np.array([[hot]], np.int32), T, u, np.array([(k + 0.5) / (V - 1)]))
        assert int(n_acc[0]) == 0 and int(nxt[0]) == others[k]


def test_sample_bonus_explicit_cdf():
    """Every draft accepted: the bonus row is sampled from its full softmax.
    Row weights 1, 1, 1, 3, 1, ... (logit ln 3 at token 3): the CDF steps are
    known exactly."""
    V = 8
    row = np.zeros(V, np.float32)
    lg = np.stack([row, row])
    lg[1, 3] = math.log(3.0)                        # bonus row (rounded to BF16; weights read back)
    bits = synth.f32_to_bf16_bits(lg[None])
    w = np.exp(orc.bf16_to_f32(bits)[0, 1].astype(np.float64))
    cdf = np.cumsum(w) / w.sum()
    for v in range(V):
        lo = cdf[v - 1] if v else 0.0
        u_next = (lo + cdf[v]) / 2
        n_acc, nxt = orc.verify_sample(bits, np.array([[0]], np.int32), 1.0, np.array([[0.0]], np.float32),
                                       np.array([u_next]))
        assert int(n_acc[0]) == 1 and int(nxt[0]) == v


def test_sample_rejects_draft_never_resampled():
    """The rejected draft token has no residual mass: it is never drawn."""
    V = 16
    rng = np.random.default_rng(5)
    bits = synth.f32_to_bf16_bits(rng.standard_normal((1, 2, V)))
    d = 7
    for u_next in np.linspace(0, 1, 97, endpoint=False):
        n_acc, nxt = orc.verify_sample(bits, np.array([[d]], np.int32), 1.0, np.array([[0.999999]], np.float32),
                                       np.array([u_next]))
        assert int(n_acc[0]) == 0 and int(nxt[0]) != d


@pytest.mark.parametrize("d", [0, 2, 5])
def test_sample_is_lossless_chi_square(d):
    """Losslessness: with a fixed draft d, the token emitted at position 0
    (d if accepted, else the residual draw) is distributed as the target
    softmax p_0.  20000 seeded draws, chi-square against p_0 at alpha 1e-4."""
    V, N = 6, 20000
    rng = np.random.default_rng(100 + d)
    logits = np.array([[0.3, -0.2, 1.1, 0.0, -1.0, 0.6], [0.0] * V], np.float32)
    bits = synth.f32_to_bf16_bits(np.repeat(logits[None], N, axis=0))
    draft = np.full((N, 1), d, np.int32)
    u = rng.random((N, 1)).astype(np.float32)
    u_next = rng.random(N)
    n_acc, nxt = orc.verify_sample(bits, draft, 1.0, u, u_next)
    emitted = np.where(n_acc == 1, d, nxt)
    z = orc.bf16_to_f32(bits)[0, 0].astype(np.float64)
    p = np.exp(z - z.max())
    p /= p.sum()
    counts = np.bincount(emitted, minlength=V)
    chi2 = float(((counts - N * p) ** 2 / (N * p)).sum())
    assert chi2 < 25.74, (chi2, counts, N * p)      # chi-square(5) upper 1e-4 point
    # a residual that kept the draft token would fail: check that it is detectable
    keep = np.where(n_acc == 1, d, np.minimum(np.searchsorted(np.cumsum(p), u_next, side="right"), V - 1))
    bad = float(((np.bincount(keep, minlength=V) - N * p) ** 2 / (N * p)).sum())
    assert bad > 100.0


# ---------------------------------------------------------------- 4-bit weights (R8)

def test_quantizer_w4_fixture():
    """Hand-derived: absmax 3.5 -> inv = 7/3.5 = 2, scale = 0.5; codes
    rne(1) = 1, rne(-3.5) = -4 (tie to even), rne(7) = 7, rne(2.5) = 2."""
    v = np.array([[0.5, -1.75, 3.5, 1.25], [0.0, 0.0, 0.0, 0.0]], np.float32)
    codes, scale = orc.quantize_rows(v, qmax=7)
    assert codes.tolist() == [[1, -4, 7, 2], [0, 0, 0, 0]]
    assert scale.tolist() == [0.5, 0.0]


def test_quantizer_w4_invariants():
    rng = np.random.default_rng(44)
    v = (rng.standard_normal((64, 300)) * rng.uniform(0.01, 10, (64, 1))).astype(np.float32)
    codes, scale = orc.quantize_rows(v, qmax=7)
    assert codes.min() >= -7 and codes.max() <= 7
    assert np.all(np.abs(codes).max(axis=1) == 7)
    err = np.abs(codes.astype(np.float64) * scale[:, None] - v)
    assert np.all(err <= scale[:, None] * (0.5 + 1e-5))


def test_pack_weights_w4_is_smoothed_quantizer():
    """Folding the smoothing factor first, then the 4-bit per-channel
    quantizer; a code of magnitude 7 in every row."""
    rng = np.random.default_rng(45)
    w = synth.f32_to_bf16_bits(rng.standard_normal((16, 64)) * 0.02)
    s = rng.uniform(0.5, 2.0, 64).astype(np.float32)
    wq, sw = orc.pack_weights_w4(w, s)
    wq_ref, sw_ref = orc.quantize_rows(orc.bf16_to_f32(w) / s[None, :], qmax=7)
    assert np.array_equal(wq, wq_ref) and np.array_equal(sw, sw_ref)
    assert np.all(np.abs(wq).max(axis=1) == 7)


# ------------------------------------------------ BF16 lm_head (reading R9)

def _bf16_value(bits):
    return Fraction(float(np.array([int(bits) << 16], np.uint32).view(np.float32)[0]))


def test_f64_to_bf16_midpoints_and_double_rounding():
    from tests.exact import round_to_bf16
    cases = [1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -30, -(1 + 2 ** -8 + 2 ** -30), 3.0, 1e-3,
             -7.123456789, 2.0 ** -100, 65504.25]
    got = orc.f64_to_bf16(np.array(cases))
    for x, g in zip(cases, got):
        assert _bf16_value(g) == round_to_bf16(Fraction(x)), x
    # exact midpoints go to the even neighbour; just above the first one rounds up, which a
    # detour through fp32 (1 + 2^-8 + 2^-30 -> 1 + 2^-8 -> 1.0) would lose
    assert [int(v) for v in got[:3]] == [0x3F80, 0x3F82, 0x3F81]


def test_f64_to_bf16_agrees_with_f32_path_on_f32_inputs():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    assert np.array_equal(orc.f64_to_bf16(x.astype(np.float64)), orc.f32_to_bf16(x))


def test_bf16_midpoint_distance_cases():
    u9 = 2.0 ** -9
    x = np.array([1 + 2 ** -8, 1.0, 2.0, 1 + 2 ** -7, 1.5, 1 - 2 ** -9, 1 + 2 ** -9, -(1 + 2 ** -7)])
    want = np.array([0, 1, 2, 2, 2, 0, 1, 2]) * u9
    assert np.array_equal(orc.bf16_midpoint_distance(x), want)


def test_lm_head_logits_exact_brute_force():
    from tests.exact import round_to_bf16
    rng = np.random.default_rng(11)
    R, K, V = 3, 16, 7
    h = orc.f32_to_bf16(rng.standard_normal((R, K)).astype(np.float32))
    w = orc.f32_to_bf16((rng.standard_normal((V, K)) * 0.05).astype(np.float32))
    got = orc.lm_head_logits(h, w, chunk=3)   # several vocabulary slices and a ragged last one
    for r in range(R):
        for v in range(V):
            exact = sum(_bf16_value(h[r, k]) * _bf16_value(w[v, k]) for k in range(K))
            assert _bf16_value(got[r, v]) == round_to_bf16(exact), (r, v)


def test_lm_head_logits_selector_closed_form():
    # W[v] = 2^s_v * e_{k_v}: logits[r][v] = 2^s_v * H[r][k_v] exactly
    rng = np.random.default_rng(12)
    R, K, V = 5, 32, 40
    h = orc.f32_to_bf16(rng.standard_normal((R, K)).astype(np.float32))
    kv = rng.integers(0, K, V)
    sv = rng.integers(-3, 4, V)
    w = np.zeros((V, K), np.float32)
    w[np.arange(V), kv] = 2.0 ** sv
    got = orc.bf16_to_f32(orc.lm_head_logits(h, orc.f32_to_bf16(w)))
    want = orc.bf16_to_f32(h)[:, kv] * (2.0 ** sv)[None, :]
    assert np.array_equal(got, want.astype(np.float32))


def test_lm_head_verify_hand_built():
    # Hidden rows pick the vocabulary row holding their maximum; W = identity
    # on the first V coordinates, so each row's argmax is where its maximum sits.
    B, D, V, K = 2, 3, 8, 8
    top = np.array([[5, 1, 6, 2], [0, 3, 3, 7]])      # argmax of rows j = 0..3 of each sequence
    h = np.zeros((B * (D + 1), K), np.float32)
    for b in range(B):
        for j in range(D + 1):
            h[b * (D + 1) + j] = -1.0
            h[b * (D + 1) + j, top[b, j]] = 2.0
    w = np.eye(V, K, dtype=np.float32)
    draft = np.array([[5, 1, 4], [0, 3, 3]], np.int32)  # seq 0 fails at j = 2; seq 1 accepts all
    n_acc, nxt = orc.lm_head_verify(orc.f32_to_bf16(h), orc.f32_to_bf16(w), draft)
    assert n_acc.tolist() == [2, 3]
    assert nxt.tolist() == [6, 7]


# ------------------------------------- MLP glue: SiLU(gate) * up (reading R10)

def test_exp_f32_constants():
    """The reduction constants and coefficients are what the algorithm says:
    log2(e), ln2 split in a head whose products with every n of the range
    are exact and a tail, and 1/k! -- each the fp32 rounding of the exact
    value (rational arithmetic)."""
    ln2 = Fraction(math.log(2))          # fp64 ln2: 2^-53 relative, far below what is checked
    hi, lo = Fraction(float(orc.EXP_LN2_HI)), Fraction(float(orc.EXP_LN2_LO))
    assert abs(hi + lo - ln2) <= ulp_f32(lo)
    assert round_to_f32(ln2 - hi) == lo
    for n in range(-126, 128):           # n * head is exact in fp32
        assert round_to_f32(n * hi) == n * hi if n else True
    assert Fraction(float(orc.EXP_LOG2E)) == round_to_f32(1 / ln2)
    for k, c in zip(range(7, 1, -1), orc.EXP_TAYLOR):
        assert Fraction(float(c)) == round_to_f32(Fraction(1, math.factorial(k)))


def test_exp_f32_within_two_ulp():
    """Against the fp64 exponential on a dense grid of the clamped range (a
    dropped Taylor term already gives ~3 ulp, a dropped ln2 tail thousands)."""
    t = np.linspace(-87.0, 88.0, 2_000_001).astype(np.float32)
    t = np.concatenate([t, np.float32(2.0) ** -np.arange(1, 40, dtype=np.float32),
                        -np.float32(2.0) ** -np.arange(1, 40, dtype=np.float32)])
    ref = np.exp(t.astype(np.float64))
    err = np.abs(orc.exp_f32(t).astype(np.float64) - ref) / np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert err.max() <= 2.0
    assert orc.exp_f32(np.float32(0.0)) == np.float32(1.0)


def test_silu_f32_closed_forms_and_accuracy():
    """silu(0) = 0; for g >= 18, e^-g < 2^-25 so 1 + e rounds to 1 and silu(g)
    is g exactly; elsewhere within 3 ulp of g / (1 + e^-g) in fp64 (exp's 2 ulp
    plus two roundings)."""
    big = np.array([18.0, 20.0, 87.5, 1000.0, 3.0e38], np.float32)
    assert np.array_equal(orc.silu_f32(big), big)
    assert orc.silu_f32(np.zeros(3, np.float32)).tolist() == [0.0, 0.0, 0.0]
    g = np.linspace(-87.0, 80.0, 1_000_001).astype(np.float32)
    g = g[g != 0]
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    err = np.abs(orc.silu_f32(g).astype(np.float64) - ref) / np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert err.max() <= 3.0
    # below the clamp the result stays a tiny negative number of the right sign
    tail = orc.silu_f32(np.array([-90.0, -1000.0], np.float32))
    assert np.all(tail < 0) and np.all(tail > -1e-30)


def test_silu_f32_rounding_sequence():
    """silu(g) = g / d with d = fp32(1 + e) and ONE correctly rounded
    division, checked in rational arithmetic on 400 BF16 gate values (a
    reciprocal-then-multiply form rounds twice and differs on some)."""
    g = orc.bf16_to_f32(synth.f32_to_bf16_bits(np.linspace(-20.0, 20.0, 400)))
    g = g[g != 0]
    e = orc.exp_f32(np.minimum(np.maximum(-g, np.float32(-87.0)), np.float32(88.0)))
    got = orc.silu_f32(g)
    for gi, ei, si in zip(g, e, got):
        d = round_to_f32(1 + Fraction(float(ei)))
        assert Fraction(float(si)) == round_to_f32(Fraction(float(gi)) / d)


def test_silu_mul_gate_up_order_by_hand():
    """Row layout [gate | up]: silu(20) * 0.5 = 10 exactly; silu(0) * 7 = 0;
    silu(2) * -1 = -2 / (1 + e^-2) = -1.761594... -> BF16 -1.7578125 (spacing
    2^-7 on [1, 2): it lies 0.00378 from -1.7578125 and 0.00403 from
    -1.765625).  Swapping gate and up changes every nonzero entry."""
    g = [20.0, 0.0, 2.0]
    u = [0.5, 7.0, -1.0]
    h = orc.silu_mul(bf16([g + u]), 3)
    assert orc.bf16_to_f32(h).tolist() == [[10.0, 0.0, -1.7578125]]
    swapped = orc.silu_mul(bf16([u + g]), 3)
    assert not np.array_equal(orc.bf16_to_f32(swapped)[0, [0, 2]], orc.bf16_to_f32(h)[0, [0, 2]])


def test_silu_mul_is_the_fp64_value_rounded_once():
    """On data shaped like a gate_up output, h equals the fp64 silu(g) * u
    rounded once to BF16 wherever that value is not within fp32 noise of a
    BF16 rounding midpoint, and is never more than one BF16 step away."""
    rng = np.random.default_rng(61)
    M, inter = 16, 4096
    gu = synth.f32_to_bf16_bits(rng.standard_normal((M, 2 * inter)) * rng.uniform(0.5, 8.0, (M, 1)))
    h = orc.silu_mul(gu, inter)
    g = orc.bf16_to_f32(gu[:, :inter]).astype(np.float64)
    u = orc.bf16_to_f32(gu[:, inter:]).astype(np.float64)
    ref = orc.silu_mul_f64(g, u)
    ref_bits = orc.f64_to_bf16(ref)
    clear = orc.bf16_midpoint_distance(ref) > 1e-6 * np.abs(ref)
    assert clear.mean() > 0.99
    assert np.array_equal(h[clear], ref_bits[clear])
    step = np.abs(orc.bf16_to_f32(h).astype(np.float64) - orc.bf16_to_f32(ref_bits))
    assert np.all(step <= np.spacing(np.abs(orc.bf16_to_f32(ref_bits))) * 65536 + 1e-38)


def test_silu_mul_smooth_quant_is_the_composition():
    """The glue step quantizes h exactly as the activation quantizer does: a
    code of magnitude 127 in every nonzero row, codes * sa within sa/2 of
    fp32(h) * smooth, and a zero gate row gives a zero row."""
    rng = np.random.default_rng(62)
    M, inter = 6, 256
    gu = synth.f32_to_bf16_bits(rng.standard_normal((M, 2 * inter)) * 3.0)
    gu[3, :inter] = 0                     # silu(0) = 0: the whole row of h is 0
    s = rng.uniform(0.25, 4.0, inter).astype(np.float32)
    xq, sa = orc.silu_mul_smooth_quant(gu, inter, s)
    hv = orc.bf16_to_f32(orc.silu_mul(gu, inter)).astype(np.float64) * s[None, :]
    assert sa[3] == 0 and not xq[3].any()
    nz = sa > 0
    assert np.all(np.abs(xq[nz]).max(axis=1) == 127)
    assert np.all(np.abs(xq.astype(np.float64) * sa[:, None] - hv) <= sa[:, None] * (0.5 + 1e-5))


# ------------------------------------------- RMSNorm ahead of qkv (reading R11)

def test_rms_norm_hand_case_intermediate_rounding():
    """x = [3, 4], eps = 0: ss = 25, ms = 12.5, r = fp32(1/sqrt(12.5)).
    t = bf16(3r) = 0.84765625 (3r = 0.848528, spacing 2^-8 on [0.5, 1)),
    bf16(4r) = 1.1328125 (4r = 1.131371, spacing 2^-7).  With gamma = 1.5:
    0.84765625 * 1.5 = 1.271484 -> 1.2734375; 1.1328125 * 1.5 = 1.69921875
    is a tie between 1.6953125 and 1.703125 -> the even 1.703125.  Rounding
    once instead (4r * 1.5 = 1.697056) would give 1.6953125."""
    x = bf16([[3.0, 4.0]])
    assert orc.bf16_to_f32(orc.rms_norm(x, bf16([1.0, 1.0]), 0.0)).tolist() == [[0.84765625, 1.1328125]]
    assert orc.bf16_to_f32(orc.rms_norm(x, bf16([1.5, 1.5]), 0.0)).tolist() == [[1.2734375, 1.703125]]
    r, r64 = orc.rms_inverse(x, 0.0)
    assert Fraction(float(r[0])) == round_to_f32(Fraction(float(r64[0])))
    assert abs(r64[0] - 1.0 / math.sqrt(12.5)) <= 1e-16


def test_rms_inverse_sum_is_correctly_rounded():
    """ss is the exact sum of the squares rounded once: checked with rational
    arithmetic on rows mixing magnitudes 2^-20 .. 2^12 (where a plain fp64
    running sum rounds)."""
    rng = np.random.default_rng(71)
    v = rng.standard_normal((4, 300)) * np.exp2(rng.integers(-20, 12, (4, 300)))
    x = synth.f32_to_bf16_bits(v)
    _, r64 = orc.rms_inverse(x, 0.0)
    for i in range(4):
        exact = sum(Fraction(float(a)) ** 2 for a in orc.bf16_to_f32(x[i]))
        ss = float(exact)                          # Fraction -> float rounds correctly
        assert r64[i] == 1.0 / math.sqrt(ss / 300.0)


def test_rms_norm_scale_invariance_zero_row_and_gamma():
    """With eps = 0 the normalisation ignores the row's scale exactly for
    powers of two; a zero row gives zeros (r = 1/sqrt(eps)); gamma = 2^j
    scales t exactly."""
    rng = np.random.default_rng(72)
    x = synth.f32_to_bf16_bits(rng.standard_normal((5, 64)))
    g = synth.f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(64))
    h = orc.rms_norm(x, g, 0.0)
    for j in (-3, 5):
        xs = synth.f32_to_bf16_bits(orc.bf16_to_f32(x).astype(np.float64) * 2.0 ** j)
        assert np.array_equal(orc.rms_norm(xs, g, 0.0), h)
    z = np.zeros((1, 64), np.uint16)
    assert not orc.bf16_to_f32(orc.rms_norm(z, g, 1e-6)).any()
    ones = bf16(np.ones(64))
    t = orc.rms_norm(x, ones, 0.0)
    assert np.array_equal(orc.bf16_to_f32(orc.rms_norm(x, bf16(np.full(64, 4.0)), 0.0)),
                          orc.bf16_to_f32(t) * 4.0)


def test_rms_norm_close_to_fp64_normalisation():
    """Within two BF16 roundings of x / sqrt(mean(x^2) + eps) * gamma in
    fp64: |h - t*gamma| <= ulp(h)/2 and |gamma| * |t - x*r| <= |gamma| *
    ulp(t)/2 <= ulp(h) (h ~ t*gamma, so ulp(t)*|gamma| <= 2 ulp(h)), 1.5 BF16
    steps in all; equal to it rounded once for most entries."""
    rng = np.random.default_rng(73)
    K = 4096
    x = synth.activations(74, 16, K, synth.outlier_channels(75, K, 41), 30.0)
    g = synth.f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(K))
    h = orc.bf16_to_f32(orc.rms_norm(x, g, 1e-6)).astype(np.float64)
    xv = orc.bf16_to_f32(x).astype(np.float64)
    ref = xv / np.sqrt((xv * xv).mean(axis=1, keepdims=True) + 1e-6) * orc.bf16_to_f32(g).astype(np.float64)[None, :]
    step = np.spacing(np.maximum(np.abs(ref), np.abs(h)).astype(np.float32)).astype(np.float64) * 65536
    assert np.all(np.abs(h - ref) <= 1.51 * step)
    assert np.mean(orc.f64_to_bf16(ref) == orc.f32_to_bf16(h.astype(np.float32))) > 0.7


def test_rms_ambiguous_band():
    """A value on an fp32 rounding midpoint is flagged, one a quarter of the
    spacing away is not, nor is an exact fp32 value."""
    one = 1.0
    mid = one + 2.0 ** -24                      # halfway between 1 and 1 + 2^-23
    flags = orc.rms_ambiguous(np.array([mid, mid * (1 + 2.0 ** -45), one + 2.0 ** -25, 0.75]))
    assert flags.tolist() == [True, True, False, False]


def test_rms_norm_smooth_quant_is_the_composition():
    rng = np.random.default_rng(76)
    x = synth.f32_to_bf16_bits(rng.standard_normal((6, 128)) * 3.0)
    x[2] = 0
    g = synth.f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(128))
    s = rng.uniform(0.25, 4.0, 128).astype(np.float32)
    xq, sa = orc.rms_norm_smooth_quant(x, g, 1e-6, s)
    assert sa[2] == 0 and not xq[2].any()
    assert np.all(np.abs(xq[sa > 0]).max(axis=1) == 127)
