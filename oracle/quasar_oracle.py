"""CPU oracle for the Quasar W8A8 verification path.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this module.  The product library never
calls it, and it shares no code with the CUDA kernels.

Source: "Quasar: Quantized Self-Speculative Acceleration for Rapid Inference
via Memory-Efficient Verification" (arXiv 2603.01399), as summarised on four
gist.science pages (pt, nl, zh, ko).  Citations below name the page language
and its technical-summary section:

  * zh §2 "方法论" / pt §2 "Metodologia": W8A8 verifier; SmoothQuant smoothing
    Y = (W·diag(s)^-1)·(diag(s)·X) with s calibrated offline; offline smooth +
    INT8 weight quantization; online smooth + quantize of the BF16
    activations; INT8 matmul; dequantize to BF16 before the nonlinear layers
    and softmax; rejection sampling on the high-precision logits.
  * pt §2: symmetric uniform quantization of weights and activations.
  * pt §4 / zh §4: greedy (T=0) and sampled (T>0) verification, acceptance
    length.

The pages leave the numeric details open.  The readings taken here are:

  R1  smooth[k] multiplies activations and divides weights (the pages'
      identity), with smooth[k] = max|W[:,k]|^(1-a) / max|X[:,k]|^a, which is
      SmoothQuant's migration factor inverted, so outlier channels shrink.
      a = 0.5.  A channel whose maximum is 0 gets smooth = 1.
  R2  weights: per output channel; activations: per token; symmetric,
      codes in [-127, 127], scale = absmax/127, code = rne(v * (127/absmax)),
      all in fp32 with correctly rounded division and multiplication; a
      zero row gets scale 0 and all-zero codes.
  R3  the INT8 products are accumulated exactly (INT32 on the device).
  R4  dequantization: y = bf16_rne((fp32(acc) * sa[m]) * sw[n]), two fp32
      multiplies in that order, no bias.
  R5  greedy acceptance: draft j is accepted iff it equals the first-index
      argmax of logits row j; the accepted length is the first rejected j
      (or D); the next token is the argmax of row n_acc.
  R6  T > 0: the drafter is deterministic, so draft j is accepted iff
      u[j] < p_j, p_j = softmax(logits_j / T)[draft_j], evaluated in fp64.
  R7  lossless output token (the pages name the rejection sampling lossless
      but do not spell out the correction; this is the standard speculative
      sampling rule with the deterministic drafter of R6, whose
      distribution is one-hot at the draft): at the first rejection j the
      next token is drawn from norm(max(0, p_j - onehot(draft_j))), i.e.
      p_j without the draft token, renormalised; after D acceptances the
      bonus token is drawn from p_D.  Drawn by inverse CDF with one uniform
      u_next per sequence: the smallest v whose cumulative weight exceeds
      u_next times the total; if no weight is left, the lowest index other
      than the draft.
  R8  4-bit weights (the pages' future ultra-low-bit verifier, a kernel
      variant only): per output channel, scale = absmax/7, code =
      clamp(rne(w' * (7/absmax)), -7, 7), in fp32 as R2; activations as R2;
      the same exact integer GEMM and dequantization (R3, R4).
  R9  BF16 lm_head (the verifier's last matmul, which the pages keep in BF16
      ahead of the high-precision acceptance test): logits = the exact
      product H·W^T of the BF16 inputs, rounded once to BF16 (nearest, ties
      to even); acceptance as R5/R6 on those logits.
  R10 the MLP glue between gate_up and down (the pages dequantize to BF16
      before the nonlinear layers; the block then re-smooths and
      re-quantizes for down): h = bf16_rne(silu(g) * u) with g, u the BF16
      gate and up halves of the gate_up output, silu(g) = g / (1 + exp(-g))
      in fp32, one rounding to BF16 at the end.  So that the quantized codes
      of h are a fixed function of the inputs, exp is a stated fp32
      algorithm (Cody and Waite's reduction t = n*ln2 + r with ln2 split in
      a 15-bit head and a tail, then the degree-7 Taylor polynomial of e^r
      by Horner, times 2^n; each step one correctly rounded fp32 operation;
      the argument clamped to [-87, 88]), within 2 fp32 ulp of the true
      exponential.  Then h is smoothed and quantized as R2.
  R11 the RMSNorm ahead of qkv and gate_up, fused with their smooth +
      quantize (the producer of those linears' BF16 input): per token,
      ss = sum_k x_k^2 (each square exact in fp64; the sum correctly
      rounded), r = fp32_rn(1 / sqrt(ss / K + eps)) in fp64 (division,
      square root and division correctly rounded, one rounding to fp32),
      t_k = bf16_rne(x_k * r), h_k = bf16_rne(t_k * gamma_k) in fp32 (the
      usual BF16 RMSNorm: normalise, round to the activation type, apply the
      BF16 weight), then h smoothed and quantized as R2.  A device sums the
      squares in its own order, which can move ss by a few fp64 ulps, so a
      row whose fp64 inverse RMS lies within 2^-38 (relative) of an fp32
      rounding midpoint is ambiguous: compared by count, not bit for bit.

Every function below is pinned by tests under ``tests/`` against hand-derived
values, closed forms, invariants or brute force (see each docstring).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F64 = np.float64
QMAX = 127


# ---------------------------------------------------------------------------
# BF16 helpers (independent of the data generator's copy on purpose).

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> fp32 values (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(F32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> BF16 bits, round to nearest, ties to even (finite inputs).

    Pinned by the BF16 rounding fixtures (257 -> 256, 259 -> 260, ...)."""
    u = np.asarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    keep = u >> 16
    rem = u & 0xFFFF
    up = (rem > 0x8000) | ((rem == 0x8000) & ((keep & 1) == 1))
    return (keep + up.astype(np.uint64)).astype(np.uint16)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> BF16 bits, rounded once (nearest, ties to even; finite inputs
    in the normal range).  Going through fp32 first would round twice.

    Pinned by exact midpoints, a value just above a midpoint that fp32 would
    collapse onto it, and agreement with f32_to_bf16 on fp32 inputs."""
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    r = np.rint(np.ldexp(m, 8))              # 8 significant bits, half to even
    y = np.ldexp(r, e - 8).astype(F32)       # exact: 8 bits fit in fp32
    return (y.view(np.uint32) >> 16).astype(np.uint16)


def bf16_midpoint_distance(x: np.ndarray) -> np.ndarray:
    """|x - nearest rounding midpoint| for BF16 rounding of fp64 x: how far x
    may move before its BF16 value can change.  0 at a midpoint; half the
    spacing at a BF16 number inside a binade; at a power of two 2^p the
    nearest midpoint is the one below, 2^p - 2^(p-9).  Pinned by those cases."""
    x = np.abs(np.asarray(x, dtype=F64))
    _, e = np.frexp(x)                       # x in [2^(e-1), 2^e)
    ulp = np.ldexp(1.0, e - 8)               # BF16 spacing on that binade
    frac = x / ulp - np.floor(x / ulp)
    inside = np.abs(frac - 0.5) * ulp
    below = x - np.ldexp(1.0, e - 1) * (1.0 - 2.0 ** -9)   # midpoint under the binade's first number
    return np.minimum(inside, below)


# ---------------------------------------------------------------------------
# Offline calibration of the smoothing vector (reading R1).

def calibrate_smooth(x_cal_bits: np.ndarray, w_bits: np.ndarray, alpha: float = 0.5) -> np.ndarray:
    """smooth[k] = max_n|W[n,k]|^(1-alpha) / max_m|X[m,k]|^alpha  (fp64, then fp32).

    zh §2: the smoothing factor s is calibrated offline from activation and
    weight statistics; with the pages' identity s multiplies X, so the factor
    that shrinks an outlier channel is the inverse of SmoothQuant's.
    Pinned: hand fixture (max|X|=4, max|W|=9 -> 1.5), degenerate columns -> 1.
    """
    x = bf16_to_f32(x_cal_bits).astype(F64)
    w = bf16_to_f32(w_bits).astype(F64)
    xmax = np.abs(x).max(axis=0)          # per input channel k, over tokens
    wmax = np.abs(w).max(axis=0)          # per input channel k, over output rows
    smooth = np.ones(x.shape[1], dtype=F64)
    ok = (xmax > 0) & (wmax > 0)
    if alpha == 0.5:
        smooth[ok] = np.sqrt(wmax[ok]) / np.sqrt(xmax[ok])
    else:
        smooth[ok] = wmax[ok] ** (1.0 - alpha) / xmax[ok] ** alpha
    return smooth.astype(F32)


# ---------------------------------------------------------------------------
# Symmetric per-row quantizer (reading R2).

def quantize_rows(v: np.ndarray, qmax: int = QMAX):
    """Quantize each row of an fp32 matrix to integer codes with one fp32 scale.

    pt §2: symmetric uniform quantization to 8 bits (qmax = 127; qmax = 7
    for the 4-bit weights of reading R8).  For a row with absmax a > 0:
    scale = a/qmax, code = clamp(rne(v * (qmax/a)), -qmax, qmax).
    Pinned: tie-rounding fixtures, |code*scale - v| <= scale/2 bound, a code
    of magnitude qmax in every nonzero row, zero rows.
    """
    QMAX = qmax
    v = np.asarray(v, dtype=F32)
    amax = np.abs(v).max(axis=1) if v.shape[1] else np.zeros(v.shape[0], F32)
    scale = np.zeros(v.shape[0], dtype=F32)
    codes = np.zeros(v.shape, dtype=np.int8)
    nz = amax > 0
    if nz.any():
        a = amax[nz]
        inv = F32(QMAX) / a                     # one correctly rounded fp32 division
        scale[nz] = a / F32(QMAX)
        q = np.rint(v[nz] * inv[:, None])       # fp32 product, round half to even
        codes[nz] = np.clip(q, -QMAX, QMAX).astype(np.int8)
    return codes, scale


def pack_weights(w_bits: np.ndarray, smooth: np.ndarray):
    """Offline weight preparation: fold diag(smooth)^-1 into W, quantize each
    output channel.  w'[n,k] = fp32(W[n,k]) / smooth[k].

    pt §2 step 1 / zh §2 "离线准备": weights are smoothed and quantized to INT8.
    Returns (Wq int8 [N][K], sw fp32 [N]).
    """
    w = bf16_to_f32(w_bits)
    wp = w / np.asarray(smooth, dtype=F32)[None, :]     # correctly rounded fp32 division
    return quantize_rows(wp)


def pack_weights_w4(w_bits: np.ndarray, smooth: np.ndarray):
    """4-bit weights (reading R8): as pack_weights with codes in [-7, 7],
    sw = absmax / 7.  Returns (Wq int8 [N][K] holding the 4-bit codes, sw)."""
    w = bf16_to_f32(w_bits)
    wp = w / np.asarray(smooth, dtype=F32)[None, :]
    return quantize_rows(wp, qmax=7)


def smooth_quant_act(x_bits: np.ndarray, smooth: np.ndarray):
    """Online activation step: x'[m,k] = fp32(X[m,k]) * smooth[k], then quantize
    each token.  pt §2 step 2 / zh §2 "在线验证".
    Returns (Xq int8 [M][K], sa fp32 [M])."""
    x = bf16_to_f32(x_bits)
    xp = x * np.asarray(smooth, dtype=F32)[None, :]
    return quantize_rows(xp)


# ---------------------------------------------------------------------------
# The MLP glue before down: SiLU(gate) * up, then smooth + quantize (R10).

def _f32_bits(b: int) -> np.float32:
    return np.array([b], dtype=np.uint32).view(F32)[0]


EXP_LOG2E = _f32_bits(0x3FB8AA3B)     # 1/ln2 rounded to fp32
EXP_LN2_HI = _f32_bits(0x3F317200)    # ln2 to 15 significant bits: n * head is exact for |n| < 2^9
EXP_LN2_LO = _f32_bits(0x35BFBE8E)    # ln2 - head, rounded to fp32
# 1/k! rounded to fp32, k = 7 down to 2 (Taylor coefficients of e^r).
EXP_TAYLOR = tuple(_f32_bits(b) for b in (0x39500D01, 0x3AB60B61, 0x3C088889, 0x3D2AAAAB, 0x3E2AAAAB, 0x3F000000))


def exp_f32(t: np.ndarray) -> np.ndarray:
    """The fp32 exponential of reading R10, for t in [-87, 88].

    Cody and Waite, "Software Manual for the Elementary Functions" (1980):
    n = rint(t / ln2), r = (t - n*ln2_head) - n*ln2_tail, then
    e^r = 1 + r(1 + r(1/2! + ... + r/7!)) by Horner and the result p * 2^n,
    every operation rounded to fp32 separately (numpy float32 arithmetic).
    Pinned: within 2 fp32 ulp of the fp64 exponential on a dense grid of the
    range, exactly 1 at 0, and the head/tail split and coefficients checked
    against ln2 and 1/k!."""
    t = np.asarray(t, dtype=F32)
    n = np.rint(t * EXP_LOG2E).astype(F32)
    r = (t - n * EXP_LN2_HI) - n * EXP_LN2_LO
    p = np.full(t.shape, EXP_TAYLOR[0], dtype=F32)
    for c in EXP_TAYLOR[1:] + (F32(1.0), F32(1.0)):
        p = p * r + c
    two_n = ((n.astype(np.int32) + 127).astype(np.uint32) << 23).view(F32)
    return (p * two_n).astype(F32)


def silu_f32(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + exp(-g)) in fp32 with exp_f32 (argument clamped to
    [-87, 88]; beyond 87 the exponential is below 2^-125 and 1 + e = 1)."""
    g = np.asarray(g, dtype=F32)
    t = np.minimum(np.maximum(-g, F32(-87.0)), F32(88.0))
    return g / (F32(1.0) + exp_f32(t))


def silu_mul(gu_bits: np.ndarray, inter: int) -> np.ndarray:
    """h = bf16_rne(silu(g) * u) (reading R10) for gate_up rows laid out as
    [gate (inter values) | up (inter values)].  Returns BF16 bits [M][inter].
    Pinned: gate/up asymmetry by hand, silu(0) = 0, silu(g) = g for large g,
    and agreement with the fp64 SiLU rounded once wherever the fp64 value is
    not within rounding noise of a BF16 midpoint."""
    gu = np.asarray(gu_bits, dtype=np.uint16)
    g = bf16_to_f32(gu[:, :inter])
    u = bf16_to_f32(gu[:, inter:2 * inter])
    return f32_to_bf16(silu_f32(g) * u)


def silu_mul_f64(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g) * u in fp64 (the accuracy yardstick and the calibration glue)."""
    g = np.asarray(g, dtype=F64)
    return g / (1.0 + np.exp(-g)) * np.asarray(u, dtype=F64)


def silu_mul_smooth_quant(gu_bits: np.ndarray, inter: int, smooth: np.ndarray):
    """The MLP glue as one step: h = silu_mul(...), then smooth_quant_act(h)."""
    return smooth_quant_act(silu_mul(gu_bits, inter), smooth)


# ---------------------------------------------------------------------------
# RMSNorm ahead of qkv / gate_up, then smooth + quantize (R11).

def rms_inverse(x_bits: np.ndarray, eps: float):
    """Per row: (r fp32, r64 fp64) with r64 = 1 / sqrt(ss / K + eps) in fp64,
    ss the correctly rounded sum of the exact fp64 squares (math.fsum), and
    r = r64 rounded once to fp32.  Pinned by an exact rational sum and by
    the scale invariance of r under powers of two (eps = 0)."""
    import math
    x = bf16_to_f32(x_bits).astype(F64)
    K = x.shape[1]
    ss = np.array([math.fsum(row) for row in x * x], dtype=F64)
    r64 = 1.0 / np.sqrt(ss / F64(K) + F64(F32(eps)))
    return r64.astype(F32), r64


def rms_ambiguous(r64: np.ndarray, band: float = 2.0 ** -38) -> np.ndarray:
    """Rows whose fp64 inverse RMS lies within `band` (relative) of an fp32
    rounding midpoint, where a few fp64 ulps of summation order could flip
    its fp32 value.  Pinned on a constructed midpoint and a value far from
    one."""
    r64 = np.asarray(r64, dtype=F64)
    m, e = np.frexp(r64)                      # r64 = m * 2^e, 0.5 <= m < 1
    scaled = np.ldexp(m, 24)                  # 24 significant bits: fp32 spacing is 1 here
    dist = np.abs(scaled - np.floor(scaled) - 0.5)
    return dist <= band * scaled


def rms_norm(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float) -> np.ndarray:
    """h = bf16(bf16(x * r) * gamma) per token (reading R11); BF16 bits.
    Pinned: a hand case where the intermediate rounding decides a tie,
    scale invariance (eps = 0), a zero row, gamma = 2^j scaling exactly, and
    agreement with the fp64 normalisation within two BF16 roundings."""
    r, _ = rms_inverse(x_bits, eps)
    t = f32_to_bf16(bf16_to_f32(x_bits) * r[:, None])
    return f32_to_bf16(bf16_to_f32(t) * bf16_to_f32(gamma_bits)[None, :])


def rms_norm_smooth_quant(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float, smooth: np.ndarray):
    """RMSNorm (R11), then smooth_quant_act.  Returns (Xq, sa)."""
    return smooth_quant_act(rms_norm(x_bits, gamma_bits, eps), smooth)


# ---------------------------------------------------------------------------
# INT8 GEMM and dequantization (readings R3, R4).

def int_gemm(xq: np.ndarray, wq: np.ndarray) -> np.ndarray:
    """acc[m,n] = sum_k Xq[m,k] * Wq[n,k], exact, as int64.

    pt §2 step 3: the matmul runs on INT8 operands.  The sum is formed with an
    fp64 matmul: every product and every partial sum is an integer of
    magnitude <= 127*127*K < 2^53, so fp64 represents each one exactly in any
    summation order.  Pinned against brute-force integer loops."""
    acc = np.asarray(xq, dtype=F64) @ np.asarray(wq, dtype=F64).T
    return np.rint(acc).astype(np.int64)


def dequant(acc: np.ndarray, sa: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """Y[m,n] = bf16_rne((fp32(acc[m,n]) * sa[m]) * sw[n]) -> BF16 bits.

    pt §2 step 4: results return to BF16 before the nonlinear layers.
    int -> fp32 is one round-to-nearest-even step (exact through fp64 for
    |acc| < 2^53).  Pinned by the dequant fixtures."""
    return f32_to_bf16(dequant_f32(acc, sa, sw))


def dequant_f32(acc, sa, sw) -> np.ndarray:
    """The fp32 value that dequant() rounds to BF16: (fp32(acc) * sa) * sw."""
    a = np.asarray(acc, dtype=np.int64).astype(F64).astype(F32)
    t = a * np.asarray(sa, dtype=F32)[:, None]
    return t * np.asarray(sw, dtype=F32)[None, :]


def w8a8_linear(xq, sa, wq, sw) -> np.ndarray:
    """The whole verify linear on quantized operands -> BF16 bits."""
    return dequant(int_gemm(xq, wq), sa, sw)


def reference_linear_f64(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """Unquantized Y = X·W^T in fp64 from the BF16 inputs (the accuracy yardstick)."""
    return bf16_to_f32(x_bits).astype(F64) @ bf16_to_f32(w_bits).astype(F64).T


def smoothed_linear_f64(x_bits, w_bits, smooth) -> np.ndarray:
    """(W·diag(s)^-1)(diag(s)·X) in fp64: the pages' identity, zh §2."""
    s = np.asarray(smooth, dtype=F64)
    x = bf16_to_f32(x_bits).astype(F64) * s[None, :]
    w = bf16_to_f32(w_bits).astype(F64) / s[None, :]
    return x @ w.T


# ---------------------------------------------------------------------------
# Verification (readings R5, R6).

def acceptance_probabilities(logits_bits: np.ndarray, draft: np.ndarray, temperature: float) -> np.ndarray:
    """p[b,j] = softmax(logits[b,j,:] / T)[draft[b,j]] in fp64, for j < D.

    zh §2 "无损拒绝采样": rejection sampling on the high-precision logits.
    Pinned by the two-level closed form p = c / (c + V - 1)."""
    lg = bf16_to_f32(logits_bits).astype(F64)
    B, R, V = lg.shape
    D = R - 1
    p = np.zeros((B, D), dtype=F64)
    for b in range(B):
        for j in range(D):
            z = lg[b, j] / temperature
            e = np.exp(z - z.max())
            p[b, j] = e[draft[b, j]] / e.sum()
    return p


def verify_accept(logits_bits: np.ndarray, draft: np.ndarray, temperature: float = 0.0,
                  u: np.ndarray | None = None):
    """Accepted prefix length per sequence (and the greedy next token).

    logits [B][D+1][V] (BF16 bits): row j scores the position drafted as
    draft[b,j]; row D is the bonus position.  T == 0: draft j is accepted iff
    it equals the lowest-index argmax of row j.  T > 0: accepted iff
    u[b,j] < p[b,j].  n_acc[b] = first rejected j, or D.  For T == 0,
    next[b] = argmax of row n_acc[b]; for T > 0 next is -1 (not produced).
    Pinned by hand-built acceptance cases.
    """
    lg = bf16_to_f32(logits_bits)
    B, R, V = lg.shape
    D = R - 1
    n_acc = np.full(B, D, dtype=np.int32)
    nxt = np.full(B, -1, dtype=np.int32)
    p = acceptance_probabilities(logits_bits, draft, temperature) if temperature > 0 else None
    for b in range(B):
        for j in range(D):
            if temperature > 0:
                ok = bool(u[b, j] < p[b, j])
            else:
                ok = int(draft[b, j]) == int(np.argmax(lg[b, j]))
            if not ok:
                n_acc[b] = j
                break
        if temperature == 0:
            nxt[b] = int(np.argmax(lg[b, n_acc[b]]))
    return n_acc, nxt


def lm_head_logits(h_bits: np.ndarray, w_bits: np.ndarray, chunk: int = 8192) -> np.ndarray:
    """logits[r][v] = bf16_rne(sum_k H[r][k] * W[v][k]) (reading R9) -> BF16 bits.

    The products of BF16 numbers are exact in fp64 and the fp64 sum of K of
    them is the exact sum up to fp64 rounding, far below a BF16 spacing; the
    vocabulary is processed in slices of `chunk` rows only to bound memory.
    Pinned by exact rational brute force on tiny inputs and by a closed form
    (weights that select and scale one hidden entry per vocabulary row)."""
    h = bf16_to_f32(h_bits).astype(F64)
    V = w_bits.shape[0]
    out = np.empty((h.shape[0], V), dtype=np.uint16)
    for v0 in range(0, V, chunk):
        w = bf16_to_f32(w_bits[v0:v0 + chunk]).astype(F64)
        out[:, v0:v0 + chunk] = f64_to_bf16(h @ w.T)
    return out


def lm_head_verify(h_bits: np.ndarray, w_bits: np.ndarray, draft: np.ndarray, temperature: float = 0.0,
                   u: np.ndarray | None = None):
    """The lm_head followed by verification: verify_accept on lm_head_logits
    (R9, then R5/R6).  h [B*(D+1)][K] holds row b*(D+1)+j for draft j of
    sequence b (j = D: the bonus position)."""
    B, D = draft.shape
    lg = lm_head_logits(h_bits, w_bits).reshape(B, D + 1, w_bits.shape[0])
    return verify_accept(lg, draft, temperature, u)


def verify_sample(logits_bits: np.ndarray, draft: np.ndarray, temperature: float, u: np.ndarray,
                  u_next: np.ndarray):
    """Accepted prefix length and the lossless next token (readings R6, R7).

    zh §2 "无损拒绝采样" (lossless rejection sampling on the high-precision
    logits).  T > 0.  n_acc as verify_accept; next[b] is drawn from the
    residual of row n_acc[b] (that row's softmax without the rejected draft
    token) or, when every draft was accepted, from the bonus row D, by
    inverse CDF on u_next[b], all in fp64.  Pinned by closed forms (two-level
    rows, explicit CDFs) and by a chi-square test that the emitted token is
    distributed as the target softmax whatever the draft (losslessness).
    """
    assert temperature > 0
    lg = bf16_to_f32(logits_bits).astype(F64)
    B, R, V = lg.shape
    D = R - 1
    n_acc, _ = verify_accept(logits_bits, draft, temperature, u)
    nxt = np.zeros(B, dtype=np.int32)
    for b in range(B):
        j = int(n_acc[b])
        z = lg[b, j] / temperature
        w = np.exp(z - z.max())
        d = int(draft[b, j]) if j < D else -1
        if 0 <= d < V:
            w[d] = 0.0
        total = w.sum()
        if total <= 0.0:
            nxt[b] = 1 if d == 0 else 0
            continue
        cdf = np.cumsum(w)
        nxt[b] = min(int(np.searchsorted(cdf, u_next[b] * total, side="right")), V - 1)
    return n_acc, nxt
