"""Seeded synthetic inputs for the W8A8 verify path.

This module only draws random numbers and lays them out as the workloads
described on the Quasar summary pages (Qwen3-8B-shaped linears, drafted
tokens, uniforms for the rejection test).  It holds none of the method's
arithmetic: no smoothing, no quantization, no matmul, no acceptance rule.
Both the CPU oracle and the CUDA path consume exactly the bytes it returns.

Every array is produced from ``numpy.random.Generator(PCG64(seed))`` so that
a (seed, shape) pair always yields the same bytes on any machine running the
same numpy release.

BF16 tensors are returned as ``uint16`` bit patterns: values are drawn in
fp64, narrowed to fp32, then rounded to BF16 (round to nearest even on the 16
dropped bits).  This is data preparation only.
"""
from __future__ import annotations

import numpy as np

# Qwen3-8B shapes used by the workloads: (in_features K, out_features N).
HIDDEN = 4096
KV_DIM = 1024
INTERMEDIATE = 12288
VOCAB = 151936

LINEARS = {
    "qkv": (HIDDEN, HIDDEN + 2 * KV_DIM),      # fused q/k/v: 4096 -> 6144
    "o": (HIDDEN, HIDDEN),                     # 4096 -> 4096
    "gate_up": (HIDDEN, 2 * INTERMEDIATE),     # fused gate/up: 4096 -> 24576
    "down": (INTERMEDIATE, HIDDEN),            # 12288 -> 4096
}

M_SWEEP = (1, 2, 4, 8, 16, 32, 64, 128, 256)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to BF16 (nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to fp32 (exact)."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def outlier_channels(seed: int, K: int, count: int) -> np.ndarray:
    """Sorted indices of ``count`` distinct input channels that carry outliers."""
    return np.sort(_rng(seed).choice(K, size=count, replace=False)).astype(np.int64)


def outlier_count(K: int, frac: float = 0.01) -> int:
    """Number of outlier channels for a fraction of K (1% of 4096 -> 41)."""
    return int(round(frac * K))


def activations(seed: int, M: int, K: int, outliers: np.ndarray | None = None,
                scale: float = 1.0) -> np.ndarray:
    """BF16 activations X[M][K] ~ N(0,1), with the ``outliers`` columns x ``scale``."""
    x = _rng(seed).standard_normal((M, K))
    if outliers is not None and len(outliers):
        x[:, outliers] *= scale
    return f32_to_bf16_bits(x.astype(np.float32))


def weights(seed: int, N: int, K: int, std: float = 0.02) -> np.ndarray:
    """BF16 weights W[N][K] ~ N(0, std^2), row-major (K contiguous)."""
    w = _rng(seed).standard_normal((N, K)) * std
    return f32_to_bf16_bits(w.astype(np.float32))


def logits(seed: int, rows: int, V: int, std: float = 1.0) -> np.ndarray:
    """BF16 logits[rows][V] ~ N(0, std^2)."""
    return f32_to_bf16_bits((_rng(seed).standard_normal((rows, V)) * std).astype(np.float32))


def draft_tokens(seed: int, B: int, D: int, V: int) -> np.ndarray:
    """Drafted token ids, uniform over [0, V), int32 [B][D]."""
    return _rng(seed).integers(0, V, size=(B, D), dtype=np.int64).astype(np.int32)


def bernoulli_mask(seed: int, shape, p: float = 0.5) -> np.ndarray:
    """Boolean mask with P(True) = p."""
    return _rng(seed).random(shape) < p


def uniforms(seed: int, shape) -> np.ndarray:
    """fp32 uniforms in [0, 1) for the rejection test."""
    u = _rng(seed).random(shape).astype(np.float32)
    # fp64 -> fp32 rounding can produce exactly 1.0; keep the half-open range.
    return np.minimum(u, np.float32(np.nextafter(np.float32(1.0), np.float32(0.0))))


# ---------------------------------------------------------------------------
# Workload recipes (shapes, seeds and value distributions only).

class LinearCase:
    """One W8A8 linear's synthetic inputs: run batch X, calibration batch, W."""

    def __init__(self, name: str, M: int, K: int, N: int, seeds, outlier_frac: float,
                 outlier_scale: float, cal_tokens: int, n_outliers: int | None = None):
        self.name, self.M, self.K, self.N = name, M, K, N
        self.seed_x, self.seed_w, self.seed_cal, self.seed_idx = seeds
        self.outlier_scale = outlier_scale
        self.cal_tokens = cal_tokens
        self.n_outliers = n_outliers if n_outliers is not None else outlier_count(K, outlier_frac)

    def outliers(self) -> np.ndarray:
        return outlier_channels(self.seed_idx, self.K, self.n_outliers)

    def x(self) -> np.ndarray:
        return activations(self.seed_x, self.M, self.K, self.outliers(), self.outlier_scale)

    def x_cal(self) -> np.ndarray:
        return activations(self.seed_cal, self.cal_tokens, self.K, self.outliers(), self.outlier_scale)

    def w(self) -> np.ndarray:
        return weights(self.seed_w, self.N, self.K)


def small_case() -> LinearCase:
    """Single linear, CPU-fast: M=8 (1 sequence x (7 drafts + 1)), K=256, N=512,
    4 outlier channels x50, 64-token calibration batch."""
    return LinearCase("small", 8, 256, 512, (101, 102, 103, 104), 0.0, 50.0, 64, n_outliers=4)


def attention_cases(M: int = 20):
    """Qwen3-8B attention projections at M = 4 x (4 + 1) = 20 tokens:
    fused qkv 4096->6144 and o_proj 4096->4096; 1% outlier channels x30."""
    out = []
    for i, name in enumerate(("qkv", "o")):
        K, N = LINEARS[name]
        out.append(LinearCase(name, M, K, N, (201 + 10 * i, 202 + 10 * i, 203 + 10 * i, 204 + 10 * i),
                              0.01, 30.0, 512))
    return out


def mlp_cases(M: int = 40):
    """Qwen3-8B MLP block at M = 8 x (4 + 1) = 40: fused gate/up 4096->24576,
    down 12288->4096."""
    out = []
    for i, name in enumerate(("gate_up", "down")):
        K, N = LINEARS[name]
        out.append(LinearCase(name, M, K, N, (301 + 10 * i, 302 + 10 * i, 303 + 10 * i, 304 + 10 * i),
                              0.01, 30.0, 512))
    return out


def sweep_case(name: str, M: int) -> LinearCase:
    """One decoder-layer linear of the M sweep (M in 1..256)."""
    K, N = LINEARS[name]
    i = list(LINEARS).index(name)
    return LinearCase(name, M, K, N, (401 + 10 * i, 402 + 10 * i, 403 + 10 * i, 404 + 10 * i),
                      0.01, 30.0, 512)


def verify_inputs(B: int, D: int, V: int, seed_logits: int = 501, seed_draft: int = 502,
                  seed_mask: int = 503, seed_u: int = 504, std: float = 1.0):
    """Logits [B][D+1][V] (BF16 bits), uniform drafts [B][D], a Bernoulli(0.5)
    mask of positions whose draft is to be forced to the target's choice, and
    uniforms u [B][D].  The caller applies the mask (it needs the argmax)."""
    lg = logits(seed_logits, B * (D + 1), V, std).reshape(B, D + 1, V)
    return (lg, draft_tokens(seed_draft, B, D, V), bernoulli_mask(seed_mask, (B, D)),
            uniforms(seed_u, (B, D)))


# ---------------------------------------------------------------------------
# The verifier's BF16 lm_head (hidden states -> logits over the vocabulary).

def hidden_states(seed: int, rows: int, K: int) -> np.ndarray:
    """BF16 final hidden states H[rows][K] ~ N(0,1) (an RMS-normalised
    activation with unit gain)."""
    return f32_to_bf16_bits(_rng(seed).standard_normal((rows, K)).astype(np.float32))


def _bf16_inplace(a: np.ndarray) -> np.ndarray:
    """fp32 -> BF16 bits (nearest, ties to even) for finite values, in 32-bit
    arithmetic on the array's own storage (large weight slices)."""
    b = a.view(np.uint32)
    b += np.uint32(0x7FFF) + ((b >> 16) & np.uint32(1))
    return (b >> 16).astype(np.uint16)


def _sliced(seed: int, V: int, K: int, chunk: int, draw) -> np.ndarray:
    """A [V][K] BF16 matrix drawn slice by slice of ``chunk`` rows, slice i
    from its own generator PCG64(SeedSequence(seed).spawn(n)[i]); slices are
    drawn on a thread pool (the bytes do not depend on the thread count)."""
    from concurrent.futures import ThreadPoolExecutor
    n_sl = (V + chunk - 1) // chunk
    seqs = np.random.SeedSequence(seed).spawn(n_sl)
    out = np.empty((V, K), dtype=np.uint16)

    def job(i):
        v0 = i * chunk
        n = min(chunk, V - v0)
        out[v0:v0 + n] = _bf16_inplace(draw(np.random.Generator(np.random.PCG64(seqs[i])), n))

    with ThreadPoolExecutor(max_workers=8) as ex:
        list(ex.map(job, range(n_sl)))
    return out


def lm_head_weight(seed: int, V: int, K: int, std: float = 0.02, chunk: int = 8192) -> np.ndarray:
    """BF16 lm_head weight W[V][K] ~ N(0, std^2), drawn directly in fp32
    (``standard_normal(dtype=float32)``) slice by slice: the Qwen3-8B
    vocabulary makes it 622 M values."""
    def draw(g, n):
        x = g.standard_normal((n, K), dtype=np.float32)
        x *= np.float32(std)
        return x
    return _sliced(seed, V, K, chunk, draw)


def grid_hidden_states(seed: int, rows: int, K: int, amp: int = 4) -> np.ndarray:
    """BF16 hidden states on an integer grid: uniform integers in [-amp, amp]."""
    return f32_to_bf16_bits(_rng(seed).integers(-amp, amp + 1, size=(rows, K)).astype(np.float32))


def grid_lm_head_weight(seed: int, V: int, K: int, amp: int = 32, shift: int = 6,
                        chunk: int = 8192) -> np.ndarray:
    """BF16 lm_head weight on a dyadic grid: uniform integers in [-amp, amp]
    times 2^-shift.  With grid_hidden_states every product is a multiple of
    2^-shift and, for K up to 4096, every partial sum of a row stays below
    2^19 of those units, so any fp32 summation order gives the exact sum."""
    def draw(g, n):
        x = g.integers(-amp, amp + 1, size=(n, K), dtype=np.int16).astype(np.float32)
        x *= np.float32(2.0 ** -shift)
        return x
    return _sliced(seed, V, K, chunk, draw)
