"""GPU parity of the verifier's BF16 lm_head with fused verification
(quasar_lm_head_verify) and of the same kernel writing its logits
(quasar_lm_head_logits), against the CPU oracle: logits are the exact
product of the BF16 inputs rounded once to BF16 (reading R9 of the oracle),
acceptance as quasar_verify_accept (R5 greedy, R6 rejection at T > 0).

Two input families:
  * a dyadic grid (hidden states integers in [-4, 4], weights integers in
    [-32, 32] times 2^-6): every partial sum of a row is a multiple of 2^-6
    below 2^19 of those units, so the tensor cores' fp32 accumulation is exact
    in any order, and logits, argmaxes and accepted lengths must match the
    oracle bit for bit;
  * the workload recipe (H ~ N(0,1), W ~ N(0, 0.02)): the fp32 accumulation
    order inside the tensor cores is unspecified, so each logit must be the
    BF16 rounding of some value within TAU of the exact sum, TAU = 2^-16 *
    sum_k |H[c][k] W[v][k]| (far above fp32 rounding over K/16 accumulation
    steps): between bf16(exact - TAU) and bf16(exact + TAU).  Away from zero
    that is the exact value's rounding or, next to a rounding midpoint, its
    neighbour one BF16 ulp away; near zero (cancellation) the sign may
    differ.  Decisions are compared with the oracle wherever no logit inside
    its interval can alter them, and bit for bit with quasar_verify_accept
    run on this kernel's own logits.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle as orc  # noqa: E402
from tests.gpu_util import dev, dev_bf16, host_bf16_bits  # noqa: E402
from tests.test_gpu_parity import _acc_uniforms, _u_next_midpoints  # noqa: E402
from w8a8_quantized_speculative_gb300 import quasar as q  # noqa: E402
from w8a8_quantized_speculative_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

TAU_REL = 2.0 ** -16
MAX_MISMATCH_FRAC = 1e-2
P_BAND_EXACT = (1e-4, 1e-7)     # |u - p| <= a*p + b is ambiguous (fp32 vs fp64 softmax)
P_BAND_ULP = (5e-2, 1e-6)       # same, when a logit may also move by one BF16 ulp
VOCAB = synth.VOCAB
HID = synth.HIDDEN


def ord16(bits):
    b = np.asarray(bits, dtype=np.int64)
    return np.where(b & 0x8000, (~b) & 0xFFFF, b | 0x8000)


def oracle_logits(h, w, chunk=8192):
    """Oracle logits (BF16 bits) and, per element, the ordered BF16 keys of
    bf16(exact - TAU) and bf16(exact + TAU): the range any fp32 summation
    order within TAU may produce."""
    lg = orc.lm_head_logits(h, w)
    habs = h & np.uint16(0x7FFF)
    lo = np.empty(lg.shape, dtype=np.int32)
    hi = np.empty(lg.shape, dtype=np.int32)
    for v0 in range(0, w.shape[0], chunk):
        ws = w[v0:v0 + chunk]
        ex = orc.reference_linear_f64(h, ws)
        tau = TAU_REL * orc.reference_linear_f64(habs, ws & np.uint16(0x7FFF))
        lo[:, v0:v0 + chunk] = ord16(orc.f64_to_bf16(ex - tau))
        hi[:, v0:v0 + chunk] = ord16(orc.f64_to_bf16(ex + tau))
    return lg, lo, hi


def row_is_clear(key, lo, hi):
    """True when the lowest-index argmax of each row is the same for every
    choice of logits inside their [lo, hi] key ranges."""
    a = np.argmax(key, axis=1)
    R, V = key.shape
    lo_a = lo[np.arange(R), a]
    idx = np.arange(V)[None, :]
    before = np.where(idx < a[:, None], hi, -1).max(axis=1)
    after = np.where(idx > a[:, None], hi, -1).max(axis=1)
    return (before < lo_a) & (after <= lo_a)


def forced_drafts(lg_bits, B, D, seed_draft, seed_mask):
    """Uniform drafts with a Bernoulli(0.5) mask forcing the oracle's argmax."""
    V = lg_bits.shape[-1]
    draft = synth.draft_tokens(seed_draft, B, D, V)
    mask = synth.bernoulli_mask(seed_mask, (B, D))
    am = np.argmax(orc.bf16_to_f32(lg_bits).reshape(B, D + 1, V)[:, :D], axis=2).astype(np.int32)
    return np.where(mask, am, draft).astype(np.int32)


def run_verify(h, w, draft, T=0.0, u=None, ldh=None):
    B, D = draft.shape
    h_d = dev_bf16(h)
    if ldh is not None:
        wide = torch.zeros(h.shape[0], ldh, dtype=torch.bfloat16, device="cuda")
        wide[:, :h.shape[1]] = h_d
        h_d = wide[:, :h.shape[1]]
    ws = q.Workspace()
    n_acc, nxt = q.lm_head_verify(h_d, q.pack_lm_head(dev_bf16(w)), dev(draft), T, None if u is None else dev(u),
                                  workspace=ws)
    torch.cuda.synchronize()
    assert q.get_device_error()[0] == q.OK
    assert not ws.buf.any().item(), "the workspace must be left zero-filled"
    return n_acc.cpu().numpy(), (None if nxt is None else nxt.cpu().numpy())


# ------------------------------------------------------------- packing

def unpack_lm_head(buf: np.ndarray, V: int, K: int) -> np.ndarray:
    """[V][K] BF16 bits from the packed layout documented in include/quasar.h:
    16 KB blocks (tile t, K block kb) at (t*KB + kb) * 16384, row r at r*128,
    its 16-byte chunk c at chunk position c ^ (r % 8)."""
    KB, T = -(-K // 64), -(-V // 128)
    blk = buf.view(np.uint16).reshape(T, KB, 128, 8, 8)        # [t][kb][row][pos][8 values]
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    rows = blk[:, :, r, c ^ (r & 7), :]                         # chunk c of row r
    full = rows.transpose(0, 2, 1, 3, 4).reshape(T * 128, KB * 64)
    return full[:V, :K], full


@pytest.mark.parametrize("V,K", [(1000, 200), (128, 64), (300, 72), (VOCAB, HID)])
def test_pack_layout(V, K):
    w = synth.grid_lm_head_weight(661, V, K) if V < VOCAB else synth.lm_head_weight(505, V, K)
    wp = q.pack_lm_head(dev_bf16(w))
    assert wp.buf.numel() == -(-V // 128) * -(-K // 64) * 16384
    got, full = unpack_lm_head(wp.buf.cpu().numpy(), V, K)
    assert np.array_equal(got, w)
    pad = full.copy()
    pad[:V, :K] = 0
    assert not pad.any(), "rows past V and K values past K must be zero"


# ------------------------------------------------------------- logits

@pytest.mark.parametrize("M,V,K", [(1, 1, 8), (3, 5, 8), (17, 130, 16), (1, 1000, 200), (20, 1000, 200),
                                   (32, 2048, 64), (256, 20000, 128),
                                   (257, 40000, 256), (300, 40000, 512), (512, 40000, 256)])
def test_logits_grid_bit_exact(M, V, K):
    h = synth.grid_hidden_states(601 + M, M, K)
    w = synth.grid_lm_head_weight(602 + V, V, K)
    got = host_bf16_bits(q.lm_head_logits(dev_bf16(h), q.pack_lm_head(dev_bf16(w))))
    want = orc.lm_head_logits(h, w)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} logits differ, first at {bad[:3].tolist()}"


@pytest.mark.parametrize("M,V,K", [(20, 1000, 200), (300, 40000, 512)])
def test_logits_recipe_within_one_ulp(M, V, K):
    h = synth.hidden_states(611, M, K)
    w = synth.lm_head_weight(612, V, K)
    _check_recipe_logits(h, w, host_bf16_bits(q.lm_head_logits(dev_bf16(h), q.pack_lm_head(dev_bf16(w)))))


def _check_recipe_logits(h, w, got, pre=None):
    want, lo, hi = oracle_logits(h, w) if pre is None else pre
    k = ord16(got)
    out = (k < lo) | (k > hi)
    assert not out.any(), f"{out.sum()} logits outside bf16(exact -/+ TAU), first at {np.argwhere(out)[:3].tolist()}"
    off = k != ord16(want)
    assert off.mean() <= MAX_MISMATCH_FRAC, f"{off.mean():.4f} of the logits differ from the oracle's"
    ex = np.concatenate([orc.reference_linear_f64(h, w[v0:v0 + 8192]) for v0 in range(0, w.shape[0], 8192)],
                        axis=1)
    rel = np.linalg.norm(orc.bf16_to_f32(got) - ex) / np.linalg.norm(ex)
    assert rel <= 2.0 ** -8


def test_logits_strided_rows_and_empty():
    M, V, K = 40, 3000, 192
    h = synth.grid_hidden_states(621, M, K)
    w = synth.grid_lm_head_weight(622, V, K)
    wide = torch.zeros(M, K + 72, dtype=torch.bfloat16, device="cuda")
    wide[:, :K] = dev_bf16(h)
    out = torch.full((M, V + 40), 7.0, dtype=torch.bfloat16, device="cuda")
    q.lm_head_logits(wide[:, :K], q.pack_lm_head(dev_bf16(w)), logits=out[:, :V])
    got = host_bf16_bits(out)
    assert np.array_equal(got[:, :V], orc.lm_head_logits(h, w))
    assert np.all(orc.bf16_to_f32(got[:, V:]) == 7.0), "columns past V must not be written"
    empty = torch.empty(0, V, dtype=torch.bfloat16, device="cuda")
    q.lm_head_logits(torch.empty(0, K, dtype=torch.bfloat16, device="cuda"), q.pack_lm_head(dev_bf16(w)),
                     logits=empty)
    torch.cuda.synchronize()


# ------------------------------------------------------------- fused verification, exact grid

@pytest.mark.parametrize("B,D,V,K", [(3, 5, 40000, 512), (4, 0, 5000, 128), (1, 7, 1000, 200), (2, 2, 5, 8),
                                     (1, 0, 1, 8),
                                     (51, 9, 40000, 256), (32, 8, VOCAB, HID)])
def test_fused_greedy_grid_matches_oracle(B, D, V, K):
    h = synth.grid_hidden_states(631 + B, B * (D + 1), K)
    w = synth.grid_lm_head_weight(632 + V, V, K)
    lg = orc.lm_head_logits(h, w)
    draft = forced_drafts(lg, B, D, 633, 634)
    n_acc, nxt = run_verify(h, w, draft, ldh=K + 64 if B == 3 else None)
    want_n, want_next = orc.verify_accept(lg.reshape(B, D + 1, V), draft)
    assert np.array_equal(n_acc, want_n)
    assert np.array_equal(nxt, want_next)


@pytest.mark.parametrize("B,D,V,K,T", [(3, 5, 40000, 512, 40.0), (32, 8, VOCAB, HID, 60.0)])
def test_fused_sampled_grid_matches_oracle(B, D, V, K, T):
    h = synth.grid_hidden_states(641 + B, B * (D + 1), K)
    w = synth.grid_lm_head_weight(642 + V, V, K)
    lg = orc.lm_head_logits(h, w)
    draft = forced_drafts(lg, B, D, 643, 644)
    p = orc.acceptance_probabilities(lg.reshape(B, D + 1, V), draft, T)
    # uniforms spread over [0, 2p]: about half the drafts pass, none near the boundary
    u = (synth.uniforms(645, (B, D)).astype(np.float64) * 2.0 * p).astype(np.float32)
    amb = np.abs(u.astype(np.float64) - p) <= P_BAND_EXACT[0] * p + P_BAND_EXACT[1]
    u = np.where(amb, np.float32(0.0), u).astype(np.float32)      # u = 0 always accepts when p > 0
    n_acc, nxt = run_verify(h, w, draft, T, u)
    assert nxt is None
    want_n, _ = orc.verify_accept(lg.reshape(B, D + 1, V), draft, T, u)
    assert np.array_equal(n_acc, want_n)
    assert 0 < want_n.mean() < D, "the case should accept some drafts and reject others"


@pytest.mark.parametrize("B,D,V,K,T", [(3, 5, 40000, 512, 40.0), (4, 0, 5000, 128, 20.0), (6, 2, 1000, 200, 8.0),
                                       (32, 8, VOCAB, HID, 60.0)])
def test_fused_sample_next_grid_matches_oracle(B, D, V, K, T):
    """The lossless next token of the fused path against the oracle's
    verify_sample on the same (exact) logits, u_next at the middle of a
    token's interval."""
    h = synth.grid_hidden_states(671 + B, B * (D + 1), K)
    w = synth.grid_lm_head_weight(672 + V, V, K)
    lg = orc.lm_head_logits(h, w).reshape(B, D + 1, V)
    draft = forced_drafts(lg, B, D, 673, 674)
    u = _acc_uniforms(lg, draft, T, 675) if D else np.zeros((B, 0), np.float32)
    n_r, _ = orc.verify_accept(lg, draft, T, u)
    u_next = _u_next_midpoints(lg, draft, T, n_r, np.random.default_rng(676))
    ws = q.Workspace()
    n_acc, nxt = q.lm_head_verify_sample(dev_bf16(h), q.pack_lm_head(dev_bf16(w)), dev(draft), T,
                                         dev(u) if D else None, dev(u_next), workspace=ws)
    torch.cuda.synchronize()
    assert q.get_device_error()[0] == q.OK
    assert not ws.buf.any().item(), "the workspace must be left zero-filled"
    n_o, nxt_o = orc.verify_sample(lg, draft, T, u, u_next.astype(np.float64))
    assert np.array_equal(n_acc.cpu().numpy(), n_o)
    assert np.array_equal(nxt.cpu().numpy(), nxt_o)
    if D:
        assert 0 < n_o.mean() < D or B < 4


def test_fused_sample_next_recipe_matches_unfused(recipe_c5):
    """On the workload recipe the fused draw equals verify_sample run on the
    same kernel's logits (u_next at interval midpoints of those logits)."""
    B, D, h, w, lg, lo, hi, draft = recipe_c5
    V = w.shape[0]
    T = 1.0
    wp = q.pack_lm_head(dev_bf16(w))
    lg_gpu = q.lm_head_logits(dev_bf16(h), wp)
    lg_bits = host_bf16_bits(lg_gpu).reshape(B, D + 1, V)
    u = _acc_uniforms(lg_bits, draft, T, 677)
    n_g, _ = orc.verify_accept(lg_bits, draft, T, u)
    u_next = _u_next_midpoints(lg_bits, draft, T, n_g, np.random.default_rng(678))
    n1, x1 = q.lm_head_verify_sample(dev_bf16(h), wp, dev(draft), T, dev(u), dev(u_next))
    n2, x2 = q.verify_sample(lg_gpu.view(B, D + 1, V), dev(draft), T, dev(u), dev(u_next))
    assert np.array_equal(n1.cpu().numpy(), n2.cpu().numpy())
    assert np.array_equal(x1.cpu().numpy(), x2.cpu().numpy())


def test_fused_empty_batch():
    w = q.pack_lm_head(dev_bf16(synth.grid_lm_head_weight(651, 1000, 64)))
    h = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    n_acc, nxt = q.lm_head_verify(h, w, torch.empty(0, 3, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert n_acc.numel() == 0 and nxt.numel() == 0


# ------------------------------------------------------------- the workload recipe at full size

@pytest.fixture(scope="module")
def recipe_c5():
    """Verification step of the workload: 32 sequences x (8 drafts + 1)
    hidden states, Qwen3-8B lm_head 4096 -> 151936."""
    B, D = 32, 8
    h = synth.hidden_states(506, B * (D + 1), HID)
    w = synth.lm_head_weight(505, VOCAB, HID)
    lg, lo, hi = oracle_logits(h, w)
    draft = forced_drafts(lg, B, D, 502, 503)
    return B, D, h, w, lg, lo, hi, draft


def test_recipe_logits_full_vocab(recipe_c5):
    B, D, h, w, lg, lo, hi, draft = recipe_c5
    got = host_bf16_bits(q.lm_head_logits(dev_bf16(h), q.pack_lm_head(dev_bf16(w))))
    _check_recipe_logits(h, w, got, (lg, lo, hi))


def test_recipe_fused_greedy(recipe_c5):
    B, D, h, w, lg, lo, hi, draft = recipe_c5
    V = w.shape[0]
    n_acc, nxt = run_verify(h, w, draft)
    # bit for bit against the unfused GPU path on this kernel's own logits
    lg_gpu = q.lm_head_logits(dev_bf16(h), q.pack_lm_head(dev_bf16(w))).view(B, D + 1, V)
    n2, x2 = q.verify_accept(lg_gpu, dev(draft))
    assert np.array_equal(n_acc, n2.cpu().numpy()) and np.array_equal(nxt, x2.cpu().numpy())
    # against the oracle wherever no logit inside its interval can change a decision
    want_n, want_next = orc.verify_accept(lg.reshape(B, D + 1, V), draft)
    clear = row_is_clear(ord16(lg), lo, hi).reshape(B, D + 1)
    comparable = np.array([clear[b, :want_n[b] + 1].all() for b in range(B)])
    assert comparable.mean() >= 0.75, f"only {comparable.sum()} of {B} sequences are unambiguous"
    assert np.array_equal(n_acc[comparable], want_n[comparable])
    assert np.array_equal(nxt[comparable], want_next[comparable])
    assert want_n.mean() > 0.5, "half of the drafts are forced to the argmax"


def test_recipe_fused_sampled(recipe_c5):
    B, D, h, w, lg, lo, hi, draft = recipe_c5
    V = w.shape[0]
    T = 1.0
    u = synth.uniforms(504, (B, D))
    n_acc, _ = run_verify(h, w, draft, T, u)
    p = orc.acceptance_probabilities(lg.reshape(B, D + 1, V), draft, T)
    want_n, _ = orc.verify_accept(lg.reshape(B, D + 1, V), draft, T, u)
    amb = np.abs(u.astype(np.float64) - p) <= P_BAND_ULP[0] * p + P_BAND_ULP[1]
    comparable = np.array([not amb[b, :min(want_n[b] + 1, D)].any() for b in range(B)])
    assert comparable.mean() >= 0.9
    assert np.array_equal(n_acc[comparable], want_n[comparable])
