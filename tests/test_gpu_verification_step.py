"""GPU test of the workload's verification step as the benchmark runs it:
32 sequences x (8 drafts + 1) = 288 token rows through four Qwen3-8B-shaped
decoder layers (RMSNorm and SiLU * up fused into this library's quantizers,
the W8A8 linears, attention and residual adds in torch BF16), the final
RMSNorm and the fused BF16 lm_head + acceptance.  The accepted prefix length
of every sequence, greedy and by rejection sampling at T = 1, must equal the
oracle's acceptance rule applied to the same hidden states' logits (the
lm_head kernel's logits mode): bit for bit for greedy (and the next token),
and at T = 1 wherever the decision is not within the fp32 / fp64 softmax band
(reading R11 of the pages: |u - p| <= 1e-4 p + 1e-9 counts as ambiguous)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402
import oracle as orc  # noqa: E402
from w8a8_quantized_speculative_gb300 import quasar as q  # noqa: E402

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def step():
    vs = bench.VerificationStep(q, torch.device("cuda", 0))
    lg = vs.logits_ours()
    vs.set_drafts(lg)
    torch.cuda.synchronize()
    yield vs, _bits(lg), vs.draft.cpu().numpy()
    del vs
    torch.cuda.empty_cache()


def _sampled_agree(lg, d, u, n_gpu, T=1.0):
    p = orc.acceptance_probabilities(lg, d, T)
    n_r, _ = orc.verify_accept(lg, d, T, u)
    B, D = d.shape
    ambiguous = 0
    for b in range(B):
        last = min(int(n_r[b]), D - 1)
        if np.any(np.abs(u[b, :last + 1].astype(np.float64) - p[b, :last + 1]) <= 1e-4 * p[b, :last + 1] + 1e-9):
            ambiguous += 1
            continue
        assert int(n_gpu[b]) == int(n_r[b]), b
    return ambiguous


def test_greedy_matches_oracle_on_same_logits(step):
    vs, lg, d = step
    n_acc, nxt = vs.step_ours(0.0)
    n_r, nxt_r = orc.verify_accept(lg, d, 0.0)
    assert np.array_equal(n_acc.cpu().numpy(), n_r)
    assert np.array_equal(nxt.cpu().numpy(), nxt_r)
    # half the drafts are forced to the greedy choice: some sequences accept
    assert n_r.max() > 0


def test_shared_workspace_gives_the_same_logits(step):
    """One workspace for every call of the chain (the one-call linear leaves
    its codes after its zero-filled part; the binding clears what a later,
    larger linear needs) gives the same logits as separate workspaces."""
    vs, lg, d = step
    sep = vs.ws_f
    vs.ws_f = vs.ws
    try:
        shared = _bits(vs.logits_ours())
    finally:
        vs.ws_f = sep
    assert np.array_equal(shared.reshape(lg.shape), lg)


def test_rejection_sampling_t1_matches_oracle(step):
    vs, lg, d = step
    n_acc, _ = vs.step_ours(1.0)
    assert _sampled_agree(lg, d, vs.u.cpu().numpy(), n_acc.cpu().numpy()) == 0


def test_rejection_sampling_t1_with_acceptances(step):
    """The same chain at T = 1 with uniforms placed away from p (0.5 p to
    accept on 80% of the positions, p + 0.5 (1 - p) to reject), so that long
    accepted prefixes occur and every position's decision is checked."""
    vs, lg, d = step
    p = orc.acceptance_probabilities(lg, d, 1.0)
    acc = np.random.default_rng(506).random(d.shape) < 0.8
    u = np.where(acc, 0.5 * p, p + 0.5 * (1 - p)).astype(np.float32)
    saved = vs.u.clone()
    vs.u.copy_(torch.from_numpy(u))
    try:
        n_acc, _ = vs.step_ours(1.0)
        n_gpu = n_acc.cpu().numpy()
    finally:
        vs.u.copy_(saved)
    assert _sampled_agree(lg, d, u, n_gpu) == 0
    assert n_gpu.max() >= 3
    st, site = q.get_device_error()
    assert st == 0, site
