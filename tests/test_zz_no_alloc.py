"""GPU test of quasar_w8a8_linear_noalloc, the W8A8 linear for callers that
cannot give the library a workspace (for example code hosted in another
runtime's plugin interface that owns all device memory, or serving loops that
may not allocate once running).  Its split-K scratch is a fixed array inside
the library, so the test checks, through the C ABI, that two calls in a row
give bit for bit the BF16 output of the workspace-taking quasar_w8a8_linear
(both dispatch to the same deterministic kernels: the register-path kernel for
a few tokens, the tcgen05 kernel above), that the device error word stays
clear, and that sizes beyond the fixed array are refused.

Kept in a file of its own that pytest collects last; it needs no state from
the other tests and also runs alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from tests.gpu_util import dev_bf16, host_bf16_bits  # noqa: E402
from w8a8_quantized_speculative_gb300 import quasar as q  # noqa: E402
from w8a8_quantized_speculative_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

QUASAR_ERR_WORKSPACE = 3
SCRATCH = 8 << 20   # QUASAR_NOALLOC_SCRATCH_BYTES


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _prepared(case):
    x, w, xc = case.x(), case.w(), case.x_cal()
    smooth = q.calibrate_smooth(dev_bf16(xc), dev_bf16(w))
    wp, sw = q.pack_weights(dev_bf16(w), smooth)
    xq, sa = q.smooth_quant_act(dev_bf16(x), smooth)
    return xq, sa, wp, sw


def _noalloc(xq, sa, wp, sw, y):
    M, K = xq.shape
    N = sw.numel()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return q.lib.quasar_w8a8_linear_noalloc(_p(xq), _p(sa), _p(wp), _p(sw), M, N, K, _p(y), y.stride(0), stream)


def _check_twice(case):
    """Two no-alloc calls in a row against the workspace entry point: equal
    output bits each time, and no device-side error."""
    xq, sa, wp, sw = _prepared(case)
    want = host_bf16_bits(q.w8a8_linear(xq, sa, wp, sw, workspace=q.Workspace()))
    for _ in range(2):
        got = torch.full((case.M, case.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(xq, sa, wp, sw, got) == 0
        torch.cuda.synchronize()
        assert np.array_equal(host_bf16_bits(got), want), case.name
    st, site = q.get_device_error()
    assert st == 0, site


def test_noalloc_matches_workspace_entry_point_twice():
    # qkv then o_proj at M = 20 (register-path kernel)
    for case in synth.attention_cases():
        _check_twice(case)


@pytest.mark.parametrize("M", [40, 64])
def test_noalloc_tcgen05_branch(M):
    # qkv (N = 6144, K = 4096) above 32 tokens: the tcgen05 kernel's split-K
    # counters and int32 sums live in the fixed array (about 1.6 MB at M = 64)
    case = synth.sweep_case("qkv", M)
    assert q.lib.quasar_w8a8_linear_workspace_size(M, case.N, case.K) <= SCRATCH
    _check_twice(case)


@pytest.mark.parametrize("name", ["qkv", "o"])
def test_noalloc_register_path_four_token_tiles(name):
    # M = 32 on a layer of <= 8192 rows: the register-path kernel with four
    # token tiles, whose partial-sum slots (5.2 MB) need the larger array
    case = synth.sweep_case(name, 32)
    assert q.lib.quasar_w8a8_linear_workspace_size(32, case.N, case.K) <= SCRATCH
    _check_twice(case)


def test_noalloc_repeated_call_same_layer():
    _check_twice(synth.small_case())


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch():
    M, N, K = 256, 24576, 4096          # needs ~25 MB of split-K scratch
    assert q.lib.quasar_w8a8_linear_workspace_size(M, N, K) > SCRATCH
    xq = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sa = torch.zeros(M, device="cuda")
    wp = torch.zeros(16, dtype=torch.int8, device="cuda")   # never read: the call is refused first
    sw = torch.zeros(N, device="cuda")
    y = torch.zeros((1, N), dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = q.lib.quasar_w8a8_linear_noalloc(_p(xq), _p(sa), _p(wp), _p(sw), M, N, K, _p(y), N, stream)
    assert rc == QUASAR_ERR_WORKSPACE
