"""Host-only checks of the C ABI: the library builds and loads without a GPU,
exports every function include/quasar.h declares, and rejects bad arguments
on the host before touching CUDA.  No compute call is made here."""
import ctypes
import os
import re

import pytest

from w8a8_quantized_speculative_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = build.build_library()
    return ctypes.CDLL(path)


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(quasar_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("quasar_pack_weights", "quasar_smooth_quant_act", "quasar_w8a8_linear", "quasar_verify_accept",
                 "quasar_calibrate_smooth", "quasar_int8_gemm_s32", "quasar_get_device_error"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.quasar_status_string.restype = ctypes.c_char_p
    assert lib.quasar_status_string(0) == b"ok"
    assert b"timed out" in lib.quasar_status_string(5)
    assert lib.quasar_status_string(99) == b"unknown status"
    assert lib.quasar_version() >> 16 == 1


def test_workspace_sizes(lib):
    lib.quasar_w8a8_linear_workspace_size.restype = ctypes.c_size_t
    lib.quasar_verify_accept_workspace_size.restype = ctypes.c_size_t
    lib.quasar_calibrate_workspace_size.restype = ctypes.c_size_t
    ws = lib.quasar_w8a8_linear_workspace_size
    # M <= 24 (register-path kernel): counters for 48 tiles x 16 (3072 B) + two
    # partial-sum slots (64 rows x 24 token columns of int32) for each of at
    # most 320 CTAs (two per SM)
    assert ws(20, 6144, 4096) == 3072 + 2 * 320 * 64 * 24 * 4
    assert ws(8, 512, 256) == 256 + 2 * 16 * 64 * 8 * 4          # 16 work items -> 16 CTAs
    # M > 24 (tcgen05 kernel): counters for the tiles x 16 warps + int32 sums M x N
    assert ws(64, 4096, 4096) == 2048 + 64 * 4096 * 4
    lib.quasar_packed_weight_bytes.restype = ctypes.c_size_t
    assert lib.quasar_packed_weight_bytes(6144, 4096) == 6144 * 4096
    assert lib.quasar_packed_weight_bytes(136, 144) == 2 * 2 * 16384
    assert ws(0, 6144, 4096) == 0
    assert ws(256, 4096, 4096) >= 256 * 4096 * 4
    # token tiles of >= 128 rows: + the fp16 token copy M x K x 2, and the
    # counters sized for the 64-row fallback tiles (4 x 192 tiles x 16 warps)
    assert ws(256, 24576, 4096) == 4 * 192 * 16 * 4 + 256 * 24576 * 4 + 256 * 4096 * 2
    assert ws(128, 6144, 4096) == 2 * 48 * 16 * 4 + 128 * 6144 * 4 + 128 * 4096 * 2
    # the prefix that must be zero on entry: counters, plus the int32 sums
    # of the tcgen05 kernel (the register path's slots and the fp16 token
    # copy need no initial content)
    zb = lib.quasar_w8a8_linear_workspace_zeroed_bytes
    zb.restype = ctypes.c_size_t
    assert zb(20, 6144, 4096) == 3072
    assert zb(64, 4096, 4096) == 2048 + 64 * 4096 * 4
    assert zb(256, 24576, 4096) == 4 * 192 * 16 * 4 + 256 * 24576 * 4
    assert zb(0, 6144, 4096) == 0
    # 25-32 tokens: the register path (counters only) on layers of <= 8192
    # rows, the tcgen05 kernel (plus its int32 sums) on wider ones
    assert zb(32, 4096, 4096) == 32 * 16 * 4
    assert zb(25, 8192, 4096) == 64 * 16 * 4
    assert zb(32, 8200, 4096) == 4352 + 32 * 8200 * 4          # 65 tiles x 16 counters, 256-byte aligned
    assert zb(32, 24576, 4096) == 192 * 16 * 4 + 32 * 24576 * 4
    assert zb(33, 6144, 4096) == 48 * 16 * 4 + 33 * 6144 * 4
    # the register path's partial-sum slots at four token tiles: 2 per CTA, 64 rows x 32 int32, 320 CTAs
    assert ws(32, 4096, 4096) == 32 * 16 * 4 + 2 * 320 * 64 * 32 * 4
    for M, N, K in [(1, 8, 16), (24, 24576, 12288), (40, 4096, 12288), (288, 6144, 4096)]:
        assert zb(M, N, K) <= ws(M, N, K)
    assert lib.quasar_calibrate_workspace_size(4096) == 8 * 4096
    assert lib.quasar_verify_accept_workspace_size(32, 8, 151936) > 0
    assert lib.quasar_verify_accept_workspace_size(0, 8, 151936) == 0


FAKE = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x10004)


def test_linear_rejects_bad_arguments(lib):
    f = lib.quasar_w8a8_linear
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                               ctypes.c_size_t, ctypes.c_void_p]
    ok_args = [FAKE, FAKE, FAKE, FAKE, 8, 128, 128, FAKE, 128, FAKE, 1 << 20, None]

    def call(**kw):
        a = list(ok_args)
        names = ["xq", "sa", "wq", "sw", "M", "N", "K", "y", "ldy", "ws", "wsb", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(xq=None) == 1
    assert call(M=-1) == 1
    assert call(K=0) == 1
    assert call(K=100) == 2          # K % 16
    assert call(N=12) == 2           # N % 8
    assert call(K=131072 + 16) == 2  # int32 overflow bound
    assert call(ldy=64) == 2         # ldy < N
    assert call(xq=FAKE_ODD) == 2    # 16-byte alignment
    assert call(ws=None) == 3
    assert call(wsb=16) == 3
    assert call(M=0) == 0            # empty batch is a no-op


def test_quant_and_verify_reject_bad_arguments(lib):
    q = lib.quasar_smooth_quant_act
    q.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    assert q(FAKE, 128, FAKE, 4, 120, FAKE, FAKE, None) == 2     # K % 16
    assert q(FAKE, 64, FAKE, 4, 128, FAKE, FAKE, None) == 2      # ldx < K
    assert q(None, 128, FAKE, 4, 128, FAKE, FAKE, None) == 1
    assert q(FAKE, 128, FAKE, 0, 128, FAKE, FAKE, None) == 0     # M == 0
    v = lib.quasar_verify_accept
    v.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_size_t, ctypes.c_void_p]
    assert v(FAKE, 1000, FAKE, 2, 3, 1000, 1.0, None, FAKE, None, FAKE, 1 << 20, None) == 1   # T>0 needs u
    assert v(FAKE, 1000, FAKE, 2, 3, 1000, 1.0, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 1   # next only for T=0
    assert v(FAKE, 1000, FAKE, 2, 3, 1000, -1.0, None, FAKE, None, FAKE, 1 << 20, None) == 1  # T<0
    assert v(FAKE, 1001, FAKE, 2, 3, 1000, 0.0, None, FAKE, None, FAKE, 1 << 20, None) == 2   # ldl % 8
    assert v(FAKE, 1000, FAKE, 2, 3, 1000, 0.0, None, FAKE, None, FAKE, 16, None) == 3        # workspace
    assert v(FAKE, 1000, FAKE, 0, 3, 1000, 0.0, None, FAKE, None, FAKE, 0, None) == 0         # B == 0


def test_silu_mul_quant_rejects_bad_arguments(lib):
    """The MLP glue entry: rows of [gate | up] need ldgu >= 2 I."""
    g = lib.quasar_silu_mul_smooth_quant
    g.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    assert g(FAKE, 256, FAKE, 4, 120, FAKE, FAKE, None) == 2     # I % 16
    assert g(FAKE, 255, FAKE, 4, 128, FAKE, FAKE, None) == 2     # ldgu < 2 I
    assert g(FAKE, 260, FAKE, 4, 128, FAKE, FAKE, None) == 2     # ldgu % 8
    assert g(FAKE, 256, FAKE, 4, 0, FAKE, FAKE, None) == 1       # I <= 0
    assert g(FAKE, 1 << 30, FAKE, 4, (1 << 29) + 16, FAKE, FAKE, None) == 1   # 2 I overflows
    assert g(None, 256, FAKE, 4, 128, FAKE, FAKE, None) == 1
    assert g(FAKE, 256, FAKE, 4, 128, FAKE, None, None) == 1
    assert g(FAKE_ODD, 256, FAKE, 4, 128, FAKE, FAKE, None) == 2  # 16-byte alignment
    assert g(FAKE, 256, FAKE, 0, 128, FAKE, FAKE, None) == 0     # M == 0: nothing launched


def test_rmsnorm_quant_rejects_bad_arguments(lib):
    r = lib.quasar_rmsnorm_smooth_quant
    r.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert r(FAKE, 128, FAKE, 1e-6, FAKE, 4, 120, FAKE, FAKE, None) == 2      # K % 16
    assert r(FAKE, 64, FAKE, 1e-6, FAKE, 4, 128, FAKE, FAKE, None) == 2       # ldx < K
    assert r(FAKE, 12304, FAKE, 1e-6, FAKE, 4, 12304, FAKE, FAKE, None) == 2  # rows beyond 12288 values
    assert r(FAKE, 128, FAKE, 0.0, FAKE, 4, 128, FAKE, FAKE, None) == 1       # eps must be > 0
    assert r(FAKE, 128, FAKE, float("inf"), FAKE, 4, 128, FAKE, FAKE, None) == 1
    assert r(FAKE, 128, None, 1e-6, FAKE, 4, 128, FAKE, FAKE, None) == 1      # gamma
    assert r(FAKE, 128, FAKE_ODD, 1e-6, FAKE, 4, 128, FAKE, FAKE, None) == 2  # gamma alignment
    assert r(FAKE, 128, FAKE, 1e-6, FAKE, 0, 128, FAKE, FAKE, None) == 0      # M == 0


def test_fused_linear_rejects_bad_arguments(lib):
    f = lib.quasar_w8a8_linear_fused
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p] + \
        [ctypes.c_int] * 3 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    names = ["x", "ldx", "smooth", "wp", "sw", "M", "N", "K", "y", "ldy", "ws", "wsb", "stream"]
    ok_args = [FAKE, 128, FAKE, FAKE, FAKE, 8, 128, 128, FAKE, 128, FAKE, 1 << 20, None]

    def call(**kw):
        a = list(ok_args)
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(x=None) == 1
    assert call(smooth=None) == 1
    assert call(M=-1) == 1
    assert call(K=100) == 2          # K % 16
    assert call(ldx=64) == 2         # ldx < K
    assert call(ldx=132) == 2        # ldx % 8
    assert call(x=FAKE_ODD) == 2     # 16-byte alignment
    assert call(smooth=FAKE_ODD) == 2
    assert call(M=0) == 0            # empty batch is a no-op
    lib.quasar_w8a8_linear_fused_workspace_size.restype = ctypes.c_size_t
    lib.quasar_w8a8_linear_workspace_size.restype = ctypes.c_size_t
    lin = lib.quasar_w8a8_linear_workspace_size(20, 24576, 4096)
    assert lib.quasar_w8a8_linear_fused_workspace_size(20, 24576, 4096) == lin + 20 * 4096 + 256


def test_verify_sample_rejects_bad_arguments(lib):
    f = lib.quasar_verify_sample
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int] * 3 + \
        [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
         ctypes.c_size_t, ctypes.c_void_p]
    names = ["lg", "ldl", "draft", "B", "D", "V", "T", "u", "un", "n_acc", "nxt", "ws", "wsb", "stream"]
    ok_args = [FAKE, 128, FAKE, 2, 3, 128, 1.0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None]

    def call(**kw):
        a = list(ok_args)
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(T=0.0) == 1             # sampling needs T > 0
    assert call(T=float("inf")) == 1
    assert call(un=None) == 1
    assert call(nxt=None) == 1
    assert call(u=None) == 1            # D > 0 needs the acceptance uniforms
    assert call(ldl=100) == 2
    assert call(B=0) == 0


def test_selftest_wait_rejects_limits_out_of_range(lib):
    f = lib.quasar_selftest_wait_timeout
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    assert f(0, None) == 1
    assert f(999, None) == 1
    assert f(10_000_000_001, None) == 1


def test_lm_head_rejects_bad_arguments(lib):
    lib.quasar_lm_head_verify_workspace_size.restype = ctypes.c_size_t
    # counters [B], row results [B*(D+1)] x 16 B, draft logits [B*(D+1)], records [B*(D+1)][ceil(V/128)] x 8 B
    assert lib.quasar_lm_head_verify_workspace_size(32, 8, 151936) == 256 + 4608 + 1280 + 288 * 1187 * 8
    f = lib.quasar_lm_head_verify
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    names = ["h", "ldh", "wp", "K", "draft", "B", "D", "V", "T", "u", "n_acc", "nxt", "ws", "wsb", "stream"]
    ok_args = [FAKE, 64, FAKE, 64, FAKE, 2, 3, 1000, 0.0, None, FAKE, FAKE, FAKE, 1 << 20, None]

    def call(**kw):
        a = list(ok_args)
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(B=-1) == 1
    assert call(T=-1.0) == 1
    assert call(T=float("inf")) == 1
    assert call(T=1.0) == 1                  # T > 0 needs u and no next token
    assert call(T=1.0, u=FAKE) == 1
    assert call(n_acc=None) == 1
    assert call(draft=None) == 1
    assert call(B=52, D=9) == 2              # 520 token rows > 512
    assert call(ws=None) == 3
    assert call(wsb=100) == 3
    assert call(K=60, ldh=64) == 2           # K % 8
    assert call(ldh=32) == 2                 # ldh < K
    assert call(h=None) == 1
    assert call(wp=None) == 1
    assert call(wp=FAKE_ODD) == 2            # 16-byte alignment
    assert call(B=0) == 0
    g = lib.quasar_lm_head_logits
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p]
    assert g(FAKE, 64, FAKE, 2, 1000, 64, FAKE, 999, None) == 2     # ldl < V
    assert g(FAKE, 64, FAKE, 513, 1000, 64, FAKE, 1000, None) == 2  # M > 512
    assert g(FAKE, 64, FAKE, 2, 1000, 64, None, 1000, None) == 1
    assert g(FAKE, 64, FAKE, 0, 1000, 64, None, 1000, None) == 0
    fs = lib.quasar_lm_head_verify_sample
    fs.restype = ctypes.c_int
    fs.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert fs(FAKE, 64, FAKE, 64, FAKE, 2, 3, 1000, 0.0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 1  # T > 0
    assert fs(FAKE, 64, FAKE, 64, FAKE, 2, 3, 1000, 1.0, FAKE, None, FAKE, FAKE, FAKE, 1 << 20, None) == 1  # u_next
    assert fs(FAKE, 64, FAKE, 64, FAKE, 2, 3, 1000, 1.0, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, None) == 1  # next
    assert fs(FAKE, 64, FAKE, 64, FAKE, 2, 3, 1000, 1.0, None, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 1  # u
    assert fs(FAKE, 64, FAKE, 64, FAKE, 0, 3, 1000, 1.0, None, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 0  # B = 0
    lib.quasar_lm_head_packed_bytes.restype = ctypes.c_size_t
    assert lib.quasar_lm_head_packed_bytes(151936, 4096) == 1187 * 64 * 16384
    assert lib.quasar_lm_head_packed_bytes(1000, 200) == 8 * 4 * 16384
    pk = lib.quasar_pack_lm_head
    pk.restype = ctypes.c_int
    pk.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    assert pk(FAKE, 64, 0, 64, FAKE, None) == 1
    assert pk(FAKE, 64, 100, 60, FAKE, None) == 2       # K % 8
    assert pk(FAKE, 32, 100, 64, FAKE, None) == 2       # ldw < K
    assert pk(FAKE_ODD, 64, 100, 64, FAKE, None) == 2
    assert pk(None, 64, 100, 64, FAKE, None) == 1


def test_tensor_probe_rejects_bad_arguments(lib):
    f = lib.quasar_probe_tensor_rate
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert f(0, 128, 16, None, 1024, None) == 1           # no output buffer
    assert f(9, 128, 16, FAKE, 1024, None) == 1           # unknown form
    assert f(7, 256, 16, FAKE, 1024, None) == 2           # pair form: accumulator would reach the A operand
    assert f(0, 128, 0, FAKE, 1024, None) == 1            # no iterations
    assert f(0, 24, 16, FAKE, 1024, None) == 2            # N not a multiple of 16
    assert f(0, 272, 16, FAKE, 1024, None) == 2           # N above 256
    assert f(5, 128, 16, FAKE, 1024, None) == 2           # four accumulators of 128 columns do not fit
