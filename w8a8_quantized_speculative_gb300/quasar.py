"""Thin ctypes binding of libquasar.so (argument marshalling only).

Every function here checks tensor dtypes/devices, allocates outputs with
torch when the caller does not pass them, and forwards raw device pointers
and the current CUDA stream to the C ABI declared in ``include/quasar.h``.
All arithmetic happens in the library's CUDA kernels.  Importing this module
raises ImportError when the library has not been built: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libquasar.so is not built ({LIB_PATH}); run "
                      "`python -m w8a8_quantized_speculative_gb300.build`")

lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGS = {
    "quasar_status_string": (ctypes.c_char_p, [_i]),
    "quasar_version": (_i, []),
    "quasar_get_device_error": (_i, [_p, ctypes.POINTER(ctypes.c_uint32)]),
    "quasar_set_wait_limit_ns": (_i, [ctypes.c_uint64]),
    "quasar_selftest_wait_timeout": (_i, [ctypes.c_uint64, _p]),
    "quasar_calibrate_workspace_size": (_sz, [_i]),
    "quasar_calibrate_smooth": (_i, [_p, _i, _i, _p, _i, _i, _i, _f, _p, _p, _sz, _p]),
    "quasar_packed_weight_bytes": (_sz, [_i, _i]),
    "quasar_pack_weights": (_i, [_p, _i, _p, _i, _i, _p, _p, _p]),
    "quasar_tile_weights": (_i, [_p, _i, _i, _p, _p]),
    "quasar_packed_weight_bytes_w4": (_sz, [_i, _i]),
    "quasar_pack_weights_w4": (_i, [_p, _i, _p, _i, _i, _p, _p, _p]),
    "quasar_tile_weights_w4": (_i, [_p, _i, _i, _p, _p]),
    "quasar_w4a8_linear": (_i, [_p, _p, _p, _p, _i, _i, _i, _p, _i, _p, _sz, _p]),
    "quasar_smooth_quant_act": (_i, [_p, _i, _p, _i, _i, _p, _p, _p]),
    "quasar_silu_mul_smooth_quant": (_i, [_p, _i, _p, _i, _i, _p, _p, _p]),
    "quasar_rmsnorm_smooth_quant": (_i, [_p, _i, _p, _f, _p, _i, _i, _p, _p, _p]),
    "quasar_w8a8_linear_workspace_size": (_sz, [_i, _i, _i]),
    "quasar_w8a8_linear_workspace_zeroed_bytes": (_sz, [_i, _i, _i]),
    "quasar_probe_tensor_rate": (_i, [_i, _i, _i, _p, _i, _p]),
    "quasar_w8a8_linear": (_i, [_p, _p, _p, _p, _i, _i, _i, _p, _i, _p, _sz, _p]),
    "quasar_w8a8_linear_fused_workspace_size": (_sz, [_i, _i, _i]),
    "quasar_w8a8_linear_fused": (_i, [_p, _i, _p, _p, _p, _i, _i, _i, _p, _i, _p, _sz, _p]),
    "quasar_int8_gemm_s32": (_i, [_p, _p, _i, _i, _i, _p, _p, _sz, _p]),
    "quasar_w8a8_linear_noalloc": (_i, [_p, _p, _p, _p, _i, _i, _i, _p, _i, _p]),
    "quasar_verify_accept_workspace_size": (_sz, [_i, _i, _i]),
    "quasar_verify_accept": (_i, [_p, _i, _p, _i, _i, _i, _f, _p, _p, _p, _p, _sz, _p]),
    "quasar_verify_sample": (_i, [_p, _i, _p, _i, _i, _i, _f, _p, _p, _p, _p, _p, _sz, _p]),
    "quasar_lm_head_verify_workspace_size": (_sz, [_i, _i, _i]),
    "quasar_lm_head_packed_bytes": (_sz, [_i, _i]),
    "quasar_pack_lm_head": (_i, [_p, _i, _i, _i, _p, _p]),
    "quasar_lm_head_verify": (_i, [_p, _i, _p, _i, _p, _i, _i, _i, _f, _p, _p, _p, _p, _sz, _p]),
    "quasar_lm_head_logits": (_i, [_p, _i, _p, _i, _i, _i, _p, ctypes.c_longlong, _p]),
    "quasar_lm_head_verify_sample": (_i, [_p, _i, _p, _i, _p, _i, _i, _i, _f, _p, _p, _p, _p, _p, _sz, _p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

OK = 0
STATUS = {0: "QUASAR_OK", 1: "QUASAR_ERR_INVALID_ARG", 2: "QUASAR_ERR_UNSUPPORTED", 3: "QUASAR_ERR_WORKSPACE",
          4: "QUASAR_ERR_CUDA", 5: "QUASAR_ERR_TIMEOUT"}


class QuasarError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.quasar_status_string(status).decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


def _check(status: int, where: str):
    if status != OK:
        raise QuasarError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _rowmajor(t: torch.Tensor, name: str):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit inner stride")
    return t.stride(0)


class Workspace:
    """Zero-filled device scratch that grows on demand.  Every call leaves
    the part of the workspace it needs zero-filled, except the one-call
    linear (w8a8_linear_fused), which leaves its codes and scales after that
    part; this object remembers that range and clears the overlap before a
    later call that needs those bytes zero, so one instance can be shared by
    consecutive calls on the same stream."""

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.buf = None
        self.dirty = None          # (lo, hi): bytes a call may have left nonzero

    def get(self, nbytes: int, zero_prefix: int | None = None, stream=None) -> torch.Tensor:
        """The buffer, at least `nbytes` long, with its first `zero_prefix`
        bytes (default: all `nbytes`) zero when the next call on `stream` starts."""
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
            self.dirty = None
        z = nbytes if zero_prefix is None else int(zero_prefix)
        if self.dirty is not None and self.dirty[0] < z:
            lo, hi = self.dirty[0], min(self.dirty[1], z)
            if stream is None:
                self.buf[lo:hi].zero_()
            else:
                with torch.cuda.stream(stream):
                    self.buf[lo:hi].zero_()
            self.dirty = (z, self.dirty[1]) if self.dirty[1] > z else None
        return self.buf

    def mark_dirty(self, lo: int, hi: int):
        if hi <= lo:
            return
        self.dirty = (lo, hi) if self.dirty is None else (min(lo, self.dirty[0]), max(hi, self.dirty[1]))

    def reset(self):
        if self.buf is not None:
            self.buf.zero_()
        self.dirty = None


_default_ws = {}


def _ws(ws, device):
    if ws is not None:
        return ws
    key = torch.device(device).index
    if key not in _default_ws:
        _default_ws[key] = Workspace(device)
    return _default_ws[key]


# ---------------------------------------------------------------- entry points

def calibrate_smooth(x_cal: torch.Tensor, w: torch.Tensor, alpha: float = 0.5, out=None, stream=None):
    """smooth[k] = max|W[:,k]|^(1-alpha) / max|Xcal[:,k]|^alpha (fp32 [K])."""
    _need(x_cal, torch.bfloat16, "x_cal")
    _need(w, torch.bfloat16, "w")
    ldx = _rowmajor(x_cal, "x_cal")
    ldw = _rowmajor(w, "w")
    K = x_cal.shape[1]
    if w.shape[1] != K:
        raise ValueError("x_cal and w disagree on K")
    out = torch.empty(K, dtype=torch.float32, device=x_cal.device) if out is None else out
    ws = torch.empty(max(int(lib.quasar_calibrate_workspace_size(K)), 16), dtype=torch.uint8, device=x_cal.device)
    _check(lib.quasar_calibrate_smooth(_ptr(x_cal), x_cal.shape[0], ldx, _ptr(w), w.shape[0], ldw, K, alpha,
                                       _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "calibrate_smooth")
    return out


def packed_weight_bytes(N: int, K: int) -> int:
    return int(lib.quasar_packed_weight_bytes(N, K))


def pack_weights(w: torch.Tensor, smooth: torch.Tensor, wp=None, sw=None, stream=None):
    """(Wp packed int8 [packed_weight_bytes], sw fp32 [N]) from BF16 W [N][K]
    and smooth [K].  The packed layout is described in include/quasar.h."""
    _need(w, torch.bfloat16, "w")
    _need(smooth, torch.float32, "smooth")
    ldw = _rowmajor(w, "w")
    N, K = w.shape
    wp = torch.empty(packed_weight_bytes(N, K), dtype=torch.int8, device=w.device) if wp is None else wp
    sw = torch.empty(N, dtype=torch.float32, device=w.device) if sw is None else sw
    _check(lib.quasar_pack_weights(_ptr(w), ldw, _ptr(smooth), N, K, _ptr(wp), _ptr(sw), _stream(stream)),
           "pack_weights")
    return wp, sw


def tile_weights(wq: torch.Tensor, wp=None, stream=None):
    """Packed int8 weights from row-major int8 codes [N][K]."""
    _need(wq, torch.int8, "wq")
    if not wq.is_contiguous():
        raise ValueError("wq must be contiguous")
    N, K = wq.shape
    wp = torch.empty(packed_weight_bytes(N, K), dtype=torch.int8, device=wq.device) if wp is None else wp
    _check(lib.quasar_tile_weights(_ptr(wq), N, K, _ptr(wp), _stream(stream)), "tile_weights")
    return wp


def packed_weight_bytes_w4(N: int, K: int) -> int:
    return int(lib.quasar_packed_weight_bytes_w4(N, K))


def pack_weights_w4(w: torch.Tensor, smooth: torch.Tensor, wp=None, sw=None, stream=None):
    """(Wp4 packed 4-bit [packed_weight_bytes_w4], sw fp32 [N]) from BF16 W [N][K]."""
    _need(w, torch.bfloat16, "w")
    _need(smooth, torch.float32, "smooth")
    ldw = _rowmajor(w, "w")
    N, K = w.shape
    wp = torch.empty(packed_weight_bytes_w4(N, K), dtype=torch.int8, device=w.device) if wp is None else wp
    sw = torch.empty(N, dtype=torch.float32, device=w.device) if sw is None else sw
    _check(lib.quasar_pack_weights_w4(_ptr(w), ldw, _ptr(smooth), N, K, _ptr(wp), _ptr(sw), _stream(stream)),
           "pack_weights_w4")
    return wp, sw


def tile_weights_w4(wq: torch.Tensor, wp=None, stream=None):
    """Packed 4-bit weights from row-major codes [N][K] in [-8, 7] (int8)."""
    _need(wq, torch.int8, "wq")
    if not wq.is_contiguous():
        raise ValueError("wq must be contiguous")
    N, K = wq.shape
    wp = torch.empty(packed_weight_bytes_w4(N, K), dtype=torch.int8, device=wq.device) if wp is None else wp
    _check(lib.quasar_tile_weights_w4(_ptr(wq), N, K, _ptr(wp), _stream(stream)), "tile_weights_w4")
    return wp


def w4a8_linear(xq, sa, wp4, sw, y=None, workspace: Workspace | None = None, stream=None):
    """Y bf16 [M][N] from INT8 codes and 4-bit packed weights (any M)."""
    _need(xq, torch.int8, "xq")
    _need(wp4, torch.int8, "wp4")
    M, K = xq.shape
    N = sw.numel()
    if wp4.numel() < packed_weight_bytes_w4(N, K) or not wp4.is_contiguous():
        raise ValueError("wp4 must be a contiguous packed 4-bit weight buffer of packed_weight_bytes_w4(N, K)")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device) if y is None else y
    ldy = _rowmajor(y, "y")
    ws = _ws(workspace, xq.device)
    buf = ws.get(int(lib.quasar_w8a8_linear_workspace_size(M, N, K)),
                 zero_prefix=int(lib.quasar_w8a8_linear_workspace_zeroed_bytes(M, N, K)), stream=stream)
    _check(lib.quasar_w4a8_linear(_ptr(xq), _ptr(sa), _ptr(wp4), _ptr(sw), M, N, K, _ptr(y), ldy, _ptr(buf),
                                  buf.numel(), _stream(stream)), "w4a8_linear")
    return y


def smooth_quant_act(x: torch.Tensor, smooth: torch.Tensor, xq=None, sa=None, stream=None):
    """(Xq int8 [M][K], sa fp32 [M]) from BF16 X [M][K] and smooth [K]."""
    _need(x, torch.bfloat16, "x")
    _need(smooth, torch.float32, "smooth")
    ldx = _rowmajor(x, "x")
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    sa = torch.empty(M, dtype=torch.float32, device=x.device) if sa is None else sa
    _check(lib.quasar_smooth_quant_act(_ptr(x), ldx, _ptr(smooth), M, K, _ptr(xq), _ptr(sa), _stream(stream)),
           "smooth_quant_act")
    return xq, sa


def rmsnorm_smooth_quant(x: torch.Tensor, gamma: torch.Tensor, smooth: torch.Tensor, eps: float = 1e-6, xq=None,
                         sa=None, stream=None):
    """(Xq int8 [M][K], sa fp32 [M]) of h = bf16(bf16(x * r) * gamma), r the
    row's inverse RMS, from BF16 x [M][K], the norm's BF16 weight gamma [K]
    and the linear's smooth [K]: RMSNorm ahead of qkv / gate_up, one launch."""
    _need(x, torch.bfloat16, "x")
    _need(gamma, torch.bfloat16, "gamma")
    _need(smooth, torch.float32, "smooth")
    ldx = _rowmajor(x, "x")
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    sa = torch.empty(M, dtype=torch.float32, device=x.device) if sa is None else sa
    _check(lib.quasar_rmsnorm_smooth_quant(_ptr(x), ldx, _ptr(gamma), float(eps), _ptr(smooth), M, K, _ptr(xq),
                                           _ptr(sa), _stream(stream)), "rmsnorm_smooth_quant")
    return xq, sa


def silu_mul_smooth_quant(gu: torch.Tensor, smooth: torch.Tensor, xq=None, sa=None, stream=None):
    """(Xq int8 [M][I], sa fp32 [M]) of h = bf16(silu(gate) * up), from the
    gate_up output gu [M][2I] (gate in columns 0..I-1, up in I..2I-1) and
    down's smooth [I]: the MLP glue before down, one launch."""
    _need(gu, torch.bfloat16, "gu")
    _need(smooth, torch.float32, "smooth")
    ldgu = _rowmajor(gu, "gu")
    M, two_i = gu.shape
    if two_i % 2:
        raise ValueError("gu must hold [gate | up] halves of equal width")
    inter = two_i // 2
    xq = torch.empty((M, inter), dtype=torch.int8, device=gu.device) if xq is None else xq
    sa = torch.empty(M, dtype=torch.float32, device=gu.device) if sa is None else sa
    _check(lib.quasar_silu_mul_smooth_quant(_ptr(gu), ldgu, _ptr(smooth), M, inter, _ptr(xq), _ptr(sa),
                                            _stream(stream)), "silu_mul_smooth_quant")
    return xq, sa


def _check_packed(wp, N, K):
    _need(wp, torch.int8, "wp")
    if wp.numel() < packed_weight_bytes(N, K) or not wp.is_contiguous():
        raise ValueError("wp must be a contiguous packed weight buffer of packed_weight_bytes(N, K)")


def w8a8_linear(xq, sa, wp, sw, y=None, workspace: Workspace | None = None, stream=None):
    """Y bf16 [M][N] = dequant(Xq · Wq^T) with the per-token / per-channel
    scales; wp is the packed weight buffer, N = len(sw)."""
    _need(xq, torch.int8, "xq")
    M, K = xq.shape
    N = sw.numel()
    _check_packed(wp, N, K)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device) if y is None else y
    ldy = _rowmajor(y, "y")
    ws = _ws(workspace, xq.device)
    need = int(lib.quasar_w8a8_linear_workspace_size(M, N, K))
    buf = ws.get(need, zero_prefix=int(lib.quasar_w8a8_linear_workspace_zeroed_bytes(M, N, K)), stream=stream)
    _check(lib.quasar_w8a8_linear(_ptr(xq), _ptr(sa), _ptr(wp), _ptr(sw), M, N, K, _ptr(y), ldy, _ptr(buf),
                                  buf.numel(), _stream(stream)), "w8a8_linear")
    return y


def w8a8_linear_fused(x, smooth, wp, sw, y=None, workspace: Workspace | None = None, stream=None):
    """Y bf16 [M][N] = w8a8_linear(*smooth_quant_act(x, smooth), wp, sw), bit-identical, in one call
    (codes and scales live in the workspace)."""
    _need(x, torch.bfloat16, "x")
    _need(smooth, torch.float32, "smooth")
    ldx = _rowmajor(x, "x")
    M, K = x.shape
    N = sw.numel()
    _check_packed(wp, N, K)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    ldy = _rowmajor(y, "y")
    ws = _ws(workspace, x.device)
    need = int(lib.quasar_w8a8_linear_fused_workspace_size(M, N, K))
    buf = ws.get(need, zero_prefix=int(lib.quasar_w8a8_linear_workspace_zeroed_bytes(M, N, K)), stream=stream)
    _check(lib.quasar_w8a8_linear_fused(_ptr(x), ldx, _ptr(smooth), _ptr(wp), _ptr(sw), M, N, K, _ptr(y), ldy,
                                        _ptr(buf), buf.numel(), _stream(stream)), "w8a8_linear_fused")
    if M > 0:
        ws.mark_dirty(int(lib.quasar_w8a8_linear_workspace_size(M, N, K)), need)
    return y


def int8_gemm_s32(xq, wp, N: int, acc=None, workspace: Workspace | None = None, stream=None):
    """acc int32 [M][N] = Xq · Wq^T, exact; wp is the packed weight buffer."""
    _need(xq, torch.int8, "xq")
    M, K = xq.shape
    _check_packed(wp, N, K)
    acc = torch.empty((M, N), dtype=torch.int32, device=xq.device) if acc is None else acc
    ws = _ws(workspace, xq.device)
    buf = ws.get(int(lib.quasar_w8a8_linear_workspace_size(M, N, K)),
                 zero_prefix=int(lib.quasar_w8a8_linear_workspace_zeroed_bytes(M, N, K)), stream=stream)
    _check(lib.quasar_int8_gemm_s32(_ptr(xq), _ptr(wp), M, N, K, _ptr(acc), _ptr(buf), buf.numel(),
                                    _stream(stream)), "int8_gemm_s32")
    return acc


def verify_accept(logits: torch.Tensor, draft: torch.Tensor, temperature: float = 0.0, u=None,
                  want_next: bool = True, n_acc=None, next_token=None, workspace: Workspace | None = None,
                  stream=None):
    """Accepted prefix length per sequence (int32 [B]) and, for T == 0, the
    next token (argmax of row n_acc) or None.  logits: bf16 [B][D+1][V]."""
    _need(logits, torch.bfloat16, "logits")
    _need(draft, torch.int32, "draft")
    if logits.dim() != 3 or logits.stride(2) != 1 or (
            logits.shape[0] > 1 and logits.stride(0) != logits.shape[1] * logits.stride(1)):
        raise ValueError("logits must be [B][D+1][V] with unit inner stride and evenly spaced rows")
    B, R, V = logits.shape
    D = R - 1
    ldl = logits.stride(1)
    n_acc = torch.empty(B, dtype=torch.int32, device=logits.device) if n_acc is None else n_acc
    sampled = temperature > 0
    if sampled:
        _need(u, torch.float32, "u")
        next_token = None
    elif want_next and next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=logits.device)
    ws = _ws(workspace, logits.device)
    buf = ws.get(int(lib.quasar_verify_accept_workspace_size(B, D, V)))
    _check(lib.quasar_verify_accept(_ptr(logits), ldl, _ptr(draft), B, D, V, float(temperature), _ptr(u),
                                    _ptr(n_acc), _ptr(next_token), _ptr(buf), buf.numel(), _stream(stream)),
           "verify_accept")
    return n_acc, next_token



def verify_sample(logits: torch.Tensor, draft: torch.Tensor, temperature: float, u, u_next, n_acc=None,
                  next_token=None, workspace: Workspace | None = None, stream=None):
    """T > 0: accepted prefix length (int32 [B]) and the lossless next token
    (int32 [B]): a draw from row n_acc's softmax without the rejected draft,
    or from the bonus row after D acceptances, by inverse CDF on u_next [B]."""
    _need(logits, torch.bfloat16, "logits")
    _need(draft, torch.int32, "draft")
    _need(u_next, torch.float32, "u_next")
    if logits.dim() != 3 or logits.stride(2) != 1 or (
            logits.shape[0] > 1 and logits.stride(0) != logits.shape[1] * logits.stride(1)):
        raise ValueError("logits must be [B][D+1][V] with unit inner stride and evenly spaced rows")
    B, R, V = logits.shape
    D = R - 1
    if D > 0:
        _need(u, torch.float32, "u")
    n_acc = torch.empty(B, dtype=torch.int32, device=logits.device) if n_acc is None else n_acc
    next_token = torch.empty(B, dtype=torch.int32, device=logits.device) if next_token is None else next_token
    ws = _ws(workspace, logits.device)
    buf = ws.get(int(lib.quasar_verify_accept_workspace_size(B, D, V)))
    _check(lib.quasar_verify_sample(_ptr(logits), logits.stride(1), _ptr(draft), B, D, V, float(temperature),
                                    _ptr(u), _ptr(u_next), _ptr(n_acc), _ptr(next_token), _ptr(buf), buf.numel(),
                                    _stream(stream)), "verify_sample")
    return n_acc, next_token

class PackedLmHead:
    """An lm_head weight W [V][K] (BF16) packed by quasar_pack_lm_head into
    the kernels' 16 KB block layout (see include/quasar.h)."""

    def __init__(self, buf: torch.Tensor, V: int, K: int):
        self.buf, self.V, self.K = buf, V, K


def pack_lm_head(w: torch.Tensor, stream=None) -> PackedLmHead:
    """Pack a BF16 lm_head weight [V][K] (offline, once)."""
    _need(w, torch.bfloat16, "w")
    ldw = _rowmajor(w, "w")
    V, K = w.shape
    buf = torch.empty(int(lib.quasar_lm_head_packed_bytes(V, K)), dtype=torch.uint8, device=w.device)
    _check(lib.quasar_pack_lm_head(_ptr(w), ldw, V, K, _ptr(buf), _stream(stream)), "pack_lm_head")
    return PackedLmHead(buf, V, K)


def lm_head_logits(h: torch.Tensor, wp: PackedLmHead, logits=None, stream=None):
    """logits[m][v] = bf16(fp32 sum_k h[m][k] * W[v][k]) (bf16 [M][V]) from
    the tcgen05 lm_head kernel.  h: bf16 [M][K]; wp: pack_lm_head(W)."""
    _need(h, torch.bfloat16, "h")
    ldh = _rowmajor(h, "h")
    M, K = h.shape
    V = wp.V
    if wp.K != K:
        raise ValueError("h and the packed weight must share K")
    if logits is None:
        logits = torch.empty(M, V, dtype=torch.bfloat16, device=h.device)
    _need(logits, torch.bfloat16, "logits")
    ldl = _rowmajor(logits, "logits")
    _check(lib.quasar_lm_head_logits(_ptr(h), ldh, _ptr(wp.buf), M, V, K, _ptr(logits), ldl, _stream(stream)),
           "lm_head_logits")
    return logits


def lm_head_verify(h: torch.Tensor, wp: PackedLmHead, draft: torch.Tensor, temperature: float = 0.0, u=None,
                   want_next: bool = True, n_acc=None, next_token=None, workspace: Workspace | None = None,
                   stream=None):
    """The BF16 lm_head and verification in one call, without writing the
    logits: accepted prefix length (int32 [B]) and, for T == 0, the next
    token.  h: bf16 [B*(D+1)][K] (row b*(D+1)+j scores draft j of sequence
    b), wp: pack_lm_head(W), draft: int32 [B][D], u: fp32 [B][D] for T > 0."""
    _need(h, torch.bfloat16, "h")
    _need(draft, torch.int32, "draft")
    ldh = _rowmajor(h, "h")
    if draft.dim() != 2 or not draft.is_contiguous():
        raise ValueError("draft must be a contiguous [B][D] tensor")
    B, D = draft.shape
    K = h.shape[1]
    V = wp.V
    if h.shape[0] != B * (D + 1) or wp.K != K:
        raise ValueError("h must be [B*(D+1)][K] with the packed weight's K")
    n_acc = torch.empty(B, dtype=torch.int32, device=h.device) if n_acc is None else n_acc
    sampled = temperature > 0
    if sampled:
        if D > 0:
            _need(u, torch.float32, "u")
        next_token = None
    elif want_next and next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=h.device)
    ws = _ws(workspace, h.device)
    buf = ws.get(int(lib.quasar_lm_head_verify_workspace_size(B, D, V)))
    _check(lib.quasar_lm_head_verify(_ptr(h), ldh, _ptr(wp.buf), K, _ptr(draft), B, D, V, float(temperature),
                                     _ptr(u), _ptr(n_acc), _ptr(next_token), _ptr(buf), buf.numel(),
                                     _stream(stream)), "lm_head_verify")
    return n_acc, next_token


def lm_head_verify_sample(h: torch.Tensor, wp: PackedLmHead, draft: torch.Tensor, temperature: float, u, u_next,
                          n_acc=None, next_token=None, workspace: Workspace | None = None, stream=None):
    """T > 0: the BF16 lm_head and the acceptance test in one call, plus the
    lossless next token (int32 [B]) drawn by inverse CDF on u_next [B], as
    verify_sample draws it; the logits are never written."""
    _need(h, torch.bfloat16, "h")
    _need(draft, torch.int32, "draft")
    _need(u_next, torch.float32, "u_next")
    ldh = _rowmajor(h, "h")
    if draft.dim() != 2 or not draft.is_contiguous():
        raise ValueError("draft must be a contiguous [B][D] tensor")
    B, D = draft.shape
    K = h.shape[1]
    if h.shape[0] != B * (D + 1) or wp.K != K:
        raise ValueError("h must be [B*(D+1)][K] with the packed weight's K")
    if D > 0:
        _need(u, torch.float32, "u")
    n_acc = torch.empty(B, dtype=torch.int32, device=h.device) if n_acc is None else n_acc
    next_token = torch.empty(B, dtype=torch.int32, device=h.device) if next_token is None else next_token
    ws = _ws(workspace, h.device)
    buf = ws.get(int(lib.quasar_lm_head_verify_workspace_size(B, D, wp.V)))
    _check(lib.quasar_lm_head_verify_sample(_ptr(h), ldh, _ptr(wp.buf), K, _ptr(draft), B, D, wp.V,
                                            float(temperature), _ptr(u), _ptr(u_next), _ptr(n_acc),
                                            _ptr(next_token), _ptr(buf), buf.numel(), _stream(stream)),
           "lm_head_verify_sample")
    return n_acc, next_token


PROBE_FORMS = {"tcgen05_ts": 0, "tcgen05_ss": 1, "tcgen05_ts_with_tmem_stores": 2, "mma_sync": 3,
               "tcgen05_ts_2chains": 4, "tcgen05_ts_4chains": 5, "tcgen05_ss_m64": 6,
               "tcgen05_ts_pair": 7, "tcgen05_ss_pair": 8}


def probe_tensor_rate(form: str, n: int = 128, iters: int = 4096, stream=None):
    """Measured rate of one MMA form on every SM (see quasar_probe_tensor_rate):
    returns dict(mac_per_clk_per_sm, cycles_per_mma, tmem_st_per_clk_per_sm)
    averaged over the SMs."""
    f = PROBE_FORMS[form]
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = torch.zeros(4 * sms, dtype=torch.int64, device="cuda")
    _check(lib.quasar_probe_tensor_rate(f, int(n), int(iters), _ptr(out), out.numel(), _stream(stream)),
           "probe_tensor_rate")
    torch.cuda.synchronize()
    o = out.view(sms, 4).cpu().numpy().astype("float64")
    ok = o[:, 0] > 0
    if not ok.any():
        raise QuasarError("probe_tensor_rate: every bounded wait ran out")
    cyc, mmas = o[ok, 0], o[ok, 1]
    if f == 3:
        macs = mmas * 16 * 8 * 16               # mmas counts every warp's mma.sync (16 x 8 x 16 each)
        per_issuer = mmas / 16                  # one issuing warp's share
    else:
        macs = mmas * (64 if f == 6 else 128) * n * 16
        per_issuer = mmas
    res = {"mac_per_clk_per_sm": float((macs / cyc).mean()), "cycles_per_mma": float((cyc / per_issuer).mean())}
    if f == 2:
        res["tmem_st_per_clk_per_sm"] = float((o[ok, 2] / o[ok, 3].clip(min=1)).mean())
    return res


def get_device_error(stream=None):
    """Synchronise and return (status, site) of the library's device error word."""
    site = ctypes.c_uint32(0)
    st = lib.quasar_get_device_error(_stream(stream), ctypes.byref(site))
    return st, site.value


def selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None):
    """Launch a kernel whose bounded wait must run out after limit_ns (the
    error word then reports QUASAR_ERR_TIMEOUT with site 12)."""
    _check(lib.quasar_selftest_wait_timeout(int(limit_ns), _stream(stream)), "selftest_wait_timeout")


def set_wait_limit_ns(ns: int):
    _check(lib.quasar_set_wait_limit_ns(ns), "set_wait_limit_ns")
