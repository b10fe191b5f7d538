"""Thin ctypes binding of libmoe.so (include/moe.h), same names as the C ABI.

Only argument marshalling lives here: torch tensors supply device pointers and
the current CUDA stream; every step of the MoE layer runs in the library's
CUDA kernels.  There is no fallback: if the library cannot be built or loaded,
importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MOE_OK = 0
MOE_LOGITS_IN = 0x1
MOE_CHECK = 0x2
MOE_WEIGHTS_PREPACKED = 0x4
MOE_SINGLE_CTA_TILES = 0x8
MOE_SHARED_SERIAL = 0x10
MOE_FP8_DISPATCH = 0x20
MOE_FP8_MX = 0x40
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_BAD_ROUTING", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_CUDA"}

# the C ABI's exported symbols (checked against include/moe.h by the tests)
SYMBOLS = ("moe_status_string", "moe_version", "moe_last_cuda_error", "moe_trace_events",
           "moe_kernel_launches", "moe_selftest_wait_timeout",
           "moe_route", "moe_dispatch", "moe_dispatch_noalloc", "moe_dispatch_fp8",
           "moe_dequant_fp8", "moe_quantize_mx", "moe_dispatch_mx", "moe_grouped_ffn_mx",
           "moe_prepack_weights", "moe_grouped_ffn", "moe_grouped_ffn_fp8",
           "moe_combine", "moe_layer_fwd", "moe_layer_bwd")

# moe_stage_t
STAGES = ("gate", "topk", "dispatch", "gateup", "down", "combine", "bwd_route", "bwd_dh", "bwd_dx",
          "bwd_wg2", "bwd_wg13", "bwd_dwg", "bwd_dxc", "shared_fwd", "shared_bwd")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, cuda_error: int = 0):
        extra = f" (cudaError {cuda_error})" if cuda_error else ""
        super().__init__(f"{where}: {STATUS.get(status, status)}{extra}")
        self.status = status
        self.cuda_error = cuda_error


_vp = ctypes.c_void_p
_i = ctypes.c_int
_u = ctypes.c_uint
_szp = ctypes.POINTER(ctypes.c_size_t)


class moe_shared_t(ctypes.Structure):
    _fields_ = [("fs", _i), ("W1", _vp), ("W3", _vp), ("W2", _vp), ("dW1", _vp), ("dW3", _vp),
                ("dW2", _vp)]


class moe_mx_weights_t(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("W1q", "W1s", "W3q", "W3s", "W2q", "W2s")]


class moe_layer_t(ctypes.Structure):
    _fields_ = [("T", _i), ("d", _i), ("E", _i), ("R", _i), ("f", _i), ("w_gate", _vp),
                ("bias", _vp), ("W1", _vp), ("W3", _vp), ("W2", _vp),
                ("shared", ctypes.POINTER(moe_shared_t)),
                ("mx", ctypes.POINTER(moe_mx_weights_t))]


class moe_saved_t(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("logits", "topk_idx", "topk_w", "counts", "offsets", "row_slot",
                                   "slot_row", "x_perm", "a", "b", "h", "o", "sa", "sb", "sh")]


def _declare(lib):
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [_i]
    lib.moe_version.restype = _i
    lib.moe_version.argtypes = []
    lib.moe_trace_events.restype = _i
    lib.moe_trace_events.argtypes = [ctypes.POINTER(_vp)]
    lib.moe_kernel_launches.restype = ctypes.c_ulonglong
    lib.moe_kernel_launches.argtypes = []
    lib.moe_selftest_wait_timeout.restype = _i
    lib.moe_selftest_wait_timeout.argtypes = [_u, _vp, _vp]
    lib.moe_route.restype = _i
    lib.moe_route.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _szp, _u, _vp]
    lib.moe_dispatch.restype = _i
    lib.moe_dispatch.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _szp, _u,
                                 _vp]
    lib.moe_dispatch_noalloc.restype = _i
    lib.moe_dispatch_noalloc.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _u,
                                         _vp]
    lib.moe_dispatch_fp8.restype = _i
    lib.moe_dispatch_fp8.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _szp, _u, _vp]
    lib.moe_dequant_fp8.restype = _i
    lib.moe_dequant_fp8.argtypes = [_vp, _vp, _i, _i, _vp, _vp]
    _ll = ctypes.c_longlong
    lib.moe_quantize_mx.restype = _i
    lib.moe_quantize_mx.argtypes = [_vp, _ll, _i, _vp, _vp, _vp]
    lib.moe_dispatch_mx.restype = _i
    lib.moe_dispatch_mx.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _szp, _u, _vp]
    lib.moe_grouped_ffn_mx.restype = _i
    lib.moe_grouped_ffn_mx.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _vp, _vp, _vp, _vp, _szp, _u, _vp]
    lib.moe_prepack_weights.restype = _i
    lib.moe_prepack_weights.argtypes = [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp]
    lib.moe_grouped_ffn.restype = _i
    lib.moe_grouped_ffn.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _szp, _u, _vp]
    lib.moe_grouped_ffn_fp8.restype = _i
    lib.moe_grouped_ffn_fp8.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _szp, _u, _vp]
    lib.moe_combine.restype = _i
    lib.moe_combine.argtypes = [_vp, _vp, _vp, _i, _i, _i, _vp, _vp]
    lib.moe_layer_fwd.restype = _i
    lib.moe_layer_fwd.argtypes = [ctypes.POINTER(moe_layer_t), _vp, _vp,
                                  ctypes.POINTER(moe_saved_t), _vp, _szp, _u, _vp]
    lib.moe_layer_bwd.restype = _i
    lib.moe_layer_bwd.argtypes = [ctypes.POINTER(moe_layer_t), _vp, ctypes.POINTER(moe_saved_t),
                                  _vp, _vp, _vp, _vp, _vp, _vp, _vp, _szp, _u, _vp]


_LIB = None


def lib():
    """The loaded library (built in-tree on first use)."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        handle = ctypes.CDLL(path)
        _declare(handle)
        _LIB = handle
    return _LIB


def library_path() -> str:
    return _build.LIB


# ---------------------------------------------------------------- marshalling
def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(st, where):
    if st != MOE_OK:
        raise MoeError(st, where, int(lib().moe_last_cuda_error()) if st == 6 else 0)


def _dt(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


# ---------------------------------------------------------------- entry points
def route_ws_bytes(T, d, E, R) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_route(None, None, None, T, d, E, R, None, None, None, None, ctypes.byref(n),
                           0, None), "moe_route(ws query)")
    return n.value


def moe_route(x, w_gate, bias, logits, topk_idx, topk_w, ws=None, flags=0, stream=None):
    """Router; ``ws`` may be None with MOE_LOGITS_IN (else see route_ws_bytes)."""
    T, E = logits.shape
    R = topk_idx.shape[1]
    d = x.shape[1] if x is not None else 0
    _dt(x, torch.bfloat16, "x"); _dt(w_gate, torch.float32, "w_gate"); _dt(bias, torch.float32, "bias")
    _dt(logits, torch.float32, "logits"); _dt(topk_idx, torch.int32, "topk_idx")
    _dt(topk_w, torch.float32, "topk_w")
    n = ctypes.c_size_t(0 if ws is None else ws.numel())
    st = lib().moe_route(_p(x), _p(w_gate), _p(bias), T, d, E, R, _p(logits), _p(topk_idx),
                         _p(topk_w), _p(ws), ctypes.byref(n), flags, _stream(stream))
    _check(st, "moe_route")


def dispatch_ws_bytes(T, d, E, R) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_dispatch(None, None, T, d, E, R, None, None, None, None, None, None,
                              ctypes.byref(n), 0, None), "moe_dispatch(ws query)")
    return n.value


def moe_dispatch(x, topk_idx, E, counts, offsets, row_slot, slot_row, x_perm, ws, flags=0,
                 stream=None):
    T, R = topk_idx.shape
    d = x.shape[1] if x is not None else (x_perm.shape[1] if x_perm is not None else 8)
    _dt(x, torch.bfloat16, "x"); _dt(x_perm, torch.bfloat16, "x_perm")
    for name, t in (("topk_idx", topk_idx), ("counts", counts), ("offsets", offsets),
                    ("row_slot", row_slot), ("slot_row", slot_row)):
        _dt(t, torch.int32, name)
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_dispatch(_p(x), _p(topk_idx), T, d, E, R, _p(counts), _p(offsets),
                            _p(row_slot), _p(slot_row), _p(x_perm), _p(ws), ctypes.byref(n),
                            flags, _stream(stream))
    _check(st, "moe_dispatch")


def moe_dispatch_noalloc(x, topk_idx, E, counts, offsets, row_slot, slot_row, x_perm, flags=0,
                         stream=None):
    """moe_dispatch with the library's static scratch (no workspace argument)."""
    T, R = topk_idx.shape
    d = x.shape[1] if x is not None else (x_perm.shape[1] if x_perm is not None else 8)
    _dt(x, torch.bfloat16, "x"); _dt(x_perm, torch.bfloat16, "x_perm")
    for name, t in (("topk_idx", topk_idx), ("counts", counts), ("offsets", offsets),
                    ("row_slot", row_slot), ("slot_row", slot_row)):
        _dt(t, torch.int32, name)
    st = lib().moe_dispatch_noalloc(_p(x), _p(topk_idx), T, d, E, R, _p(counts), _p(offsets),
                                    _p(row_slot), _p(slot_row), _p(x_perm), flags,
                                    _stream(stream))
    _check(st, "moe_dispatch_noalloc")


def moe_dispatch_fp8(x, topk_idx, E, counts, offsets, row_slot, slot_row, xq_perm, xscale_perm,
                     ws, flags=0, stream=None):
    """Block-scaled fp8 dispatch: E4M3 codes (uint8 [N,d]) and fp32 scales [N, d/128]."""
    T, R = topk_idx.shape
    d = x.shape[1]
    _dt(x, torch.bfloat16, "x"); _dt(xq_perm, torch.uint8, "xq_perm")
    _dt(xscale_perm, torch.float32, "xscale_perm")
    for name, t in (("topk_idx", topk_idx), ("counts", counts), ("offsets", offsets),
                    ("row_slot", row_slot), ("slot_row", slot_row)):
        _dt(t, torch.int32, name)
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_dispatch_fp8(_p(x), _p(topk_idx), T, d, E, R, _p(counts), _p(offsets),
                                _p(row_slot), _p(slot_row), _p(xq_perm), _p(xscale_perm), _p(ws),
                                ctypes.byref(n), flags, _stream(stream))
    _check(st, "moe_dispatch_fp8")


def moe_dequant_fp8(xq, xscale, out, stream=None):
    N, d = xq.shape
    _dt(xq, torch.uint8, "xq"); _dt(xscale, torch.float32, "xscale"); _dt(out, torch.bfloat16, "out")
    _check(lib().moe_dequant_fp8(_p(xq), _p(xscale), N, d, _p(out), _stream(stream)),
           "moe_dequant_fp8")


def grouped_ffn_ws_bytes(N, d, f, E) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_grouped_ffn(None, None, N, d, f, E, None, None, None, None, None, None, None,
                                 None, None, ctypes.byref(n), 0, None), "moe_grouped_ffn(ws query)")
    return n.value


def moe_grouped_ffn(x_perm, offsets, W1, W3, W2, h, out, ws, a_save=None, b_save=None, flags=0,
                    stream=None, row_scale=None):
    N, d = x_perm.shape
    E, f, _ = W1.shape
    for name, t in (("x_perm", x_perm), ("W1", W1), ("W3", W3), ("W2", W2), ("h", h),
                    ("out", out), ("a_save", a_save), ("b_save", b_save)):
        _dt(t, torch.bfloat16, name)
    _dt(offsets, torch.int32, "offsets")
    _dt(row_scale, torch.float32, "row_scale")
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_grouped_ffn(_p(x_perm), _p(offsets), N, d, f, E, _p(W1), _p(W3), _p(W2),
                               _p(row_scale), _p(a_save), _p(b_save), _p(h), _p(out), _p(ws),
                               ctypes.byref(n), flags, _stream(stream))
    _check(st, "moe_grouped_ffn")


def grouped_ffn_fp8_ws_bytes(N, d, f, E) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_grouped_ffn_fp8(None, None, None, N, d, f, E, None, None, None, None, None,
                                     None, None, None, None, ctypes.byref(n), 0, None),
           "moe_grouped_ffn_fp8(ws query)")
    return n.value


def moe_grouped_ffn_fp8(xq_perm, xscale_perm, offsets, W1, W3, W2, h, out, ws, a_save=None,
                        b_save=None, flags=0, stream=None, row_scale=None):
    """moe_grouped_ffn on block-scaled fp8 rows (uint8 codes [N, d], fp32 scales [N, d/128])."""
    N, d = xq_perm.shape
    E, f, _ = W1.shape
    _dt(xq_perm, torch.uint8, "xq_perm")
    _dt(xscale_perm, torch.float32, "xscale_perm")
    for name, t in (("W1", W1), ("W3", W3), ("W2", W2), ("h", h), ("out", out),
                    ("a_save", a_save), ("b_save", b_save)):
        _dt(t, torch.bfloat16, name)
    _dt(offsets, torch.int32, "offsets")
    _dt(row_scale, torch.float32, "row_scale")
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_grouped_ffn_fp8(_p(xq_perm), _p(xscale_perm), _p(offsets), N, d, f, E, _p(W1),
                                   _p(W3), _p(W2), _p(row_scale), _p(a_save), _p(b_save), _p(h),
                                   _p(out), _p(ws), ctypes.byref(n), flags, _stream(stream))
    _check(st, "moe_grouped_ffn_fp8")


def mx_scale_row_bytes(K: int) -> int:
    """Bytes per row of microscaled fp8 scales: K/32, rounded up to a multiple of 16."""
    return -(-K // 512) * 16


def moe_quantize_mx(W, codes, scales, stream=None):
    """Microscaled fp8 codes (uint8 [rows, K]) and scales (uint8 [rows, sk]) of a bf16
    matrix [..., K] along its last dimension."""
    K = W.shape[-1]
    rows = W.numel() // K
    _dt(W, torch.bfloat16, "W"); _dt(codes, torch.uint8, "codes"); _dt(scales, torch.uint8, "scales")
    _check(lib().moe_quantize_mx(_p(W), rows, K, _p(codes), _p(scales), _stream(stream)),
           "moe_quantize_mx")


def moe_dispatch_mx(x, topk_idx, E, counts, offsets, row_slot, slot_row, xq_perm, xscale_perm, ws,
                    flags=0, stream=None):
    """Dispatch with rows in microscaled fp8: codes uint8 [N, d], scales uint8 [N, sk(d)]."""
    T, R = topk_idx.shape
    d = x.shape[1]
    _dt(x, torch.bfloat16, "x"); _dt(xq_perm, torch.uint8, "xq_perm")
    _dt(xscale_perm, torch.uint8, "xscale_perm")
    for name, t in (("topk_idx", topk_idx), ("counts", counts), ("offsets", offsets),
                    ("row_slot", row_slot), ("slot_row", slot_row)):
        _dt(t, torch.int32, name)
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_dispatch_mx(_p(x), _p(topk_idx), T, d, E, R, _p(counts), _p(offsets),
                               _p(row_slot), _p(slot_row), _p(xq_perm), _p(xscale_perm), _p(ws),
                               ctypes.byref(n), flags, _stream(stream))
    _check(st, "moe_dispatch_mx")


def grouped_ffn_mx_ws_bytes(N, d, f, E) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_grouped_ffn_mx(None, None, None, N, d, f, E, None, None, None, None, None,
                                    None, None, None, None, None, None, ctypes.byref(n), 0, None),
           "moe_grouped_ffn_mx(ws query)")
    return n.value


def moe_grouped_ffn_mx(xq, xs, offsets, W1q, W1s, W3q, W3s, W2q, W2s, out, ws, hq=None, hs=None,
                       row_scale=None, flags=0, stream=None):
    """The grouped SwiGLU FFN on microscaled fp8 operands (see include/moe.h).
    W1q, W3q: uint8 [E, f, d] (scales [E, f, sk(d)]); W2q: uint8 [E, d, f] (scales [E, d, sk(f)])."""
    N, d = xq.shape
    E, f, _ = W1q.shape
    for name, t in (("xq", xq), ("xs", xs), ("W1q", W1q), ("W1s", W1s), ("W3q", W3q),
                    ("W3s", W3s), ("W2q", W2q), ("W2s", W2s), ("hq", hq), ("hs", hs)):
        _dt(t, torch.uint8, name)
    _dt(out, torch.bfloat16, "out")
    _dt(offsets, torch.int32, "offsets")
    _dt(row_scale, torch.float32, "row_scale")
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_grouped_ffn_mx(_p(xq), _p(xs), _p(offsets), N, d, f, E, _p(W1q), _p(W1s),
                                  _p(W3q), _p(W3s), _p(W2q), _p(W2s), _p(row_scale), _p(hq),
                                  _p(hs), _p(out), _p(ws), ctypes.byref(n), flags, _stream(stream))
    _check(st, "moe_grouped_ffn_mx")


def moe_prepack_weights(W1, W3, W2, W1p, W3p, W2p, stream=None):
    """Forward weight tiles (see include/moe.h); returns nothing, fills W1p, W3p, W2p."""
    E, f, d = W1.shape
    for name, t in (("W1", W1), ("W3", W3), ("W2", W2), ("W1p", W1p), ("W3p", W3p), ("W2p", W2p)):
        _dt(t, torch.bfloat16, name)
    _check(lib().moe_prepack_weights(_p(W1), _p(W3), _p(W2), E, d, f, _p(W1p), _p(W3p), _p(W2p),
                                     _stream(stream)), "moe_prepack_weights")


def moe_combine(expert_out, slot_row, topk_w, y, R, stream=None):
    T, d = y.shape
    _dt(expert_out, torch.bfloat16, "expert_out"); _dt(y, torch.bfloat16, "y")
    _dt(slot_row, torch.int32, "slot_row"); _dt(topk_w, torch.float32, "topk_w")
    st = lib().moe_combine(_p(expert_out), _p(slot_row), _p(topk_w), T, d, R, _p(y),
                           _stream(stream))
    _check(st, "moe_combine")


# ---------------------------------------------------------------- layer
class Shared:
    """A shared expert (moe_shared_t): bf16 weights W1, W3 [fs, d], W2 [d, fs]
    and, for moe_layer_bwd, fp32 gradient buffers of the same shapes."""

    def __init__(self, W1, W3, W2, dW1=None, dW3=None, dW2=None):
        self.W1, self.W3, self.W2 = W1, W3, W2
        self.dW1, self.dW3, self.dW2 = dW1, dW3, dW2
        self.fs = W1.shape[0]
        self.c = moe_shared_t(self.fs, _p(W1), _p(W3), _p(W2), _p(dW1), _p(dW3), _p(dW2))


class MxWeights:
    """The expert weights in microscaled fp8 (moe_mx_weights_t), quantised on the device
    from bf16 W1, W3 [E, f, d] and W2 [E, d, f] with moe_quantize_mx."""

    def __init__(self, W1, W3, W2, stream=None):
        def q(W):
            K = W.shape[-1]
            codes = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
            scales = torch.empty(W.shape[:-1] + (mx_scale_row_bytes(K),), dtype=torch.uint8,
                                 device=W.device)
            moe_quantize_mx(W, codes, scales, stream)
            return codes, scales
        (self.W1q, self.W1s), (self.W3q, self.W3s), (self.W2q, self.W2s) = q(W1), q(W3), q(W2)
        self.c = moe_mx_weights_t(*[_p(getattr(self, n)) for n, _ in moe_mx_weights_t._fields_])


class Layer:
    """Parameters of one MoE layer (device tensors) and their C struct."""

    def __init__(self, w_gate, bias, W1, W3, W2, R, T, shared: Shared = None,
                 mx: MxWeights = None):
        self.w_gate, self.bias, self.W1, self.W3, self.W2 = w_gate, bias, W1, W3, W2
        self.E, self.f, self.d = W1.shape
        self.R, self.T = R, T
        self.shared = shared
        self.mx = mx
        self.c = moe_layer_t(T, self.d, self.E, R, self.f, _p(w_gate), _p(bias), _p(W1), _p(W3),
                             _p(W2), ctypes.pointer(shared.c) if shared is not None else None,
                             ctypes.pointer(mx.c) if mx is not None else None)

    def with_tokens(self, T):
        return Layer(self.w_gate, self.bias, self.W1, self.W3, self.W2, self.R, T, self.shared,
                     self.mx)


class Saved:
    """Caller-owned forward intermediates (allocated here with torch)."""

    def __init__(self, layer: Layer, device, train=True):
        T, d, E, R, f = layer.T, layer.d, layer.E, layer.R, layer.f
        N = T * R
        z = dict(device=device)
        self.logits = torch.empty((T, E), dtype=torch.float32, **z)
        self.topk_idx = torch.empty((T, R), dtype=torch.int32, **z)
        self.topk_w = torch.empty((T, R), dtype=torch.float32, **z)
        self.counts = torch.empty((E,), dtype=torch.int32, **z)
        self.offsets = torch.empty((E + 1,), dtype=torch.int32, **z)
        self.row_slot = torch.empty((N,), dtype=torch.int32, **z)
        self.slot_row = torch.empty((N,), dtype=torch.int32, **z)
        self.x_perm = torch.empty((N, d), dtype=torch.bfloat16, **z)
        self.a = torch.empty((N, f), dtype=torch.bfloat16, **z) if train else None
        self.b = torch.empty((N, f), dtype=torch.bfloat16, **z) if train else None
        self.h = torch.empty((N, f), dtype=torch.bfloat16, **z)
        self.o = torch.empty((N, d), dtype=torch.bfloat16, **z)
        fs = layer.shared.fs if layer.shared is not None else 0
        for n in ("sa", "sb", "sh"):
            setattr(self, n, torch.empty((T, fs), dtype=torch.bfloat16, **z)
                    if fs and train else None)
        self.c = moe_saved_t(*[_p(getattr(self, n)) for n, _ in moe_saved_t._fields_])


def layer_fwd_ws_bytes(layer: Layer, flags=0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_layer_fwd(ctypes.byref(layer.c), None, None, None, None, ctypes.byref(n),
                               flags, None), "moe_layer_fwd(ws query)")
    return n.value


def layer_bwd_ws_bytes(layer: Layer) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_layer_bwd(ctypes.byref(layer.c), None, None, None, None, None, None, None,
                               None, None, ctypes.byref(n), 0, None), "moe_layer_bwd(ws query)")
    return n.value


def workspace(nbytes: int, device="cuda"):
    """A device byte buffer for the workspace arguments (torch allocates it)."""
    return torch.empty((max(int(nbytes), 256),), dtype=torch.uint8, device=device)


def moe_layer_fwd(layer: Layer, x, y, saved: Saved, ws, flags=0, stream=None):
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_layer_fwd(ctypes.byref(layer.c), _p(x), _p(y), ctypes.byref(saved.c), _p(ws),
                             ctypes.byref(n), flags, _stream(stream))
    _check(st, "moe_layer_fwd")


def moe_layer_bwd(layer: Layer, x, saved: Saved, dy, dx, dW_gate, dW1, dW3, dW2, ws, flags=0,
                  stream=None):
    n = ctypes.c_size_t(ws.numel())
    st = lib().moe_layer_bwd(ctypes.byref(layer.c), _p(x), ctypes.byref(saved.c), _p(dy), _p(dx),
                             _p(dW_gate), _p(dW1), _p(dW3), _p(dW2), _p(ws), ctypes.byref(n),
                             flags, _stream(stream))
    _check(st, "moe_layer_bwd")


class StageTrace:
    """CUDA events recorded by the library around each layer stage (moe_trace_events).

    ``arm()`` makes the library record into this trace's events until
    ``disarm()``; ``elapsed_ms()`` (after the work completed) gives each
    stage's device time, or None for stages that did not run.
    """

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(STAGES))]
        self._arr = None

    def arm(self):
        # torch creates an event's CUDA handle at its first record(): record every
        # event once (unused stages then read as ~0) before handing the handles over
        for e in self.events:
            e.record()
        self._arr = (_vp * len(self.events))(*[e.cuda_event for e in self.events])
        _check(lib().moe_trace_events(self._arr), "moe_trace_events")

    @staticmethod
    def disarm():
        _check(lib().moe_trace_events(None), "moe_trace_events")

    def elapsed_ms(self):
        out = {}
        for i, name in enumerate(STAGES):
            out[name] = self.events[2 * i].elapsed_time(self.events[2 * i + 1])
        return out


def kernel_launches() -> int:
    return int(lib().moe_kernel_launches())


def status_string(st: int) -> str:
    return lib().moe_status_string(st).decode()


def loaded_path() -> str:
    return os.path.realpath(_build.LIB)
