"""Thin ctypes binding of libmlp_tp.so (include/mlp_tp.h), same names as the C ABI.

Argument marshalling only: tensors become device pointers, the stream defaults to torch's
current stream, and a non-OK status raises MlpError. Every step of the block runs in the
library's CUDA kernels; there is no Python or CPU fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmlp_tp.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "mlp_tp.h")

_lock = threading.Lock()
_lib = None

_STATUS = {0: "MLP_OK", 1: "MLP_EINVAL", 2: "MLP_ESHAPE", 3: "MLP_EALIGN", 4: "MLP_ECUDA",
           5: "MLP_ETIMEOUT", 6: "MLP_EUNSUPPORTED", 7: "MLP_EWORKSPACE"}
STATUS_CODES = {v: k for k, v in _STATUS.items()}


class MlpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = _STATUS.get(status, f"status {status}")
        msg = lib().mlp_tp_status_string(status).decode()
        super().__init__(f"{where}: {msg}")


def header_functions() -> list[str]:
    """Names of the functions include/mlp_tp.h declares."""
    src = open(HEADER).read()
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mlp_tp_\w+)\s*\(", src, re.M)


def lib() -> ctypes.CDLL:
    """Load libmlp_tp.so (built by build.py); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m megatron_tensor_transformer_tcgen05_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, sz, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_ulonglong
            L.mlp_tp_forward.restype = i32
            L.mlp_tp_forward.argtypes = [vp] * 5 + [i32] * 4 + [vp] * 3 + [vp, sz, vp]
            L.mlp_tp_forward_workspace_bytes.restype = sz
            L.mlp_tp_forward_workspace_bytes.argtypes = []
            L.mlp_tp_backward.restype = i32
            L.mlp_tp_backward.argtypes = [vp] * 6 + [i32] * 4 + [vp] * 5 + [vp, sz, vp]
            L.mlp_tp_workspace_bytes.restype = sz
            L.mlp_tp_workspace_bytes.argtypes = [i32] * 4
            L.mlp_tp_query_device_status.restype = i32
            L.mlp_tp_query_device_status.argtypes = [vp]
            L.mlp_tp_last_device_code.restype = i32
            L.mlp_tp_last_device_code.argtypes = []
            L.mlp_tp_last_device_where.restype = i32
            L.mlp_tp_last_device_where.argtypes = [vp, vp, vp, vp]
            L.mlp_tp_status_string.restype = ctypes.c_char_p
            L.mlp_tp_status_string.argtypes = [i32]
            L.mlp_tp_launch_count.restype = ctypes.c_longlong
            L.mlp_tp_launch_count.argtypes = []
            L.mlp_tp_selftest_wait_timeout.restype = i32
            L.mlp_tp_selftest_wait_timeout.argtypes = [u64, vp]
            L.mlp_tp_timing_enable.restype = i32
            L.mlp_tp_timing_enable.argtypes = [i32]
            L.mlp_tp_timing_collect.restype = i32
            L.mlp_tp_timing_collect.argtypes = [vp, vp]
            L.mlp_tp_kernel_name.restype = ctypes.c_char_p
            L.mlp_tp_kernel_name.argtypes = [i32]
            L.mlp_tp_forward_residual_dropout.restype = i32
            L.mlp_tp_forward_residual_dropout.argtypes = ([vp] * 6 + [i32] * 4 + [ctypes.c_double, u64, u64] +
                                                          [vp] * 3 + [vp])
            L.mlp_tp_dropout_backward.restype = i32
            L.mlp_tp_dropout_backward.argtypes = [vp, i32, i32, ctypes.c_double, u64, u64, vp, vp]
            L.mlp_tp_swiglu_forward.restype = i32
            L.mlp_tp_swiglu_forward.argtypes = [vp] * 4 + [i32] * 4 + [vp] * 4 + [vp, sz, vp]
            L.mlp_tp_swiglu_backward.restype = i32
            L.mlp_tp_swiglu_backward.argtypes = [vp] * 8 + [i32] * 4 + [vp] * 5 + [sz, vp]
            L.mlp_tp_swiglu_workspace_bytes.restype = sz
            L.mlp_tp_swiglu_workspace_bytes.argtypes = [i32] * 4
            L.mlp_tp_bias_grads_noalloc.restype = i32
            L.mlp_tp_bias_grads_noalloc.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
            L.mlp_tp_attn_forward.restype = i32
            L.mlp_tp_attn_forward.argtypes = [vp] * 3 + [i32] * 7 + [vp] * 4 + [vp, sz, vp]
            L.mlp_tp_attn_workspace_bytes.restype = sz
            L.mlp_tp_attn_workspace_bytes.argtypes = [i32] * 6
            L.mlp_tp_attn_backward.restype = i32
            L.mlp_tp_attn_backward.argtypes = [vp] * 7 + [i32] * 7 + [vp] * 4 + [sz, vp]
            L.mlp_tp_recompute_workspace_bytes.restype = sz
            L.mlp_tp_recompute_workspace_bytes.argtypes = [i32] * 4
            L.mlp_tp_backward_recompute.restype = i32
            L.mlp_tp_backward_recompute.argtypes = [vp] * 5 + [i32] * 4 + [vp] * 5 + [vp, sz, vp]
            L.mlp_tp_forward_recompute.restype = i32
            L.mlp_tp_forward_recompute.argtypes = [vp] * 5 + [i32] * 4 + [vp] * 2 + [vp, sz, vp]
            _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MlpError(status, where)


def mlp_tp_forward(X, A, a, B, b, T: int, h: int, f: int, t: int, H, G, Y, workspace, workspace_bytes: int,
                   stream=None) -> None:
    _check(lib().mlp_tp_forward(_ptr(X), _ptr(A), _ptr(a), _ptr(B), _ptr(b), T, h, f, t,
                                _ptr(H), _ptr(G), _ptr(Y), _ptr(workspace), workspace_bytes, _stream(stream)),
           "mlp_tp_forward")


def mlp_tp_forward_workspace_bytes() -> int:
    return int(lib().mlp_tp_forward_workspace_bytes())


def mlp_tp_backward(X, A, B, H, G, dY, T: int, h: int, f: int, t: int, dX, dA, dB, da, db,
                    workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib().mlp_tp_backward(_ptr(X), _ptr(A), _ptr(B), _ptr(H), _ptr(G), _ptr(dY), T, h, f, t,
                                 _ptr(dX), _ptr(dA), _ptr(dB), _ptr(da), _ptr(db), _ptr(workspace),
                                 workspace_bytes, _stream(stream)), "mlp_tp_backward")


def mlp_tp_workspace_bytes(T: int, h: int, f: int, t: int) -> int:
    return int(lib().mlp_tp_workspace_bytes(T, h, f, t))


def mlp_tp_query_device_status(stream=None) -> int:
    """Returns the raw mlp_status (0 = OK, 5 = a device wait ran out)."""
    return int(lib().mlp_tp_query_device_status(_stream(stream)))


def mlp_tp_last_device_code() -> int:
    return int(lib().mlp_tp_last_device_code())


def mlp_tp_last_device_where() -> dict:
    """Where the bounded wait behind the last MLP_ETIMEOUT gave up."""
    v = [ctypes.c_int() for _ in range(4)]
    code = lib().mlp_tp_last_device_where(*[ctypes.byref(x) for x in v])
    return {"code": int(code), "block": v[0].value, "thread": v[1].value, "tile": v[2].value,
            "kblock": v[3].value}


def mlp_tp_status_string(status: int) -> str:
    return lib().mlp_tp_status_string(status).decode()


def mlp_tp_launch_count() -> int:
    return int(lib().mlp_tp_launch_count())


def mlp_tp_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(lib().mlp_tp_selftest_wait_timeout(limit_ns, _stream(stream)),
           "mlp_tp_selftest_wait_timeout")


MLP_NUM_KERNELS = 19


def mlp_tp_timing_enable(on: bool) -> None:
    _check(lib().mlp_tp_timing_enable(int(bool(on))), "mlp_tp_timing_enable")


def mlp_tp_timing_collect() -> tuple[list[float], list[int]]:
    ms = (ctypes.c_double * MLP_NUM_KERNELS)()
    counts = (ctypes.c_int * MLP_NUM_KERNELS)()
    _check(lib().mlp_tp_timing_collect(ms, counts), "mlp_tp_timing_collect")
    return list(ms), list(counts)


def mlp_tp_kernel_name(kernel: int) -> str:
    return lib().mlp_tp_kernel_name(kernel).decode()


def mlp_tp_bias_grads_noalloc(dH, dY, T: int, h: int, f: int, da, db, stream=None) -> None:
    """da = colsum(dH), db = colsum(dY) with no workspace: the library's fixed device
    scratch array holds the partial sums (see include/mlp_tp.h for its limit)."""
    _check(lib().mlp_tp_bias_grads_noalloc(_ptr(dH), _ptr(dY), T, h, f, _ptr(da), _ptr(db),
                                           _stream(stream)), "mlp_tp_bias_grads_noalloc")


def mlp_tp_forward_residual_dropout(X, A, a, B, b, R, T: int, h: int, f: int, t: int, p: float, seed: int,
                                    offset: int, H, G, Z, stream=None) -> None:
    _check(lib().mlp_tp_forward_residual_dropout(_ptr(X), _ptr(A), _ptr(a), _ptr(B), _ptr(b), _ptr(R), T, h,
                                                 f, t, float(p), int(seed), int(offset), _ptr(H), _ptr(G),
                                                 _ptr(Z), _stream(stream)), "mlp_tp_forward_residual_dropout")


def mlp_tp_dropout_backward(dZ, T: int, h: int, p: float, seed: int, offset: int, dY, stream=None) -> None:
    _check(lib().mlp_tp_dropout_backward(_ptr(dZ), T, h, float(p), int(seed), int(offset), _ptr(dY),
                                         _stream(stream)), "mlp_tp_dropout_backward")


def mlp_tp_swiglu_forward(X, A, Wg, B, T: int, h: int, f: int, t: int, Ha, Hg, U, Y, workspace, workspace_bytes: int,
                          stream=None) -> None:
    _check(lib().mlp_tp_swiglu_forward(_ptr(X), _ptr(A), _ptr(Wg), _ptr(B), T, h, f, t, _ptr(Ha), _ptr(Hg),
                                       _ptr(U), _ptr(Y), _ptr(workspace), workspace_bytes, _stream(stream)),
           "mlp_tp_swiglu_forward")


def mlp_tp_swiglu_backward(X, A, Wg, B, Ha, Hg, U, dY, T: int, h: int, f: int, t: int, dX, dA, dWg, dB,
                           workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib().mlp_tp_swiglu_backward(_ptr(X), _ptr(A), _ptr(Wg), _ptr(B), _ptr(Ha), _ptr(Hg), _ptr(U), _ptr(dY),
                                        T, h, f, t, _ptr(dX), _ptr(dA), _ptr(dWg), _ptr(dB), _ptr(workspace),
                                        workspace_bytes, _stream(stream)), "mlp_tp_swiglu_backward")


def mlp_tp_swiglu_workspace_bytes(T: int, h: int, f: int, t: int) -> int:
    return int(lib().mlp_tp_swiglu_workspace_bytes(T, h, f, t))


def mlp_tp_attn_forward(X, Wqkv, Wo, b: int, s: int, h: int, a: int, d: int, t: int, causal: bool, QKV, C, L, Y,
                        workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib().mlp_tp_attn_forward(_ptr(X), _ptr(Wqkv), _ptr(Wo), b, s, h, a, d, t, int(bool(causal)), _ptr(QKV),
                                     _ptr(C), _ptr(L), _ptr(Y), _ptr(workspace), workspace_bytes, _stream(stream)),
           "mlp_tp_attn_forward")


def mlp_tp_attn_workspace_bytes(b: int, s: int, h: int, a: int, d: int, t: int) -> int:
    return int(lib().mlp_tp_attn_workspace_bytes(b, s, h, a, d, t))


def mlp_tp_attn_backward(X, Wqkv, Wo, QKV, C, L, dY, b: int, s: int, h: int, a: int, d: int, t: int, causal: bool,
                         dX, dWqkv, dWo, workspace, workspace_bytes: int, stream=None) -> None:
    _check(lib().mlp_tp_attn_backward(_ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(QKV), _ptr(C), _ptr(L), _ptr(dY), b, s, h,
                                      a, d, t, int(bool(causal)), _ptr(dX), _ptr(dWqkv), _ptr(dWo), _ptr(workspace),
                                      workspace_bytes, _stream(stream)), "mlp_tp_attn_backward")


def mlp_tp_forward_recompute(X, A, a, B, b, T: int, h: int, f: int, t: int, H, Y, workspace, workspace_bytes: int,
                             stream=None) -> None:
    _check(lib().mlp_tp_forward_recompute(_ptr(X), _ptr(A), _ptr(a), _ptr(B), _ptr(b), T, h, f, t, _ptr(H), _ptr(Y),
                                          _ptr(workspace), workspace_bytes, _stream(stream)), "mlp_tp_forward_recompute")


def mlp_tp_recompute_workspace_bytes(T: int, h: int, f: int, t: int) -> int:
    return int(lib().mlp_tp_recompute_workspace_bytes(T, h, f, t))


def mlp_tp_backward_recompute(X, A, B, H, dY, T: int, h: int, f: int, t: int, dX, dA, dB, da, db, workspace,
                              workspace_bytes: int, stream=None) -> None:
    _check(lib().mlp_tp_backward_recompute(_ptr(X), _ptr(A), _ptr(B), _ptr(H), _ptr(dY), T, h, f, t, _ptr(dX),
                                           _ptr(dA), _ptr(dB), _ptr(da), _ptr(db), _ptr(workspace), workspace_bytes,
                                           _stream(stream)), "mlp_tp_backward_recompute")
