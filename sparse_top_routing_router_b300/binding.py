"""ctypes binding of libmoe.so: the same names as the C ABI (include/moe.h), taking
torch tensors.  Argument marshalling only - every step of the forward runs in the
library's CUDA kernels.  There is no fallback: if the library is missing, `lib()`
raises.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_DEVICE_INDEX = -5
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_DTYPE_BF16, MOE_DTYPE_F32 = 0, 1
MOE_TEST_HOOK_NONE, MOE_TEST_HOOK_WITHHOLD_LOAD = 0, 1

KERNEL_NAMES = ["router_logits", "router_select", "dispatch_count", "dispatch_scan",
                "dispatch_scatter", "dispatch_gather", "expert_gate_up", "expert_down",
                "combine", "balance_stats", "bias_update"]
MOE_KERNEL_COUNT = len(KERNEL_NAMES)

EXPORTS = ["moe_ctx_create", "moe_ctx_destroy", "moe_workspace_bytes", "moe_workspace_init",
           "moe_capacity", "moe_router_topk", "moe_dispatch", "moe_dispatch_static",
           "moe_grouped_swiglu",
           "moe_combine", "moe_balance_stats", "moe_bias_update", "moe_get_device_status",
           "moe_expert_choice", "moe_gather_rows", "moe_quantize_fp8",
           "moe_grouped_swiglu_fp8",
           "moe_ctx_set_tracing", "moe_ctx_trace_read", "moe_ctx_set_test_hook",
           "moe_kernel_name",
           "moe_status_string", "moe_last_error_detail", "moe_version"]


class RouterDesc(C.Structure):
    _fields_ = [("T", C.c_int), ("H", C.c_int), ("E", C.c_int), ("k", C.c_int),
                ("score", C.c_int), ("renorm", C.c_int), ("x_dtype", C.c_int),
                ("n_groups", C.c_int), ("topk_groups", C.c_int)]


class ExpertDesc(C.Structure):
    _fields_ = [("T", C.c_int), ("H", C.c_int), ("E", C.c_int), ("I", C.c_int),
                ("k", C.c_int), ("dtype", C.c_int), ("has_shared", C.c_int)]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn}: status {status} ({status_string(status)}): {detail}")
        self.status = status


_lib: Optional[C.CDLL] = None


def lib() -> C.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run "
                           "`python -m sparse_top_routing_router_b300.build`")
    L = C.CDLL(LIB_PATH)
    vp, i, sz, d = C.c_void_p, C.c_int, C.c_size_t, C.c_double
    L.moe_ctx_create.argtypes = [C.POINTER(vp), i]
    L.moe_ctx_destroy.argtypes = [vp]
    L.moe_ctx_destroy.restype = None
    L.moe_workspace_bytes.argtypes = [i] * 7
    L.moe_workspace_bytes.restype = sz
    L.moe_workspace_init.argtypes = [vp, sz, vp]
    L.moe_capacity.argtypes = [d, i, i, i]
    L.moe_router_topk.argtypes = [vp, C.POINTER(RouterDesc), vp, vp, vp, vp, vp, vp, vp, vp,
                                  vp, sz, vp]
    L.moe_dispatch.argtypes = [vp, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_dispatch_static.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_grouped_swiglu.argtypes = [vp, C.POINTER(ExpertDesc)] + [vp] * 12 + [sz, vp]
    L.moe_combine.argtypes = [vp, i, i, i, vp, vp, vp, vp, vp, vp, vp]
    L.moe_balance_stats.argtypes = [vp, i, i, i, vp, vp, vp, d, vp, vp, vp, vp]
    L.moe_bias_update.argtypes = [vp, i, i, i, vp, C.c_float, vp, vp]
    L.moe_expert_choice.argtypes = [vp, C.POINTER(RouterDesc), vp, vp, vp, vp, vp, vp, vp,
                                    vp, vp, sz, vp]
    L.moe_gather_rows.argtypes = [vp, i, i, i, i, vp, vp, i, vp, vp, vp]
    L.moe_quantize_fp8.argtypes = [vp, i, i, i, vp, vp, vp, vp]
    L.moe_grouped_swiglu_fp8.argtypes = [vp, C.POINTER(ExpertDesc)] + [vp] * 18 + [sz, vp]
    L.moe_get_device_status.argtypes = [vp, vp, C.POINTER(i), i, vp]
    L.moe_ctx_set_tracing.argtypes = [vp, i]
    L.moe_ctx_set_test_hook.argtypes = [vp, i, i]
    L.moe_ctx_trace_read.argtypes = [vp, C.POINTER(i), C.POINTER(d), i]
    L.moe_kernel_name.argtypes = [i]
    L.moe_kernel_name.restype = C.c_char_p
    L.moe_status_string.argtypes = [i]
    L.moe_status_string.restype = C.c_char_p
    L.moe_last_error_detail.argtypes = []
    L.moe_last_error_detail.restype = C.c_char_p
    L.moe_version.argtypes = []
    for name in EXPORTS:
        if name not in ("moe_ctx_destroy", "moe_workspace_bytes", "moe_kernel_name",
                        "moe_status_string", "moe_last_error_detail"):
            getattr(L, name).restype = C.c_int
    _lib = L
    return L


def status_string(s: int) -> str:
    return lib().moe_status_string(s).decode()


def last_error_detail() -> str:
    return lib().moe_last_error_detail().decode()


def _check(fn: str, s: int) -> None:
    if s != MOE_OK:
        raise MoEError(fn, s, last_error_detail())


def _p(t: Optional[torch.Tensor]):
    """Device pointer of a contiguous CUDA tensor (None stays None).  A host tensor or a
    strided view is refused here: the kernels would read its address as device memory
    laid out row-major."""
    if t is None:
        return None
    if t.device.type != "cuda":
        raise TypeError(f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got strides {t.stride()}")
    return C.c_void_p(t.data_ptr())


def _req(t: Optional[torch.Tensor], name: str, dtype: torch.dtype, numel: int) -> None:
    """`t` (if given) holds `dtype` elements, at least `numel` of them: the library takes
    its sizes from the shapes passed beside the pointers and cannot check the buffers."""
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, the call needs {numel}")


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def x_dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    if t.dtype == torch.float32:
        return MOE_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


class Context:
    """Owns one moe_ctx bound to a CUDA device."""

    def __init__(self, device: int = 0):
        self.device = device
        h = C.c_void_p()
        _check("moe_ctx_create", lib().moe_ctx_create(C.byref(h), device))
        self.handle = h

    def close(self):
        if self.handle:
            lib().moe_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_tracing(self, enable: bool) -> None:
        _check("moe_ctx_set_tracing", lib().moe_ctx_set_tracing(self.handle, int(enable)))

    def set_test_hook(self, hook: int, wait_limit_ms: int = 0) -> None:
        _check("moe_ctx_set_test_hook",
               lib().moe_ctx_set_test_hook(self.handle, hook, wait_limit_ms))

    def trace_read(self) -> dict:
        n = MOE_KERNEL_COUNT
        launches = (C.c_int * n)()
        ms = (C.c_double * n)()
        _check("moe_ctx_trace_read", lib().moe_ctx_trace_read(self.handle, launches, ms, n))
        return {KERNEL_NAMES[i]: (launches[i], ms[i]) for i in range(n)}


def moe_workspace_bytes(T, H, E, I, k, dtype, has_shared) -> int:
    return int(lib().moe_workspace_bytes(T, H, E, I, k, dtype, int(has_shared)))


def moe_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check("moe_workspace_init", lib().moe_workspace_init(_p(ws), ws.numel() * ws.element_size(),
                                                          _stream(stream)))


def moe_capacity(c: float, T: int, k: int, E: int) -> int:
    r = lib().moe_capacity(float(c), T, k, E)
    if r < 0:
        raise MoEError("moe_capacity", r, last_error_detail())
    return r


def moe_router_topk(ctx: Context, X, Wg, k: int, score: int, renorm: bool, topk_idx,
                    topk_gate, ws, bias=None, logit_bias=None, key_gap=None,
                    prob_colsum=None, stream=None, n_groups: int = 0,
                    topk_groups: int = 0) -> None:
    T, H = X.shape
    E = Wg.shape[1]
    _req(Wg, "Wg", torch.float32, H * E)
    _req(bias, "bias", torch.float32, E)
    _req(logit_bias, "logit_bias", torch.float32, E)
    _req(topk_idx, "topk_idx", torch.int32, T * k)
    _req(topk_gate, "topk_gate", torch.float32, T * k)
    _req(key_gap, "key_gap", torch.float32, T)
    _req(prob_colsum, "prob_colsum", torch.float64, E)
    d = RouterDesc(T, H, E, k, score, int(renorm), x_dtype_code(X), n_groups, topk_groups)
    _check("moe_router_topk", lib().moe_router_topk(
        ctx.handle, C.byref(d), _p(X), _p(Wg), _p(bias), _p(logit_bias), _p(topk_idx),
        _p(topk_gate), _p(key_gap), _p(prob_colsum), _p(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_expert_choice(ctx: Context, X, Wg, k: int, score: int, offsets, row_of_slot,
                      slot_of_row, slot_gate, ws, logit_bias=None, col_gap=None,
                      stream=None) -> None:
    T, H = X.shape
    E = Wg.shape[1]
    _req(Wg, "Wg", torch.float32, H * E)
    _req(logit_bias, "logit_bias", torch.float32, E)
    _req(offsets, "offsets", torch.int32, E + 1)
    _req(row_of_slot, "row_of_slot", torch.int32, T * E)
    _req(slot_of_row, "slot_of_row", torch.int32, T * k)
    _req(slot_gate, "slot_gate", torch.float32, T * E)
    _req(col_gap, "col_gap", torch.float32, E)
    d = RouterDesc(T, H, E, k, score, 0, x_dtype_code(X), 0, 0)
    _check("moe_expert_choice", lib().moe_expert_choice(
        ctx.handle, C.byref(d), _p(X), _p(Wg), _p(logit_bias), _p(offsets), _p(row_of_slot),
        _p(slot_of_row), _p(slot_gate), _p(col_gap), _p(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_gather_rows(ctx: Context, slot_of_row, k: int, X, Xperm, ws, stream=None) -> None:
    R = slot_of_row.shape[0]
    T, H = X.shape
    _req(slot_of_row, "slot_of_row", torch.int32, R)
    _req(Xperm, "Xperm", X.dtype, R * H)
    _check("moe_gather_rows", lib().moe_gather_rows(
        ctx.handle, R, k, H, x_dtype_code(X), _p(slot_of_row), _p(X), T, _p(Xperm), _p(ws),
        _stream(stream)))


def moe_dispatch(ctx: Context, topk_idx, E: int, capacity: int, counts, offsets,
                 row_of_slot, slot_of_row, ws, X=None, Xperm=None, stream=None,
                 H: Optional[int] = None) -> None:
    T, k = topk_idx.shape
    if H is None:
        H = X.shape[1] if X is not None else 0
    xd = x_dtype_code(X) if X is not None else MOE_DTYPE_BF16
    _req(topk_idx, "topk_idx", torch.int32, T * k)
    _req(counts, "counts", torch.int32, E)
    _req(offsets, "offsets", torch.int32, E + 1)
    _req(row_of_slot, "row_of_slot", torch.int32, T * k)
    _req(slot_of_row, "slot_of_row", torch.int32, T * k)
    if X is not None:
        _req(X, "X", X.dtype, T * H)
        _req(Xperm, "Xperm", X.dtype, T * k * H)
    _check("moe_dispatch", lib().moe_dispatch(
        ctx.handle, T, k, E, H, xd, capacity, _p(topk_idx), _p(X), _p(counts), _p(offsets),
        _p(row_of_slot), _p(slot_of_row), _p(Xperm), _p(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_grouped_swiglu(ctx: Context, X, Xperm, offsets, W_gate, W_up, W_down, O, ws, k: int,
                       Ws_gate=None, Ws_up=None, Ws_down=None, O_shared=None,
                       stream=None) -> None:
    T, H = X.shape
    E, I, _ = W_gate.shape
    has_shared = Ws_gate is not None
    dt = X.dtype
    _req(Xperm, "Xperm", dt, T * k * H)
    _req(offsets, "offsets", torch.int32, E + 1)
    for name, w in (("W_gate", W_gate), ("W_up", W_up), ("W_down", W_down)):
        _req(w, name, dt, E * I * H)
    for name, w in (("Ws_gate", Ws_gate), ("Ws_up", Ws_up), ("Ws_down", Ws_down)):
        _req(w, name, dt, I * H)
    _req(O, "O", torch.float32, T * k * H)
    _req(O_shared, "O_shared", torch.float32, T * H)
    d = ExpertDesc(T, H, E, I, k, x_dtype_code(X), int(has_shared))
    _check("moe_grouped_swiglu", lib().moe_grouped_swiglu(
        ctx.handle, C.byref(d), _p(X), _p(Xperm), _p(offsets), _p(W_gate), _p(W_up),
        _p(W_down), _p(Ws_gate), _p(Ws_up), _p(Ws_down), _p(O), _p(O_shared), _p(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_quantize_fp8(ctx: Context, W, q, scale, stream=None) -> None:
    """W [..., cols] -> q (uint8, same shape) and scale [...]: one scale per row."""
    cols = W.shape[-1]
    rows = W.numel() // cols
    _req(q, "q", torch.uint8, W.numel())
    _req(scale, "scale", torch.float32, rows)
    _check("moe_quantize_fp8", lib().moe_quantize_fp8(
        ctx.handle, rows, cols, x_dtype_code(W), _p(W), _p(q), _p(scale), _stream(stream)))


def moe_grouped_swiglu_fp8(ctx: Context, X, Xperm, offsets, fp8, O, ws, k: int,
                           O_shared=None, stream=None) -> None:
    """fp8: dict of codes and scales Q_gate, S_gate, Q_up, S_up, Q_down, S_down (and
    Qs_* / Ss_* for a shared expert)."""
    T, H = X.shape
    E, I, _ = fp8["Q_gate"].shape
    has_shared = "Qs_gate" in fp8
    _req(Xperm, "Xperm", X.dtype, T * k * H)
    _req(offsets, "offsets", torch.int32, E + 1)
    sizes = {"gate": (I * H, I), "up": (I * H, I), "down": (H * I, H)}
    for m, (n_codes, n_scales) in sizes.items():
        _req(fp8.get("Q_" + m), "Q_" + m, torch.uint8, E * n_codes)
        _req(fp8.get("S_" + m), "S_" + m, torch.float32, E * n_scales)
        _req(fp8.get("Qs_" + m), "Qs_" + m, torch.uint8, n_codes)
        _req(fp8.get("Ss_" + m), "Ss_" + m, torch.float32, n_scales)
    _req(O, "O", torch.float32, T * k * H)
    _req(O_shared, "O_shared", torch.float32, T * H)
    d = ExpertDesc(T, H, E, I, k, MOE_DTYPE_BF16, int(has_shared))
    names = ["Q_gate", "S_gate", "Q_up", "S_up", "Q_down", "S_down",
             "Qs_gate", "Ss_gate", "Qs_up", "Ss_up", "Qs_down", "Ss_down"]
    _check("moe_grouped_swiglu_fp8", lib().moe_grouped_swiglu_fp8(
        ctx.handle, C.byref(d), _p(X), _p(Xperm), _p(offsets),
        *[_p(fp8.get(n)) for n in names], _p(O), _p(O_shared), _p(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_combine(ctx: Context, O, row_of_slot, topk_gate, Y, O_shared=None, Y_bf16=None,
                stream=None) -> None:
    T, k = topk_gate.shape
    H = Y.shape[1]
    _req(topk_gate, "topk_gate", torch.float32, T * k)
    _req(row_of_slot, "row_of_slot", torch.int32, T * k)
    _req(O, "O", torch.float32, 0)
    _req(O_shared, "O_shared", torch.float32, T * H)
    _req(Y, "Y", torch.float32, T * H)
    _req(Y_bf16, "Y_bf16", torch.bfloat16, T * H)
    _check("moe_combine", lib().moe_combine(
        ctx.handle, T, k, H, _p(O), _p(O_shared), _p(row_of_slot), _p(topk_gate), _p(Y),
        _p(Y_bf16), _stream(stream)))


def moe_balance_stats(ctx: Context, T: int, k: int, counts, prob_colsum, alpha: float, f, p,
                      out, offsets=None, stream=None) -> None:
    E = counts.shape[0]
    _req(counts, "counts", torch.int32, E)
    _req(offsets, "offsets", torch.int32, E + 1)
    _req(prob_colsum, "prob_colsum", torch.float64, E)
    for name, t, n in (("f", f, E), ("p", p, E), ("out", out, 4)):
        _req(t, name, torch.float64, n)
    _check("moe_balance_stats", lib().moe_balance_stats(
        ctx.handle, T, k, E, _p(counts), _p(offsets), _p(prob_colsum), float(alpha), _p(f),
        _p(p), _p(out), _stream(stream)))


def moe_bias_update(ctx: Context, T: int, k: int, counts, gamma: float, bias,
                    stream=None) -> None:
    E = counts.shape[0]
    _req(counts, "counts", torch.int32, E)
    _req(bias, "bias", torch.float32, E)
    _check("moe_bias_update", lib().moe_bias_update(
        ctx.handle, T, k, E, _p(counts), float(gamma), _p(bias), _stream(stream)))


def moe_get_device_status(ctx: Context, ws, reset: bool = True, stream=None) -> int:
    st = C.c_int(0)
    _check("moe_get_device_status", lib().moe_get_device_status(
        ctx.handle, _p(ws), C.byref(st), int(reset), _stream(stream)))
    return st.value
