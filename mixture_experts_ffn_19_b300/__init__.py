"""Python binding of libmoe, the B300 (sm_103a) MoE-FFN forward-layer library.

Argument marshalling only: every step of the layer runs in the CUDA kernels
behind the C ABI declared in ``include/moe.h``.  Functions keep the C names
(``moe_route``, ``moe_dispatch``, ``moe_expert_ffn``, ``moe_combine``,
``moe_forward`` ...) and accept torch tensors (device pointers are taken with
``data_ptr()``); PyTorch only provides device memory and streams.  A missing
library raises at import of the first call, there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_DEVICE = -6

MOE_ACT_GELU, MOE_ACT_SWIGLU = 0, 1
MOE_F32, MOE_BF16 = 0, 1
MOE_CAP_NONE, MOE_CAP_DROP, MOE_CAP_REROUTE = 0, 1, 2
MOE_BIAS_LOGIT, MOE_BIAS_SELECT = 0, 1
MOE_SEGMENT_ALIGN = 128


class MoeError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call}: {status_string(status)} ({status})")
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("act", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("cap_mode", ctypes.c_int32), ("alpha", ctypes.c_double),
                ("has_ffn_bias", ctypes.c_int32), ("has_router_bias", ctypes.c_int32),
                ("bias_mode", ctypes.c_int32)]


class moe_stats(ctypes.Structure):
    _fields_ = [("expert_freq", ctypes.c_void_p), ("mean_prob", ctypes.c_void_p),
                ("l_bal", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("n_dropped", ctypes.c_void_p), ("n_rerouted", ctypes.c_void_p),
                ("z_loss", ctypes.c_void_p), ("router_entropy", ctypes.c_void_p)]


class moe_timing(ctypes.Structure):
    _fields_ = [("events", ctypes.c_void_p * 6)]


class moe_views(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_w", "probs", "final_idx", "pos", "offsets", "perm",
                 "x_perm", "h", "y_perm")]


_lib = None
_P = ctypes.c_void_p
_CFG = ctypes.POINTER(moe_config)
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_validate_config": (ctypes.c_int, [_CFG]),
    "moe_capacity": (ctypes.c_int32, [_CFG]),
    "moe_max_rows": (ctypes.c_int64, [_CFG]),
    "moe_max_total_rows": (ctypes.c_int64, [_CFG]),
    "moe_workspace_size": (ctypes.c_size_t, [_CFG]),
    "moe_workspace_views": (ctypes.c_int, [_CFG, _P, ctypes.c_size_t, ctypes.POINTER(moe_views)]),
    "moe_route": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, ctypes.POINTER(moe_stats), _P,
                                 ctypes.c_size_t, _P]),
    "moe_dispatch": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P,
                                    ctypes.POINTER(moe_stats), _P, ctypes.c_size_t, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                      ctypes.c_size_t, _P]),
    "moe_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P]),
    "moe_forward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   ctypes.POINTER(moe_stats), _P, ctypes.c_size_t, _P,
                                   ctypes.POINTER(moe_timing)]),
    "moe_router_bias_update": (ctypes.c_int, [_CFG, _P, ctypes.c_size_t, _P, ctypes.c_float, _P]),
    "moe_quantize_fp8": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, _P, _P,
                                        _P]),
    "moe_expert_ffn_fp8": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          ctypes.c_size_t, _P]),
    "moe_forward_fp8": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P,
                                       ctypes.POINTER(moe_stats), _P, ctypes.c_size_t, _P,
                                       ctypes.POINTER(moe_timing)]),
    "moe_selftest_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    "moe_selftest_barrier_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint32,
                                                    ctypes.c_uint32, _P]),
    "moe_device_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_kernel_launches": (ctypes.c_int64, []),
}


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mixture_experts_ffn_19_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().moe_status_string(st).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name: str, st: int) -> int:
    if st != MOE_OK:
        raise MoeError(name, st)
    return st


def make_config(n_tokens, d_model, n_experts, top_k, d_ff, n_shared=0, act=MOE_ACT_SWIGLU,
                dtype=MOE_BF16, cap_mode=MOE_CAP_NONE, alpha=0.0, has_ffn_bias=False,
                has_router_bias=False, bias_mode=MOE_BIAS_LOGIT) -> moe_config:
    return moe_config(int(n_tokens), int(d_model), int(n_experts), int(top_k), int(d_ff),
                      int(n_shared), int(act), int(dtype), int(cap_mode), float(alpha),
                      int(bool(has_ffn_bias)), int(bool(has_router_bias)), int(bias_mode))


def make_stats(expert_freq=None, mean_prob=None, l_bal=None, counts=None, n_dropped=None,
               n_rerouted=None, z_loss=None, router_entropy=None) -> moe_stats:
    return moe_stats(_ptr(expert_freq), _ptr(mean_prob), _ptr(l_bal), _ptr(counts),
                     _ptr(n_dropped), _ptr(n_rerouted), _ptr(z_loss), _ptr(router_entropy))


def moe_validate_config(cfg: moe_config) -> int:
    return lib().moe_validate_config(ctypes.byref(cfg))


def moe_capacity(cfg: moe_config) -> int:
    return lib().moe_capacity(ctypes.byref(cfg))


def moe_max_rows(cfg: moe_config) -> int:
    return lib().moe_max_rows(ctypes.byref(cfg))


def moe_max_total_rows(cfg: moe_config) -> int:
    return lib().moe_max_total_rows(ctypes.byref(cfg))


def moe_workspace_size(cfg: moe_config) -> int:
    return lib().moe_workspace_size(ctypes.byref(cfg))


def moe_workspace_views(cfg, workspace) -> moe_views:
    v = moe_views()
    _check("moe_workspace_views", lib().moe_workspace_views(
        ctypes.byref(cfg), _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(v)))
    return v


def moe_route(cfg, x, w_router, router_bias, topk_idx, topk_w, probs=None, stats=None,
              workspace=None, stream=None) -> int:
    return _check("moe_route", lib().moe_route(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(topk_idx),
        _ptr(topk_w), _ptr(probs), ctypes.byref(stats) if stats is not None else None,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_dispatch(cfg, topk_idx, probs, x, final_idx, pos, offsets, perm, x_perm, stats=None,
                 workspace=None, stream=None) -> int:
    return _check("moe_dispatch", lib().moe_dispatch(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(probs), _ptr(x), _ptr(final_idx), _ptr(pos),
        _ptr(offsets), _ptr(perm), _ptr(x_perm),
        ctypes.byref(stats) if stats is not None else None,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_expert_ffn(cfg, x, x_perm, offsets, counts, w_gate, w_up, w_down, b1, b2, y_perm,
                   workspace=None, stream=None) -> int:
    return _check("moe_expert_ffn", lib().moe_expert_ffn(
        ctypes.byref(cfg), _ptr(x), _ptr(x_perm), _ptr(offsets), _ptr(counts), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(b1), _ptr(b2), _ptr(y_perm), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_combine(cfg, y_perm, offsets, final_idx, pos, topk_w, y, stream=None) -> int:
    return _check("moe_combine", lib().moe_combine(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(offsets), _ptr(final_idx), _ptr(pos),
        _ptr(topk_w), _ptr(y), _stream(stream)))


def moe_forward(cfg, x, w_router, router_bias, w_gate, w_up, w_down, b1, b2, y, stats=None,
                workspace=None, stream=None, timing=None) -> int:
    return _check("moe_forward", lib().moe_forward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(b1), _ptr(b2), _ptr(y),
        ctypes.byref(stats) if stats is not None else None,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream),
        ctypes.byref(timing) if timing is not None else None))


def moe_router_bias_update(cfg, workspace, router_bias, gamma, stream=None) -> int:
    return _check("moe_router_bias_update", lib().moe_router_bias_update(
        ctypes.byref(cfg), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(router_bias), float(gamma), _stream(stream)))


def moe_quantize_fp8(w, q, scales, stream=None) -> int:
    """w [n_mat, rows, cols] bf16 -> q (uint8, same shape), scales [n_mat] fp32."""
    n_mat, rows, cols = w.shape
    return _check("moe_quantize_fp8", lib().moe_quantize_fp8(
        _ptr(w), int(n_mat), int(rows), int(cols), _ptr(q), _ptr(scales), _stream(stream)))


def moe_expert_ffn_fp8(cfg, x, x_perm, offsets, counts, w_gate, w_up, w_down, scales, y_perm,
                       workspace=None, stream=None) -> int:
    return _check("moe_expert_ffn_fp8", lib().moe_expert_ffn_fp8(
        ctypes.byref(cfg), _ptr(x), _ptr(x_perm), _ptr(offsets), _ptr(counts), _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(scales), _ptr(y_perm), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_forward_fp8(cfg, x, w_router, router_bias, w_gate, w_up, w_down, scales, y, stats=None,
                    workspace=None, stream=None, timing=None) -> int:
    return _check("moe_forward_fp8", lib().moe_forward_fp8(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(scales), _ptr(y),
        ctypes.byref(stats) if stats is not None else None,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream),
        ctypes.byref(timing) if timing is not None else None))


def moe_selftest_timeout(workspace, limit_us, stream=None) -> int:
    return _check("moe_selftest_timeout", lib().moe_selftest_timeout(
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(limit_us),
        _stream(stream)))


def moe_selftest_barrier_timeout(workspace, limit_us, n_barriers, stream=None) -> int:
    return _check("moe_selftest_barrier_timeout", lib().moe_selftest_barrier_timeout(
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(limit_us),
        int(n_barriers), _stream(stream)))


def moe_device_status(workspace, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("moe_device_status", lib().moe_device_status(_ptr(workspace), _stream(stream),
                                                        ctypes.byref(out)))
    return out.value


def moe_kernel_launches() -> int:
    return lib().moe_kernel_launches()


def alloc_workspace(cfg, device="cuda"):
    """A zero-filled uint8 workspace tensor of moe_workspace_size(cfg) bytes."""
    import torch
    n = moe_workspace_size(cfg)
    if n == 0:
        raise MoeError("moe_workspace_size", moe_validate_config(cfg) or MOE_ERR_INVALID_ARG)
    return torch.zeros(n, dtype=torch.uint8, device=device)
