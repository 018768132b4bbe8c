"""CPU oracle for the MoE-FFN forward layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow C++17 restatement of what the layer computes (``oracle/*.cpp``:
loops only, double accumulation, OpenMP over tokens and over the output
features of each expert row), used to check the CUDA path.  This module is
its ctypes binding: argument marshalling and result packaging only, every step
of the arithmetic runs in ``libmoe_oracle.so``.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` may
import it; the product library never calls it and shares no code with it.

Pages cited (by title; section numbers are the ones printed in each page):
  [P1] «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» (mhpn.cn)
  [P2] «项目概述：为什么MoE成了大模型突围的“秘密武器”» (mooersco.com)
  [P3] «DeepSeek-V2: A Strong, Economical, and Efficient Mixture-of-Experts
       Language Model» — paper summary page (wzjinhao.cn)
  [P4] «GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token.» —
       rebuttal page (l189.com)
  [P5] «为什么MoE有效？稀疏激活的数学直觉与工程实践» (ai.learningdata.cn)

Readings taken where the pages are silent or disagree (R1..R17) are stated
in the C++ sources beside the step they decide.  ``numpy_oracle.py`` is an
independent float64 NumPy restatement kept only as one more pin of this one
(``tests/test_oracle_cross.py``).  Parity status per function: ``PINS``.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

__all__ = [
    "widen", "router_logits", "softmax_fp32", "topk_select", "topk_margin",
    "renormalise", "balance_stats", "alpha_for_batch", "capacity",
    "apply_capacity_drop", "apply_capacity_reroute", "route", "dispatch",
    "gelu_erf", "silu", "expert_ffn", "combine_token", "moe_forward",
    "router_z_loss", "router_entropy", "selection_keys", "router_bias_update",
    "e4m3_encode", "e4m3_decode", "quantize_fp8", "dequantize_fp8",
    "set_threads", "threads", "hardware_concurrency", "PINS",
]

# Parity pins: which CPU test pins each function to something other than itself.
PINS = {
    "router_logits": "tests/test_oracle_router.py: E=k special case, zero router, "
                     "permutation of experts, one dot product written out longhand",
    "softmax_fp32": "tests/test_oracle_router.py: scipy.special.softmax, shift invariance",
    "topk_select": "tests/test_oracle_router.py: brute force over all C(E,k) subsets",
    "renormalise": "tests/test_oracle_router.py: sum to 1, E=k gives w=p, golden case",
    "balance_stats": "tests/test_oracle_stats.py: L_bal=1 under uniform routing "
                     "([P3] §2.2), golden hand case",
    "capacity": "tests/test_oracle_capacity.py: [P1] §5.3 worked example C=1, "
                "[P5] exercise 1 (250), workload values 1280 / 2048",
    "apply_capacity_drop": "tests/test_oracle_capacity.py: counts<=C, all-to-one keeps "
                           "lowest tokens, C>=N*k is identity, golden hand case",
    "apply_capacity_reroute": "tests/test_oracle_reroute.py: hand-worked golden cases, "
                              "counts<=C, no duplicate expert, next-best and "
                              "maximality properties, brute-force replay on tiny inputs",
    "expert_ffn": "tests/test_oracle_ffn.py: erf/exp special values, torch dense FFN",
    "combine_token": "tests/test_oracle_forward.py: linearity in the routed outputs, "
                     "dropped slots contribute nothing, shared-only layer",
    "router_z_loss": "tests/test_oracle_next.py: zero logits give 0.001*(ln E)^2, "
                     "scipy.special.logsumexp, shift by c adds c to lse",
    "router_entropy": "tests/test_oracle_next.py: equal gates give log2 k, one gate "
                      "gives 0, hand case (0.75, 0.25) -> 0.8112781 bits",
    "selection_keys": "tests/test_oracle_next.py: zero bias reduces to the plain "
                      "router, brute force over subsets of p+b, gates from unbiased p",
    "router_bias_update": "tests/test_oracle_next.py: hand case of signs, balanced "
                          "picks leave the bias unchanged",
    "e4m3_encode": "tests/test_oracle_fp8.py: torch float8_e4m3fn cast (library) on "
                   "random, tie and subnormal values; saturation and signed zero by hand",
    "e4m3_decode": "tests/test_oracle_fp8.py: all 256 codes vs torch float8_e4m3fn, "
                   "encode(decode(c)) == c for every finite code",
    "quantize_fp8": "tests/test_oracle_fp8.py: largest element maps to 448, error "
                    "<= half a step, zero matrix, hand case",
    "dequantize_fp8": "tests/test_oracle_fp8.py: product of the decoded code and the scale",
    "moe_forward": "tests/test_oracle_forward.py: E=1 dense layer, shared-only dense "
                   "layer, k=E layer = probability-weighted dense mixture of every "
                   "expert (logit and selection-only bias; a gate rotated to the "
                   "wrong expert fails), token-permutation equivariance, linearity "
                   "in the routed outputs, dropped slots contribute nothing; no page "
                   "prints a numeric layer output, so the pins are these special "
                   "cases and invariants",
}

ORC_F32, ORC_BF16, ORC_F64, ORC_E4M3 = 0, 1, 2, 3

_P = C.c_void_p
_I32, _I64, _F32, _F64 = C.c_int32, C.c_int64, C.c_float, C.c_double


class _Mat(C.Structure):
    _fields_ = [("data", _P), ("dtype", _I32), ("scale", _F32)]


class _RouteOut(C.Structure):
    _fields_ = [("logits", _P), ("p", _P), ("key", _P), ("idx", _P), ("w", _P),
                ("margin", _P), ("freq", _P), ("mean_prob", _P), ("picks", _P),
                ("l_bal", _F64), ("z_loss", _F64), ("router_entropy", _F64)]


class _DispatchOut(C.Structure):
    _fields_ = [("final_idx", _P), ("members", _P), ("member_start", _P),
                ("n_dropped", _I64), ("n_rerouted", _I64), ("rounds", _I64)]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = C.CDLL(path)
        sig = {
            "orc_set_threads": (C.c_int, [C.c_int]),
            "orc_threads": (C.c_int, []),
            "orc_hardware_concurrency": (C.c_int, []),
            "orc_widen": (None, [_P, _I32, _I64, _P]),
            "orc_e4m3_encode": (None, [_P, _I64, _P]),
            "orc_e4m3_decode": (None, [_P, _I64, _P]),
            "orc_quantize_fp8": (None, [_P, _I32, _I64, _P, _P]),
            "orc_dequantize_fp8": (None, [_P, _I64, _F32, _P]),
            "orc_router_logits": (None, [_I32, _I32, _I32, _P, _I32, _P, _I32, _P, _P]),
            "orc_softmax_fp32": (None, [_I32, _I32, _P, _P]),
            "orc_topk": (None, [_I32, _I32, _I32, _P, _P]),
            "orc_topk_margin": (None, [_I32, _I32, _I32, _P, _P]),
            "orc_renormalise": (None, [_I32, _I32, _I32, _P, _P, _P]),
            "orc_balance_stats": (None, [_I32, _I32, _I32, _P, _P, _P, _P, _P, _P]),
            "orc_z_loss": (_F64, [_I32, _I32, _P]),
            "orc_router_entropy": (_F64, [_I32, _I32, _P]),
            "orc_selection_keys": (None, [_I32, _I32, _P, _P, _P]),
            "orc_router_bias_update": (None, [_I32, _P, _P, _I64, _I32, _F32, _P]),
            "orc_route": (None, [_I32, _I32, _I32, _I32, _P, _I32, _P, _I32, _P, _I32, _P,
                                 C.POINTER(_RouteOut)]),
            "orc_alpha_for_batch": (_F64, [_I64]),
            "orc_capacity": (_I64, [_I64, _I32, _I32, _F64]),
            "orc_dispatch": (C.c_int, [_I32, _I32, _I32, _I32, _I64, _P, _P,
                                       C.POINTER(_DispatchOut)]),
            "orc_gelu_n": (None, [_P, _I64, _P]),
            "orc_silu_n": (None, [_P, _I64, _P]),
            "orc_expert_ffn": (None, [_I32, _I32, _I32, _I64, _P, _Mat, _Mat, _Mat, _Mat,
                                      _Mat, _P]),
            "orc_combine_token": (None, [_I32, _I32, _P, _I32, _P, _P, _P]),
            "orc_layer_rows": (C.c_int, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _I32,
                                         _P, _P, _P, _I64, _P, _P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _LIB = lib
    return _LIB


# ----------------------------------------------------------------------------- marshalling

def _ptr(a):
    return None if a is None else a.ctypes.data


def _typed(a):
    """A contiguous array and its ORC_* element code (bf16 arrives as uint16 bit
    patterns; other types are made float64, exactly for every integer and float
    type the tests pass)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, ORC_BF16
    if a.dtype == np.float32:
        return a, ORC_F32
    return np.ascontiguousarray(a, dtype=np.float64), ORC_F64


def _mat(v, keep):
    """A weight entry -> _Mat.  v: None, an array (bf16 bits / f32 / f64), or a
    (codes uint8, scale) pair of FP8 E4M3 codes and their per-matrix scale."""
    if v is None:
        return _Mat(None, 0, 0.0)
    if isinstance(v, tuple):
        codes = np.ascontiguousarray(v[0], dtype=np.uint8)
        keep.append(codes)
        return _Mat(codes.ctypes.data, ORC_E4M3, float(np.float32(v[1])))
    a, dt = _typed(v)
    keep.append(a)
    return _Mat(a.ctypes.data, dt, 1.0)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def set_threads(n: int) -> int:
    """OpenMP threads the oracle uses from now on (n <= 0: leave as is)."""
    return int(_lib().orc_set_threads(int(n)))


def threads() -> int:
    return int(_lib().orc_threads())


def hardware_concurrency() -> int:
    return int(_lib().orc_hardware_concurrency())


# ----------------------------------------------------------------------------- inputs

def widen(a):
    """bf16 bit patterns (uint16) or float32 -> float64, exactly."""
    if a is None:
        return None
    a, dt = _typed(a)
    out = np.empty(a.shape, dtype=np.float64)
    _lib().orc_widen(_ptr(a), dt, a.size, _ptr(out))
    return out


# ----------------------------------------------------------------------------- router

def router_logits(x, w_router, router_bias=None):
    """z[t,e] = sum_j x[t,j] Wr[e,j] (+ b[e]) in double -- [P5] §2.2, [P3] §2.2."""
    x, xd = _typed(x)
    wr, wd = _typed(w_router)
    N, d = x.shape
    E = wr.shape[0]
    b = None if router_bias is None else _f32(router_bias)
    z = np.empty((N, E), dtype=np.float64)
    _lib().orc_router_logits(N, d, E, _ptr(x), xd, _ptr(wr), wd, _ptr(b), _ptr(z))
    return z


def softmax_fp32(z):
    """p = exp(z - max z) / sum in double, rounded to float32 -- [P5] §2.2."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    p = np.empty(z.shape, dtype=np.float32)
    _lib().orc_softmax_fp32(z.shape[0], z.shape[1], _ptr(z), _ptr(p))
    return p


def topk_select(p, k):
    """k largest per token, largest first, ties to the lower index (reading R1)."""
    p = _f32(p)
    idx = np.empty((p.shape[0], k), dtype=np.int32)
    _lib().orc_topk(p.shape[0], p.shape[1], k, _ptr(p), _ptr(idx))
    return idx


def topk_margin(p, k):
    """Smallest gap between consecutive scores among the k+1 largest (reading R17)."""
    p = _f32(p)
    m = np.empty(p.shape[0], dtype=np.float64)
    _lib().orc_topk_margin(p.shape[0], p.shape[1], k, _ptr(p), _ptr(m))
    return m


def renormalise(p, idx):
    """w = p[idx] / sum_j p[idx_j] in double, then float32 -- [P5] §2.2."""
    p, idx = _f32(p), _i32(idx)
    w = np.empty(idx.shape, dtype=np.float32)
    _lib().orc_renormalise(p.shape[0], p.shape[1], idx.shape[1], _ptr(p), _ptr(idx), _ptr(w))
    return w


def balance_stats(p, idx, n_experts):
    """(expert_freq[E], mean_prob[E], L_bal) -- [P3] §2.2 (reading R5)."""
    p, idx = _f32(p), _i32(idx)
    N, k = idx.shape
    f = np.empty(n_experts)
    m = np.empty(n_experts)
    lb = C.c_double()
    picks = np.empty(n_experts, dtype=np.int64)
    _lib().orc_balance_stats(N, n_experts, k, _ptr(p), _ptr(idx), _ptr(f), _ptr(m),
                             C.addressof(lb), _ptr(picks))
    return f, m, float(lb.value)


def router_z_loss(z):
    """L_z = 0.001 mean_t logsumexp(z_t)^2 -- [P2] §3.3 (reading R13)."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    return float(_lib().orc_z_loss(z.shape[0], z.shape[1], _ptr(z)))


def router_entropy(w):
    """mean_t -sum_j w_j log2 w_j in bits -- [P4] §2.3 (reading R14)."""
    w = _f32(w)
    return float(_lib().orc_router_entropy(w.shape[0], w.shape[1], _ptr(w)))


def selection_keys(p, router_bias):
    """key = p + b in float32 -- [P5] §2.4 (reading R15)."""
    p, b = _f32(p), _f32(router_bias)
    key = np.empty(p.shape, dtype=np.float32)
    _lib().orc_selection_keys(p.shape[0], p.shape[1], _ptr(p), _ptr(b), _ptr(key))
    return key


def router_bias_update(router_bias, picks, n_tokens, k, gamma):
    """b_e -/+ gamma by pre-capacity picks against N k / E -- [P5] §2.4."""
    b = _f32(router_bias)
    picks = np.ascontiguousarray(picks, dtype=np.int64)
    out = np.empty_like(b)
    _lib().orc_router_bias_update(len(b), _ptr(b), _ptr(picks), int(n_tokens), int(k),
                                  float(np.float32(gamma)), _ptr(out))
    return out


def route(x, w_router, router_bias, k, bias_mode=0, idx_given=None):
    """Router stage: logits, float32 probabilities, top-k, gates, statistics.

    bias_mode 0 adds the bias to the logits ([P3] §2.2), 1 lets it steer the
    selection only (reading R15); "key" is what top-k and reroute rank by.
    idx_given replaces the top-k selection (see orc_route)."""
    x, xd = _typed(x)
    wr, wd = _typed(w_router)
    N, d = x.shape
    E = wr.shape[0]
    b = None if router_bias is None else _f32(router_bias)
    o = {"logits": np.empty((N, E)), "p": np.empty((N, E), np.float32),
         "key": np.empty((N, E), np.float32), "idx": np.empty((N, k), np.int32),
         "w": np.empty((N, k), np.float32), "margin": np.empty(N),
         "expert_freq": np.empty(E), "mean_prob": np.empty(E),
         "picks": np.empty(E, np.int64)}
    ro = _RouteOut(_ptr(o["logits"]), _ptr(o["p"]), _ptr(o["key"]), _ptr(o["idx"]),
                   _ptr(o["w"]), _ptr(o["margin"]), _ptr(o["expert_freq"]),
                   _ptr(o["mean_prob"]), _ptr(o["picks"]), 0.0, 0.0, 0.0)
    given = None if idx_given is None else _i32(idx_given)
    if given is not None and given.shape != (N, k):
        raise ValueError("idx_given must be [N, k]")
    _lib().orc_route(N, d, E, k, _ptr(x), xd, _ptr(wr), wd, _ptr(b), int(bias_mode),
                     _ptr(given), C.byref(ro))
    o.update(l_bal=ro.l_bal, z_loss=ro.z_loss, router_entropy=ro.router_entropy)
    return o


# ----------------------------------------------------------------------------- fp8 weights

E4M3_MAX = 448.0


def e4m3_encode(v):
    """float32 -> FP8 E4M3 codes, nearest-even, saturated at 448 (reading R16)."""
    v = _f32(v)
    out = np.empty(v.shape, dtype=np.uint8)
    _lib().orc_e4m3_encode(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(code):
    """FP8 E4M3 codes -> float64 values (NaN for S.1111.111)."""
    c = np.ascontiguousarray(code, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _lib().orc_e4m3_decode(_ptr(c), c.size, _ptr(out))
    return out


def quantize_fp8(w):
    """One expert matrix -> (codes uint8, scale float32): scale = amax/448, codes of
    the float32 quotients (reading R16)."""
    a, dt = _typed(w)
    if dt == ORC_F64:
        raise TypeError("quantize_fp8 takes bf16 bit patterns or float32")
    codes = np.empty(a.shape, dtype=np.uint8)
    s = C.c_float()
    _lib().orc_quantize_fp8(_ptr(a), dt, a.size, _ptr(codes), C.addressof(s))
    return codes, np.float32(s.value)


def dequantize_fp8(codes, scale):
    """scale * value(code), float64 (exact)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _lib().orc_dequantize_fp8(_ptr(c), c.size, float(np.float32(scale)), _ptr(out))
    return out


# ----------------------------------------------------------------------------- capacity

def alpha_for_batch(n_tokens):
    """alpha = 1 + 0.5 log2(N/256) -- [P1] §3.1."""
    return float(_lib().orc_alpha_for_batch(int(n_tokens)))


def capacity(n_tokens, n_experts, k, alpha):
    """C = floor(floor(k N / E) * alpha) -- [P1] §3.1 (reading R2)."""
    return int(_lib().orc_capacity(int(n_tokens), int(n_experts), int(k), float(alpha)))


def _dispatch(idx, key, n_experts, cap_mode, cap):
    idx = _i32(idx)
    N, k = idx.shape
    key = None if key is None else _f32(key)
    final = np.empty((N, k), dtype=np.int32)
    members = np.empty(N * k, dtype=np.int32)
    start = np.empty(n_experts + 1, dtype=np.int32)
    do = _DispatchOut(_ptr(final), _ptr(members), _ptr(start), 0, 0, 0)
    big = np.iinfo(np.int64).max
    rc = _lib().orc_dispatch(N, n_experts, k, int(cap_mode), big if cap is None else int(cap),
                             _ptr(idx), _ptr(key), C.byref(do))
    if rc != 0:
        raise ValueError(f"orc_dispatch: bad arguments (cap_mode {cap_mode})")
    mem = [members[start[e]:start[e + 1]].copy() for e in range(n_experts)]
    return final, mem, int(do.n_rerouted), int(do.n_dropped), int(do.rounds)


def apply_capacity_drop(idx, n_experts, cap):
    """Each expert keeps its first ``cap`` tokens in token order ([P1] §4.2,
    reading R3); ``cap=None`` means no limit.  Returns (final_idx, members)."""
    final, mem, _, _, _ = _dispatch(idx, None, n_experts, 0 if cap is None else 1, cap)
    return final, mem


def apply_capacity_reroute(idx, p, n_experts, cap):
    """Drop, then reroute overflow to the next-best unfilled expert (reading R4).
    Returns (final_idx, members, n_rerouted, n_dropped, rounds)."""
    return _dispatch(idx, p, n_experts, 2, cap)


def dispatch(idx, p, n_experts, cap_mode, cap):
    """Capacity stage.  cap_mode: 0 none, 1 drop, 2 reroute."""
    final, mem, nr, nd, _ = _dispatch(idx, p if cap_mode == 2 else None, n_experts, cap_mode,
                                      cap if cap_mode else None)
    counts = np.array([len(m) for m in mem], dtype=np.int32)
    return {"final": final, "members": mem, "counts": counts, "n_dropped": nd,
            "n_rerouted": nr}


# ----------------------------------------------------------------------------- experts

def gelu_erf(a):
    """GELU(a) = 0.5 a (1 + erf(a / sqrt 2)) -- reading R7."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape)
    _lib().orc_gelu_n(_ptr(a), a.size, _ptr(out))
    return out


def silu(a):
    """silu(a) = a / (1 + e^-a) -- reading R6."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape)
    _lib().orc_silu_n(_ptr(a), a.size, _ptr(out))
    return out


def expert_ffn(x_rows, wts, act):
    """One expert applied to rows of x (float64 in, float64 out).

    act 0: GELU(x W1^T + b1) W2^T + b2 with W1 = wts['w_gate'], W2 = wts['w_down'];
    act 1: (silu(x Wg^T) * (x Wu^T)) Wd^T.  Weight entries: bf16 bits, float32,
    float64, or (E4M3 codes, scale)."""
    x = np.ascontiguousarray(x_rows, dtype=np.float64)
    R, d = x.shape
    wg = wts["w_gate"]
    F = (wg[0] if isinstance(wg, tuple) else wg).shape[0]
    keep = []
    mats = [_mat(wts.get(key), keep) for key in ("w_gate", "w_up", "w_down", "b1", "b2")]
    if act == 1 and not mats[1].data:
        raise ValueError("SwiGLU expert needs w_up")
    y = np.empty((R, d), dtype=np.float64)
    _lib().orc_expert_ffn(int(act), d, F, R, _ptr(x), *mats, _ptr(y))
    return y


def combine_token(shared_rows, routed_rows, gates):
    """y = sum_s shared_s + sum_j g_j routed_j -- [P5] §2.1, [P3] §2.3."""
    rows = [np.ascontiguousarray(r, dtype=np.float64) for r in list(shared_rows) + list(routed_rows)]
    if not rows:
        return 0.0
    d = rows[0].shape[0]
    S = len(shared_rows)
    ptrs = (C.c_void_p * max(len(rows), 1))(*[r.ctypes.data for r in rows])
    sh = C.cast(ptrs, C.c_void_p)
    rt = C.c_void_p(C.addressof(ptrs) + S * C.sizeof(C.c_void_p))
    g = _f32(np.asarray(gates, dtype=np.float32).reshape(-1))
    y = np.empty(d)
    _lib().orc_combine_token(d, S, sh, len(rows) - S, rt, _ptr(g), _ptr(y))
    return y


# ----------------------------------------------------------------------------- layer

_KEYS = ("w_gate", "w_up", "w_down", "b1", "b2")


def moe_forward(cfg, inputs, tokens=None, get_expert=None, idx_given=None):
    """Whole layer: route, capacity, experts, combine, statistics.

    cfg: object with n_tokens, d_model, n_experts, top_k, d_ff, n_shared, act,
         cap_mode, alpha, bias_mode (the synth ``Workload`` fields).
    inputs: dict from ``synth.make_inputs`` (expert arrays may be omitted when
         ``get_expert(e)`` supplies one expert's weights on demand).
    tokens: the tokens whose output rows to compute (default: all).  Routing
         and capacity always run over the whole batch; each output row then
         depends on its own token only.
    idx_given: a top-k selection to use instead of the oracle's own (one of
         several equally valid selections of near-tied tokens).
    Returns a dict with routing tensors, statistics and y [len(tokens), d] float64.
    """
    N, E, k, S = cfg.n_tokens, cfg.n_experts, cfg.top_k, cfg.n_shared
    r = route(inputs["x"], inputs["w_router"], inputs.get("router_bias"), k,
              getattr(cfg, "bias_mode", 0), idx_given=idx_given)
    cap = capacity(N, E, k, cfg.alpha) if cfg.cap_mode != 0 else None
    dsp = dispatch(r["idx"], r["key"], E, cfg.cap_mode, cap)
    out = dict(r)
    out.update(dsp)
    out["capacity"] = cap

    if get_expert is None:
        def get_expert(e):
            return {key: (inputs[key][e] if inputs.get(key) is not None else None)
                    for key in _KEYS}

    tokens = np.arange(N, dtype=np.int64) if tokens is None else \
        np.ascontiguousarray(tokens, dtype=np.int64)
    used = set(int(e) for e in np.unique(dsp["final"][tokens]) if e >= 0) | \
        set(range(E, E + S))
    keep = []
    mats = (_Mat * (5 * (E + S)))()
    for e in sorted(used):
        wts = get_expert(e)
        for i, key in enumerate(_KEYS):
            mats[5 * e + i] = _mat(wts.get(key), keep)
    x, xd = _typed(inputs["x"])
    y = np.empty((len(tokens), cfg.d_model), dtype=np.float64)
    rc = _lib().orc_layer_rows(N, cfg.d_model, E, k, cfg.d_ff, S, int(cfg.act), _ptr(x), xd,
                               _ptr(dsp["final"]), _ptr(r["w"]), _ptr(tokens), len(tokens),
                               C.cast(mats, C.c_void_p), _ptr(y))
    if rc != 0:
        raise ValueError(f"orc_layer_rows failed ({rc})")
    out["tokens"] = tokens
    out["y"] = y
    return out
