"""Seeded synthetic inputs for the MoE-FFN forward layer.

This module produces the *inputs* of a layer (token activations, router and
expert weights, router bias) and nothing else: it holds none of the layer's
arithmetic.  Both the oracle side (tests, CPU baseline) and the CUDA side
(tests, bench) draw their inputs from here, so the two see the same bytes.

Random numbers come from NumPy's PCG64 generator (O'Neill, "PCG: A Family of
Simple Fast Space-Efficient Statistically Good Algorithms for Random Number
Generation", 2014), one independent stream per (workload, tensor, expert)
via ``numpy.random.SeedSequence``.  Normal draws use NumPy's ziggurat sampler
in float32; bf16 tensors are the float32 draws rounded to nearest-even on the
top 16 bits, stored as ``uint16`` bit patterns.

Workload shapes follow the model families the pages describe: a tiny fp32
GELU layer, a Mixtral-like 8-expert top-2 SwiGLU layer, a DeepSeek-V2-like
160-routed + 2-shared top-6 layer, a 64-expert top-2 layer skewed by
log-Zipf router offsets, and two decode-sized batches.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

ACT_GELU = 0
ACT_SWIGLU = 1
DT_F32 = 0
DT_BF16 = 1
CAP_NONE = 0
CAP_DROP = 1
CAP_REROUTE = 2

# Router-bias laws.
BIAS_NONE = "none"
BIAS_UNIFORM = "uniform_0.1"     # expert_bias ~ U(-0.1, 0.1)
BIAS_LOGZIPF = "logzipf_1.1"     # b[e] = -1.1 * ln(r_e), r a seeded permutation of 1..E
BIAS_UNIFORM_P = "uniform_p"     # b ~ U(-1/(2E), 1/(2E)): half the mean probability


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_tokens: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    n_shared: int
    act: int
    dtype: int
    cap_mode: int
    alpha: float
    has_ffn_bias: bool
    bias_law: str
    seed: int
    bias_mode: int = 0          # 0: bias added to the logits, 1: selection only
    fp8_weights: bool = False   # expert weights quantised to FP8 E4M3 by the library

    @property
    def has_router_bias(self) -> bool:
        return self.bias_law != BIAS_NONE

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workload families.  ``seed`` values are arbitrary fixed integers.
WORKLOADS = {
    # Tiny fp32 layer: Linear(128,256)+GELU+Linear(256,128) experts with biases.
    "tiny_fp32": Workload("tiny_fp32", 256, 128, 8, 2, 256, 0, ACT_GELU, DT_F32,
                          CAP_NONE, 0.0, True, BIAS_NONE, 0x4D6F4501),
    # Mixtral-like prefill, capacity alpha=1.25 with drop.
    "mixtral_prefill": Workload("mixtral_prefill", 4096, 4096, 8, 2, 14336, 0, ACT_SWIGLU,
                                DT_BF16, CAP_DROP, 1.25, False, BIAS_NONE, 0x4D6F4502),
    # DeepSeek-V2-like: 160 routed top-6 + 2 shared, expert_bias ~ U(-0.1,0.1).
    "dsv2": Workload("dsv2", 8192, 5120, 160, 6, 1536, 2, ACT_SWIGLU, DT_BF16,
                     CAP_NONE, 0.0, False, BIAS_UNIFORM, 0x4D6F4503),
    # 64 experts top-2, log-Zipf skew, alpha = 1 + 0.5*log2(16384/256) = 4.0, reroute.
    "e64_reroute": Workload("e64_reroute", 16384, 2048, 64, 2, 1408, 0, ACT_SWIGLU, DT_BF16,
                            CAP_REROUTE, 4.0, False, BIAS_LOGZIPF, 0x4D6F4504),
    # Decode-sized batches (weight-bandwidth bound), log-Zipf skew, no capacity.
    "decode_mixtral": Workload("decode_mixtral", 64, 4096, 8, 2, 14336, 0, ACT_SWIGLU,
                               DT_BF16, CAP_NONE, 0.0, False, BIAS_LOGZIPF, 0x4D6F4505),
    "decode_dsv2": Workload("decode_dsv2", 32, 5120, 160, 6, 1536, 2, ACT_SWIGLU, DT_BF16,
                            CAP_NONE, 0.0, False, BIAS_LOGZIPF, 0x4D6F4506),
    # The decode layers with FP8 E4M3 expert weights (same draws, quantised by
    # the library with one scale per expert matrix).
    "decode_mixtral_fp8": Workload("decode_mixtral_fp8", 64, 4096, 8, 2, 14336, 0, ACT_SWIGLU,
                                   DT_BF16, CAP_NONE, 0.0, False, BIAS_LOGZIPF, 0x4D6F4505,
                                   fp8_weights=True),
    "decode_dsv2_fp8": Workload("decode_dsv2_fp8", 32, 5120, 160, 6, 1536, 2, ACT_SWIGLU, DT_BF16,
                                CAP_NONE, 0.0, False, BIAS_LOGZIPF, 0x4D6F4506, fp8_weights=True),
    # The DeepSeek-V2-like layer with the bias steering selection only
    # (DeepSeek-V3 style): same shapes and x / weights as "dsv2"; the bias is
    # added to probabilities here, so it is drawn on their scale (a tilt that
    # reorders close experts without overriding the router).
    "dsv2_select": Workload("dsv2_select", 8192, 5120, 160, 6, 1536, 2, ACT_SWIGLU, DT_BF16,
                            CAP_NONE, 0.0, False, BIAS_UNIFORM_P, 0x4D6F4503, bias_mode=1),
}

# Tensor identifiers inside one workload's seed space.
_T_X, _T_WR, _T_BIAS, _T_WG, _T_WU, _T_WD, _T_B1, _T_B2 = range(1, 9)


def _rng(seed: int, tensor: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor, sub])))


def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Inputs are finite (normal draws), so no NaN handling is needed."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def _normal(seed, tensor, sub, shape, std, dtype):
    g = _rng(seed, tensor, sub)
    a = g.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(std)
    return round_to_bf16_bits(a) if dtype == DT_BF16 else a


def _uniform(seed, tensor, sub, shape, bound, dtype):
    g = _rng(seed, tensor, sub)
    a = g.uniform(-bound, bound, size=shape).astype(np.float32)
    return round_to_bf16_bits(a) if dtype == DT_BF16 else a


def _per_expert(n, fn, threads):
    """Run fn(e) for e in range(n) on a thread pool (PCG64 fills release the GIL)."""
    if threads <= 1 or n <= 1:
        return [fn(e) for e in range(n)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, range(n)))


def router_bias(w: Workload) -> np.ndarray | None:
    """Per-expert router offsets [E] float32, or None."""
    E = w.n_experts
    if w.bias_law == BIAS_NONE:
        return None
    if w.bias_law == BIAS_UNIFORM:
        return _rng(w.seed, _T_BIAS).uniform(-0.1, 0.1, size=E).astype(np.float32)
    if w.bias_law == BIAS_UNIFORM_P:
        h = 0.5 / E
        return _rng(w.seed, _T_BIAS).uniform(-h, h, size=E).astype(np.float32)
    if w.bias_law == BIAS_LOGZIPF:
        # Zipf popularity over a seeded ranking of the experts: weight r^-s for the
        # expert of rank r; its log is -s*ln(r).  The normalising constant is dropped
        # (a constant shift of every logit).
        ranks = _rng(w.seed, _T_BIAS).permutation(E) + 1
        return (-1.1 * np.log(ranks.astype(np.float64))).astype(np.float32)
    raise ValueError(w.bias_law)


def make_inputs(w: Workload, with_experts: bool = True, threads: int | None = None) -> dict:
    """All inputs of one forward pass as numpy arrays.

    bf16 tensors are uint16 bit patterns; fp32 tensors are float32.
      x        [N, d]
      w_router [E, d]          ~ N(0, 1/d)
      router_bias [E] float32 or None
      w_gate, w_up [E+S, F, d] ~ N(0, 1/d)   (SwiGLU)   | w1 [E, F, d] (GELU)
      w_down   [E+S, d, F]     ~ N(0, 1/F)              | w2 [E, d, F]
      b1 [E, F], b2 [E, d]     ~ U(+-1/sqrt(fan_in))    (GELU layer only)
    Shared experts are stored as experts E..E+S-1 of the expert arrays.
    """
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    N, d, E, F, S = w.n_tokens, w.d_model, w.n_experts, w.d_ff, w.n_shared
    out = {
        "x": _normal(w.seed, _T_X, 0, (N, d), 1.0, w.dtype),
        "w_router": _normal(w.seed, _T_WR, 0, (E, d), 1.0 / math.sqrt(d), w.dtype),
        "router_bias": router_bias(w),
    }
    if not with_experts:
        return out
    ET = E + S
    if w.act == ACT_SWIGLU:
        out["w_gate"] = np.stack(_per_expert(
            ET, lambda e: _normal(w.seed, _T_WG, e, (F, d), 1.0 / math.sqrt(d), w.dtype), threads))
        out["w_up"] = np.stack(_per_expert(
            ET, lambda e: _normal(w.seed, _T_WU, e, (F, d), 1.0 / math.sqrt(d), w.dtype), threads))
    else:
        out["w_gate"] = np.stack(_per_expert(
            ET, lambda e: _normal(w.seed, _T_WG, e, (F, d), 1.0 / math.sqrt(d), w.dtype), threads))
        out["w_up"] = None
    out["w_down"] = np.stack(_per_expert(
        ET, lambda e: _normal(w.seed, _T_WD, e, (d, F), 1.0 / math.sqrt(F), w.dtype), threads))
    if w.has_ffn_bias:
        out["b1"] = np.stack([_uniform(w.seed, _T_B1, e, (F,), 1.0 / math.sqrt(d), w.dtype)
                              for e in range(ET)])
        out["b2"] = np.stack([_uniform(w.seed, _T_B2, e, (d,), 1.0 / math.sqrt(F), w.dtype)
                              for e in range(ET)])
    else:
        out["b1"] = None
        out["b2"] = None
    return out


def expert_weights(w: Workload, e: int) -> dict:
    """The weights of one expert (routed e < E, shared E..E+S-1), drawn from the same
    streams as ``make_inputs`` so a sampled check never needs every expert resident."""
    d, F = w.d_model, w.d_ff
    r = {
        "w_gate": _normal(w.seed, _T_WG, e, (F, d), 1.0 / math.sqrt(d), w.dtype),
        "w_up": (_normal(w.seed, _T_WU, e, (F, d), 1.0 / math.sqrt(d), w.dtype)
                 if w.act == ACT_SWIGLU else None),
        "w_down": _normal(w.seed, _T_WD, e, (d, F), 1.0 / math.sqrt(F), w.dtype),
        "b1": None, "b2": None,
    }
    if w.has_ffn_bias:
        r["b1"] = _uniform(w.seed, _T_B1, e, (F,), 1.0 / math.sqrt(d), w.dtype)
        r["b2"] = _uniform(w.seed, _T_B2, e, (d,), 1.0 / math.sqrt(F), w.dtype)
    return r


def small_workload(name: str, **kw) -> Workload:
    """A reduced copy of a workload family (same dtype/activation/capacity/bias law)."""
    return WORKLOADS[name].replace(name=name + "_small", **kw)
