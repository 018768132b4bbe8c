"""Shared helpers for the tests: workload -> C config, uploads, comparisons."""
from __future__ import annotations

import numpy as np

import mixture_experts_ffn_19_b300 as moe
import synth


def config_of(w: synth.Workload) -> moe.moe_config:
    return moe.make_config(w.n_tokens, w.d_model, w.n_experts, w.top_k, w.d_ff, w.n_shared,
                           act=w.act, dtype=w.dtype, cap_mode=w.cap_mode, alpha=w.alpha,
                           has_ffn_bias=w.has_ffn_bias, has_router_bias=w.has_router_bias)


def to_dev(a, device="cuda"):
    """numpy array (bf16 bits as uint16, or float32/int32) -> torch device tensor."""
    import torch
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_f64(t):
    """torch tensor (bf16/fp32) -> float64 numpy."""
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def rel_err_inf(y, ref):
    """||y - ref||_inf / ||ref||_inf (norm-wise relative error)."""
    return float(np.max(np.abs(y - ref)) / max(np.max(np.abs(ref)), 1e-30))


def segment_rows(offsets, counts, E):
    """Per-expert row ranges [offsets[e], offsets[e] + counts[e])."""
    return [(int(offsets[e]), int(offsets[e]) + int(counts[e])) for e in range(E)]
