"""Shared helpers for the tests: workload -> C config, uploads, comparisons."""
from __future__ import annotations

import numpy as np

import mixture_experts_ffn_19_b300 as moe
import synth


def config_of(w: synth.Workload) -> moe.moe_config:
    return moe.make_config(w.n_tokens, w.d_model, w.n_experts, w.top_k, w.d_ff, w.n_shared,
                           act=w.act, dtype=w.dtype, cap_mode=w.cap_mode, alpha=w.alpha,
                           has_ffn_bias=w.has_ffn_bias, has_router_bias=w.has_router_bias,
                           bias_mode=w.bias_mode)


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


def a128(n):
    return (n + 127) // 128 * 128


def host_layout(w, members):
    """Segment offsets [E+S+1] for the given per-expert member lists (128-row padding)."""
    E, S, N = w.n_experts, w.n_shared, w.n_tokens
    offsets, row = [], 0
    for e in range(E):
        offsets.append(row)
        row += a128(len(members[e]))
    for s in range(S):
        offsets.append(row)
        row += a128(N)
    offsets.append(row)
    return np.array(offsets, dtype=np.int32)


def upload_experts(w, device):
    """Expert weights as device arrays [E+S, ...], drawn and copied one expert at a time."""
    import concurrent.futures as cf
    import torch
    ET, F, d = w.n_experts + w.n_shared, w.d_ff, w.d_model
    dt = torch.bfloat16 if w.dtype == synth.DT_BF16 else torch.float32
    dev = {"w_gate": torch.empty((ET, F, d), dtype=dt, device=device),
           "w_up": torch.empty((ET, F, d), dtype=dt, device=device)
           if w.act == synth.ACT_SWIGLU else None,
           "w_down": torch.empty((ET, d, F), dtype=dt, device=device),
           "b1": torch.empty((ET, F), dtype=dt, device=device) if w.has_ffn_bias else None,
           "b2": torch.empty((ET, d), dtype=dt, device=device) if w.has_ffn_bias else None}
    with cf.ThreadPoolExecutor(8) as ex:
        for e, r in zip(range(ET), ex.map(lambda e: synth.expert_weights(w, e), range(ET))):
            for key, t in dev.items():
                if t is not None:
                    t[e].copy_(to_dev(r[key], device))
    return dev


NEAR_TIE = 1e-6


def valid_selection(key_row, sel, tol=NEAR_TIE):
    """True when `sel` (slot order) is a top-k of key_row once keys closer than
    `tol` are taken as equal: slots descend within tol, and no unselected key
    exceeds a selected one by tol or more."""
    key_row = np.asarray(key_row, dtype=np.float64)
    sel = list(int(e) for e in sel)
    if len(set(sel)) != len(sel) or min(sel) < 0 or max(sel) >= len(key_row):
        return False
    vals = key_row[sel]
    if np.any(vals[1:] > vals[:-1] + tol):
        return False
    rest = np.delete(key_row, sel)
    return rest.size == 0 or rest.max() < vals.min() + tol


def adopt_near_ties(o, idx_dev):
    """Where the oracle's top-k and the device's differ, require the token to be
    a counted near-tie (oracle margin < 1e-6) and the device's selection to be
    one of the valid selections under that tie; return the oracle's selection
    with those tokens' selections replaced (the tie resolution the downstream
    stages are then compared under) and the flipped tokens."""
    flips = np.nonzero(np.any(idx_dev != o["idx"], axis=1))[0]
    near = o["margin"] < NEAR_TIE
    assert np.all(near[flips]), f"top-k differs on tokens without a near-tie: " \
                                f"{flips[~near[flips]][:10]}"
    for t in flips:
        assert valid_selection(o["key"][t], idx_dev[t]), \
            f"token {t}: device selection {idx_dev[t]} is not a valid tie resolution"
    adopted = o["idx"].copy()
    adopted[flips] = idx_dev[flips]
    return adopted, flips


def elementwise_err(y, ref):
    """max |y - ref| / max(|ref|, 1e-3 rms(ref)): the element-wise relative error
    with a floor, reported beside the norm-wise one."""
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    floor = 1e-3 * float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(y - ref) / np.maximum(np.abs(ref), max(floor, 1e-300))))


PARITY_REPORT = []


def report(name, **fields):
    """One line of the parity report printed at the end of the test session."""
    PARITY_REPORT.append((name, fields))
