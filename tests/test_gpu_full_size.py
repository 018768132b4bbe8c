"""Whole-layer parity at the full workload sizes, through moe_forward as bench.py
calls it.

Routing, statistics and the dispatch layout are compared over the whole batch
(a top-k that differs from the oracle's must be a valid resolution of a counted
near-tie; capacity and layout are then compared under it); the output rows of
a token sample that puts a checked row in every 128-row tile of every GEMM
segment are compared with the oracle, which evaluates only the experts those
tokens use.  Expert weights are drawn one expert at a time and uploaded; the
oracle draws the ones it needs again from the same seeded streams, so no host
copy of every expert is ever held.
"""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import oracle
import synth
from helpers import (NEAR_TIE, adopt_near_ties, config_of, elementwise_err, rel_err_inf,
                     report, to_dev, to_f64, upload_experts)

pytestmark = pytest.mark.gpu

SAMPLE = 24
FULL = ["mixtral_prefill", "dsv2", "dsv2_select", "e64_reroute", "decode_mixtral",
        "decode_dsv2", "tiny_fp32"]


def sample_tokens(w, members):
    """Tokens whose output rows are checked: the first and last token, a seeded
    random sample, and for every segment of the GEMMs' row layout (each routed
    expert's kept rows in row order, then each shared expert's N rows in token
    order) the token of its first and last row and the token of the first row
    of every 128-row tile, so that every tile the GEMMs compute holds a checked
    row."""
    rng = np.random.default_rng(w.seed)
    n = min(SAMPLE, w.n_tokens)
    mid = rng.choice(np.arange(1, max(w.n_tokens - 1, 1)), size=max(n - 2, 0), replace=False) \
        if w.n_tokens > 2 else np.array([], dtype=np.int64)
    picks = [0, w.n_tokens - 1, *mid.tolist()]
    segments = [np.asarray(m) for m in members] + \
        [np.arange(w.n_tokens)] * w.n_shared
    for seg in segments:
        if len(seg) == 0:
            continue
        picks += seg[::128].tolist() + [int(seg[-1])]
    return np.unique(np.asarray(picks, dtype=np.int64))


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size_sampled(cuda, name):
    w = synth.WORKLOADS[name]
    N, E, k, S = w.n_tokens, w.n_experts, w.top_k, w.n_shared
    inp = synth.make_inputs(w, with_experts=False)
    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], k, w.bias_mode)
    C = oracle.capacity(N, E, k, w.alpha) if w.cap_mode else None
    wdev = upload_experts(w, cuda)

    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    xd = to_dev(inp["x"])
    y = torch.zeros((N, w.d_model), dtype=xd.dtype, device=cuda)
    f32 = dict(dtype=torch.float32, device=cuda)
    i32 = dict(dtype=torch.int32, device=cuda)
    st_t = {"expert_freq": torch.zeros(E, **f32), "mean_prob": torch.zeros(E, **f32),
            "l_bal": torch.zeros(1, **f32), "counts": torch.zeros(E, **i32),
            "n_dropped": torch.zeros(1, **i32), "n_rerouted": torch.zeros(1, **i32),
            "z_loss": torch.zeros(1, **f32), "router_entropy": torch.zeros(1, **f32)}
    moe.moe_forward(cfg, xd, to_dev(inp["w_router"]), to_dev(inp["router_bias"]),
                    wdev["w_gate"], wdev["w_up"], wdev["w_down"], wdev["b1"], wdev["b2"], y,
                    moe.make_stats(**st_t), ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    s = {key: v.cpu().numpy() for key, v in st_t.items()}

    # routing over the whole batch
    v = moe.moe_workspace_views(cfg, ws)
    i32v = ws.view(torch.int32)
    base = ws.data_ptr()

    def view(ptr, n):
        off = (ptr - base) // 4
        return i32v[off:off + n].cpu().numpy()

    idx = view(v.topk_idx, N * k).reshape(N, k)
    final = view(v.final_idx, N * k).reshape(N, k)
    adopted, flips = adopt_near_ties(r, idx)
    near = int((r["margin"] < NEAR_TIE).sum())
    if len(flips):
        r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], k, w.bias_mode,
                         idx_given=adopted)
    dsp = oracle.dispatch(r["idx"], r["key"], E, w.cap_mode, C)
    print(f"{name}: near-ties {near}, flipped {len(flips)}")
    np.testing.assert_array_equal(final, dsp["final"])
    np.testing.assert_array_equal(s["counts"], dsp["counts"])
    assert s["n_dropped"][0] == dsp["n_dropped"]
    assert s["n_rerouted"][0] == dsp["n_rerouted"]
    np.testing.assert_allclose(s["mean_prob"], r["mean_prob"], rtol=1e-5, atol=1e-9)
    np.testing.assert_allclose(s["l_bal"][0], r["l_bal"], rtol=1e-5)
    np.testing.assert_allclose(s["z_loss"][0], r["z_loss"], rtol=2e-5)

    # output rows of a sample that puts a checked row in every 128-row GEMM tile
    toks = sample_tokens(w, dsp["members"])
    o = oracle.moe_forward(w, inp, tokens=toks, get_expert=lambda e: synth.expert_weights(w, e),
                           idx_given=adopted if len(flips) else None)
    np.testing.assert_array_equal(o["final"], dsp["final"])
    got = to_f64(y)[toks]
    err = rel_err_inf(got, o["y"])
    tol = 1e-4 if w.dtype == synth.DT_F32 else 2e-2
    tiles = sum((len(m) + 127) // 128 for m in dsp["members"]) + S * ((N + 127) // 128)
    report(f"full-size {name}", tokens=len(toks), gemm_row_tiles=tiles, rel_err_inf=err,
           elementwise_err=elementwise_err(got, o["y"]), near_ties=near, flipped=len(flips))
    print(f"{name}: y rel err {err:.3g} over {len(toks)} sampled tokens ({tiles} row tiles)")
    assert err <= tol
