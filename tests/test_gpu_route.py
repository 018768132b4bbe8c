"""Router parity: CUDA moe_route vs the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import oracle
import synth
from helpers import config_of, report, to_dev, valid_selection

pytestmark = pytest.mark.gpu

NEAR_TIE = 1e-6


def run_route(w, inp, device):
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, device)
    N, k, E = w.n_tokens, w.top_k, w.n_experts
    idx = torch.full((N, k), -7, dtype=torch.int32, device=device)
    gw = torch.zeros((N, k), dtype=torch.float32, device=device)
    probs = torch.zeros((N, E), dtype=torch.float32, device=device)
    freq = torch.zeros(E, dtype=torch.float32, device=device)
    mp = torch.zeros(E, dtype=torch.float32, device=device)
    lb = torch.zeros(1, dtype=torch.float32, device=device)
    zl = torch.full((1,), -1.0, dtype=torch.float32, device=device)
    ent = torch.full((1,), -1.0, dtype=torch.float32, device=device)
    st = moe.make_stats(expert_freq=freq, mean_prob=mp, l_bal=lb, z_loss=zl, router_entropy=ent)
    moe.moe_route(cfg, to_dev(inp["x"]), to_dev(inp["w_router"]), to_dev(inp["router_bias"]),
                  idx, gw, probs, st, ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    out = {k_: v.cpu().numpy() for k_, v in
           dict(idx=idx, w=gw, p=probs, freq=freq, mean_prob=mp, l_bal=lb, z_loss=zl,
                entropy=ent).items()}
    out["ws"] = ws
    return out


def check_route(w, inp, g):
    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], w.top_k, w.bias_mode)
    near = r["margin"] < NEAR_TIE
    same = np.all(g["idx"] == r["idx"], axis=1)
    mism = np.nonzero(~same)[0]
    print(f"{w.name}: near-tie tokens {near.sum()}, index mismatches {len(mism)}, "
          f"max |dp| {np.max(np.abs(g['p'] - r['key'])):.3g}")
    # every mismatch must be a counted near-tie, resolved in one of its valid ways
    assert np.all(near[mism]), f"mismatch on non-near-tie tokens {mism[~near[mism]][:10]}"
    for t in mism:
        assert valid_selection(r["key"][t], g["idx"][t]), f"token {t}: invalid selection"
    report(f"route {w.name} N={w.n_tokens} E={w.n_experts} k={w.top_k}",
           near_ties=int(near.sum()), flipped=len(mism),
           max_abs_dp=float(np.max(np.abs(g["p"] - r["key"]))))
    ok = same & ~near
    np.testing.assert_allclose(g["w"][ok], r["w"][ok], rtol=1e-5, atol=1e-7)
    # probs holds the selection scores: p, or p + b under selection-only bias
    np.testing.assert_allclose(g["p"], r["key"], rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(g["mean_prob"], r["mean_prob"], rtol=1e-5, atol=1e-9)
    if len(mism) == 0:
        np.testing.assert_array_equal(g["freq"], r["expert_freq"].astype(np.float32))
    np.testing.assert_allclose(g["l_bal"][0], r["l_bal"], rtol=1e-5)
    assert np.allclose(g["w"].astype(np.float64).sum(1), 1.0, atol=1e-6)
    # z-loss (fp32 logsumexp per token); entropy (a flipped near-tie token may
    # move its own term by at most log2 k)
    np.testing.assert_allclose(g["z_loss"][0], r["z_loss"], rtol=2e-5)
    tol = 1e-5 * r["router_entropy"] + len(mism) * np.log2(max(w.top_k, 2)) / w.n_tokens
    assert abs(g["entropy"][0] - r["router_entropy"]) <= tol + 1e-7
    return r


SMALL = [
    synth.small_workload("tiny_fp32"),
    synth.small_workload("tiny_fp32", n_tokens=77, d_model=72, n_experts=3, top_k=3),
    synth.small_workload("dsv2", n_tokens=300, d_model=520, n_experts=37, top_k=6),
    synth.small_workload("e64_reroute", n_tokens=1000, d_model=256),
    synth.small_workload("mixtral_prefill", n_tokens=1, d_model=64, n_experts=1, top_k=1),
    synth.small_workload("dsv2", n_tokens=129, d_model=64, n_experts=256, top_k=8),
    # selection-only bias (DeepSeek-V3 style), fp32 and bf16
    synth.small_workload("dsv2_select", n_tokens=700, d_model=256, n_experts=64, top_k=6),
    synth.small_workload("tiny_fp32", n_tokens=150, bias_law=synth.BIAS_UNIFORM_P, bias_mode=1),
    # each lane-group width of the finish kernel: 8 lanes per token up to 64
    # experts (above), 16 up to 128, 32 beyond; the upper bounds of each, a
    # ragged group, both dtypes, selection-only bias, and a batch large enough
    # for many CTAs of 8-token warps
    synth.small_workload("dsv2", n_tokens=333, d_model=256, n_experts=65, top_k=6),
    synth.small_workload("dsv2", n_tokens=2500, d_model=128, n_experts=100, top_k=4),
    synth.small_workload("dsv2_select", n_tokens=400, d_model=128, n_experts=128, top_k=8),
    synth.small_workload("tiny_fp32", n_tokens=300, n_experts=97, top_k=5),
    synth.small_workload("dsv2", n_tokens=600, d_model=128, n_experts=200, top_k=6),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"{w.name}-N{w.n_tokens}-E{w.n_experts}")
def test_route_small(cuda, w):
    inp = synth.make_inputs(w, with_experts=False)
    check_route(w, inp, run_route(w, inp, cuda))


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_route_full_size(cuda, name):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, with_experts=False)
    check_route(w, inp, run_route(w, inp, cuda))


def test_zero_router_uniform(cuda):
    w = synth.small_workload("e64_reroute", n_tokens=256, d_model=64)
    inp = synth.make_inputs(w, with_experts=False)
    inp["w_router"][:] = 0
    inp["router_bias"] = None
    w = w.replace(bias_law=synth.BIAS_NONE)
    g = run_route(w, inp, cuda)
    assert np.all(g["idx"] == np.arange(2)[None, :])          # ties -> lowest indices
    assert g["l_bal"][0] == 1.0
    assert np.all(g["p"] == np.float32(1 / 64))


def test_z_loss_entropy_closed_form(cuda):
    # zero router: lse = ln E for every token, equal gates give log2 k bits
    w = synth.small_workload("e64_reroute", n_tokens=300, d_model=64, top_k=4)
    inp = synth.make_inputs(w, with_experts=False)
    inp["w_router"][:] = 0
    inp["router_bias"] = None
    w = w.replace(bias_law=synth.BIAS_NONE)
    g = run_route(w, inp, cuda)
    np.testing.assert_allclose(g["z_loss"][0], 0.001 * np.log(64) ** 2, rtol=1e-6)
    np.testing.assert_allclose(g["entropy"][0], 2.0, rtol=1e-6)


@pytest.mark.parametrize("w", [
    synth.small_workload("dsv2_select", n_tokens=700, d_model=256, n_experts=64, top_k=6),
    synth.small_workload("e64_reroute", n_tokens=1000, d_model=256),
    synth.small_workload("mixtral_prefill", n_tokens=0, d_model=64),
], ids=lambda w: f"{w.name}-N{w.n_tokens}")
def test_router_bias_update(cuda, w):
    """b_e -/+ gamma from the picks of the last route on the workspace."""
    inp = synth.make_inputs(w, with_experts=False)
    if inp["router_bias"] is None:
        inp["router_bias"] = np.zeros(w.n_experts, dtype=np.float32)
        w = w.replace(bias_law=synth.BIAS_UNIFORM_P)
    cfg = config_of(w)
    g = run_route(w, inp, cuda) if w.n_tokens else {"ws": moe.alloc_workspace(cfg, cuda)}
    gamma = 1e-3
    b = torch.from_numpy(inp["router_bias"].copy()).to(cuda)
    moe.moe_router_bias_update(cfg, g["ws"], b, gamma)
    got = b.cpu().numpy()
    if w.n_tokens == 0:
        assert np.array_equal(got, inp["router_bias"])
        return
    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], w.top_k, w.bias_mode)
    # the device's own picks (equal to the oracle's unless a near-tie flipped)
    picks = np.rint(g["freq"].astype(np.float64) * w.n_tokens * w.top_k).astype(np.int64)
    if np.array_equal(g["idx"], r["idx"]):
        assert np.array_equal(picks, r["picks"])
    expect = oracle.router_bias_update(inp["router_bias"], picks, w.n_tokens, w.top_k, gamma)
    assert np.array_equal(got, expect)


def test_bias_update_rejects_bad_args(cuda):
    w = synth.small_workload("dsv2_select", n_tokens=64, d_model=64, n_experts=16, top_k=2)
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    b = torch.zeros(16, device=cuda)
    with pytest.raises(moe.MoeError):
        moe.moe_router_bias_update(cfg, ws, b, float("nan"))
    bad = config_of(w)
    bad.bias_mode = 7
    with pytest.raises(moe.MoeError):
        moe.moe_router_bias_update(bad, ws, b, 1e-3)
