"""Expert-FFN and combine parity: the CUDA stages fed layouts built on the host
from the oracle's routing, vs the oracle's float64 expert outputs."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import oracle
import synth
from helpers import config_of, host_layout, rel_err_inf, to_dev, to_f64

pytestmark = pytest.mark.gpu


def oracle_routing(w, inp):
    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], w.top_k, w.bias_mode)
    C = oracle.capacity(w.n_tokens, w.n_experts, w.top_k, w.alpha) if w.cap_mode else None
    d = oracle.dispatch(r["idx"], r["key"], w.n_experts, w.cap_mode, C)
    return r, d


def run_ffn(w, inp, members, device, with_counts=True):
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, device)
    offsets = host_layout(w, members)
    R, RT = moe.moe_max_rows(cfg), moe.moe_max_total_rows(cfg)
    x = inp["x"]
    xp = np.zeros((R, w.d_model), dtype=x.dtype)
    for e, m in enumerate(members):
        xp[offsets[e]:offsets[e] + len(m)] = x[m]
    xd = to_dev(x)
    y_perm = torch.zeros((RT, w.d_model), dtype=xd.dtype, device=device)
    counts = to_dev(np.array([len(m) for m in members], dtype=np.int32)) if with_counts else None
    moe.moe_expert_ffn(cfg, xd, to_dev(xp), to_dev(offsets), counts, to_dev(inp["w_gate"]),
                       to_dev(inp["w_up"]), to_dev(inp["w_down"]), to_dev(inp["b1"]),
                       to_dev(inp["b2"]), y_perm, ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    return offsets, to_f64(y_perm)


def expert(inp, e):
    return {k: (inp[k][e] if inp.get(k) is not None else None)
            for k in ("w_gate", "w_up", "w_down", "b1", "b2")}


def tol(w):
    return 1e-4 if w.dtype == synth.DT_F32 else 2e-2


CASES = [
    synth.small_workload("mixtral_prefill", n_tokens=128, d_model=64, n_experts=1, top_k=1, d_ff=128),
    synth.small_workload("mixtral_prefill", n_tokens=300, d_model=256, n_experts=4, top_k=2, d_ff=384),
    synth.small_workload("dsv2", n_tokens=300, d_model=256, n_experts=4, top_k=2, d_ff=384, n_shared=1),
    synth.small_workload("mixtral_prefill", n_tokens=1000, d_model=512, n_experts=8, top_k=2, d_ff=1024),
    synth.small_workload("mixtral_prefill", n_tokens=333, d_model=200, n_experts=3, top_k=2, d_ff=200),
    synth.small_workload("dsv2", n_tokens=200, d_model=320, n_experts=16, top_k=6, d_ff=192, n_shared=2),
    synth.small_workload("dsv2", n_tokens=37, d_model=128, n_experts=160, top_k=6, d_ff=128, n_shared=2),
    synth.small_workload("tiny_fp32"),
    synth.small_workload("tiny_fp32", n_tokens=100, d_model=72, n_experts=5, top_k=3, d_ff=136),
    synth.small_workload("tiny_fp32", n_tokens=90, d_model=64, n_experts=4, top_k=2, d_ff=96,
                         act=synth.ACT_SWIGLU, has_ffn_bias=False, n_shared=1),
    # many rows per expert: odd row-tile counts, shared expert,
    # K and N tails
    synth.small_workload("mixtral_prefill", n_tokens=1100, d_model=256, n_experts=2, top_k=2, d_ff=384),
    synth.small_workload("dsv2", n_tokens=800, d_model=200, n_experts=2, top_k=2, d_ff=136, n_shared=1),
    # decode-sized batches: few tokens per expert (weights-as-M variant)
    synth.small_workload("decode_dsv2", d_model=256, d_ff=320),
    synth.small_workload("decode_mixtral", d_model=512, d_ff=1024),
    synth.small_workload("decode_mixtral", n_tokens=200, d_model=192, top_k=1, d_ff=200),
    synth.small_workload("decode_dsv2", n_tokens=300, d_model=128, n_experts=64, top_k=2,
                         d_ff=136, n_shared=1),
]


@pytest.mark.parametrize("with_counts", [True, False], ids=["counts", "nocounts"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.name}-N{w.n_tokens}-d{w.d_model}-E{w.n_experts}-F{w.d_ff}")
def test_expert_ffn(cuda, w, with_counts):
    inp = synth.make_inputs(w)
    _, dsp = oracle_routing(w, inp)
    offsets, y = run_ffn(w, inp, dsp["members"], cuda, with_counts)
    x = oracle.widen(inp["x"])
    worst = 0.0
    for e, m in enumerate(dsp["members"]):
        if len(m) == 0:
            continue
        ref = oracle.expert_ffn(x[m], expert(inp, e), w.act)
        got = y[offsets[e]:offsets[e] + len(m)]
        err = rel_err_inf(got, ref)
        worst = max(worst, err)
        assert err <= tol(w), f"expert {e}: rel err {err:.3g}"
    for s in range(w.n_shared):
        ref = oracle.expert_ffn(x, expert(inp, w.n_experts + s), w.act)
        got = y[offsets[w.n_experts + s]:offsets[w.n_experts + s] + w.n_tokens]
        err = rel_err_inf(got, ref)
        worst = max(worst, err)
        assert err <= tol(w), f"shared {s}: rel err {err:.3g}"
    print(f"{w.name}: worst per-expert rel err {worst:.3g}")


COMBINE_CASES = [
    CASES[2], CASES[5], CASES[7],
    # rows of 128-256 16-byte vectors with at most 4 per token take two
    # vectors per thread: a full row (the 64-expert shape), a ragged one with a
    # shared expert, and an fp32 one
    synth.small_workload("e64_reroute", n_tokens=300, d_model=2048, alpha=1.5),
    synth.small_workload("dsv2", n_tokens=150, d_model=1040, n_experts=12, top_k=3, n_shared=1),
    synth.small_workload("tiny_fp32", n_tokens=120, d_model=1000, n_experts=6, top_k=2),
    # fewer than 1024 tokens with rows wider than one CTA pass: several CTAs
    # per token, each over its own range of the row (3 here, the last ragged)
    synth.small_workload("dsv2", n_tokens=64, d_model=5136, n_experts=24, top_k=6, n_shared=2),
]


@pytest.mark.parametrize("w", COMBINE_CASES, ids=lambda w: f"{w.name}-d{w.d_model}")
def test_combine(cuda, w):
    inp = synth.make_inputs(w, with_experts=False)
    r, dsp = oracle_routing(w, inp)
    cfg = config_of(w)
    offsets = host_layout(w, dsp["members"])
    RT = moe.moe_max_total_rows(cfg)
    rng = np.random.default_rng(11)
    yp = rng.standard_normal((RT, w.d_model)).astype(np.float32)
    if w.dtype == synth.DT_BF16:
        yp = synth.round_to_bf16_bits(yp)
    pos = np.full((w.n_tokens, w.top_k), -1, dtype=np.int32)
    for e, m in enumerate(dsp["members"]):
        where = {int(t): i for i, t in enumerate(m)}
        ts, js = np.nonzero(dsp["final"] == e)
        for t, j in zip(ts, js):
            pos[t, j] = offsets[e] + where[int(t)]
    y = torch.zeros((w.n_tokens, w.d_model), dtype=torch.float32 if w.dtype == 0 else torch.bfloat16,
                    device=cuda)
    moe.moe_combine(cfg, to_dev(yp), to_dev(offsets), to_dev(dsp["final"].astype(np.int32)),
                    to_dev(pos), to_dev(r["w"]), y)
    torch.cuda.synchronize()
    Y = oracle.widen(yp)
    got = to_f64(y)
    for t in range(w.n_tokens):
        kept = [j for j in range(w.top_k) if dsp["final"][t, j] >= 0]
        ref = oracle.combine_token([Y[offsets[w.n_experts + s] + t] for s in range(w.n_shared)],
                                   [Y[pos[t, j]] for j in kept], [r["w"][t, j] for j in kept])
        bound = 1e-6 if w.dtype == 0 else 2 ** -8
        assert np.max(np.abs(got[t] - ref)) <= bound * max(1.0, np.max(np.abs(ref))) * 2
