"""Dispatch parity: CUDA moe_dispatch fed the oracle's routing, vs oracle.dispatch.

Both sides see identical inputs (the oracle's top-k indices and float32
probabilities are uploaded), so every integer output must match bit for bit."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import oracle
import synth
from helpers import config_of, to_dev

pytestmark = pytest.mark.gpu


def run_dispatch(w, inp, idx, p, device):
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, device)
    N, k, E, S, d = w.n_tokens, w.top_k, w.n_experts, w.n_shared, w.d_model
    R = moe.moe_max_rows(cfg)
    x = to_dev(inp["x"])
    out = dict(
        final=torch.full((N, k), -9, dtype=torch.int32, device=device),
        pos=torch.full((N, k), -9, dtype=torch.int32, device=device),
        offsets=torch.full((E + S + 1,), -9, dtype=torch.int32, device=device),
        perm=torch.full((R,), -9, dtype=torch.int32, device=device),
        x_perm=torch.zeros((R, d), dtype=x.dtype, device=device),
        counts=torch.full((E,), -9, dtype=torch.int32, device=device),
        nd=torch.full((1,), -9, dtype=torch.int32, device=device),
        nr=torch.full((1,), -9, dtype=torch.int32, device=device))
    st = moe.make_stats(counts=out["counts"], n_dropped=out["nd"], n_rerouted=out["nr"])
    moe.moe_dispatch(cfg, to_dev(idx.astype(np.int32)), to_dev(p.astype(np.float32)), x,
                     out["final"], out["pos"], out["offsets"], out["perm"], out["x_perm"], st, ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    g = {k_: v.cpu() for k_, v in out.items()}
    g["x"] = x.cpu()
    return g


def check_dispatch(w, inp, idx, p, g):
    E, S, N, k = w.n_experts, w.n_shared, w.n_tokens, w.top_k
    C = oracle.capacity(N, E, k, w.alpha) if w.cap_mode else None
    o = oracle.dispatch(idx, p, E, w.cap_mode, C)
    final = g["final"].numpy()
    np.testing.assert_array_equal(final, o["final"])
    np.testing.assert_array_equal(g["counts"].numpy(), o["counts"])
    assert int(g["nd"][0]) == o["n_dropped"] and int(g["nr"][0]) == o["n_rerouted"]
    off = g["offsets"].numpy()
    perm = g["perm"].numpy()
    pos = g["pos"].numpy()
    row = 0
    for e in range(E):
        assert off[e] == row
        c = o["counts"][e]
        np.testing.assert_array_equal(perm[off[e]:off[e] + c], o["members"][e])
        assert np.all(perm[off[e] + c:off[e] + (c + 127) // 128 * 128] == -1)
        row += (c + 127) // 128 * 128
    for s in range(S):
        assert off[E + s] == row
        row += (N + 127) // 128 * 128
    assert off[E + S] == row
    # pos: row of each kept slot inside its expert's member list; -1 when dropped
    for e in range(E):
        where = {int(t): i for i, t in enumerate(o["members"][e])}
        ts, js = np.nonzero(o["final"] == e)
        for t, j in zip(ts, js):
            assert pos[t, j] == off[e] + where[int(t)]
    assert np.all(pos[o["final"] < 0] == -1)
    # x_perm rows are copies of x
    kept = pos[pos >= 0]
    toks = perm[kept]
    assert torch.equal(g["x_perm"][torch.from_numpy(kept.astype(np.int64))],
                       g["x"][torch.from_numpy(toks.astype(np.int64))])
    return o


def routed(w, inp):
    # the reroute ranks candidates by the selection scores (p, or p + b)
    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], w.top_k, w.bias_mode)
    return r["idx"], r["key"]


CASES = [
    synth.small_workload("tiny_fp32"),
    synth.small_workload("mixtral_prefill", n_tokens=700, d_model=64, alpha=0.6),
    synth.small_workload("mixtral_prefill", n_tokens=300, d_model=64, n_experts=5, top_k=3, alpha=0.3),
    synth.small_workload("e64_reroute", n_tokens=2000, d_model=64, alpha=1.0),
    synth.small_workload("e64_reroute", n_tokens=513, d_model=64, n_experts=16, top_k=4, alpha=0.8),
    synth.small_workload("e64_reroute", n_tokens=700, d_model=64, n_experts=8, top_k=1, alpha=0.4),
    synth.small_workload("e64_reroute", n_tokens=300, d_model=64, n_experts=8, top_k=2, alpha=0.3),
    synth.small_workload("dsv2", n_tokens=333, d_model=64, n_experts=160, top_k=6, n_shared=2),
    synth.small_workload("dsv2", n_tokens=1, d_model=64),
    # either side of the one-kernel dispatch's limit (N k <= 4096, no reroute), with drops
    synth.small_workload("mixtral_prefill", n_tokens=2048, d_model=64, alpha=0.7),
    synth.small_workload("mixtral_prefill", n_tokens=2049, d_model=64, alpha=0.7),
    synth.small_workload("e64_reroute", n_tokens=2500, d_model=64, n_experts=256, top_k=8, alpha=1.0),
    # reroute ranked by p + b (selection-only bias)
    synth.small_workload("e64_reroute", n_tokens=1500, d_model=64, alpha=0.7,
                         bias_law=synth.BIAS_UNIFORM_P, bias_mode=1),
    # the reroute kernel's other paths: a per-chunk count table too large for
    # every CTA to sum (71 chunks x 256 experts), more 128-token chunks than
    # co-resident CTAs (313), and both at once
    synth.small_workload("e64_reroute", n_tokens=9000, d_model=64, n_experts=256, alpha=0.5),
    synth.small_workload("e64_reroute", n_tokens=40000, d_model=64, n_experts=32, alpha=0.5),
    synth.small_workload("e64_reroute", n_tokens=40000, d_model=64, n_experts=64, alpha=0.7),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.name}-N{w.n_tokens}-E{w.n_experts}k{w.top_k}a{w.alpha}")
def test_dispatch_small(cuda, w):
    inp = synth.make_inputs(w, with_experts=False)
    idx, p = routed(w, inp)
    o = check_dispatch(w, inp, idx, p, run_dispatch(w, inp, idx, p, cuda))
    print(w.name, "dropped", o["n_dropped"], "rerouted", o["n_rerouted"])


@pytest.mark.parametrize("name", ["mixtral_prefill", "dsv2", "e64_reroute", "decode_dsv2"])
def test_dispatch_full_size(cuda, name):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, with_experts=False)
    idx, p = routed(w, inp)
    o = check_dispatch(w, inp, idx, p, run_dispatch(w, inp, idx, p, cuda))
    print(name, "dropped", o["n_dropped"], "rerouted", o["n_rerouted"])


def test_all_tokens_on_one_expert_keeps_lowest(cuda):
    w = synth.small_workload("mixtral_prefill", n_tokens=1000, d_model=64, n_experts=4, top_k=1,
                             alpha=0.5)
    inp = synth.make_inputs(w, with_experts=False)
    idx = np.zeros((1000, 1), dtype=np.int32)
    p = np.tile(np.array([[0.7, 0.1, 0.1, 0.1]], dtype=np.float32), (1000, 1))
    check_dispatch(w, inp, idx, p, run_dispatch(w, inp, idx, p, cuda))


def test_reroute_hand_cases(cuda):
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "reroute_hand_case.json")))
    for c in g["cases"]:
        p = np.array(c["p"], dtype=np.float32)
        N = p.shape[0]
        # alpha chosen so that floor(floor(k*N/E)*alpha) equals the case's capacity
        base = (c["k"] * N) // c["E"]
        w = synth.small_workload("e64_reroute", n_tokens=N, d_model=64, n_experts=c["E"],
                                 top_k=c["k"], alpha=(c["C"] + 0.5) / base)
        assert oracle.capacity(N, c["E"], c["k"], w.alpha) == c["C"]
        inp = synth.make_inputs(w, with_experts=False)
        idx = oracle.topk_select(p, c["k"])
        r = run_dispatch(w, inp, idx, p, cuda)
        assert r["final"].numpy().tolist() == c["final"], c["name"]
        assert int(r["nr"][0]) == c["n_rerouted"] and int(r["nd"][0]) == c["n_dropped"]
