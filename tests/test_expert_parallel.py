"""Expert-parallel exchange logic on CPU ranks: capacity decisions identical to
one device, consistent send/receive counts and segments, and (world size 2,
gloo) a whole expert-parallel layer equal to the single-device oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
from mixture_experts_ffn_19_b300 import expert_parallel as ep


def _split(N, R, seed):
    """Uneven, seeded contiguous split of N tokens over R ranks."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, N), size=R - 1, replace=False))
    return np.split(np.arange(N), cuts)


def _simulate(idx, key, E, cap_mode, cap, parts):
    """Every rank's plan in one process: the collectives become stacks."""
    R = len(parts)
    hist_all = np.stack([np.bincount(idx[p].ravel(), minlength=E) for p in parts])
    plans = [ep.primary_plan(idx[p], hist_all, r, cap) for r, p in enumerate(parts)]
    finals = [pl[0] for pl in plans]
    blocks = [pl[1] for pl in plans]
    pending = [pl[2] for pl in plans]
    n_dropped = sum(len(p) for p in pending) if cap_mode == 1 else 0
    n_rerouted = 0
    if cap_mode == 2:
        fill = np.minimum(cap, hist_all.sum(axis=0))
        while sum(len(p) for p in pending):
            full = fill >= cap
            props = []
            for r in range(R):
                pr, dr = ep.propose(finals[r], key[parts[r]], pending[r], full)
                n_dropped += len(dr)
                props.append(pr)
            ph_all = np.stack([np.bincount([e for (_, _, e) in pr], minlength=E) for pr in props])
            new_fill = None
            for r in range(R):
                acc, pending[r], new_fill = ep.reroute_round(props[r], ph_all, r, fill, cap)
                for (t, j, e) in acc:
                    finals[r][t, j] = e
                    blocks[r][e].append((t, j))
                n_rerouted += len(acc)
            fill = new_fill
    kept_all = np.stack([[len(b) for b in bl] for bl in blocks])
    return np.concatenate(finals), blocks, kept_all, n_dropped, n_rerouted


CASES = [
    ("drop", 1, 0.6, 2), ("drop", 1, 0.9, 3), ("reroute", 2, 0.7, 2), ("reroute", 2, 0.5, 4),
    ("none", 0, 0.0, 3),
]


@pytest.mark.parametrize("name,cap_mode,alpha,R", CASES)
def test_capacity_plan_matches_one_device(name, cap_mode, alpha, R):
    rng = np.random.default_rng(R * 10 + cap_mode)
    N, E, k = 300, 12, 3
    z = rng.standard_normal((N, E)) - 1.1 * np.log(rng.permutation(E) + 1.0)
    p = oracle.softmax_fp32(z)
    idx = oracle.topk_select(p, k)
    cap = ep.capacity_for(N, E, k, cap_mode, alpha)
    assert cap == (oracle.capacity(N, E, k, alpha) if cap_mode else None)
    one = oracle.dispatch(idx, p, E, cap_mode, cap)
    final, blocks, kept_all, nd, nr = _simulate(idx, p, E, cap_mode, cap, _split(N, R, R))
    assert np.array_equal(final, one["final"])
    assert np.array_equal(kept_all.sum(axis=0), one["counts"])
    assert (nd, nr) == (one["n_dropped"], one["n_rerouted"])
    if cap_mode:
        assert (one["final"] < 0).any() or one["n_rerouted"] > 0


@pytest.mark.parametrize("R", [2, 3, 4])
def test_exchange_plan_moves_every_kept_row_to_its_owner_and_back(R):
    rng = np.random.default_rng(R)
    N, E, k = 200, 10, 2
    p = oracle.softmax_fp32(rng.standard_normal((N, E)))
    idx = oracle.topk_select(p, k)
    cap = ep.capacity_for(N, E, k, 1, 0.8)
    parts = _split(N, R, 7)
    final, blocks, kept_all, _, _ = _simulate(idx, p, E, 1, cap, parts)
    owner = ep.expert_owner(E, R)
    assert sorted(np.bincount(owner, minlength=R)) == sorted(
        [len(ep.local_experts(E, R, r)) for r in range(R)])
    plans = [ep.exchange_plan(blocks[r], kept_all, r) for r in range(R)]
    # what each source sends to each owner is what that owner expects from it
    sent = np.stack([pl["send_counts"] for pl in plans])       # [source, owner]
    recvd = np.stack([pl["recv_counts"] for pl in plans])      # [owner, source]
    assert np.array_equal(sent, recvd.T)
    # deliver labels (global token, slot) and check every segment row
    bufs = []
    for r in range(R):
        labels = [(int(parts[r][t]), j) for (t, j) in plans[r]["send_slots"]]
        cuts = np.cumsum(plans[r]["send_counts"])[:-1]
        bufs.append(np.split(np.array(labels, dtype=np.int64).reshape(-1, 2), cuts))
    for o in range(R):
        recv = np.concatenate([bufs[r][o] for r in range(R)])
        for e, seg in plans[o]["segments"].items():
            assert owner[e] == o and len(seg) == kept_all[:, e].sum()
            for (t, j) in recv[seg]:
                assert final[t, j] == e
            # sources ascending inside the segment (global token order within a source block)
            src = np.searchsorted(np.cumsum([len(q) for q in parts]), recv[seg][:, 0], side="right")
            assert np.all(np.diff(src) >= 0)
        assert len(recv) == sum(len(s) for s in plans[o]["segments"].values())
    # every kept slot is sent exactly once
    all_sent = sorted((int(parts[r][t]), j) for r in range(R) for (t, j) in plans[r]["send_slots"])
    assert all_sent == sorted((int(t), int(j)) for t, j in zip(*np.nonzero(final >= 0)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, wname, overrides, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.small_workload(wname, **overrides)
        inp = synth.make_inputs(w)
        part = _split(w.n_tokens, world, 11)[rank]
        r = oracle.route(inp["x"][part], inp["w_router"], inp["router_bias"], w.top_k,
                         w.bias_mode)
        E, S = w.n_experts, w.n_shared

        def expert(e):
            return {key: (inp[key][e] if inp.get(key) is not None else None)
                    for key in ("w_gate", "w_up", "w_down", "b1", "b2")}

        def expert_fn(e, rows):
            assert ep.expert_owner(E, world)[e] == rank
            return oracle.expert_ffn(oracle.widen(rows.numpy().view(np.uint16)), expert(e), w.act)

        def shared_fn(xr):
            xs = oracle.widen(xr.numpy().view(np.uint16))
            y = np.zeros(xs.shape)
            for s in range(S):
                y = y + oracle.expert_ffn(xs, expert(E + s), w.act)
            return y

        x = torch.from_numpy(inp["x"][part].view(np.int16))
        y, info = ep.ep_forward(x, r["idx"], r["w"], r["key"], E, w.cap_mode, w.alpha, expert_fn,
                                shared_fn if S else None)
        out[rank] = (part, y, info["final"], info["counts"], info["n_dropped"], info["n_rerouted"],
                     info["send_counts"], info["recv_counts"])
    finally:
        dist.destroy_process_group()


EP_CASES = [
    ("mixtral_prefill", dict(n_tokens=160, d_model=32, n_experts=6, d_ff=24, alpha=0.7)),
    ("e64_reroute", dict(n_tokens=200, d_model=32, n_experts=8, d_ff=24, alpha=0.6)),
    ("dsv2", dict(n_tokens=90, d_model=32, n_experts=10, top_k=3, d_ff=24, n_shared=2)),
]


@pytest.mark.parametrize("wname,overrides", EP_CASES, ids=[c[0] for c in EP_CASES])
def test_two_rank_expert_parallel_layer_equals_one_device(wname, overrides):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), wname, overrides, out), nprocs=world,
             join=True)
    w = synth.small_workload(wname, **overrides)
    inp = synth.make_inputs(w)
    one = oracle.moe_forward(w, inp)
    y = np.zeros((w.n_tokens, w.d_model))
    final = np.zeros((w.n_tokens, w.top_k), dtype=np.int32)
    for rank in range(world):
        part, yr, fr, counts, nd, nr, sc, rc = out[rank]
        y[part], final[part] = yr, fr
        assert np.array_equal(counts, one["counts"])
        assert (nd, nr) == (one["n_dropped"], one["n_rerouted"])
    assert np.array_equal(out[0][6], [out[0][7][0], out[1][7][0]])    # rank 0's sends
    assert np.array_equal(final, one["final"])
    np.testing.assert_allclose(y, one["y"], rtol=1e-12, atol=1e-12)
    if w.cap_mode == 2:
        assert one["n_rerouted"] > 0
    if w.cap_mode == 1:
        assert one["n_dropped"] > 0
