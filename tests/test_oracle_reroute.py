"""Pins for the reroute rule (next-best unfilled expert)."""
import json
import os

import numpy as np
import pytest

import oracle


def test_hand_cases(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "reroute_hand_case.json")))
    for c in g["cases"]:
        p = np.array(c["p"], dtype=np.float32)
        idx = oracle.topk_select(p, c["k"])
        final, members, nr, nd, rounds = oracle.apply_capacity_reroute(idx, p, c["E"], c["C"])
        assert final.tolist() == c["final"], c["name"]
        assert [m.tolist() for m in members] == c["members"], c["name"]
        assert (nr, nd, rounds) == (c["n_rerouted"], c["n_dropped"], c["rounds"]), c["name"]


def _case(seed, N, E, k, C, skew):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((N, E)) - skew * np.log(rng.permutation(E) + 1.0)
    p = oracle.softmax_fp32(z)
    idx = oracle.topk_select(p, k)
    return p, idx, oracle.apply_capacity_reroute(idx, p, E, C)


@pytest.mark.parametrize("seed,N,E,k,C,skew", [
    (0, 200, 8, 2, 30, 1.1), (1, 300, 16, 2, 20, 1.1), (2, 97, 6, 3, 40, 2.0),
    (3, 64, 8, 1, 4, 1.1), (4, 150, 12, 4, 25, 0.5)])
def test_invariants(seed, N, E, k, C, skew):
    p, idx, (final, members, nr, nd, rounds) = _case(seed, N, E, k, C, skew)
    counts = np.array([len(m) for m in members])
    assert np.all(counts <= C)
    # conservation: kept + rerouted + dropped = N*k, and the members match final
    assert int((final >= 0).sum()) == counts.sum()
    assert int((final < 0).sum()) == nd
    assert int(((final >= 0) & (final != idx)).sum()) == nr
    for e in range(E):
        assert sorted(members[e].tolist()) == sorted(
            t for t in range(N) for j in range(k) if final[t, j] == e)
    for t in range(N):
        held = [e for e in final[t] if e >= 0]
        assert len(held) == len(set(held)), "a token holds an expert twice"
    # primary assignments keep the earliest tokens of each expert
    for e in range(E):
        users = [t for t in range(N) if e in idx[t]]
        assert members[e][:min(C, len(users))].tolist() == users[:C]
    full = counts >= C
    for t in range(N):
        held = set(int(e) for e in final[t] if e >= 0)
        for j in range(k):
            e_new = final[t, j]
            if e_new < 0:
                # maximality: a dropped slot has no expert left with room it could take
                assert all(full[e] or e in held for e in range(E))
            elif e_new != idx[t, j]:
                # next-best: every expert it prefers (and does not hold) ended full
                better = [e for e in range(E)
                          if (p[t, e] > p[t, e_new] or (p[t, e] == p[t, e_new] and e < e_new))]
                assert all(full[e] or e in held for e in better)


def test_room_everywhere_means_no_reroute():
    p, idx, (final, members, nr, nd, rounds) = _case(7, 100, 8, 2, 200, 1.1)
    assert np.array_equal(final, idx) and nr == 0 and nd == 0 and rounds == 0
