"""Pins for expert capacity and the drop rule."""
import json
import os

import numpy as np
import pytest

import oracle


def test_capacity_worked_examples(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "capacity_examples.json")))
    for c in g["capacity"]:
        assert oracle.capacity(c["N"], c["E"], c["k"], c["alpha"]) == c["C"], c["cite"]
    for a in g["alpha_for_batch"]:
        assert oracle.alpha_for_batch(a["N"]) == a["alpha"], a["cite"]


def test_drop_hand_case(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "drop_hand_case.json")))
    idx = np.array(g["idx"], dtype=np.int32)
    final, members = oracle.apply_capacity_drop(idx, g["E"], g["C"])
    assert final.tolist() == g["final"]
    assert [m.tolist() for m in members] == g["members"]
    assert int((final < 0).sum()) == g["n_dropped"]


def _random_idx(rng, N, E, k, skew):
    z = rng.standard_normal((N, E)) + skew * np.linspace(2, 0, E)
    return oracle.topk_select(oracle.softmax_fp32(z), k)


@pytest.mark.parametrize("C", [0, 1, 5, 17])
def test_counts_never_exceed_capacity_and_kept_are_earliest(C):
    rng = np.random.default_rng(C)
    N, E, k = 120, 6, 2
    idx = _random_idx(rng, N, E, k, 1.5)
    final, members = oracle.apply_capacity_drop(idx, E, C)
    for e in range(E):
        assert len(members[e]) <= C
        users = [t for t in range(N) if e in idx[t]]
        assert members[e].tolist() == users[:C]
    # a kept slot keeps its expert, a dropped slot is -1
    assert np.all((final == idx) | (final == -1))


def test_capacity_at_least_Nk_is_identity():
    rng = np.random.default_rng(2)
    N, E, k = 50, 5, 3
    idx = _random_idx(rng, N, E, k, 3.0)
    final, _ = oracle.apply_capacity_drop(idx, E, N * k)
    assert np.array_equal(final, idx)


def test_all_tokens_on_one_expert_keeps_lowest_indices():
    N, E, C = 40, 4, 7
    idx = np.zeros((N, 1), dtype=np.int32)
    final, members = oracle.apply_capacity_drop(idx, E, C)
    assert members[0].tolist() == list(range(C))
    assert (final[:, 0] == 0).sum() == C and np.all(final[C:, 0] == -1)
