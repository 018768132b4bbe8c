"""Pins for the oracle's router steps (logits, softmax, top-k, renormalisation)."""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle


def _rand_p(rng, n, e):
    z = rng.standard_normal((n, e))
    return oracle.softmax_fp32(z)


def test_softmax_matches_scipy_and_is_shift_invariant():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((64, 13)) * 3
    p = oracle.softmax_fp32(z)
    ref = scipy.special.softmax(z, axis=1).astype(np.float32)
    assert np.array_equal(p, ref) or np.max(np.abs(p - ref) / ref) < 2 ** -23
    p2 = oracle.softmax_fp32(z + 123.25)
    assert np.max(np.abs(p2 - p) / p) < 4 * 2 ** -24


@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 2), (8, 3), (7, 6)])
def test_topk_equals_brute_force_over_subsets(E, k):
    rng = np.random.default_rng(E * 10 + k)
    p = _rand_p(rng, 200, E)
    idx = oracle.topk_select(p, k)
    for t in range(p.shape[0]):
        best = max(itertools.combinations(range(E), k),
                   key=lambda s: sum(float(p[t, e]) for e in s))
        assert set(idx[t]) == set(best)
        # slot order: descending probability
        vals = p[t, idx[t]]
        assert np.all(vals[:-1] >= vals[1:])


def test_topk_ties_go_to_lower_index(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "router_hand_cases.json")))
    for case in g["ties"]:
        p = np.array([case["p"]], dtype=np.float32)
        assert oracle.topk_select(p, case["k"])[0].tolist() == case["idx"]


def test_renormalise_hand_case_and_sum_to_one(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "router_hand_cases.json")))
    for case in g["renorm"]:
        p = np.array([case["p"]], dtype=np.float32)
        idx = oracle.topk_select(p, case["k"])
        assert idx[0].tolist() == case["idx"]
        w = oracle.renormalise(p, idx)
        np.testing.assert_allclose(w[0], case["w"], rtol=1e-6)
    rng = np.random.default_rng(3)
    p = _rand_p(rng, 500, 16)
    w = oracle.renormalise(p, oracle.topk_select(p, 4))
    assert np.max(np.abs(w.astype(np.float64).sum(1) - 1.0)) <= 4 * 2 ** -24


def test_k_equals_E_every_expert_fires_and_gates_equal_p():
    rng = np.random.default_rng(4)
    E = 6
    p = _rand_p(rng, 100, E)
    idx = oracle.topk_select(p, E)
    assert all(sorted(r) == list(range(E)) for r in idx.tolist())
    w = oracle.renormalise(p, idx)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=2e-7)
    # with k == E only the slot order can flip: the margin is the smallest gap
    srt = -np.sort(-p.astype(np.float64), axis=1)
    np.testing.assert_array_equal(oracle.topk_margin(p, E), np.min(srt[:, :-1] - srt[:, 1:], axis=1))


def test_zero_router_gives_uniform_probabilities():
    x = np.random.default_rng(5).standard_normal((10, 32)).astype(np.float32)
    for E in (8, 64):
        p = oracle.softmax_fp32(oracle.router_logits(x, np.zeros((E, 32), np.float32)))
        assert np.all(p == np.float32(1.0 / E))


def test_router_bias_shifts_logits_and_expert_permutation_commutes():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((20, 16)).astype(np.float32)
    wr = rng.standard_normal((5, 16)).astype(np.float32)
    b = rng.uniform(-1, 1, 5).astype(np.float32)
    z0 = oracle.router_logits(x, wr)
    z1 = oracle.router_logits(x, wr, b)
    np.testing.assert_allclose(z1 - z0, np.broadcast_to(b.astype(np.float64), z0.shape), atol=1e-12)
    perm = rng.permutation(5)
    zp = oracle.router_logits(x, wr[perm], b[perm])
    np.testing.assert_allclose(zp, z1[:, perm], atol=1e-12)
    # a single dot product written out longhand
    assert abs(z0[3, 2] - sum(float(x[3, j]) * float(wr[2, j]) for j in range(16))) < 1e-12


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x3E80], dtype=np.uint16)
    assert oracle.widen(bits).tolist() == [1.0, -1.0, 3.140625, 0.0, 0.25]


def test_margin_flags_near_ties():
    p = np.array([[0.5, 0.25, 0.25 - 2 ** -25, 0.0]], dtype=np.float32)
    m = oracle.topk_margin(p, 2)
    assert 0 < m[0] < 1e-6
    # a near-tie inside the selected set (slot order) is flagged too
    q = np.array([[0.4, 0.4 - 2 ** -24, 0.1, 0.1 - 0.05]], dtype=np.float32)
    assert 0 < oracle.topk_margin(q, 2)[0] < 1e-6
    assert oracle.topk_margin(np.array([[0.5, 0.3, 0.2, 0.0]], np.float32), 2)[0] == \
        np.float64(np.float32(0.3)) - np.float64(np.float32(0.2))
