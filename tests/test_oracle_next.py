"""Pins of the oracle's router extras: z-loss, router entropy, selection-only
bias and the bias update (CPU only).

Each pin is something other than the oracle's own formula: a closed form, a
library routine (scipy.special.logsumexp), brute force over subsets, or a
hand-worked case.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle as O


def test_z_loss_zero_logits_closed_form():
    # all logits 0: logsumexp = ln E for every token
    for E in (2, 8, 160):
        z = np.zeros((7, E))
        assert O.router_z_loss(z) == pytest.approx(0.001 * math.log(E) ** 2, rel=1e-14)


def test_z_loss_matches_scipy_and_shift():
    rng = np.random.default_rng(3)
    z = rng.normal(size=(50, 16)) * 3.0
    ref = 0.001 * np.mean(logsumexp(z, axis=1) ** 2)
    assert O.router_z_loss(z) == pytest.approx(ref, rel=1e-13)
    # a constant shift c moves every lse by c
    c = 2.5
    ref_c = 0.001 * np.mean((logsumexp(z, axis=1) + c) ** 2)
    assert O.router_z_loss(z + c) == pytest.approx(ref_c, rel=1e-13)


def test_z_loss_ignores_expert_bias():
    # the z-loss is taken on the router's own logits: the bias changes p, not L_z
    rng = np.random.default_rng(4)
    x = rng.normal(size=(20, 8)).astype(np.float32)
    wr = rng.normal(size=(6, 8)).astype(np.float32)
    b = rng.uniform(-1, 1, size=6).astype(np.float32)
    r0 = O.route(x, wr, None, 2)
    r1 = O.route(x, wr, b, 2)
    assert r0["z_loss"] == r1["z_loss"]
    assert not np.array_equal(r0["p"], r1["p"])


def test_entropy_closed_forms():
    k = 4
    w = np.full((5, k), 1.0 / k, dtype=np.float32)
    assert O.router_entropy(w) == pytest.approx(math.log2(k), rel=1e-7)
    one = np.zeros((3, 2), dtype=np.float32)
    one[:, 0] = 1.0
    assert O.router_entropy(one) == 0.0
    hand = np.array([[0.75, 0.25]], dtype=np.float32)
    assert O.router_entropy(hand) == pytest.approx(0.8112781244591328, rel=1e-12)


def test_entropy_of_top2_softmax():
    # [P4] §3.1 code: softmax of the two selected logits, then -sum p log2 p
    z = np.array([[2.0, 0.5, -1.0, 1.0]])
    a, b = 2.0, 1.0
    pa = math.exp(a) / (math.exp(a) + math.exp(b))
    ref = -(pa * math.log2(pa) + (1 - pa) * math.log2(1 - pa))
    x = np.array([[1, 0, 0, 0]], dtype=np.float32)
    wr = np.zeros((4, 4), dtype=np.float32)
    wr[:, 0] = z[0]                          # z = x Wr^T with x = e_0
    r = O.route(x, wr, None, 2)
    assert list(r["idx"][0]) == [0, 3]
    assert r["router_entropy"] == pytest.approx(ref, rel=1e-6)


def test_selection_bias_zero_reduces_to_plain_router():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(40, 12)).astype(np.float32)
    wr = (rng.normal(size=(9, 12)) / 4).astype(np.float32)
    zero = np.zeros(9, dtype=np.float32)
    r0 = O.route(x, wr, None, 3)
    r1 = O.route(x, wr, zero, 3, bias_mode=1)
    for key in ("idx", "w", "p"):
        assert np.array_equal(r0[key], r1[key])


def test_selection_bias_brute_force_and_gates():
    rng = np.random.default_rng(6)
    E, k = 6, 2
    x = rng.normal(size=(30, 10)).astype(np.float32)
    wr = (rng.normal(size=(E, 10)) / 3).astype(np.float32)
    b = rng.uniform(-0.2, 0.2, size=E).astype(np.float32)
    r = O.route(x, wr, b, k, bias_mode=1)
    z = x.astype(np.float64) @ wr.astype(np.float64).T
    p = np.exp(z - z.max(1, keepdims=True))
    p = (p / p.sum(1, keepdims=True)).astype(np.float32)
    assert np.array_equal(r["p"], p)             # the bias leaves p alone
    key = p.astype(np.float64) + b.astype(np.float64)
    for t in range(len(x)):
        best = max(itertools.combinations(range(E), k),
                   key=lambda S: (sum(key[t, e] for e in S), [-e for e in S]))
        assert set(r["idx"][t]) == set(best)
        sel = p[t, r["idx"][t]].astype(np.float64)
        np.testing.assert_allclose(r["w"][t], sel / sel.sum(), rtol=1e-6)
    # mean_prob is the mean of the unbiased p
    np.testing.assert_allclose(r["mean_prob"], p.astype(np.float64).mean(0), rtol=1e-12)


def test_selection_bias_large_bias_forces_expert():
    rng = np.random.default_rng(7)
    x = rng.normal(size=(25, 8)).astype(np.float32)
    wr = rng.normal(size=(5, 8)).astype(np.float32)
    b = np.array([0, 0, 0, 5.0, 0], dtype=np.float32)
    r = O.route(x, wr, b, 2, bias_mode=1)
    assert np.all(r["idx"][:, 0] == 3)           # selected first by the key ...
    assert np.all(r["w"][:, 0] < 1.0)             # ... but gated by its own p


def test_bias_update_hand_case():
    # E=4, N=4, k=2: mean load N*k/E = 2 picks per expert
    b = np.array([0.1, -0.2, 0.0, 0.5], dtype=np.float32)
    picks = np.array([5, 1, 2, 0])
    out = O.router_bias_update(b, picks, 4, 2, 0.01)
    expect = np.array([np.float32(0.1) - np.float32(0.01), np.float32(-0.2) + np.float32(0.01),
                       np.float32(0.0), np.float32(0.5) + np.float32(0.01)], dtype=np.float32)
    assert np.array_equal(out, expect)


def test_bias_update_balanced_is_identity_and_fractional_mean():
    b = np.array([0.3, -0.1, 0.2], dtype=np.float32)
    assert np.array_equal(O.router_bias_update(b, [2, 2, 2], 3, 2, 0.5), b)
    # N*k/E = 7/3: 2 picks is under, 3 picks is over
    out = O.router_bias_update(np.zeros(3, np.float32), [2, 3, 2], 7, 1, 0.25)
    assert list(out) == [0.25, -0.25, 0.25]
