"""Pins for the load-balance statistics ([P3] §2.2 form)."""
import json
import os

import numpy as np

import oracle


def test_uniform_routing_gives_exactly_one():
    # zero router -> p = 1/E exactly; ties -> experts 0..k-1 for every token
    for E, N, k in ((8, 256, 2), (64, 128, 2), (4, 100, 4)):
        x = np.random.default_rng(E).standard_normal((N, 16)).astype(np.float32)
        r = oracle.route(x, np.zeros((E, 16), np.float32), None, k)
        assert r["l_bal"] == 1.0
        assert np.all(r["mean_prob"] == 1.0 / E)


def test_uniform_mean_prob_gives_one_for_any_selection():
    E, N, k = 8, 64, 2
    p = np.full((N, E), 1.0 / E, dtype=np.float32)
    idx = np.random.default_rng(0).integers(0, E, (N, k)).astype(np.int32)
    _, _, l = oracle.balance_stats(p, idx, E)
    assert abs(l - 1.0) < 1e-15


def test_hand_cases(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "router_hand_cases.json")))
    for case in g["balance"]:
        p = np.array(case["p"], dtype=np.float32)
        idx = oracle.topk_select(p, case["k"])
        f, m, l = oracle.balance_stats(p, idx, p.shape[1])
        assert f.tolist() == case["freq"]
        np.testing.assert_allclose(m, case["mean_prob"], rtol=1e-7)
        assert abs(l - case["l_bal"]) < 1e-7


def test_freq_counts_picks_over_N_times_k():
    rng = np.random.default_rng(9)
    E, N, k = 10, 300, 3
    p = oracle.softmax_fp32(rng.standard_normal((N, E)))
    idx = oracle.topk_select(p, k)
    f, _, _ = oracle.balance_stats(p, idx, E)
    assert abs(f.sum() - 1.0) < 1e-12
    for e in range(E):
        assert round(f[e] * N * k) == sum(1 for t in range(N) for j in range(k) if idx[t, j] == e)
