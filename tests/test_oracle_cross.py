"""The C++ oracle against an independent float64 NumPy restatement of the same
steps (``oracle/numpy_oracle.py``: library matmul, argsort and erf as steps).

The two were written separately from the pages, so a slip in either (a dropped
term, a wrong index, a reroute rule taken in another order) shows up as a
disagreement.  Routing decisions must agree exactly wherever the float32
probabilities agree; the outputs agree to float64 rounding.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import numpy_oracle as NP

CASES = [
    synth.small_workload("tiny_fp32", n_tokens=96),
    synth.small_workload("mixtral_prefill", n_tokens=150, d_model=48, n_experts=6, d_ff=40,
                         alpha=0.6),
    synth.small_workload("dsv2", n_tokens=80, d_model=40, n_experts=12, top_k=4, d_ff=24,
                         n_shared=2),
    synth.small_workload("e64_reroute", n_tokens=300, d_model=32, n_experts=16, d_ff=24,
                         alpha=0.7),
    synth.small_workload("dsv2_select", n_tokens=90, d_model=32, n_experts=10, top_k=3, d_ff=24,
                         n_shared=1, cap_mode=synth.CAP_REROUTE, alpha=0.9),
    synth.small_workload("decode_dsv2", d_model=64, d_ff=32),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_layer_agrees_with_numpy_restatement(w):
    inp = synth.make_inputs(w)
    a = oracle.moe_forward(w, inp)
    b = NP.moe_forward(w, inp)
    # probabilities: the logits' sums run in another order, so a float32 rounding
    # may differ by one ulp
    assert np.max(np.abs(a["p"].astype(np.float64) - b["p"]) / b["p"]) <= 2 ** -23
    same_p = np.all(a["p"] == b["p"], axis=1)
    assert same_p.mean() > 0.9
    for key in ("idx", "w", "final"):
        assert np.array_equal(a[key][same_p], b[key][same_p]), key
    if same_p.all():
        assert np.array_equal(a["counts"], b["counts"])
        assert (a["n_dropped"], a["n_rerouted"]) == (b["n_dropped"], b["n_rerouted"])
        for ma, mb in zip(a["members"], b["members"]):
            assert np.array_equal(ma, mb)
        np.testing.assert_allclose(a["y"], b["y"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(a["mean_prob"], b["mean_prob"], rtol=1e-6)
    assert a["l_bal"] == pytest.approx(b["l_bal"], rel=1e-6)
    assert a["z_loss"] == pytest.approx(b["z_loss"], rel=1e-12)
    assert a["router_entropy"] == pytest.approx(b["router_entropy"], rel=1e-6)


@pytest.mark.parametrize("seed,N,E,k,C", [(0, 40, 6, 2, 5), (1, 64, 8, 3, 9), (2, 16, 4, 2, 3),
                                          (3, 120, 12, 4, 11), (4, 33, 5, 1, 2)])
def test_reroute_agrees_with_numpy_restatement(seed, N, E, k, C):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((N, E)) - 1.1 * np.log(rng.permutation(E) + 1.0)
    p = oracle.softmax_fp32(z)
    idx = oracle.topk_select(p, k)
    got = oracle.apply_capacity_reroute(idx, p, E, C)
    ref = NP.apply_capacity_reroute(idx, p, E, C)
    assert np.array_equal(got[0], ref[0])
    assert all(np.array_equal(x, y) for x, y in zip(got[1], ref[1]))
    assert got[2:] == ref[2:]


def test_fp8_codec_agrees_with_numpy_restatement():
    rng = np.random.default_rng(21)
    v = np.concatenate([rng.normal(size=5000).astype(np.float32) * np.float32(100.0),
                        rng.uniform(-0.02, 0.02, size=2000).astype(np.float32)])
    assert np.array_equal(oracle.e4m3_encode(v), NP.e4m3_encode(v))
    w = synth.round_to_bf16_bits(rng.normal(size=(37, 48)).astype(np.float32) * np.float32(0.05))
    qa, sa = oracle.quantize_fp8(w)
    qb, sb = NP.quantize_fp8(w)
    assert sa == sb and np.array_equal(qa, qb)
