"""Whole-layer pins: special cases that reduce to a dense FFN, equivariance, linearity."""
import numpy as np
import torch

import oracle
import synth


def _small(name, **kw):
    return synth.small_workload(name, **kw)


def test_one_expert_top1_is_a_dense_ffn():
    w = _small("dsv2", n_tokens=33, d_model=64, n_experts=1, top_k=1, d_ff=96, n_shared=0)
    inp = synth.make_inputs(w)
    out = oracle.moe_forward(w, inp)
    x = torch.tensor(oracle.widen(inp["x"]))
    wg, wu, wd = (torch.tensor(oracle.widen(inp[k][0])) for k in ("w_gate", "w_up", "w_down"))
    ref = torch.nn.functional.silu(x @ wg.T) * (x @ wu.T) @ wd.T
    assert np.all(out["w"] == 1.0)
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_gelu_one_expert_is_a_dense_ffn_with_biases():
    w = _small("tiny_fp32", n_tokens=20, n_experts=1, top_k=1)
    inp = synth.make_inputs(w)
    out = oracle.moe_forward(w, inp)
    seq = torch.nn.Sequential(torch.nn.Linear(128, 256), torch.nn.GELU(), torch.nn.Linear(256, 128)).double()
    with torch.no_grad():
        seq[0].weight.copy_(torch.tensor(inp["w_gate"][0]))
        seq[0].bias.copy_(torch.tensor(inp["b1"][0]))
        seq[2].weight.copy_(torch.tensor(inp["w_down"][0]))
        seq[2].bias.copy_(torch.tensor(inp["b2"][0]))
        ref = seq(torch.tensor(oracle.widen(inp["x"]))).numpy()
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_shared_only_is_a_dense_ffn():
    w = _small("dsv2", n_tokens=17, d_model=32, n_experts=4, top_k=2, d_ff=48, n_shared=1)
    inp = synth.make_inputs(w)
    for key in ("w_gate", "w_up", "w_down"):
        inp[key][:4] = 0                      # routed experts output exactly zero
    out = oracle.moe_forward(w, inp)
    x = torch.tensor(oracle.widen(inp["x"]))
    wg, wu, wd = (torch.tensor(oracle.widen(inp[k][4])) for k in ("w_gate", "w_up", "w_down"))
    ref = torch.nn.functional.silu(x @ wg.T) * (x @ wu.T) @ wd.T
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_token_permutation_equivariance_without_capacity():
    w = _small("dsv2", n_tokens=40, d_model=32, n_experts=8, top_k=3, d_ff=32, n_shared=1)
    inp = synth.make_inputs(w)
    out = oracle.moe_forward(w, inp)
    perm = np.random.default_rng(0).permutation(40)
    inp2 = dict(inp, x=inp["x"][perm])
    out2 = oracle.moe_forward(w, inp2)
    assert np.array_equal(out2["idx"], out["idx"][perm])
    np.testing.assert_allclose(out2["y"], out["y"][perm], rtol=1e-12, atol=1e-12)


def test_linear_in_routed_expert_output():
    w = _small("dsv2", n_tokens=30, d_model=32, n_experts=4, top_k=2, d_ff=32, n_shared=1)
    inp = synth.make_inputs(w)
    base = oracle.moe_forward(w, inp)
    wd = oracle.widen(inp["w_down"])
    wd2 = wd.copy()
    wd2[:4] *= 2.0                             # doubles every routed expert's output
    inp2 = dict(inp, w_down=wd2.astype(np.float32))
    inp1 = dict(inp, w_down=wd.astype(np.float32))
    y1 = oracle.moe_forward(w, inp1)["y"]
    y2 = oracle.moe_forward(w, inp2)["y"]
    wd0 = wd.copy()
    wd0[:4] = 0
    y0 = oracle.moe_forward(w, dict(inp, w_down=wd0.astype(np.float32)))["y"]   # shared only
    np.testing.assert_allclose(y2 - y0, 2 * (y1 - y0), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(y1, base["y"], rtol=1e-12, atol=1e-12)


def test_dropped_slot_contributes_nothing():
    w = _small("mixtral_prefill", n_tokens=64, d_model=32, n_experts=4, top_k=2, d_ff=32)
    inp = synth.make_inputs(w)
    out = oracle.moe_forward(w.replace(alpha=0.25), inp)
    assert (out["final"] < 0).any()
    # recompute by hand from the routed rows
    for t in range(8):
        y = 0.0
        for j in range(2):
            e = out["final"][t, j]
            if e >= 0:
                wts = {k: inp[k][e] for k in ("w_gate", "w_up", "w_down")}
                y = y + float(out["w"][t, j]) * oracle.expert_ffn(oracle.widen(inp["x"][t:t + 1]), wts, 1)[0]
        np.testing.assert_allclose(out["y"][t], y if not np.isscalar(y) else np.zeros(32), atol=1e-12)



def _dense_mixture(w, inp, bias_in_weights, roll=0):
    """y = sum_e p_e(x) FFN_e(x) + shared FFN(x), every expert evaluated densely
    with torch, p from scipy's softmax of the router logits (float64).  Returns y
    and the elementwise bound sum_e |FFN_e(x)| that gate errors are scaled by.
    roll != 0 pairs expert e with the gate of expert e + roll (a planted mistake)."""
    from scipy.special import softmax
    x = torch.tensor(oracle.widen(inp["x"]))
    z = (x @ torch.tensor(oracle.widen(inp["w_router"])).T).numpy()
    if bias_in_weights and inp["router_bias"] is not None:
        z = z + np.asarray(inp["router_bias"], dtype=np.float64)
    p = np.roll(softmax(z, axis=1), -roll, axis=1)
    y = np.zeros((w.n_tokens, w.d_model))
    scale = np.zeros_like(y)
    for e in range(w.n_experts + w.n_shared):
        wg, wu, wd = (torch.tensor(oracle.widen(inp[k][e])) for k in ("w_gate", "w_up", "w_down"))
        f = (torch.nn.functional.silu(x @ wg.T) * (x @ wu.T) @ wd.T).numpy()
        y += f * (p[:, e:e + 1] if e < w.n_experts else 1.0)
        scale += np.abs(f)
    return y, scale


def _check_mixture(w, inp, bias_in_weights):
    out = oracle.moe_forward(w, inp)
    ref, scale = _dense_mixture(w, inp, bias_in_weights)
    # the oracle's probabilities are float32 (the pages' fp32 softmax): a few
    # ulps of each gate, times the expert outputs they scale
    tol = 1e-6 * scale
    assert np.all(np.abs(out["y"] - ref) <= tol)
    wrong, _ = _dense_mixture(w, inp, bias_in_weights, roll=1)
    assert np.mean(np.abs(out["y"] - wrong) > tol) > 0.9     # the pin tells them apart


def test_all_experts_firing_is_the_probability_weighted_mixture():
    # k = E and no capacity: every expert fires and the renormalised gates are
    # the softmax probabilities themselves, distinct per expert, so a gate
    # paired with the wrong expert's output (or a lost bias) changes y
    w = _small("dsv2", n_tokens=25, d_model=32, n_experts=6, top_k=6, d_ff=40, n_shared=1,
               cap_mode=synth.CAP_NONE)
    inp = synth.make_inputs(w)
    assert inp["router_bias"] is not None and np.ptp(inp["router_bias"]) > 0
    _check_mixture(w, inp, bias_in_weights=True)


def test_selection_bias_with_all_experts_firing_leaves_the_weights_unbiased():
    # selection-only bias: with k = E the selection is everything, and the
    # gates are the unbiased softmax probabilities
    w = _small("dsv2_select", n_tokens=25, d_model=32, n_experts=6, top_k=6, d_ff=40,
               n_shared=1, cap_mode=synth.CAP_NONE)
    inp = synth.make_inputs(w)
    assert w.bias_mode == 1 and np.ptp(inp["router_bias"]) > 0
    _check_mixture(w, inp, bias_in_weights=False)
    # and the biased softmax would not pass
    out = oracle.moe_forward(w, inp)
    biased, scale = _dense_mixture(w, inp, bias_in_weights=True)
    assert np.mean(np.abs(out["y"] - biased) > 1e-6 * scale) > 0.9
