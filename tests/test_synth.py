"""The input generator is deterministic and has the stated laws."""
import numpy as np

import oracle
import synth


def test_deterministic_and_independent_streams():
    w = synth.small_workload("dsv2", n_tokens=64, d_model=64, n_experts=8, d_ff=32, n_shared=2)
    a = synth.make_inputs(w)
    b = synth.make_inputs(w, threads=1)
    for k in a:
        if a[k] is None:
            assert b[k] is None
        else:
            assert np.array_equal(a[k], b[k])
    e = synth.expert_weights(w, 9)
    assert np.array_equal(e["w_gate"], a["w_gate"][9])
    assert not np.array_equal(a["w_gate"][0], a["w_up"][0])


def test_distribution_laws():
    w = synth.small_workload("mixtral_prefill", n_tokens=512, d_model=256, n_experts=4, d_ff=128)
    a = synth.make_inputs(w)
    x = oracle.widen(a["x"])
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    wg = oracle.widen(a["w_gate"])
    assert abs(wg.std() * np.sqrt(256) - 1) < 0.02
    wd = oracle.widen(a["w_down"])
    assert abs(wd.std() * np.sqrt(128) - 1) < 0.02


def test_bias_laws():
    u = synth.router_bias(synth.WORKLOADS["dsv2"])
    assert u.shape == (160,) and u.min() >= -0.1 and u.max() <= 0.1
    z = synth.router_bias(synth.WORKLOADS["e64_reroute"])
    assert z.max() == 0.0
    assert np.allclose(np.sort(z)[::-1], -1.1 * np.log(np.arange(1, 65)), atol=1e-6)


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9], dtype=np.float32)
    bits = synth.round_to_bf16_bits(f)
    assert oracle.widen(bits).tolist() == [1.0, 1.0, 1.0 + 2 ** -6 * 1.0, 1.0]
