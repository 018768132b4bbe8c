"""Pins for the expert activations and the expert FFN."""
import math

import numpy as np
import torch

import oracle


def test_gelu_erf_special_values_and_library():
    a = np.array([0.0, 1.0, -1.0, 3.0, -3.0, 0.5])
    g = oracle.gelu_erf(a)
    ref = [0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in a]
    np.testing.assert_allclose(g, ref, rtol=1e-15, atol=1e-300)
    assert g[0] == 0.0
    # Phi(1) = 0.841344746...: GELU(1) = Phi(1)
    assert abs(g[1] - 0.8413447460685429) < 1e-15
    t = torch.nn.functional.gelu(torch.tensor(a, dtype=torch.float64)).numpy()
    np.testing.assert_allclose(g, t, rtol=1e-14, atol=1e-300)


def test_silu_special_values_and_library():
    a = np.linspace(-6, 6, 41)
    s = oracle.silu(a)
    assert s[20] == 0.0
    np.testing.assert_allclose(s, torch.nn.functional.silu(torch.tensor(a)).numpy(), rtol=1e-14)
    # silu(a) - silu(-a) = a  (since sigmoid(a) + sigmoid(-a) = 1)
    np.testing.assert_allclose(s - oracle.silu(-a), a, atol=1e-14)


def test_swiglu_expert_against_torch_dense():
    rng = np.random.default_rng(0)
    d, F = 24, 40
    x = rng.standard_normal((7, d))
    w = {"w_gate": rng.standard_normal((F, d)).astype(np.float32),
         "w_up": rng.standard_normal((F, d)).astype(np.float32),
         "w_down": rng.standard_normal((d, F)).astype(np.float32)}
    y = oracle.expert_ffn(x, w, 1)
    X = torch.tensor(x)
    G = torch.nn.functional.linear(X, torch.tensor(w["w_gate"], dtype=torch.float64))
    U = torch.nn.functional.linear(X, torch.tensor(w["w_up"], dtype=torch.float64))
    ref = torch.nn.functional.linear(torch.nn.functional.silu(G) * U,
                                     torch.tensor(w["w_down"], dtype=torch.float64))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_gelu_expert_against_torch_sequential():
    rng = np.random.default_rng(1)
    d, F = 16, 32
    lin1 = torch.nn.Linear(d, F).double()
    lin2 = torch.nn.Linear(F, d).double()
    seq = torch.nn.Sequential(lin1, torch.nn.GELU(), lin2)
    x = rng.standard_normal((9, d))
    w = {"w_gate": lin1.weight.detach().numpy(), "b1": lin1.bias.detach().numpy(),
         "w_down": lin2.weight.detach().numpy(), "b2": lin2.bias.detach().numpy()}
    y = oracle.expert_ffn(x, w, 0)
    np.testing.assert_allclose(y, seq(torch.tensor(x)).detach().numpy(), rtol=1e-12, atol=1e-12)
