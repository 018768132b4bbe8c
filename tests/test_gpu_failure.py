"""Failure detection without a GPU fault: a bounded device wait that runs out
(on an mbarrier that nothing arrives on, or at a grid barrier one CTA never
reaches) records MOE_ERR_TIMEOUT in the workspace status word; the host reads
and clears it, and the context stays usable for the layer afterwards."""
import time

import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import oracle
import synth
from helpers import config_of, rel_err_inf, to_dev, to_f64

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_context_survives(cuda):
    w = synth.small_workload("mixtral_prefill", n_tokens=300, d_model=128, n_experts=4, d_ff=256)
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    t0 = time.perf_counter()
    moe.moe_selftest_timeout(ws, 20000)                 # 20 ms
    st = moe.moe_device_status(ws)                      # synchronises
    dt = time.perf_counter() - t0
    assert st == moe.MOE_ERR_TIMEOUT
    assert 0.015 < dt < 10.0
    assert moe.moe_device_status(ws) == moe.MOE_OK      # reading cleared it
    # the same workspace and context run the layer afterwards
    inp = synth.make_inputs(w)
    y = torch.zeros((w.n_tokens, w.d_model), dtype=torch.bfloat16, device=cuda)
    moe.moe_forward(cfg, to_dev(inp["x"]), to_dev(inp["w_router"]), to_dev(inp["router_bias"]),
                    to_dev(inp["w_gate"]), to_dev(inp["w_up"]), to_dev(inp["w_down"]), None, None,
                    y, None, ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    o = oracle.moe_forward(w, inp)
    assert rel_err_inf(to_f64(y), o["y"]) <= 2e-2


def test_selftest_argument_checks(cuda):
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda)
    for bad in (0, 2_000_000):
        with pytest.raises(moe.MoeError):
            moe.moe_selftest_timeout(ws, bad)


def test_grid_barrier_timeout_costs_one_limit(cuda):
    """CTA 0 of a cooperative grid never reaches the barrier; the others run a
    chain of 64 barriers with a 50 ms limit.  Without the abort flag that would
    take 64 limits (3.2 s); with it the grid leaves after about one."""
    w = synth.small_workload("e64_reroute", n_tokens=1500, d_model=128, n_experts=16, d_ff=128,
                             alpha=0.8)
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    t0 = time.perf_counter()
    moe.moe_selftest_barrier_timeout(ws, 50000, 64)      # 50 ms, 64 barriers
    st = moe.moe_device_status(ws)                       # synchronises
    dt = time.perf_counter() - t0
    assert st == moe.MOE_ERR_TIMEOUT
    assert 0.045 < dt < 1.0
    assert moe.moe_device_status(ws) == moe.MOE_OK
    # the cooperative reroute kernel then runs normally on the same workspace
    inp = synth.make_inputs(w)
    y = torch.zeros((w.n_tokens, w.d_model), dtype=torch.bfloat16, device=cuda)
    moe.moe_forward(cfg, to_dev(inp["x"]), to_dev(inp["w_router"]), to_dev(inp["router_bias"]),
                    to_dev(inp["w_gate"]), to_dev(inp["w_up"]), to_dev(inp["w_down"]), None, None,
                    y, None, ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    o = oracle.moe_forward(w, inp)
    assert o["n_rerouted"] > 0
    assert rel_err_inf(to_f64(y), o["y"]) <= 2e-2


def test_barrier_selftest_argument_checks(cuda):
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda)
    for lim, nb in ((0, 4), (2_000_000, 4), (1000, 0), (1000, 5000)):
        with pytest.raises(moe.MoeError):
            moe.moe_selftest_barrier_timeout(ws, lim, nb)
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_barrier_timeout(ws[:16], 1000, 1)
