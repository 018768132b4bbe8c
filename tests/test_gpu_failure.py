"""Failure detection without a GPU fault: a bounded device wait that runs out
(on an mbarrier that nothing arrives on) records MOE_ERR_TIMEOUT in the
workspace status word; the host reads and clears it, and the context stays
usable for the layer afterwards."""
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
