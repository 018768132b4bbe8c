"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device
memory, checked through the C ABI against moe_dispatch on the same inputs, two
calls in a row (the fixed scratch array keeps the previous call's contents)."""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import oracle
import synth
from helpers import config_of, to_dev

pytestmark = pytest.mark.gpu

_P = ctypes.c_void_p


def _noalloc():
    f = moe.lib().moe_dispatch_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(moe.moe_config), _P, _P, _P, _P, _P, _P, _P, _P,
                  ctypes.POINTER(moe.moe_stats), _P, _P]
    return f


def _outputs(w, cfg, x, device):
    N, k, E, S = w.n_tokens, w.top_k, w.n_experts, w.n_shared
    R = moe.moe_max_rows(cfg)
    return dict(final=torch.full((N, k), -9, dtype=torch.int32, device=device),
                pos=torch.full((N, k), -9, dtype=torch.int32, device=device),
                offsets=torch.full((E + S + 1,), -9, dtype=torch.int32, device=device),
                perm=torch.full((R,), -9, dtype=torch.int32, device=device),
                x_perm=torch.zeros((R, w.d_model), dtype=x.dtype, device=device),
                counts=torch.full((E,), -9, dtype=torch.int32, device=device),
                nd=torch.full((1,), -9, dtype=torch.int32, device=device),
                nr=torch.full((1,), -9, dtype=torch.int32, device=device))


def _stats(o):
    return moe.make_stats(counts=o["counts"], n_dropped=o["nd"], n_rerouted=o["nr"])


def _compare(a, b):
    for key in ("final", "pos", "offsets", "counts", "nd", "nr"):
        assert torch.equal(a[key], b[key]), key
    kept = a["pos"][a["pos"] >= 0].long()
    assert torch.equal(a["perm"][kept], b["perm"][kept])
    assert torch.equal(a["x_perm"][kept].view(torch.int16), b["x_perm"][kept].view(torch.int16))


CASES = [
    synth.small_workload("e64_reroute", n_tokens=2000, d_model=64, alpha=1.0),
    synth.small_workload("mixtral_prefill", n_tokens=700, d_model=64, alpha=0.6),
    synth.small_workload("dsv2", n_tokens=333, d_model=64, n_experts=160, top_k=6, n_shared=2),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_dispatch_matches_workspace_dispatch(cuda, w):
    f = _noalloc()
    cfg = config_of(w)
    inp = synth.make_inputs(w, with_experts=False)
    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], w.top_k)
    idx = to_dev(r["idx"].astype(np.int32))
    probs = to_dev(r["p"].astype(np.float32))
    x = to_dev(inp["x"])
    ws = moe.alloc_workspace(cfg, cuda)
    ref = _outputs(w, cfg, x, cuda)
    moe.moe_dispatch(cfg, idx, probs, x, ref["final"], ref["pos"], ref["offsets"], ref["perm"],
                     ref["x_perm"], _stats(ref), ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):                       # two calls in a row share the scratch array
        got = _outputs(w, cfg, x, cuda)
        status = torch.full((1,), -1, dtype=torch.int32, device=cuda)
        st = f(ctypes.byref(cfg), idx.data_ptr(), probs.data_ptr(), x.data_ptr(),
               got["final"].data_ptr(), got["pos"].data_ptr(), got["offsets"].data_ptr(),
               got["perm"].data_ptr(), got["x_perm"].data_ptr(), ctypes.byref(_stats(got)),
               status.data_ptr(), stream)
        assert st == moe.MOE_OK
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        _compare(got, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda):
    f = _noalloc()
    cfg = moe.make_config(1 << 20, 64, 256, 8, 64, cap_mode=moe.MOE_CAP_REROUTE, alpha=1.0)
    st = f(ctypes.byref(cfg), 16, 16, 16, 16, 16, 16, 16, 16, None, 16,
           torch.cuda.current_stream().cuda_stream)
    assert st == moe.MOE_ERR_WORKSPACE
    # a null device_status is refused: device-side failures would go unreported
    small = moe.make_config(64, 64, 8, 2, 64)
    st = f(ctypes.byref(small), 16, 16, 16, 16, 16, 16, 16, 16, None, None,
           torch.cuda.current_stream().cuda_stream)
    assert st == moe.MOE_ERR_INVALID_ARG
