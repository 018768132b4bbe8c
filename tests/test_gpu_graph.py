"""The layer inside a CUDA graph: moe_forward (bf16 and E4M3 weights, with the
cooperative reroute) enqueues only stream-ordered work, so a captured forward
replays to the bit-identical output of an eager call."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import synth
from helpers import config_of, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [
    synth.small_workload("e64_reroute", n_tokens=1024, d_model=256, d_ff=256, alpha=0.8),
    synth.small_workload("decode_mixtral", d_model=512, d_ff=1024),
    synth.small_workload("dsv2_select", n_tokens=300, d_model=256, n_experts=32, top_k=4, d_ff=256),
], ids=lambda w: w.name)
@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_forward_replays_in_cuda_graph(cuda, w, fp8):
    inp = synth.make_inputs(w)
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    x = to_dev(inp["x"])
    wr, rb = to_dev(inp["w_router"]), to_dev(inp["router_bias"])
    wts = [to_dev(inp[k]) for k in ("w_gate", "w_up", "w_down")]
    if fp8:
        q, sc = [], []
        for t in wts:
            qq = torch.empty(t.shape, dtype=torch.uint8, device=cuda)
            ss = torch.empty(t.shape[0], dtype=torch.float32, device=cuda)
            moe.moe_quantize_fp8(t, qq, ss)
            q.append(qq)
            sc.append(ss)
        scales = torch.stack(sc).contiguous()
    lb = torch.zeros(1, device=cuda)
    st = moe.make_stats(l_bal=lb)

    def fwd(y, stream):
        if fp8:
            moe.moe_forward_fp8(cfg, x, wr, rb, q[0], q[1], q[2], scales, y, st, ws, stream)
        else:
            moe.moe_forward(cfg, x, wr, rb, wts[0], wts[1], wts[2], None, None, y, st, ws, stream)

    y_eager = torch.empty((w.n_tokens, w.d_model), dtype=x.dtype, device=cuda)
    fwd(y_eager, None)
    torch.cuda.synchronize()
    assert moe.moe_device_status(ws) == moe.MOE_OK

    y_graph = torch.zeros_like(y_eager)
    side = torch.cuda.Stream(cuda)
    side.wait_stream(torch.cuda.current_stream(cuda))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fwd(y_graph, side)
    for _ in range(3):
        y_graph.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert moe.moe_device_status(ws) == moe.MOE_OK
    assert torch.equal(y_graph.view(torch.int16), y_eager.view(torch.int16))
