"""Guard bands around every output buffer, in place of a memory sanitizer: each
output (and the workspace) is a window of a larger byte buffer whose margins
hold a fixed pattern; after the four stage calls and the whole forward, every
margin must be unchanged.  The shapes are odd on purpose (N not a multiple of
128, d and F not multiples of 64, ragged expert segments, shared experts,
empty experts, the largest top-k), so tails and limits are exercised."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import synth
from helpers import config_of, to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """Byte buffers with guard margins; .new() hands out typed windows."""

    def __init__(self, device):
        self.device = device
        self.bufs = []

    def new(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        buf = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=self.device)
        self.bufs.append((buf, n))
        return buf[GUARD:GUARD + n].view(dtype).view(*shape)

    def check(self):
        for i, (buf, n) in enumerate(self.bufs):
            head, tail = buf[:GUARD], buf[GUARD + n:]
            assert torch.all(head == PATTERN), f"buffer {i}: bytes before the window written"
            assert torch.all(tail == PATTERN), f"buffer {i}: bytes after the window written"


def stats_of(g, E):
    f32, i32 = torch.float32, torch.int32
    return moe.make_stats(expert_freq=g.new((E,), f32), mean_prob=g.new((E,), f32),
                          l_bal=g.new((1,), f32), counts=g.new((E,), i32),
                          n_dropped=g.new((1,), i32), n_rerouted=g.new((1,), i32),
                          z_loss=g.new((1,), f32), router_entropy=g.new((1,), f32))


CASES = [
    synth.small_workload("mixtral_prefill", n_tokens=333, d_model=80, n_experts=5, top_k=3,
                         d_ff=96, alpha=0.7),
    synth.small_workload("e64_reroute", n_tokens=257, d_model=64, n_experts=16, d_ff=80,
                         alpha=0.8),
    synth.small_workload("dsv2", n_tokens=129, d_model=64, n_experts=37, top_k=6, d_ff=48,
                         n_shared=2),
    synth.small_workload("dsv2", n_tokens=5, d_model=64, n_experts=160, top_k=8, d_ff=64,
                         n_shared=2),
    synth.small_workload("tiny_fp32", n_tokens=77, n_experts=3, top_k=3),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.name}-N{w.n_tokens}-E{w.n_experts}")
def test_no_write_outside_outputs(cuda, w):
    cfg = config_of(w)
    inp = synth.make_inputs(w)
    N, d, E, k, S = w.n_tokens, w.d_model, w.n_experts, w.top_k, w.n_shared
    dt = torch.bfloat16 if w.dtype == synth.DT_BF16 else torch.float32
    g = Guarded(cuda)
    ws = g.new((moe.moe_workspace_size(cfg),), torch.uint8)
    ws.zero_()
    x, wr, rb = to_dev(inp["x"]), to_dev(inp["w_router"]), to_dev(inp["router_bias"])
    wg, wu, wd = to_dev(inp["w_gate"]), to_dev(inp["w_up"]), to_dev(inp["w_down"])
    b1, b2 = to_dev(inp["b1"]), to_dev(inp["b2"])
    i32, f32 = torch.int32, torch.float32
    max_rows, max_total = moe.moe_max_rows(cfg), moe.moe_max_total_rows(cfg)

    # the four stages
    topk_idx, topk_w = g.new((N, k), i32), g.new((N, k), f32)
    probs = g.new((N, E), f32)
    st = stats_of(g, E)
    moe.moe_route(cfg, x, wr, rb, topk_idx, topk_w, probs, st, ws)
    final_idx, pos = g.new((N, k), i32), g.new((N, k), i32)
    offsets, perm = g.new((E + S + 1,), i32), g.new((max_rows,), i32)
    x_perm = g.new((max_rows, d), dt)
    counts = g.new((E,), i32)
    moe.moe_dispatch(cfg, topk_idx, probs, x, final_idx, pos, offsets, perm, x_perm,
                     moe.make_stats(counts=counts, n_dropped=g.new((1,), i32),
                                    n_rerouted=g.new((1,), i32)), ws)
    y_perm = g.new((max_total, d), dt)
    moe.moe_expert_ffn(cfg, x, x_perm, offsets, counts, wg, wu, wd, b1, b2, y_perm, ws)
    y = g.new((N, d), dt)
    moe.moe_combine(cfg, y_perm, offsets, final_idx, pos, topk_w, y)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    g.check()

    # the whole layer
    y2 = g.new((N, d), dt)
    moe.moe_forward(cfg, x, wr, rb, wg, wu, wd, b1, b2, y2, stats_of(g, E), ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    g.check()
    assert torch.isfinite(y2.float()).all()
    assert torch.equal(y2.view(torch.uint8), y.view(torch.uint8))   # stages == forward
