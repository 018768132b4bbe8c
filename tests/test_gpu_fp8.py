"""FP8 (E4M3) expert weights: the CUDA quantiser's codes and scales bit-exact
with the oracle's, and the expert FFNs and the whole layer vs the oracle run
on the dequantised weights (scale * code value)."""
import numpy as np
import pytest
import torch

import mixture_experts_ffn_19_b300 as moe
import oracle
import synth
from helpers import (adopt_near_ties, config_of, elementwise_err, host_layout, rel_err_inf,
                     report, to_dev, to_f64, upload_experts)

pytestmark = pytest.mark.gpu

KEYS = ("w_gate", "w_up", "w_down")


def device_quantize(wt, device):
    """bf16 device tensor [n_mat, rows, cols] -> (codes uint8, scales fp32) on the device."""
    q = torch.empty(wt.shape, dtype=torch.uint8, device=device)
    s = torch.empty(wt.shape[0], dtype=torch.float32, device=device)
    moe.moe_quantize_fp8(wt, q, s)
    return q, s


def quantize_all(wdev, device):
    """Device codes [E+S, ...] per matrix kind and scales [3, E+S]."""
    qs, ss = {}, []
    for key in KEYS:
        q, s = device_quantize(wdev[key], device)
        qs[key] = q
        ss.append(s)
    return qs, torch.stack(ss).contiguous()


def oracle_expert(w_bits, e):
    """Oracle codes, scales and dequantised weights of expert e (bf16 bit arrays in)."""
    out, codes, scales = {"b1": None, "b2": None}, {}, {}
    for key in KEYS:
        c, s = oracle.quantize_fp8(w_bits[key])
        codes[key], scales[key] = c, s
        out[key] = oracle.dequantize_fp8(c, s)
    return out, codes, scales


def check_codes(qdev, sdev, e, codes, scales):
    for i, key in enumerate(KEYS):
        assert np.array_equal(qdev[key][e].cpu().numpy(), codes[key]), f"{key} codes, expert {e}"
        assert sdev[i, e].item() == scales[key], f"{key} scale, expert {e}"


def test_quantiser_special_values(cuda):
    # scale 1 (amax 448): exact midpoints between neighbouring codes, signs,
    # subnormals, zero; then an all-zero matrix (scale 1, all codes 0)
    finite = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (finite[:-1] + finite[1:]) / 2
    vals = np.concatenate([[448.0], finite, -finite, mids, -mids, [2.0 ** -12, -(2.0 ** -11)]])
    vals = vals[:len(vals) // 16 * 16].astype(np.float32)
    bits = synth.round_to_bf16_bits(vals)
    assert np.array_equal(oracle.widen(bits), vals.astype(np.float64))   # exact in bf16
    mats = np.stack([bits.reshape(-1, 16), np.zeros_like(bits).reshape(-1, 16)])
    q, s = device_quantize(to_dev(mats), cuda)
    for m in range(2):
        c, sc = oracle.quantize_fp8(mats[m])
        assert s[m].item() == sc
        assert np.array_equal(q[m].cpu().numpy(), c)


@pytest.mark.parametrize("shape", [(3, 48, 64), (1, 16, 16), (5, 200, 96)])
def test_quantiser_random(cuda, shape):
    rng = np.random.default_rng(sum(shape))
    a = rng.normal(size=shape).astype(np.float32) * np.float32(0.03)
    a[0, 0, :5] = [0.0, 1e-30, -1e-8, 3.0, -2.5]                 # tiny values and the max
    bits = synth.round_to_bf16_bits(a)
    q, s = device_quantize(to_dev(bits), cuda)
    for m in range(shape[0]):
        c, sc = oracle.quantize_fp8(bits[m])
        assert s[m].item() == sc
        assert np.array_equal(q[m].cpu().numpy(), c)


CASES = [
    synth.small_workload("decode_mixtral", d_model=512, d_ff=1024),
    synth.small_workload("decode_dsv2", d_model=256, d_ff=320),
    synth.small_workload("decode_dsv2", n_tokens=300, d_model=128, n_experts=64, top_k=2,
                         d_ff=144, n_shared=1),
    # many tokens per expert: several 64-token chunks per expert, K tail (d=208)
    synth.small_workload("mixtral_prefill", n_tokens=700, d_model=208, n_experts=4, top_k=2,
                         d_ff=256, alpha=0.0, cap_mode=synth.CAP_NONE),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.name}-N{w.n_tokens}-d{w.d_model}-E{w.n_experts}")
def test_expert_ffn_fp8(cuda, w):
    inp = synth.make_inputs(w)
    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], w.top_k, w.bias_mode)
    C = oracle.capacity(w.n_tokens, w.n_experts, w.top_k, w.alpha) if w.cap_mode else None
    dsp = oracle.dispatch(r["idx"], r["key"], w.n_experts, w.cap_mode, C)
    members = dsp["members"]
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    offsets = host_layout(w, members)
    R, RT = moe.moe_max_rows(cfg), moe.moe_max_total_rows(cfg)
    xp = np.zeros((R, w.d_model), dtype=inp["x"].dtype)
    for e, m in enumerate(members):
        xp[offsets[e]:offsets[e] + len(m)] = inp["x"][m]
    wdev = {key: to_dev(inp[key]) for key in KEYS}
    qd, sd = quantize_all(wdev, cuda)
    y = torch.zeros((RT, w.d_model), dtype=torch.bfloat16, device=cuda)
    counts = to_dev(np.array([len(m) for m in members], dtype=np.int32))
    moe.moe_expert_ffn_fp8(cfg, to_dev(inp["x"]), to_dev(xp), to_dev(offsets), counts,
                           qd["w_gate"], qd["w_up"], qd["w_down"], sd, y, ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    y = to_f64(y)
    x = oracle.widen(inp["x"])
    worst = 0.0
    ET = w.n_experts + w.n_shared
    for e in range(ET):
        rows = members[e] if e < w.n_experts else np.arange(w.n_tokens)
        if len(rows) == 0:
            continue
        deq, codes, scales = oracle_expert({k: inp[k][e] for k in KEYS}, e)
        check_codes(qd, sd, e, codes, scales)
        ref = oracle.expert_ffn(x[rows], deq, w.act)
        got = y[offsets[e]:offsets[e] + len(rows)]
        err = rel_err_inf(got, ref)
        worst = max(worst, err)
        assert err <= 2e-2, f"expert {e}: rel err {err:.3g}"
    print(f"{w.name}: worst per-expert rel err {worst:.3g}")


def run_forward_fp8(w, inp, wdev, cuda):
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    qd, sd = quantize_all(wdev, cuda)
    xd = to_dev(inp["x"])
    y = torch.zeros((w.n_tokens, w.d_model), dtype=torch.bfloat16, device=cuda)
    moe.moe_forward_fp8(cfg, xd, to_dev(inp["w_router"]), to_dev(inp["router_bias"]),
                        qd["w_gate"], qd["w_up"], qd["w_down"], sd, y, None, ws)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    v = moe.moe_workspace_views(cfg, ws)
    nk = w.n_tokens * w.top_k
    off = (v.final_idx - ws.data_ptr()) // 4
    final = ws.view(torch.int32)[off:off + nk].cpu().numpy()
    off = (v.topk_idx - ws.data_ptr()) // 4
    idx = ws.view(torch.int32)[off:off + nk].cpu().numpy()
    return y, qd, sd, final.reshape(w.n_tokens, w.top_k), idx.reshape(w.n_tokens, w.top_k)


@pytest.mark.parametrize("w", [
    synth.small_workload("decode_mixtral", d_model=512, d_ff=1024),
    synth.small_workload("dsv2", n_tokens=300, d_model=256, n_experts=16, top_k=4, d_ff=256),
    synth.WORKLOADS["decode_mixtral"],
    synth.WORKLOADS["decode_dsv2"],
], ids=lambda w: w.name)
def test_forward_fp8(cuda, w):
    """Whole layer, every output row (the decode batches are small enough)."""
    inp = synth.make_inputs(w, with_experts=False)
    wdev = upload_experts(w, cuda)
    y, qd, sd, final, idx_dev = run_forward_fp8(w, inp, wdev, cuda)
    toks = np.arange(w.n_tokens)                 # every token, full-size decode batches too
    cache = {}

    def get_expert(e):
        if e not in cache:
            _, codes, scales = oracle_expert(synth.expert_weights(w, e), e)
            check_codes(qd, sd, e, codes, scales)
            # the oracle reads the E4M3 codes and scales themselves
            cache[e] = {key: (codes[key], scales[key]) for key in KEYS}
        return cache[e]

    r = oracle.route(inp["x"], inp["w_router"], inp["router_bias"], w.top_k, w.bias_mode)
    adopted, flips = adopt_near_ties(r, idx_dev)
    o = oracle.moe_forward(w, inp, tokens=toks, get_expert=get_expert,
                           idx_given=adopted if len(flips) else None)
    np.testing.assert_array_equal(final, o["final"])
    got = to_f64(y)[toks]
    err = rel_err_inf(got, o["y"])
    report(f"fp8 forward {w.name}", tokens=len(toks), rel_err_inf=err,
           elementwise_err=elementwise_err(got, o["y"]), flipped=len(flips),
           experts_checked=len(cache))
    print(f"{w.name}: y rel err {err:.3g} over {len(toks)} tokens, {len(cache)} experts checked")
    assert err <= 2e-2


def test_fp8_rejects_unsupported(cuda):
    w = synth.small_workload("tiny_fp32")
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    b = torch.zeros(16, dtype=torch.uint8, device=cuda)
    s = torch.ones(3 * 8, device=cuda)
    x = torch.zeros((w.n_tokens, w.d_model), device=cuda)
    with pytest.raises(moe.MoeError):       # fp32 layer
        moe.moe_forward_fp8(cfg, x, x, None, b, b, b, s, x, None, ws)
    w2 = synth.small_workload("decode_mixtral", d_model=520, d_ff=1024)   # d not a multiple of 16
    cfg2 = config_of(w2)
    ws2 = moe.alloc_workspace(cfg2, cuda)
    xb = torch.zeros((w2.n_tokens, 520), dtype=torch.bfloat16, device=cuda)
    with pytest.raises(moe.MoeError):
        moe.moe_forward_fp8(cfg2, xb, xb, None, b, b, b, s, xb, None, ws2)
    with pytest.raises(moe.MoeError):       # rows * cols not a multiple of 16
        moe.moe_quantize_fp8(torch.zeros((1, 3, 5), dtype=torch.bfloat16, device=cuda),
                             torch.zeros((1, 3, 5), dtype=torch.uint8, device=cuda),
                             torch.zeros(1, device=cuda))


def test_fp8_activation_past_f16_range_is_reported(cuda):
    """The E4M3 path multiplies f16 copies of the token rows: a finite value
    past 65504 has no f16 form, so it sets the device status; the next call on
    the same workspace starts clean."""
    w = synth.small_workload("decode_mixtral", d_model=512, d_ff=1024)
    inp = synth.make_inputs(w, with_experts=False)
    wdev = upload_experts(w, cuda)
    cfg = config_of(w)
    ws = moe.alloc_workspace(cfg, cuda)
    qd, sd = quantize_all(wdev, cuda)
    xd = to_dev(inp["x"])
    y = torch.zeros((w.n_tokens, w.d_model), dtype=torch.bfloat16, device=cuda)
    rest = (to_dev(inp["w_router"]), to_dev(inp["router_bias"]), qd["w_gate"], qd["w_up"],
            qd["w_down"], sd, y, None, ws)
    moe.moe_forward_fp8(cfg, xd, *rest)
    assert moe.moe_device_status(ws) == moe.MOE_OK
    big = xd.clone()
    big[3, 7] = 1.0e5
    moe.moe_forward_fp8(cfg, big, *rest)
    assert moe.moe_device_status(ws) == moe.MOE_ERR_DEVICE
    moe.moe_forward_fp8(cfg, xd, *rest)
    assert moe.moe_device_status(ws) == moe.MOE_OK
