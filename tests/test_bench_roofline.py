"""The roofline numerator bench.py reports: algorithmic FLOPs and bytes of the
gate/up GEMM, against values worked out by hand for the benchmark shapes, and
the rule that names the kernel those figures belong to."""
import numpy as np

import bench
import synth


def test_mixtral_prefill_flops():
    w = synth.WORKLOADS["mixtral_prefill"]
    work = bench.layer_work(w, counts_kept=8192, n_dropped=0)
    # every kept row: x (4096) against 2 x 14336 gate/up rows, 2 FLOP per MAC
    assert work["gemm1_flop"] == 2 * 8192 * 4096 * 2 * 14336 == 1_924_145_348_608
    assert work["gemm2_flop"] == work["gemm1_flop"] / 2
    assert work["router_flop"] == 2 * 4096 * 4096 * 8
    assert work["rows"] == 8192


def test_shared_rows_count_once_per_token():
    w = synth.WORKLOADS["dsv2"]                    # 2 shared experts
    work = bench.layer_work(w, counts_kept=100, n_dropped=0)
    assert work["rows"] == 100 + 2 * w.n_tokens


def test_gemm1_bytes_decode_fp8():
    w = synth.WORKLOADS["decode_mixtral_fp8"]      # 64 tokens, every expert touched
    counts = np.full(8, 16)
    got = bench.gemm1_bytes(w, counts, rows=128)
    weights = 8 * 2 * 14336 * 4096                 # one byte per E4M3 code
    assert got == weights + 128 * 4096 * 2 + 128 * 14336 * 2
    # the recorded DRAM traffic of that launch is within 1 % of it
    rec = bench.measured_traffic("ffn_tc_swap_kernel<0,fp8>", "decode_mixtral_fp8")
    if rec is not None:
        assert abs(rec / got - 1) < 0.01


def test_gemm1_bytes_skip_untouched_experts():
    w = synth.WORKLOADS["decode_dsv2"]             # bf16, 2 shared experts
    counts = np.zeros(160, dtype=np.int64)
    counts[[3, 7, 9]] = [1, 2, 5]
    got = bench.gemm1_bytes(w, counts, rows=8 + 2 * 32)
    assert got == (3 + 2) * 2 * 1536 * 5120 * 2 + 72 * 5120 * 2 + 72 * 1536 * 2


def test_kernel_rule():
    names = {n: bench.gemm1_kernel(w) for n, w in synth.WORKLOADS.items()}
    assert names["mixtral_prefill"] == names["dsv2"] == names["e64_reroute"] == "ffn_tc_kernel<0>"
    assert names["decode_mixtral"] == names["decode_dsv2"] == "ffn_tc_swap_kernel<0>"
    assert names["decode_mixtral_fp8"] == names["decode_dsv2_fp8"] == "ffn_tc_swap_kernel<0,fp8>"
    assert names["tiny_fp32"] == "ffn_simt_kernel<1>"


def test_tensor_peak_rule():
    """The burst peak for a short timed region or one that ran uncapped; the
    sustained peak only for a second or more under the power cap."""
    pk = {"bf16_tflops": 1808.6, "bf16_tflops_sustained": 1390.4, "hbm_gbs": 6425.0,
          "source": "measured"}
    assert bench.tensor_peak(pk, 0.43, {"reasons": ["sw_power_cap"]})[0] == 1808.6
    assert bench.tensor_peak(pk, 0.43, {"reasons": []})[0] == 1808.6
    assert bench.tensor_peak(pk, 5.0, {"reasons": []})[0] == 1808.6
    assert bench.tensor_peak(pk, 5.0, {"reasons": ["sw_power_cap"]})[0] == 1390.4
    assert "burst" in bench.tensor_peak(pk, 0.43, {"reasons": None})[1]


def test_gemm1_roofline_picks_binding_bound():
    pk = {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0,
          "source": "measured"}
    w = synth.WORKLOADS["mixtral_prefill"]
    counts = np.full(8, 1024)
    flop = 2 * 8192 * 4096 * 2 * 14336
    r = bench.gemm1_roofline(w, counts, 8192, flop, 1.36, 0.43, {"sm_mhz": 2032,
                                                                    "reasons": []}, pk)
    assert r["bound"] == "tensor" and r["peak"] == 1800.0
    assert abs(r["frac"] - flop / 1.36e-3 / 1e12 / 1800.0) < 1e-12
    wd = synth.WORKLOADS["decode_mixtral"]
    r2 = bench.gemm1_roofline(wd, np.full(8, 16), 128, 2 * 128 * 4096 * 2 * 14336, 0.33, 0.1,
                              {"sm_mhz": 2032, "reasons": []}, pk)
    assert r2["bound"] == "hbm" and r2["unit"] == "GB/s"


def test_traffic_records_follow_code_not_comments(tmp_path, monkeypatch):
    # an ncu capture stays valid through comment and layout edits of the
    # kernel's sources and lapses with any change to the code itself
    assert bench.strip_c_comments('a = 1; // x\n/* y\n */  b = "//z/*";\nc = \'"\';') == \
        'a = 1; b = "//z/*"; c = \'"\';'
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("int f(int a) {\n  return a + 1;  // one more\n}\n")
    d0 = bench.code_digest(["k.cu"])
    src.write_text("/* header */\nint f(int a) {\n    return a + 1;  // plus one\n}\n")
    assert bench.code_digest(["k.cu"]) == d0
    src.write_text("int f(int a) {\n  return a + 2;  // one more\n}\n")
    assert bench.code_digest(["k.cu"]) != d0
