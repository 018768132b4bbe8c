"""Benchmark of the MoE-FFN forward layer on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

A step is one moe_forward (router -> dispatch -> expert GEMMs -> combine) over
one batch of the workload, inputs resident in HBM.  L2 is flushed between
steps (a 512 MB write, outside the timed events).  With --gpus N > 1 (launched
by torch.distributed.run) every rank runs an independent replica on its own
GPU: the single-GPU layer has no exchange step, so there is no collective
on the data path; the barrier and the max over ranks of the timed region are
the only cross-rank steps.

--impl reference times the CPU oracle (C++17, double accumulation, OpenMP) on
the host cores on a bounded sample of the same workload.

The default run (headline workload, one GPU) also times the decode, DeepSeek-V2
and 64-expert layers and reports each under "workloads", and times the oracle
on one thread over the whole tiny fp32 and decode batches.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s @1 B300; grouped-GEMM TFLOP/s & HBM GB/s vs roofline"
HEADLINE = "mixtral_prefill"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def throughput(tokens_per_step: int, steps: int, world: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch (weak scaling)."""
    return tokens_per_step * steps * world / (total_ms * 1e-3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


class _Nvml:
    """Minimal read-only NVML binding over ctypes (libnvidia-ml ships with the driver)."""

    CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("libnvidia-ml not found")
        self.lib = lib
        self._ok(lib.nvmlInit_v2())

    def _ok(self, rc):
        if rc != 0:
            raise RuntimeError(f"NVML error {rc}")

    def handle(self, torch_device):
        import torch
        c = self.c
        h = c.c_void_p()
        props = torch.cuda.get_device_properties(torch_device)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(c.c_char_p(bus.encode()), c.byref(h)) != 0:
            self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(c.c_uint(0), c.byref(h)))
        return h

    def clock(self, h):
        v = self.c.c_uint()
        self._ok(self.lib.nvmlDeviceGetClockInfo(h, self.c.c_int(self.CLOCK_SM), self.c.byref(v)))
        return v.value

    def max_clock(self, h):
        v = self.c.c_uint()
        self._ok(self.lib.nvmlDeviceGetMaxClockInfo(h, self.c.c_int(self.CLOCK_SM), self.c.byref(v)))
        return v.value

    def reasons(self, h):
        v = self.c.c_ulonglong()
        f = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._ok(f(h, self.c.byref(v)))
        return v.value


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled through NVML every
    10 ms while the timed region runs (read-only queries)."""

    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.stop = threading.Event()
        self.nvml = None

    def _run(self):
        while not self.stop.is_set():
            try:
                self.samples.append(self.nvml.clock(self.h))
                r = self.nvml.reasons(self.h)
                for n, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(n)
            except Exception:
                pass
            time.sleep(0.01)

    def __enter__(self):
        try:
            self.nvml = _Nvml()
            self.h = self.nvml.handle(self.dev)
            self.max_mhz = self.nvml.max_clock(self.h)
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        except Exception as exc:  # clocks are then reported as unavailable
            self.error = repr(exc)
            self.nvml = None
        return self

    def __exit__(self, *a):
        self.stop.set()
        if self.nvml is not None:
            self.thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0, "error": getattr(self, "error", "no samples")}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


def layer_work(w, counts_kept, n_dropped):
    """Algorithmic FLOPs of one forward (kept assignments and shared rows only)."""
    N, d, E, k, F, S = w.n_tokens, w.d_model, w.n_experts, w.top_k, w.d_ff, w.n_shared
    rows = int(counts_kept) + S * N
    g1 = 2.0 * rows * d * (2 * F if w.act == synth.ACT_SWIGLU else F)
    g2 = 2.0 * rows * F * d
    router = 2.0 * N * d * E
    return {"rows": rows, "gemm1_flop": g1, "gemm2_flop": g2, "router_flop": router,
            "total_flop": g1 + g2 + router}


def gemm1_bytes(w, counts, rows: int) -> float:
    """Algorithmic bytes of one gate/up GEMM launch: the gate (and up) weights of
    every touched expert (routed experts with at least one kept row, plus the
    shared ones), the launch's input rows and its output rows of H."""
    es = 2 if w.dtype == synth.DT_BF16 else 4
    wes = 1 if w.fp8_weights else es             # bytes per expert-weight element
    touched = int((np.asarray(counts) > 0).sum()) + w.n_shared
    nmat1 = 2 if w.act == synth.ACT_SWIGLU else 1
    return float(touched * nmat1 * w.d_ff * w.d_model * wes + rows * w.d_model * es
                 + rows * w.d_ff * es)


def gemm1_kernel(w) -> str:
    """The gate/up GEMM kernel the library launches for this workload: the
    weights-as-M (swap-AB) kernel for E4M3 weights and for batches with at most
    64 assignments per expert on average (and, with shared experts, at most 512
    tokens); the 128-row-tile kernel otherwise (the rule in csrc/ffn_tc.cu)."""
    if w.dtype != synth.DT_BF16:
        return "ffn_simt_kernel<1>"
    if w.fp8_weights:
        return "ffn_tc_swap_kernel<0,fp8>"
    if w.n_tokens * w.top_k <= 64 * w.n_experts and (w.n_shared == 0 or w.n_tokens <= 512):
        return "ffn_tc_swap_kernel<0>"
    return "ffn_tc_kernel<0>"


def strip_c_comments(text: str) -> str:
    """C/C++/CUDA source without its comments, every whitespace run collapsed to
    one space (string and character literals kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                               # literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def code_digest(srcs) -> str:
    """sha256 of the sources' code (comments and layout left out): an edit of a
    comment keeps an ncu capture valid, any change to the code voids it."""
    import hashlib
    h = hashlib.sha256()
    for src in srcs:
        with open(os.path.join(ROOT, src), encoding="utf-8") as f:
            h.update(strip_c_comments(f.read()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu capture
    (profiles/ncu_traffic.json), or None when there is none or the kernel's code
    has changed since it was taken (code_digest of its source files)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[workload][kernel]
        if code_digest(entry["sources"]) != entry["source_sha256"]:
            return None
        return float(entry["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


_GEMM_SOURCES = ["mixture_experts_ffn_19_b300/csrc/ffn_tc.cu",
                 "mixture_experts_ffn_19_b300/csrc/common.cuh"]
TRAFFIC_SOURCES = {
    "ffn_tc_kernel<0>": _GEMM_SOURCES,
    "ffn_tc_swap_kernel<0>": _GEMM_SOURCES,
    "ffn_tc_swap_kernel<0,fp8>": _GEMM_SOURCES,
}


def record_traffic(workload: str, kernel: str, nbytes: float, command: str) -> None:
    """Store one ncu capture's DRAM bytes per launch in profiles/ncu_traffic.json with
    the code digest of the kernel's sources (read back by measured_traffic)."""
    srcs = TRAFFIC_SOURCES[kernel]
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    data = json.load(open(path)) if os.path.exists(path) else {}
    data.setdefault(workload, {})[kernel] = {
        "dram_bytes_per_launch": float(nbytes), "sources": srcs,
        "source_sha256": code_digest(srcs), "command": command}
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)


def to_dev(a, device):
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def oracle_experts(w, inp):
    """The oracle's expert weights: None (take them from `inp`), or for E4M3
    workloads a getter that hands the oracle each matrix's E4M3 codes and scale
    (made by the oracle's own quantiser from the bf16 draws)."""
    if not w.fp8_weights:
        return None
    import oracle
    cache = {}

    def get(e):
        # quantised once per expert, as the library's weights are before timing
        if e not in cache:
            out = {"b1": None, "b2": None}
            for key in ("w_gate", "w_up", "w_down"):
                out[key] = oracle.quantize_fp8(inp[key][e])
            cache[e] = out
        return cache[e]
    return get


def prepared_experts(w, inp):
    """oracle_experts with every expert prepared up front (outside any timing)."""
    get = oracle_experts(w, inp)
    if get is not None:
        for e in range(w.n_experts + w.n_shared):
            get(e)
    return get


def oracle_threads_info():
    import oracle
    return {"cores": oracle.threads(), "hardware_concurrency": oracle.hardware_concurrency()}


def run_cpu_oracle(w, inp, budget_s=20.0, max_tokens=None):
    """Time the oracle (as it stands, on every host thread OpenMP gives it) on a
    bounded token sample; returns the cpu_baseline record (tokens/s)."""
    import oracle
    get = prepared_experts(w, inp)
    oracle.set_threads(oracle.hardware_concurrency())
    # grow the token sample until one timed run takes about a third of the budget
    n, dt = 1, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.moe_forward(w, inp, tokens=np.arange(n), get_expert=get)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 3 or n >= w.n_tokens or (max_tokens and n >= max_tokens):
            break
        n = min(w.n_tokens, max(2 * n, int(n * budget_s / 3 / max(dt, 1e-3))))
        if max_tokens:
            n = min(n, max_tokens)
    info = oracle_threads_info()
    return {"value": n / dt, "unit": "tokens/s", "cores": info["cores"], "kind": "oracle",
            "hardware_concurrency": info["hardware_concurrency"],
            "oracle": "C++17 loops, double accumulation, OpenMP",
            "sample": f"routing and capacity over all {w.n_tokens} tokens, expert FFNs and "
                      f"combine for the first {n} tokens ({dt:.1f} s, {info['cores']} threads)"}


def oracle_single_thread(w, inp):
    """The oracle on one thread over the workload's whole batch (seconds, tokens/s)."""
    import oracle
    get = prepared_experts(w, inp)
    before = oracle.threads()
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.moe_forward(w, inp, get_expert=get)
        dt = time.perf_counter() - t0
    finally:
        oracle.set_threads(before)
    return {"seconds": dt, "tokens_per_s": w.n_tokens / dt, "threads": 1,
            "sample": f"whole batch of {w.n_tokens} tokens"}


def bench_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    inp = synth.make_inputs(w)
    budget = args.ref_budget if args.ref_budget else min(15.0, max(1.0, 150.0 / (args.warmup + args.steps)))
    info = run_cpu_oracle(w, inp, budget_s=3 * budget, max_tokens=args.ref_tokens)
    n = int(info["sample"].split("first ")[1].split(" ")[0])
    per_step = []
    get = prepared_experts(w, inp)
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.moe_forward(w, inp, tokens=np.arange(n), get_expert=get)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            per_step.append(dt)
    value = n * len(per_step) / sum(per_step)
    sample = (f"routing and capacity over all {w.n_tokens} tokens, expert FFNs and combine "
              f"for the first {n} tokens, {statistics.mean(per_step):.2f} s per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.mean(per_step), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": info["cores"],
                             "hardware_concurrency": info["hardware_concurrency"],
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def tensor_peak(pk, timed_s: float, clocks: dict):
    """The bf16 tensor peak a kernel's TFLOP/s is reported against.

    The burst peak (cuBLAS timed alone, clocks free) applies to a short timed
    region or one that ran at full clock without power capping; the sustained
    peak (seconds of back-to-back GEMMs under the power cap) applies only to a
    timed region of a second or more during which the power cap was active."""
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    if timed_s >= 1.0 and capped:
        return pk["bf16_tflops_sustained"], (
            f"{pk['source']} bf16 sustained: timed region {timed_s:.2f} s with sw_power_cap active")
    why = f"timed region {timed_s:.2f} s" if timed_s < 1.0 else "no sw_power_cap sample"
    return pk["bf16_tflops"], f"{pk['source']} bf16 burst: {why}"


L2_BYTES = 126 * 1024 * 1024        # B300 L2


def workload_config(w, world):
    return {"workload": w.name, "n_tokens": w.n_tokens, "d_model": w.d_model,
            "n_experts": w.n_experts, "top_k": w.top_k, "d_ff": w.d_ff, "n_shared": w.n_shared,
            "activation": "swiglu" if w.act == synth.ACT_SWIGLU else "gelu",
            "capacity": ["none", "drop", "reroute"][w.cap_mode],
            "alpha": w.alpha if w.cap_mode else None, "router_bias": w.bias_law,
            "router_bias_mode": "selection" if w.bias_mode else "logit",
            "expert_weights": "fp8_e4m3" if w.fp8_weights else
            ("bf16" if w.dtype == synth.DT_BF16 else "f32"),
            "l2_flush": True, "parallelism": f"replicas{world}" if world > 1 else "single"}


class Layer:
    """One workload's layer resident on the device: inputs, weights (bf16, or E4M3
    codes and scales made by the library), output, workspace and statistics."""

    def __init__(self, w, dev, inp=None):
        import torch
        import mixture_experts_ffn_19_b300 as moe
        self.w, self.dev, self.moe = w, dev, moe
        self.cfg = moe.make_config(w.n_tokens, w.d_model, w.n_experts, w.top_k, w.d_ff,
                                   w.n_shared, act=w.act, dtype=w.dtype, cap_mode=w.cap_mode,
                                   alpha=w.alpha, has_ffn_bias=w.has_ffn_bias,
                                   has_router_bias=w.has_router_bias, bias_mode=w.bias_mode)
        self.inp = synth.make_inputs(w) if inp is None else inp
        inp = self.inp
        self.x = to_dev(inp["x"], dev)
        self.wr = to_dev(inp["w_router"], dev)
        self.rb = to_dev(inp["router_bias"], dev)
        wg, wu, wd = (to_dev(inp[k], dev) for k in ("w_gate", "w_up", "w_down"))
        self.b1, self.b2 = to_dev(inp["b1"], dev), to_dev(inp["b2"], dev)
        self.y = torch.empty((w.n_tokens, w.d_model), dtype=self.x.dtype, device=dev)
        self.ws = moe.alloc_workspace(self.cfg, dev)
        E = w.n_experts
        self.st_t = {"expert_freq": torch.zeros(E, device=dev),
                     "mean_prob": torch.zeros(E, device=dev),
                     "l_bal": torch.zeros(1, device=dev),
                     "counts": torch.zeros(E, dtype=torch.int32, device=dev),
                     "n_dropped": torch.zeros(1, dtype=torch.int32, device=dev),
                     "n_rerouted": torch.zeros(1, dtype=torch.int32, device=dev),
                     "z_loss": torch.zeros(1, device=dev),
                     "router_entropy": torch.zeros(1, device=dev)}
        self.stats = moe.make_stats(**self.st_t)
        self.stream = torch.cuda.current_stream(dev)
        if w.fp8_weights:
            # E4M3 codes and per-expert-matrix scales, made by the library before timing
            qw, sc = [], []
            for t in (wg, wu, wd):
                q = torch.empty(t.shape, dtype=torch.uint8, device=dev)
                s_ = torch.empty(t.shape[0], dtype=torch.float32, device=dev)
                moe.moe_quantize_fp8(t, q, s_, self.stream)
                qw.append(q)
                sc.append(s_)
            self.qw, self.scales = qw, torch.stack(sc).contiguous()
            del wg, wu, wd
            torch.cuda.synchronize()
        else:
            self.wg, self.wu, self.wd = wg, wu, wd

    def forward(self, x_arg=None, timing=None, y_arg=None):
        moe = self.moe
        x_arg = self.x if x_arg is None else x_arg
        y_arg = self.y if y_arg is None else y_arg
        if self.w.fp8_weights:
            return moe.moe_forward_fp8(self.cfg, x_arg, self.wr, self.rb, self.qw[0], self.qw[1],
                                       self.qw[2], self.scales, y_arg, self.stats, self.ws,
                                       self.stream, timing=timing)
        return moe.moe_forward(self.cfg, x_arg, self.wr, self.rb, self.wg, self.wu, self.wd,
                               self.b1, self.b2, y_arg, self.stats, self.ws, self.stream,
                               timing=timing)

    def weight_bytes(self):
        w = self.w
        es_w = 1 if w.fp8_weights else (2 if w.dtype == synth.DT_BF16 else 4)
        nmat = 3 if w.act == synth.ACT_SWIGLU else 2
        return (w.n_experts + w.n_shared) * nmat * w.d_ff * w.d_model * es_w


STAGES = ["route", "dispatch", "gemm1", "gemm2", "combine"]


def time_device(layer, steps, warmup, flush, world):
    """W untimed forwards, then two timed passes of K forwards on the launching
    stream, L2 flushed (a 512 MB write) before each step outside the events,
    NVML clocks sampled throughout.  Pass 1 has one event pair around each
    forward: the step times (an event recorded between two kernels ends their
    chained launch, so events at the stage boundaries would lengthen the step).
    Pass 2 has an event at every stage boundary: the stage and kernel times."""
    import torch
    moe = layer.moe
    for _ in range(warmup):
        layer.forward()
    torch.cuda.synchronize()
    if moe.moe_device_status(layer.ws) != moe.MOE_OK:
        raise RuntimeError(f"{layer.w.name}: device status not ok after warm-up")
    plain = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    timings = []
    for s in range(steps):
        t = moe.moe_timing()
        for i in range(6):
            evs[s][i].record(layer.stream)    # torch creates the CUDA event on first record
            t.events[i] = evs[s][i].cuda_event
        timings.append(t)
    torch.cuda.synchronize()
    assert all(e.cuda_event for row in evs for e in row)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = moe.moe_kernel_launches()
    with ClockSampler(layer.dev) as clk:
        for s in range(steps):
            flush.fill_(s & 0xFF)
            plain[s][0].record(layer.stream)
            layer.forward()
            plain[s][1].record(layer.stream)
        torch.cuda.synchronize()
        launches = moe.moe_kernel_launches() - launches0
        for s in range(steps):
            flush.fill_(s & 0xFF)
            layer.forward(timing=timings[s])
        torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    st = moe.moe_device_status(layer.ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"{layer.w.name}: device status {moe.status_string(st)}")
    step_ms = [a.elapsed_time(b) for a, b in plain]
    staged_ms = [evs[s][0].elapsed_time(evs[s][5]) for s in range(steps)]
    stage = {n: [evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)]
             for i, n in enumerate(STAGES)}
    return {"step_ms": step_ms, "staged_step_ms": staged_ms, "stage": stage, "launches": launches,
            "clocks": clk.summary()}


def gemm1_roofline(w, counts, rows, gemm1_flop, g1_ms, timed_s, clocks, pk):
    """Roofline of the dominant kernel (the gate/up GEMM): the binding one of its
    tensor (algorithmic FLOPs) and HBM (algorithmic bytes) fractions."""
    g1_bytes = gemm1_bytes(w, counts, rows)
    g1_tflops = gemm1_flop / (g1_ms * 1e-3) / 1e12
    g1_gbs = g1_bytes / (g1_ms * 1e-3) / 1e9
    peak_t, src_t = tensor_peak(pk, timed_s, clocks)
    frac_t = g1_tflops / peak_t
    frac_b = g1_gbs / pk["hbm_gbs"]
    mhz = clocks.get("sm_mhz")
    if frac_t >= frac_b:
        roof = {"bound": "tensor", "achieved": g1_tflops, "peak": peak_t, "unit": "TFLOP/s",
                "frac": frac_t, "peak_source": src_t,
                "frac_of_burst_peak": g1_tflops / pk["bf16_tflops"],
                "frac_of_sustained_peak": g1_tflops / pk["bf16_tflops_sustained"],
                "algorithmic_per_launch": gemm1_flop}
    else:
        roof = {"bound": "hbm", "achieved": g1_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": frac_b, "peak_source": f"{pk['source']} copy bandwidth",
                "algorithmic_per_launch": g1_bytes}
    kname = gemm1_kernel(w)
    roof.update({"kernel": kname + " (gate/up GEMM + SwiGLU)", "kernel_ms": g1_ms,
                 "sm_mhz_median": mhz,
                 "kernel_mcycles": None if mhz is None else g1_ms * 1e-3 * mhz,
                 "traffic": measured_traffic(kname, w.name),
                 "algorithmic_bytes_per_launch": g1_bytes})
    return roof


def summarise(layer, t, world, pk):
    """The measured figures of one workload from its device timing."""
    w = layer.w
    steps = len(t["step_ms"])
    total_ms = max_over_ranks(sum(t["step_ms"]), layer.dev)
    counts = layer.st_t["counts"].cpu().numpy()
    kept = int(counts.sum())
    nd = int(layer.st_t["n_dropped"][0])
    work = layer_work(w, kept, nd)
    stage_ms = {k: statistics.mean(v) for k, v in t["stage"].items()}
    staged_ms = max_over_ranks(sum(t["staged_step_ms"]), layer.dev)
    # both passes ran back to back: the GEMM times of pass 2 were taken that
    # far into the run (which decides the peak they are held against)
    timed_s = (total_ms + staged_ms) * 1e-3
    roof = gemm1_roofline(w, counts, work["rows"], work["gemm1_flop"], stage_ms["gemm1"],
                          timed_s, t["clocks"], pk)
    wes = 1 if w.fp8_weights else (2 if w.dtype == synth.DT_BF16 else 4)
    touched = int((counts > 0).sum()) + w.n_shared
    nmat1 = 2 if w.act == synth.ACT_SWIGLU else 1
    wbytes = touched * (nmat1 + 1) * w.d_ff * w.d_model * wes
    step_s = total_ms / steps * 1e-3
    return {
        "value": throughput(w.n_tokens, steps, world, total_ms), "unit": "tokens/s",
        "steps": steps, "ms_per_step": total_ms / steps, "timed_region_s": timed_s,
        "ms_per_step_with_stage_events": staged_ms / steps,
        "roofline": roof, "clocks": t["clocks"], "gpu_launches": t["launches"],
        "stages_ms": stage_ms,
        "layer_tflops": work["total_flop"] / step_s / 1e12,
        "layer_weight_gbs": wbytes / step_s / 1e9,
        "layer_weight_frac_hbm": wbytes / step_s / 1e9 / pk["hbm_gbs"],
        "experts_touched": touched, "kept_assignments": kept, "dropped": nd,
        "rerouted": int(layer.st_t["n_rerouted"][0]),
        "router_stats": {"l_bal": float(layer.st_t["l_bal"][0]),
                         "z_loss": float(layer.st_t["z_loss"][0]),
                         "router_entropy_bits": float(layer.st_t["router_entropy"][0])},
    }


def time_e2e(layer, steps, warmup, flush, world):
    """End to end through the public API with host buffers, run the way a
    serving loop runs it: every step copies its x from pinned host memory,
    runs the layer and copies its y back to pinned host memory, all inside the
    timed region; two device buffers and copy-in / compute / copy-out streams
    let one step's copies overlap its neighbours' compute.  Between steps L2
    holds nothing useful when the expert weights (streamed every step) exceed
    it several times over; otherwise the flush runs on the compute stream
    before each forward, inside the timed region."""
    import torch
    w, x, y, stream = layer.w, layer.x, layer.y, layer.stream
    weight_bytes = layer.weight_bytes()
    e2e_flush = weight_bytes < 4 * L2_BYTES
    inp_x = layer.inp["x"]
    x_host = torch.from_numpy(inp_x.view(np.int16) if inp_x.dtype == np.uint16
                              else inp_x).pin_memory()
    hdt = torch.int16 if w.dtype else torch.float32
    y_host = [torch.empty((w.n_tokens, w.d_model), dtype=hdt).pin_memory() for _ in range(2)]
    x_in = [torch.empty_like(x) for _ in range(2)]
    y_out = [torch.empty_like(y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(layer.dev), torch.cuda.Stream(layer.dev)
    nst = warmup + steps
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(nst)] for _ in range(3))
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for s in range(nst):
        b = s & 1
        if s == warmup:
            t_start.record(s_in)
        if s >= 2:
            s_in.wait_event(ev_comp[s - 2])          # x_in[b] read by step s-2
        with torch.cuda.stream(s_in):
            x_in[b].view(x_host.dtype).copy_(x_host, non_blocking=True)
            ev_in[s].record(s_in)
        stream.wait_event(ev_in[s])
        if s >= 2:
            stream.wait_event(ev_out[s - 2])         # y_out[b] copied out by step s-2
        if e2e_flush:
            flush.fill_(s & 0xFF)
        layer.forward(x_in[b], None, y_out[b])
        ev_comp[s].record(stream)
        s_out.wait_event(ev_comp[s])
        with torch.cuda.stream(s_out):
            y_host[b].copy_(y_out[b].view(hdt), non_blocking=True)
            ev_out[s].record(s_out)
    t_end.record(s_out)
    t_end.synchronize()
    e2e_total = max_over_ranks(t_start.elapsed_time(t_end), layer.dev)
    return {"value": throughput(w.n_tokens, steps, world, e2e_total), "unit": "tokens/s",
            "h2d_bytes_per_step": int(x.numel() * x.element_size()),
            "d2h_bytes_per_step": int(y.numel() * y.element_size()),
            "copies": "pinned host buffers, overlapped with neighbouring steps' compute",
            "l2": "flushed before each forward" if e2e_flush else
            f"not flushed: {weight_bytes / 1e9:.2f} GB of expert weights streamed per step"}


# Workloads timed beside the headline in the default run, each with the figure
# that bounds it (the decode layers: the HBM fraction of the weights they
# stream; the prefill layers: the gate/up GEMM's roofline).
SECONDARY = ["decode_mixtral", "decode_dsv2", "dsv2", "e64_reroute"]


def secondary_record(name, dev, args, flush, pk):
    import torch
    w = synth.WORKLOADS[name]
    layer = Layer(w, dev)
    steps = max(10, min(args.steps, 100))
    t = time_device(layer, steps, max(3, min(args.warmup, 10)), flush, 1)
    rec = summarise(layer, t, 1, pk)
    rec["config"] = workload_config(w, 1)
    if name.startswith("decode") and not args.no_cpu_baseline:
        rec["oracle_single_thread"] = oracle_single_thread(w, layer.inp)
    del layer
    torch.cuda.empty_cache()
    return rec


def bench_ours(args, w):
    import torch
    rank, local, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    layer = Layer(w, dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    pk = peaks()
    t = time_device(layer, args.steps, args.warmup, flush, world)
    rec = summarise(layer, t, world, pk)
    e2e = time_e2e(layer, args.steps, args.warmup, flush, world)

    line = {
        "metric": METRIC, "value": rec["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == synth.DT_BF16 else "f32", "data": "synthetic",
        "config": workload_config(w, world),
        "roofline": rec["roofline"],
        "e2e": e2e,
        "gpu_launches": rec["gpu_launches"],
        "clocks": rec["clocks"],
    }
    line.update({k: rec[k] for k in ("timed_region_s", "ms_per_step_with_stage_events",
                                      "stages_ms", "layer_tflops",
                                      "layer_weight_gbs", "layer_weight_frac_hbm",
                                      "experts_touched", "kept_assignments", "dropped",
                                      "rerouted", "router_stats")})
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_oracle(w, layer.inp, budget_s=args.ref_budget or 15.0,
                                              max_tokens=args.ref_tokens)
        small = synth.WORKLOADS["tiny_fp32"]
        line["cpu_baseline"]["single_thread"] = {"tiny_fp32": oracle_single_thread(
            small, synth.make_inputs(small))}
    if world == 1 and w.name == HEADLINE and not args.headline_only:
        del layer
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name in SECONDARY:
            rec2 = secondary_record(name, dev, args, flush, pk)
            st = rec2.pop("oracle_single_thread", None)
            if st is not None and "cpu_baseline" in line:
                line["cpu_baseline"]["single_thread"][name] = st
            line["workloads"][name] = rec2
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=list(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the secondary workloads timed after the headline")
    ap.add_argument("--ref-budget", type=float, default=None,
                    help="seconds of oracle work per step (default: ~150 s over the run, "
                         "15 s for the cpu_baseline leg)")
    ap.add_argument("--ref-tokens", type=int, default=None)
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="override a workload field (e.g. n_experts=2) for a smaller case")
    ap.add_argument("--record-traffic", nargs=4, metavar=("WORKLOAD", "KERNEL", "BYTES", "COMMAND"),
                    help="store an ncu capture's DRAM bytes per launch for the roofline record")
    args = ap.parse_args(argv)
    if args.record_traffic:
        wl, kern, nb, cmd = args.record_traffic
        record_traffic(wl, kern, float(nb), cmd)
        return 0
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    w = synth.WORKLOADS[args.workload]
    for kv in args.set:
        key, val = kv.split("=", 1)
        cur = getattr(w, key)
        w = w.replace(**{key: type(cur)(float(val)) if isinstance(cur, (int, float)) else val},
                      name=w.name + f"[{key}={val}]")
    if args.impl == "reference":
        return bench_reference(args, w)
    return bench_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
