"""Benchmark of the MoE-FFN forward layer on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

A step is one moe_forward (router -> dispatch -> expert GEMMs -> combine) over
one batch of the workload, inputs resident in HBM.  L2 is flushed between
steps (a 512 MB write, outside the timed events).  With --gpus N > 1 (launched
by torch.distributed.run) every rank runs an independent replica on its own
GPU: the layer has no exchange step in this build, so there is no collective
on the data path; the barrier and the max over ranks of the timed region are
the only cross-rank steps.

--impl reference times the CPU oracle (float64 NumPy) on the host cores on a
bounded sample of the same workload.
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


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu capture
    (profiles/ncu_traffic.json), or None when there is none or the kernel's source
    has changed since it was taken (sha256 of its source files)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[workload][kernel]
        h = hashlib.sha256()
        for src in entry["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != entry["source_sha256"]:
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
    the sha256 of the kernel's sources (read back by measured_traffic)."""
    import hashlib
    srcs = TRAFFIC_SOURCES[kernel]
    h = hashlib.sha256()
    for s in srcs:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    data = json.load(open(path)) if os.path.exists(path) else {}
    data.setdefault(workload, {})[kernel] = {
        "dram_bytes_per_launch": float(nbytes), "sources": srcs,
        "source_sha256": h.hexdigest(), "command": command}
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
    workloads a getter that quantises and dequantises an expert on each call."""
    if not w.fp8_weights:
        return None
    import oracle

    def get(e):
        out = {"b1": None, "b2": None}
        for key in ("w_gate", "w_up", "w_down"):
            codes, scale = oracle.quantize_fp8(inp[key][e])
            out[key] = oracle.dequantize_fp8(codes, scale)
        return out
    return get


def run_cpu_oracle(w, inp, budget_s=20.0, max_tokens=None):
    """Time the oracle (as it stands) on a bounded token sample; returns tokens/s."""
    import oracle
    get = oracle_experts(w, inp)
    try:
        from threadpoolctl import threadpool_info
        cores = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        cores = os.cpu_count() or 1
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
    return {"value": n / dt, "unit": "tokens/s", "cores": int(cores), "kind": "oracle",
            "sample": f"routing and capacity over all {w.n_tokens} tokens, expert FFNs and "
                      f"combine for the first {n} tokens ({dt:.1f} s)"}


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
    get = oracle_experts(w, inp)
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
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


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


def bench_ours(args, w):
    import torch
    import mixture_experts_ffn_19_b300 as moe
    rank, local, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = moe.make_config(w.n_tokens, w.d_model, w.n_experts, w.top_k, w.d_ff, w.n_shared,
                          act=w.act, dtype=w.dtype, cap_mode=w.cap_mode, alpha=w.alpha,
                          has_ffn_bias=w.has_ffn_bias, has_router_bias=w.has_router_bias,
                          bias_mode=w.bias_mode)
    inp = synth.make_inputs(w)
    x = to_dev(inp["x"], dev)
    wr = to_dev(inp["w_router"], dev)
    rb = to_dev(inp["router_bias"], dev)
    wg, wu, wd = (to_dev(inp[k], dev) for k in ("w_gate", "w_up", "w_down"))
    b1, b2 = to_dev(inp["b1"], dev), to_dev(inp["b2"], dev)
    y = torch.empty((w.n_tokens, w.d_model), dtype=x.dtype, device=dev)
    ws = moe.alloc_workspace(cfg, dev)
    E = w.n_experts
    st_t = {"expert_freq": torch.zeros(E, device=dev), "mean_prob": torch.zeros(E, device=dev),
            "l_bal": torch.zeros(1, device=dev),
            "counts": torch.zeros(E, dtype=torch.int32, device=dev),
            "n_dropped": torch.zeros(1, dtype=torch.int32, device=dev),
            "n_rerouted": torch.zeros(1, dtype=torch.int32, device=dev),
            "z_loss": torch.zeros(1, device=dev), "router_entropy": torch.zeros(1, device=dev)}
    stats = moe.make_stats(**st_t)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    if w.fp8_weights:
        # E4M3 codes and per-expert-matrix scales, made by the library before timing
        qw, sc = [], []
        for t in (wg, wu, wd):
            q = torch.empty(t.shape, dtype=torch.uint8, device=dev)
            s_ = torch.empty(t.shape[0], dtype=torch.float32, device=dev)
            moe.moe_quantize_fp8(t, q, s_, stream)
            qw.append(q)
            sc.append(s_)
        scales = torch.stack(sc).contiguous()
        del wg, wu, wd
        torch.cuda.synchronize()

    def forward(x_arg, timing=None, y_arg=None):
        y_arg = y if y_arg is None else y_arg
        if w.fp8_weights:
            return moe.moe_forward_fp8(cfg, x_arg, wr, rb, qw[0], qw[1], qw[2], scales, y_arg,
                                       stats, ws, stream, timing=timing)
        return moe.moe_forward(cfg, x_arg, wr, rb, wg, wu, wd, b1, b2, y_arg, stats, ws, stream,
                               timing=timing)

    # warm-up
    for _ in range(args.warmup):
        forward(x)
    torch.cuda.synchronize()
    if moe.moe_device_status(ws) != moe.MOE_OK:
        raise RuntimeError("device status not ok after warm-up")
    kept = int(st_t["counts"].sum())
    nd = int(st_t["n_dropped"][0])
    work = layer_work(w, kept, nd)

    # timed region: K steps, per-step and per-stage CUDA events, L2 flush between steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    timings = []
    for s in range(args.steps):
        t = moe.moe_timing()
        for i in range(6):
            evs[s][i].record(stream)          # torch creates the CUDA event on first record
            t.events[i] = evs[s][i].cuda_event
        timings.append(t)
    torch.cuda.synchronize()
    assert all(e.cuda_event for row in evs for e in row)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = moe.moe_kernel_launches()
    with ClockSampler(dev) as clk:
        for s in range(args.steps):
            flush.fill_(s & 0xFF)
            forward(x, timings[s])
        torch.cuda.synchronize()
    launches = moe.moe_kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    step_ms = [evs[s][0].elapsed_time(evs[s][5]) for s in range(args.steps)]
    stage = {n: [evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps)]
             for i, n in enumerate(["route", "dispatch", "gemm1", "gemm2", "combine"])}
    total_ms = max_over_ranks(sum(step_ms), dev)
    st = moe.moe_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {moe.status_string(st)}")

    # end to end through the public API with host buffers, run the way a
    # serving loop runs it: every step copies its x from pinned host memory,
    # runs the layer and copies its y back to pinned host memory, all inside
    # the timed region; two device buffers and copy-in / compute / copy-out
    # streams let one step's copies overlap its neighbours' compute.  Between
    # steps L2 holds nothing useful when the expert weights (streamed every
    # step) exceed it several times over; otherwise the flush runs on the
    # compute stream before each forward, inside the timed region.
    es_w = 1 if w.fp8_weights else (2 if w.dtype == synth.DT_BF16 else 4)
    nmat = 3 if w.act == synth.ACT_SWIGLU else 2
    weight_bytes = (w.n_experts + w.n_shared) * nmat * w.d_ff * w.d_model * es_w
    e2e_flush = weight_bytes < 4 * L2_BYTES
    x_host = torch.from_numpy(inp["x"].view(np.int16) if inp["x"].dtype == np.uint16
                              else inp["x"]).pin_memory()
    hdt = torch.int16 if w.dtype else torch.float32
    y_host = [torch.empty((w.n_tokens, w.d_model), dtype=hdt).pin_memory() for _ in range(2)]
    x_in = [torch.empty_like(x) for _ in range(2)]
    y_out = [torch.empty_like(y) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nst = args.warmup + args.steps
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(nst)] for _ in range(3))
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for s in range(nst):
        b = s & 1
        if s == args.warmup:
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
        forward(x_in[b], None, y_out[b])
        ev_comp[s].record(stream)
        s_out.wait_event(ev_comp[s])
        with torch.cuda.stream(s_out):
            y_host[b].copy_(y_out[b].view(hdt), non_blocking=True)
            ev_out[s].record(s_out)
    t_end.record(s_out)
    t_end.synchronize()
    e2e_ms = [t_start.elapsed_time(t_end)]
    e2e_total = max_over_ranks(sum(e2e_ms), dev)

    pk = peaks()
    counts = st_t["counts"].cpu().numpy()
    wes = 1 if w.fp8_weights else (2 if w.dtype == synth.DT_BF16 else 4)
    touched = int((counts > 0).sum()) + w.n_shared
    nmat1 = 2 if w.act == synth.ACT_SWIGLU else 1
    g1_wbytes = touched * nmat1 * w.d_ff * w.d_model * wes
    g2_wbytes = touched * w.d_ff * w.d_model * wes
    g1_bytes = gemm1_bytes(w, counts, work["rows"])
    g1_ms = statistics.mean(stage["gemm1"])
    g1_tflops = work["gemm1_flop"] / (g1_ms * 1e-3) / 1e12
    g1_gbs = g1_bytes / (g1_ms * 1e-3) / 1e9
    peak_t = pk["bf16_tflops_sustained"]
    frac_t = g1_tflops / peak_t
    frac_b = g1_gbs / pk["hbm_gbs"]
    if frac_t >= frac_b:
        roof = {"bound": "tensor", "achieved": g1_tflops, "peak": peak_t, "unit": "TFLOP/s",
                "frac": frac_t, "peak_source": f"{pk['source']} bf16 sustained",
                "frac_of_burst_peak": g1_tflops / pk["bf16_tflops"],
                "algorithmic_per_launch": work["gemm1_flop"]}
    else:
        roof = {"bound": "hbm", "achieved": g1_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": frac_b, "peak_source": f"{pk['source']} copy bandwidth",
                "algorithmic_per_launch": g1_bytes}
    kname = gemm1_kernel(w)
    roof.update({"kernel": kname + " (gate/up GEMM + SwiGLU)",
                 "traffic": measured_traffic(kname, w.name),
                 "algorithmic_bytes_per_launch": g1_bytes})
    step_s = total_ms / args.steps * 1e-3
    value = throughput(w.n_tokens, args.steps, world, total_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == synth.DT_BF16 else "f32", "data": "synthetic",
        "config": workload_config(w, world),
        "roofline": roof,
        "e2e": {"value": throughput(w.n_tokens, args.steps, world, e2e_total), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x.numel() * x.element_size()),
                "d2h_bytes_per_step": int(y.numel() * y.element_size()),
                "copies": "pinned host buffers, overlapped with neighbouring steps' compute",
                "l2": "flushed before each forward" if e2e_flush else
                f"not flushed: {weight_bytes / 1e9:.2f} GB of expert weights streamed per step"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "stages_ms": {k: statistics.mean(v) for k, v in stage.items()},
        "layer_tflops": work["total_flop"] / step_s / 1e12,
        "layer_weight_gbs": (g1_wbytes + g2_wbytes) / step_s / 1e9,
        "layer_weight_frac_hbm": (g1_wbytes + g2_wbytes) / step_s / 1e9 / pk["hbm_gbs"],
        "experts_touched": touched, "kept_assignments": kept, "dropped": nd,
        "router_stats": {"l_bal": float(st_t["l_bal"][0]), "z_loss": float(st_t["z_loss"][0]),
                         "router_entropy_bits": float(st_t["router_entropy"][0])},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_oracle(w, inp, budget_s=args.ref_budget or 15.0,
                                              max_tokens=args.ref_tokens)
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
