"""Throughput of the chunkwise GDN forward on one GB300 (or N, one process each).

A step is one gdn_chunk_fwd call over the B=4, H=16, T=4096, Dk=Dv=128 bf16
workload (chunk 64, fp32 state): decay cumsum, decay-masked KK^T, triangular
inverse, w/u, the state scan and the output, all inside the library's kernels.
Inputs stay resident in HBM; each step reads 192 MiB and writes 64 MiB, more
than the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Rank 0 prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on
a bounded sample of the same workload (the method has no runnable reference
implementation) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# the backward passes on bf16 at D = 128: what runs where
BWD_PATH = ("WY factors, state chains and every product of the gradient step on tcgen05; "
            "elementwise gradient terms and row sums on the CUDA cores (fp32)")

WORKLOAD = "gdn_b4h16t4096d128_bf16"
METRIC = "GDN fwd tokens/s (B4,H16,T4096,D128 bf16) + % of binding roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
SCAN_SOURCES = ("scan_simt.cu", "scan_tc.cu")


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0}, "fallback"


def gdn_bytes_per_token_head(D, s_in=2, s_out=2):
    """Algorithmic HBM bytes per (token, head): q, k, v in, beta (dtype) and g
    (fp32) in, o out; the fp32 state never leaves the chip."""
    return 3 * D * s_in + s_in + 4 + D * s_out


def cam_scan_bytes_per_token_head(D, s=2):
    """Algorithmic HBM bytes per (token, head) of the frame-level scan: q, k, v
    and beta in, o out (the per-frame decay and the state are negligible)."""
    return 3 * D * s + s + D * s


def gdn_flops_per_token_head(D, C):
    """w.S, k^T v_new and q.S (2 D^2 each) + triangular-half KK^T, T.(beta k),
    T.(beta v), q k^T and P.v_new (C.D each) + the C^3/3 inverse amortised."""
    return 6 * D * D + 5 * C * D + C * C // 3


def make_workspace(binding, w, dev):
    """The library's device scratch for workload w (None when it needs none),
    allocated once so that no step allocates."""
    import torch
    r = w.r if w.kind == "deltaproduct" else 1
    n = binding.workspace_bytes(w.B, w.H, w.T, w.D, w.D, w.chunk, r)
    return torch.empty(n, dtype=torch.uint8, device=dev) if n else None


def max_over_ranks(x, world, device):
    """The largest of each rank's value (a step time): the job is as slow as
    its slowest replica.  Needs an initialised process group when world > 1."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens(tokens_per_replica, world):
    """Tokens one step processes over all ranks: each rank runs its own replica
    of the workload (independent heads, no collective on the data path)."""
    return tokens_per_replica * world


def workload_config(w, world):
    """The `config` object of both arms' JSON lines: the workload by name and
    sizes (the same keys whichever arm runs it)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "Dk": w.D, "Dv": w.D, "chunk": w.chunk,
            "state": "fp32", "parallelism": f"replicas x{world} (no collective)",
            "l2": "no flush: each step touches 270 MB > 129 MB L2"}


def median_step_ms(events):
    """Per-step times from consecutive CUDA events recorded between steps on
    the launching stream: (median, mean) in ms."""
    per = [a.elapsed_time(b) for a, b in zip(events[:-1], events[1:])]
    return statistics.median(per), sum(per) / len(per)


def source_sha():
    h = hashlib.sha256()
    for name in SCAN_SOURCES:
        p = os.path.join(ROOT, "gated_delta_rule_47_gb300", "csrc", name)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per launch of the scan kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "scan_traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_sha") != source_sha():
        return None, d.get("kernel")
    return d.get("dram_bytes_per_launch"), d.get("kernel")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"unavailable": "nvidia-smi not found"}
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"unavailable": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(inp, n_heads, B, H, T):
    """Time the fp64 oracle, as it stands, on n_heads whole heads of the
    workload; returns (tokens/s scaled to the full workload, seconds, threads)."""
    import oracle
    from gated_delta_rule_47_gb300.inputs import to_f64
    idx = list(range(n_heads))

    def sub(x):
        return to_f64(x).reshape(B * H, *x.shape[2:])[idx][None]

    args = [sub(inp[k]) for k in ("q", "k", "v", "beta", "g")]
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.gdn_fwd(*args, return_final_state=False)
    dt = time.perf_counter() - t0
    tokens = B * T * n_heads / (B * H)
    return tokens / dt, dt, threads


def run_reference(args, rank, world):
    """Reference arm: the fp64 CPU oracle on a bounded sample of the workload."""
    if rank != 0:
        return 0
    from gated_delta_rule_47_gb300.inputs import WORKLOADS
    w = WORKLOADS[WORKLOAD]
    inp = w.make()
    n_heads = args.ref_heads
    vals, secs = [], []
    threads = None
    for i in range(args.warmup + args.steps):
        v, dt, threads = cpu_oracle_sample(inp, n_heads, w.B, w.H, w.T)
        if i >= args.warmup:
            vals.append(v)
            secs.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; q,k unit-norm, v~N(0,1), beta=sigmoid(N), g=logsigmoid(N)/16)",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "cpu_count": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{n_heads} of {w.B * w.H} heads, full T={w.T}, per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from gated_delta_rule_47_gb300 import binding, build
    from gated_delta_rule_47_gb300.inputs import WORKLOADS

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build.build()
    lib = binding.load()
    w = WORKLOADS[WORKLOAD]
    inp_cpu = w.make()
    d = {k: v.to(dev) for k, v in inp_cpu.items()}
    o = torch.empty(w.B, w.H, w.T, w.D, dtype=torch.bfloat16, device=dev)
    ws = make_workspace(binding, w, dev)
    stream = torch.cuda.current_stream()

    def step():
        binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], chunk=w.chunk, o=o, workspace=ws)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    # The sampler runs over a busy window of at least `clock_window` seconds:
    # untimed steps before and after the timed ones keep the GPU on this
    # workload so that nvidia-smi sees the clocks it runs at.
    with ClockSampler(local_rank) as clk:
        t_win = time.perf_counter()
        while time.perf_counter() - t_win < args.clock_window / 2:
            step()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        n0 = binding.launch_count()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        evs[0].record(stream)
        for i in range(args.steps):
            step()
            evs[i + 1].record(stream)
        launches = binding.launch_count() - n0  # kernels the library launched in the timed steps
        torch.cuda.synchronize()
        while time.perf_counter() - t_win < args.clock_window:
            step()
            torch.cuda.synchronize()
    barrier()
    med_ms, mean_ms = median_step_ms(evs)
    ms = max_over_ranks(med_ms, world, dev)
    tokens_per_step = whole_job_tokens(w.B * w.T, world)
    value = tokens_per_step / (ms * 1e-3)

    # End to end through the same C-ABI call: every step copies its inputs in
    # from pinned host memory and its output back, inside the timed region.
    # Steps are pipelined two deep on double-buffered device tensors: the
    # input copies of step i+1 and the output copy of step i-1 run while
    # step i computes (host-to-device and device-to-host copies use both
    # directions of the link at once).
    host = {k: v.pin_memory() for k, v in inp_cpu.items()}
    o_hosts = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_hosts[0].numel() * o_hosts[0].element_size()
    dsets = [d, {k: torch.empty_like(v) for k, v in d.items()}]
    osets = [o, torch.empty_like(o)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    done_k = [None, None]    # kernel of the last step that used each buffer set
    done_out = [None, None]  # output copy of the last step that used each set

    def e2e_step(i):
        j = i & 1
        dd, oo = dsets[j], osets[j]
        s_in.wait_stream(stream) if done_k[j] is None else s_in.wait_event(done_k[j])
        with torch.cuda.stream(s_in):
            for k in host:
                dd[k].copy_(host[k], non_blocking=True)
        ev_in = torch.cuda.Event()
        ev_in.record(s_in)
        stream.wait_event(ev_in)
        if done_out[j] is not None:
            stream.wait_event(done_out[j])
        binding.gdn_chunk_fwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], chunk=w.chunk, o=oo, workspace=ws)
        ek = torch.cuda.Event()
        ek.record(stream)
        done_k[j] = ek
        s_out.wait_event(ek)
        with torch.cuda.stream(s_out):
            o_hosts[j].copy_(oo, non_blocking=True)
        eo = torch.cuda.Event()
        eo.record(s_out)
        done_out[j] = eo

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    e_s = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    e_s.record(stream)
    e2e_steps = max(1, min(args.steps, 20))
    s_in.wait_event(e_s)
    s_out.wait_event(e_s)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    e_e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, world, dev)
    e2e_value = tokens_per_step / (e2e_ms * 1e-3)

    if rank != 0:
        return 0
    peaks, peak_kind = measured_peaks()
    th = w.B * w.H * w.T
    alg_bytes = th * gdn_bytes_per_token_head(w.D)
    alg_flops = th * gdn_flops_per_token_head(w.D, w.chunk)
    launches_per_step = launches / args.steps
    kernel_ms = ms / max(launches_per_step, 1.0)
    achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    traffic, traffic_kernel = ncu_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "ms_mean": mean_ms,
        "timing": "median of per-step CUDA-event times on the launching stream",
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,k unit-norm, v~N(0,1), beta=sigmoid(N), g=logsigmoid(N)/16)",
        "config": workload_config(w, world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "alg_bytes_per_launch": alg_bytes, "alg_flops_per_launch": alg_flops,
                     "kernel": traffic_kernel or "scan", "kernel_ms": kernel_ms},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "2 steps in flight: step i+1's input copies and step i-1's output copy overlap step i",
                "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": dict(clk.summary(), window_s=args.clock_window),
    }
    if args.secondary:
        line["secondary"] = secondary(args, dev)
    if not args.no_cpu_baseline and world == 1:
        v, dt, threads = cpu_oracle_sample(inp_cpu, args.ref_heads, w.B, w.H, w.T)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads, "cpu_count": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{args.ref_heads} of {w.B * w.H} heads, full T={w.T} "
                                          f"({dt:.1f} s), scaled to the whole workload"}
    print(json.dumps(line), flush=True)
    return 0


def secondary(args, dev):
    """Device time of the other workloads (not the headline): long-sequence
    GDN, DeltaProduct r=2, the block-masked variant, the GDN backward, and the
    camera branch (prep, scans, backward passes, fused path)."""
    import torch
    from gated_delta_rule_47_gb300 import binding
    from gated_delta_rule_47_gb300.inputs import WORKLOADS
    peaks, _ = measured_peaks()
    out = {}
    steps = max(10, min(args.steps, 50))

    def timeit(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record()
        for i in range(steps):
            fn()
            evs[i + 1].record()
        torch.cuda.synchronize()
        return median_step_ms(evs)[0]

    # the small fp32 workload (CUDA-core path; launch-latency bound, reported only)
    w = WORKLOADS["gdn_tiny_f32"]
    d = {k: v.to(dev) for k, v in w.make().items()}
    o = torch.empty(w.B, w.H, w.T, w.D, dtype=torch.float32, device=dev)
    ms = timeit(lambda: binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], chunk=w.chunk, o=o))
    out[w.name] = {"ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3),
                   "hbm_frac": w.B * w.H * w.T * gdn_bytes_per_token_head(w.D, 4, 4) / (ms * 1e-3) / 1e9
                   / peaks["hbm_gbs"], "dtype": "f32"}

    for name in ("gdn_long_b1h32t32768d128_bf16", "deltaproduct_r2_b4h16t4096d128_bf16"):
        w = WORKLOADS[name]
        d = {k: v.to(dev) for k, v in w.make().items()}
        o = torch.empty(w.B, w.H, w.T, w.D, dtype=torch.bfloat16, device=dev)
        wsw = make_workspace(binding, w, dev)
        if w.kind == "gdn":
            fn = lambda: binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], chunk=w.chunk, o=o,
                                               workspace=wsw)
            nbytes = w.B * w.H * w.T * gdn_bytes_per_token_head(w.D)
        else:
            fn = lambda: binding.deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"],
                                                        chunk=w.chunk, o=o, workspace=wsw)
            nbytes = w.B * w.H * w.T * (w.D * (1 + 2 * w.r) * 2 + 2 * w.r + 4 + 2 * w.D)
        ms = timeit(fn)
        out[name] = {"ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3),
                     "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        del d, o, wsw
        torch.cuda.empty_cache()
    # the block-masked DeltaProduct variant (WY factors, state chain and output on tcgen05)
    w = WORKLOADS["masked_dp_r2_b4h16t4096d128_bf16"]
    d = {k: v.to(dev) for k, v in w.make().items()}
    o = torch.empty(w.B, w.H, w.T, w.D, dtype=torch.bfloat16, device=dev)
    wsm = torch.empty(binding.masked_deltaproduct_workspace_bytes(w.B, w.H, w.T, w.r, w.D, w.D), dtype=torch.uint8,
                      device=dev)
    ms = timeit(lambda: binding.masked_deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"],
                                                              chunk=w.chunk, o=o, workspace=wsm))
    nbytes = w.B * w.H * w.T * gdn_bytes_per_token_head(w.D)
    out[w.name] = {"ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3),
                   "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                   "path": "WY factors, state chain and output on tcgen05",
                   "launches_per_call": 3}
    # its backward
    gom = torch.randn(w.B, w.H, w.T, w.D, device=dev).to(torch.bfloat16)
    wsmb = torch.empty(binding.load().masked_deltaproduct_chunk_bwd_workspace_bytes(w.B, w.H, w.T, w.r, w.D, w.D, 1),
                       dtype=torch.uint8, device=dev)
    ms = timeit(lambda: binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"],
                                                              gom, workspace=wsmb))
    nbytes = w.B * w.H * w.T * (14 * w.D + 14)  # q, k, v, beta, g, do in; dq, dk, dv, dbeta, dg out
    out["masked_dp_bwd_r2_b4h16t4096d128_bf16"] = {"ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3),
                                                   "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                                   "path": BWD_PATH, "launches_per_call": 4}
    del d, o, wsm, gom, wsmb
    torch.cuda.empty_cache()
    # the chunkwise GDN backward on the headline's shape
    w = WORKLOADS["gdn_b4h16t4096d128_bf16"]
    d = {k: v.to(dev) for k, v in w.make().items()}
    gen = torch.Generator(device=dev).manual_seed(3)
    go = torch.randn(w.B, w.H, w.T, w.D, device=dev, generator=gen).to(torch.bfloat16)
    wsg = torch.empty(binding.gdn_chunk_bwd_workspace_bytes(w.B, w.H, w.T, w.D, w.D), dtype=torch.uint8,
                      device=dev)
    ms = timeit(lambda: binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], go, workspace=wsg))
    nbytes = w.B * w.H * w.T * (14 * w.D + 14)  # q, k, v, beta, g, do in; dq, dk, dv, dbeta, dg out
    out["gdn_bwd_b4h16t4096d128_bf16"] = {"ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3),
                                          "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                          "launches_per_call": 4, "path": BWD_PATH}
    del d, go, wsg
    torch.cuda.empty_cache()
    w = WORKLOADS["cam_b2n32760h16d128_bf16"]
    d = {k: (v.to(dev) if v is not None else None) for k, v in w.make().items()}
    outs = tuple(torch.empty(w.B, w.H, w.T, w.D, dtype=torch.bfloat16, device=dev) for _ in range(3))
    o = torch.empty(w.B, w.H, w.T, w.D, dtype=torch.bfloat16, device=dev)

    def prep():
        return binding.cam_prep_fwd(d["q_raw"], d["k_raw"], d["v_raw"], d["proj_q"], d["proj_kv"],
                                    d["q_norm_w"], d["k_norm_w"], d["rope_cos"], d["rope_sin"], outs=outs)

    pre_ms = timeit(prep)
    C = w.H * w.D
    prep_bytes = w.B * w.T * (6 * C * 2 + 2 * 16 * 4 + 2 * w.H * 4)
    wsc = make_workspace(binding, w, dev)
    scan_ms = timeit(lambda: binding.gdn_chunk_fwd(outs[0], outs[1], outs[2], d["beta"], d["g"],
                                                   chunk=w.chunk, l2norm=True, o=o, workspace=wsc))
    out[w.name] = {"prep_ms": pre_ms, "prep_gbs": prep_bytes / (pre_ms * 1e-3) / 1e9,
                   "prep_hbm_frac": prep_bytes / (pre_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                   "scan_ms": scan_ms, "tokens_per_s": w.B * w.T / ((pre_ms + scan_ms) * 1e-3)}
    # the prep's backward at the same size (gradients of q, k, v out -> raw)
    gq, gk, gv = (torch.randn(w.B, w.H, w.T, w.D, device=dev, dtype=torch.bfloat16) for _ in range(3))
    bwd_ms = timeit(lambda: binding.cam_prep_bwd(d["q_raw"], d["k_raw"], d["proj_q"], d["proj_kv"], gq, gk, gv,
                                                 None, None, d["q_norm_w"], d["k_norm_w"], d["rope_cos"],
                                                 d["rope_sin"]))
    bwd_bytes = w.B * w.T * (2 * C * 2 + 3 * C * 2 + 3 * C * 2 + 2 * 16 * 4)  # raw q, k + 3 grads in, 3 out
    out["cam_prep_bwd_b2n32760h16d128_bf16"] = {"ms": bwd_ms, "gbs": bwd_bytes / (bwd_ms * 1e-3) / 1e9,
                                                "hbm_frac": bwd_bytes / (bwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                                "path": "streamed: persistent CTAs fed by bulk copies"}
    del gq, gk, gv
    # the camera branch's own frame-level scan on the prep output: 21 frames of
    # 30 x 52 tokens, unit-norm q and k, beta / S per token, one decay per frame
    from gated_delta_rule_47_gb300.inputs import frame_gates
    F, S = 21, 30 * 52
    beta_f, decay_f = (x.to(dev) for x in frame_gates(w.B, w.H, F, S, seed=w.seed))
    wsf = torch.empty(binding.cam_scan_workspace_bytes(w.B, w.H, F, S, w.D, w.D), dtype=torch.uint8, device=dev)
    frame_bytes = w.B * w.H * w.T * cam_scan_bytes_per_token_head(w.D)
    res = {}
    for rev in (False, True):
        ms = timeit(lambda: binding.cam_scan_fwd(outs[0], outs[1], outs[2], beta_f, decay_f, l2norm=True, o=o,
                                                 workspace=wsf, reverse=rev))
        res["reverse" if rev else "forward"] = {
            "ms": ms, "gbs": frame_bytes / (ms * 1e-3) / 1e9,
            "hbm_frac": frame_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "tokens_per_s_with_prep": w.B * w.T / ((pre_ms + ms) * 1e-3)}
    out["cam_frames_b2f21s1560h16d128_bf16"] = dict(res, alg_bytes=frame_bytes, launches_per_call=3)
    # the frame scan's backward (CUDA cores, fp32), on the same inputs
    gob = torch.randn(w.B, w.H, w.T, w.D, device=dev, dtype=torch.bfloat16)
    wsb = torch.empty(binding.load().cam_scan_bwd_workspace_bytes(w.B, w.H, F, S, w.D, w.D, 1), dtype=torch.uint8,
                      device=dev)
    bms = timeit(lambda: binding.cam_scan_bwd(outs[0], outs[1], outs[2], beta_f, decay_f, gob, l2norm=True,
                                              workspace=wsb))
    out["cam_frames_bwd_b2f21s1560h16d128_bf16"] = {"ms": bms, "tokens_per_s": w.B * w.T / (bms * 1e-3),
                                                    "path": "tcgen05 for the frame products, the chains and the token gradients"}
    del gob, wsb
    # the prep fused into the frame scan: raw q, k, v in, o out, one call
    wsx = torch.empty(binding.cam_prep_scan_workspace_bytes(w.B, w.T, w.H, w.D, F), dtype=torch.uint8, device=dev)
    C = w.H * w.D
    fused_bytes = w.B * w.T * (3 * C * 2 + 2 * 16 * 4 + C * 2 + w.H * 2)
    ms = timeit(lambda: binding.cam_prep_scan_fwd(d["q_raw"], d["k_raw"], d["v_raw"], d["proj_q"], d["proj_kv"],
                                                  beta_f, decay_f, d["q_norm_w"], d["k_norm_w"], rope_base=10000.0,
                                                  o=o, workspace=wsx))
    out["cam_prep_frames_fused_b2n32760h16d128_bf16"] = {
        "ms": ms, "gbs": fused_bytes / (ms * 1e-3) / 1e9, "hbm_frac": fused_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "alg_bytes": fused_bytes, "tokens_per_s": w.B * w.T / (ms * 1e-3),
        "unfused_ms": pre_ms + res["forward"]["ms"], "launches_per_call": 4}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--ref-heads", type=int, default=64,
                    help="heads of the workload the CPU oracle runs per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-window", type=float, default=0.6,
                    help="seconds of GPU activity around the timed steps during which clocks are sampled")
    ap.add_argument("--secondary", action=argparse.BooleanOptionalAction, default=True)
    args = ap.parse_args()
    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local_rank = env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
