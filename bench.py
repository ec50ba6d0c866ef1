"""Benchmark: LA forward + backward throughput on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: the paper's standalone shape (B=4, H=16, N=4096, D=128, bf16 storage, fp32 accumulation;
"Transformer Based Linear Attention with Optimized GPU Kernel Implementation", sciencestack.ai page,
Figures 2 and 3), synthetic Gaussian inputs (Q, K ~ N(0, 1/D), V, dO ~ N(0, 1)).  One step is one pass
of the whole hot path over one batch: causal forward + backward, then non-causal forward + backward,
so a step processes 2 * B * N tokens.  Every input tensor (67 MB) and the set of them (268 MB) is larger
than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `value` is whole-job tokens/s with inputs resident in HBM; `e2e` is the
same metric through the public API with pinned host buffers copied in and results copied out inside
the timed region; `roofline` is for the call that takes the largest share of the step; `cpu_baseline`
is the fp64 oracle on a bounded sample of heads on this host's cores; `cpu_prefix_baseline` is the oracle's
O(N D^2) running-state form on the whole workload (the "CPU O(N D^2) baseline").  `--impl reference` times that
oracle alone, on the same workload and metric.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

B, H, N, D = 4, 16, 4096, 128
ELEM = 2  # bf16
METRIC = "LA fwd+bwd tokens/s and TFLOP/s, % of roofline, at B=4 H=16 D=128 N=4096"
WORKLOAD = "LA fwd+bwd (causal + non-causal) B=4 H=16 N=4096 D=128 bf16"
PASSES = ("causal", "noncausal")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")


def config_dict():
    return {"workload": WORKLOAD.replace("N=4096", f"N={N}"), "B": B, "H": H, "N": N, "D": D,
            "passes_per_step": list(PASSES),
            "tokens_per_step": 2 * B * N, "l2": "inputs larger than L2 (4 x 67 MB per step), no flush",
            "backward": "la_backward_with_forward_state: per-piece K^T V sums taken from the forward's workspace",
            "seed": 1}


def alg_bytes(kind: str) -> int:
    """Algorithmic HBM bytes of one call: fwd reads Q,K,V and writes O and the fp32 normaliser; bwd reads
    Q,K,V,O,dO and writes dQ,dK,dV."""
    t = B * H * N * D * ELEM
    return 4 * t + 4 * B * H * N if kind == "fwd" else 8 * t


def alg_flops(kind: str) -> int:
    """Algorithmic flops of one call: 4 D^2 per head-row forward (state update + read-out), 10 D^2 backward."""
    return (4 if kind == "fwd" else 10) * D * D * B * H * N


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bwd_la_fwd_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clocks and throttle reasons while the GPU is loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------- CPU baseline ---

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample_step(host, n_heads: int) -> float:
    """The explicit fp64 oracle, as it stands, on the first n_heads heads of the batch: causal and
    non-causal forward + backward.  The 4 * n_heads calls (one head each, single-threaded) run
    concurrently, one per core.  Returns seconds."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from bwd_la_fwd_gb300 import inputs
    f = {k: inputs.to_f64(v.reshape(B * H, N, D)[:n_heads], "bf16") for k, v in host.items()}
    tasks = []
    for h in range(n_heads):
        q, k, v, do = (f[n][h].reshape(1, 1, N, D) for n in ("Q", "K", "V", "dO"))
        for causal in (True, False):
            tasks.append((oracle.forward, (q, k, v, causal), {"threads": 1}))
            tasks.append((oracle.backward, (q, k, v, do, causal), {"threads": 1}))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=len(tasks)) as ex:
        for fut in [ex.submit(fn, *a, **kw) for fn, a, kw in tasks]:
            fut.result()
    return time.perf_counter() - t0


def sample_heads(cores: int) -> int:
    """Heads per oracle sample: four single-threaded calls per head, at most one call per core."""
    return max(1, min(B * H, cores // 4))


def sample_tokens(n_heads: int) -> float:
    """Tokens covered by a sample of n_heads head-sequences over both passes (a token spans H heads)."""
    return 2.0 * n_heads * N / H


def cpu_prefix_baseline(host):
    """The oracle's O(N D^2) running-state form (fp64, C, all host cores), as it stands, on the whole
    workload: causal and non-causal forward + backward of every head."""
    import oracle
    from bwd_la_fwd_gb300 import inputs
    oracle.build()
    f = {k: inputs.to_f64(v, "bf16") for k, v in host.items()}
    t0 = time.perf_counter()
    for causal in (True, False):
        oracle.prefix_forward(f["Q"], f["K"], f["V"], causal)
        oracle.prefix_backward(f["Q"], f["K"], f["V"], f["dO"], causal)
    dt = time.perf_counter() - t0
    return {"value": 2 * B * N / dt, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle prefix form",
            "sample": f"the whole step (all {B * H} heads, both passes, fwd+bwd) in fp64; {dt:.1f} s"}


def cpu_baseline(host):
    import oracle
    oracle.build()
    cores = host_cores()
    n_heads = sample_heads(cores)
    dt = oracle_sample_step(host, n_heads)
    return {"value": sample_tokens(n_heads) / dt, "unit": "tokens/s", "cores": min(cores, 4 * n_heads),
            "kind": "oracle",
            "sample": f"explicit fp64 oracle, causal + non-causal fwd+bwd on {n_heads} of {B * H} heads, one call per core "
                      f"(N={N}, D={D}); {dt:.1f} s"}


# ---------------------------------------------------------------------------------- our arm ---

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, device) -> float:
    """The largest x over the ranks of the job (its time is that of its slowest replica); x alone without
    a process group."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(ms_max: float, world: int) -> float:
    """Whole-job throughput: every replica processes one step of 2 B N tokens in the slowest one's time."""
    return world * 2 * B * N / (ms_max * 1e-3)


def run_ours(args):
    import numpy as np
    import torch

    from bwd_la_fwd_gb300 import inputs, la
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    la.load_library()

    host = inputs.generate(B, H, N, D, seed=1, dtype="bf16")
    pinned = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory() for k, v in host.items()}
    Q, K, V, dO = (pinned[n].to(dev) for n in ("Q", "K", "V", "dO"))
    ws = la.new_workspace(B, H, N, D, True, la.LA_BF16, True, dev)
    outs = {p: {"O": torch.empty_like(Q), "g": torch.empty(B, H, N, device=dev), "dQ": torch.empty_like(Q),
                "dK": torch.empty_like(Q), "dV": torch.empty_like(Q)} for p in PASSES}
    if args.layout == "bnhd":  # every [B,H,N,D] operand as a view of a [B,N,H,D] tensor (strided entry points)
        def bnhd(t):
            return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
        Q, K, V, dO = (bnhd(t) for t in (Q, K, V, dO))
        outs = {p: {k: (bnhd(v) if v.dim() == 4 else v) for k, v in o.items()} for p, o in outs.items()}
    stream = torch.cuda.current_stream()

    def step(evs=None, Q=Q, K=K, V=V, dO=dO, outs=outs):
        for p in PASSES:
            o = outs[p]
            causal = p == "causal"
            if evs is not None:
                evs[p + "_fwd"][0].record(stream)
            la.la_forward(Q, K, V, causal, O=o["O"], normaliser=o["g"], workspace=ws)
            if evs is not None:
                evs[p + "_fwd"][1].record(stream)
                evs[p + "_bwd"][0].record(stream)
            # the backward takes the per-piece state sums the forward just left in `ws` (a training step's
            # saved activations), as la_backward_with_forward_state allows
            la.la_backward(Q, K, V, o["O"], dO, causal, dQ=o["dQ"], dK=o["dK"], dV=o["dV"], workspace=ws,
                           reuse_forward_state=True)
            if evs is not None:
                evs[p + "_bwd"][1].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    sampler = ClockSampler(local)
    if not args.profile:
        sampler.start()
    t_spin = time.time()
    while not args.profile and time.time() - t_spin < 1.0:  # bring clocks up before warm-up (untimed)
        step()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = la.la_get_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {la.la_status_string(st)}")

    calls = [p + s for p in PASSES for s in ("_fwd", "_bwd")]
    per_call = {c: 0.0 for c in calls}
    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = la.la_launch_count()
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev_start.record(stream)
    evsets = []
    for _ in range(args.steps):
        evs = {c: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for c in calls}
        step(evs)
        evsets.append(evs)
    ev_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    launches = la.la_launch_count() - launches0
    sampler.stop()
    st = la.la_get_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after timed region: {la.la_status_string(st)}")
    ms = ev_start.elapsed_time(ev_end) / args.steps
    samples = {c: [evs[c][0].elapsed_time(evs[c][1]) for evs in evsets] for c in calls}
    for c in calls:
        per_call[c] = sum(samples[c]) / args.steps
    per_call_median = {c: statistics.median(samples[c]) for c in calls}
    ms = max_over_ranks(ms, dev)
    value = job_tokens_per_s(ms, world)
    clocks = sampler.summary(t_spin, t_wall1)
    clocks["window"] = "spin-up + warm-up + timed region"
    if args.profile:  # hot path only (for profilers): no end-to-end leg, memory probe or CPU baseline
        return {"profile": True, "ms_per_step": ms, "calls_us": {c: per_call[c] * 1e3 for c in calls},
                "gpu_launches": int(launches)} if rank == 0 else None

    # End to end through the public API, run the way an application pipelines it: every step copies its
    # inputs in from pinned host memory (copy-in stream) and every result back out (copy-out stream) while
    # the compute stream works on the neighbouring step; two device buffer sets alternate.  All copies of
    # every timed step are inside the timed region.
    host_out = {p: {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs[p].items()}
                for p in PASSES}
    dev_in = [{"Q": Q, "K": K, "V": V, "dO": dO}, {n: torch.empty_like(Q) for n in ("Q", "K", "V", "dO")}]
    dev_out = [outs, {p: {k: torch.empty_like(v) for k, v in outs[p].items()} for p in PASSES}]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_steps(n_steps):
        read_done = [None, None]  # compute of the step that last used input set b
        out_done = [None, None]   # copy-out of the step that last used output set b
        for i in range(n_steps):
            b = i % 2
            if read_done[b] is not None:
                s_in.wait_event(read_done[b])
            with torch.cuda.stream(s_in):
                for n in ("Q", "K", "V", "dO"):
                    dev_in[b][n].copy_(pinned[n], non_blocking=True)
            stream.wait_stream(s_in)
            if out_done[b] is not None:
                stream.wait_event(out_done[b])
            step(Q=dev_in[b]["Q"], K=dev_in[b]["K"], V=dev_in[b]["V"], dO=dev_in[b]["dO"], outs=dev_out[b])
            read_done[b] = torch.cuda.Event()
            read_done[b].record(stream)
            s_out.wait_event(read_done[b])
            with torch.cuda.stream(s_out):
                for p in PASSES:
                    for k, v in dev_out[b][p].items():
                        host_out[p][k].copy_(v, non_blocking=True)
            out_done[b] = torch.cuda.Event()
            out_done[b].record(s_out)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    e2e_steps(2)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    e2e_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    st = la.la_get_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after the end-to-end leg: {la.la_status_string(st)}")
    e2e_ms = max_over_ranks(e2e_ms, dev)
    tb = B * H * N * D * ELEM
    h2d = 4 * tb
    d2h = sum(v.numel() * v.element_size() for p in PASSES for v in outs[p].values())

    # peak device memory of one causal fwd + bwd against the O(BHND) I/O floor
    del host_out
    peak = peak_memory(dev)

    if rank != 0:
        return None
    hbm, tfl, peak_kind = measured_peaks()
    dom = max(per_call, key=per_call.get)
    kind = "fwd" if dom.endswith("_fwd") else "bwd"
    achieved = alg_bytes(kind) / (per_call[dom] * 1e-3) / 1e9
    roof = {"bound": "hbm", "call": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": traffic_for(dom), "peak_source": peak_kind,
            "alg_bytes_per_launch": alg_bytes(kind), "avg_us": per_call[dom] * 1e3}
    flops = sum(alg_flops("fwd" if c.endswith("_fwd") else "bwd") for c in calls)
    roof_time = sum(max(alg_bytes(k) / (hbm * 1e9), alg_flops(k) / (tfl * 1e12))
                    for k in ("fwd", "bwd", "fwd", "bwd"))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_dict(),
        "tflops": flops / (ms * 1e-3) / 1e12,
        "roofline_frac_step": roof_time / (ms * 1e-3),
        "calls_us": {c: per_call[c] * 1e3 for c in calls},
        "calls_us_median": {c: per_call_median[c] * 1e3 for c in calls},
        "roofline": roof,
        "e2e": {"value": job_tokens_per_s(e2e_ms, world), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "peak_memory": peak,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(host)
        line["cpu_prefix_baseline"] = cpu_prefix_baseline(host)
    return line


def peak_memory(dev):
    import torch

    from bwd_la_fwd_gb300 import la
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    Q, K, V, dO = (torch.randn(B, H, N, D, device=dev, dtype=torch.bfloat16) for _ in range(4))
    ws = la.new_workspace(B, H, N, D, True, la.LA_BF16, True, dev)
    O, g = la.la_forward(Q, K, V, True, workspace=ws)
    grads = la.la_backward(Q, K, V, O, dO, True, workspace=ws)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated(dev) - base
    floor = 8 * B * H * N * D * ELEM + 4 * B * H * N
    del Q, K, V, dO, ws, O, g, grads
    return {"bytes": int(peak), "floor": int(floor), "ratio": peak / floor,
            "what": "causal fwd+bwd, all tensors and workspace allocated by torch"}


def traffic_for(call: str):
    """DRAM bytes per launch of this call from the committed ncu summary, if taken on the current source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        t = json.load(f)
    if t.get("source_hash") != kernel_source_hash():
        return None
    return t.get("calls", {}).get(call)


# ---------------------------------------------------------------------------- reference arm ---

def run_reference(args):
    from bwd_la_fwd_gb300 import inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    host = inputs.generate(B, H, N, D, seed=1, dtype="bf16")
    cores = host_cores()
    n_heads = args.ref_heads or sample_heads(cores)
    for _ in range(args.warmup):
        oracle_sample_step(host, n_heads)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_sample_step(host, n_heads)
    sec = total / args.steps
    value = sample_tokens(n_heads) / sec
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_dict(),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, 4 * n_heads),
                             "kind": "oracle", "sample": f"each step: explicit fp64 oracle, causal + non-causal fwd+bwd on "
                                       f"{n_heads} of {B * H} heads (N={N}, D={D})"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------- decode workload ---

DEC_B, DEC_H = 256, 16  # sequences decoded together, heads each (D as above, bf16 tokens, fp32 state)


# ------------------------------------------------------------------------------ config sweep ---

SWEEP_CASES = (
    # (name, B, H, N, D, layers, seed): the head-size sweep, the sequence-length sweep and the
    # 24-layer decoder training step, all causal bf16 (the standard shape is the default line's)
    *[(f"head_size_D{d}", 4, 16, 4096, d, 1, 2) for d in (32, 64, 256)],
    *[(f"seq_len_N{n}", 4, 16, n, 128, 1, 3) for n in (1024, 2048, 8192, 16384, 32768, 65536)],
    ("decoder_24_layers", 8, 16, 2048, 128, 24, 4),
)


def shape_roofline_s(b, h, n, d, hbm, tfl):
    """Roofline time (seconds) of one causal forward + backward of one layer at this shape: per call the
    slower of its algorithmic bytes at the HBM peak and its algorithmic flops at the bf16 peak."""
    t = b * h * n * d * ELEM
    fwd = max((4 * t + 4 * b * h * n) / (hbm * 1e9), 4 * d * d * b * h * n / (tfl * 1e12))
    bwd = max(8 * t / (hbm * 1e9), 10 * d * d * b * h * n / (tfl * 1e12))
    return fwd, bwd


def run_sweep(args):
    """The other workloads of the method's measurements, one JSON line each (rank 0 only): causal
    forward + backward per layer, timed with CUDA events (median over the timed steps), against the
    roofline of the shape, with the peak device memory of the case against its I/O floor.  Inputs are
    drawn on the device (torch's generator; Q, K ~ N(0, 1/D), V, dO ~ N(0, 1)); the 24-layer case draws
    every layer's tensors separately and runs the 24 forwards, then the 24 backwards in reverse order,
    each backward reusing its layer's forward sums from that layer's own workspace."""
    import torch

    from bwd_la_fwd_gb300 import la
    rank, _, local = dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    la.load_library()
    hbm, tfl, peak_kind = measured_peaks()
    stream = torch.cuda.current_stream()
    for name, b, h, n, d, layers, seed in SWEEP_CASES:
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        gen = torch.Generator(device=dev).manual_seed(seed)

        def layer():
            x = {}
            for op in ("Q", "K", "V", "dO"):
                t = torch.randn(b, h, n, d, device=dev, generator=gen)
                x[op] = (t.div_(d ** 0.5) if op in ("Q", "K") else t).to(torch.bfloat16)
            x.update({"O": torch.empty_like(x["Q"]), "g": torch.empty(b, h, n, device=dev),
                      "dQ": torch.empty_like(x["Q"]), "dK": torch.empty_like(x["Q"]), "dV": torch.empty_like(x["Q"]),
                      "ws": la.new_workspace(b, h, n, d, True, la.LA_BF16, True, dev)})
            return x

        L = [layer() for _ in range(layers)]

        def step(evs=None):
            for i, x in enumerate(L):
                if evs is not None and i == 0:
                    evs[0].record(stream)
                la.la_forward(x["Q"], x["K"], x["V"], True, O=x["O"], normaliser=x["g"], workspace=x["ws"])
            if evs is not None:
                evs[1].record(stream)
            for x in reversed(L):
                la.la_backward(x["Q"], x["K"], x["V"], x["O"], x["dO"], True, dQ=x["dQ"], dK=x["dK"],
                               dV=x["dV"], workspace=x["ws"], reuse_forward_state=True)
            if evs is not None:
                evs[2].record(stream)

        # working sets below twice the 129 MB L2 are flushed between timed steps (outside the events)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if layers * 8 * b * h * n * d * ELEM < (256 << 20) else None
        torch.cuda.reset_peak_memory_stats(dev)  # from here: the case's tensors, workspaces and what the calls add
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        evsets = []
        for _ in range(args.steps):
            if flush is not None:
                flush.zero_()
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            step(evs)
            evsets.append(evs)
        torch.cuda.synchronize()
        st = [la.la_get_status(x["ws"]) for x in L]
        if any(st):
            raise RuntimeError(f"{name}: device status {[la.la_status_string(s) for s in st if s]}")
        fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evsets)
        bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evsets)
        peak = torch.cuda.max_memory_allocated(dev) - base - (flush.numel() if flush is not None else 0)
        floor = layers * (8 * b * h * n * d * ELEM + 4 * b * h * n)
        rf, rb = shape_roofline_s(b, h, n, d, hbm, tfl)
        step_ms = fwd_ms + bwd_ms
        line = {"workload": "sweep", "case": name, "B": b, "H": h, "N": n, "D": d, "layers": layers,
                "causal": True, "dtype": "bf16", "seed": seed, "steps": args.steps, "warmup": args.warmup,
                "path": ("tensor cores" if d in (32, 64, 128) else
                         "tensor cores, wide kernels (one CTA per head and 128-column output half)" if d == 256
                         else "CUDA cores"),
                "fwd_us": fwd_ms * 1e3, "bwd_us": bwd_ms * 1e3, "step_ms": step_ms,
                "tokens_per_s": b * n / (step_ms * 1e-3),
                "tflops": layers * 14 * d * d * b * h * n / (step_ms * 1e-3) / 1e12,
                "roofline_us": layers * (rf + rb) * 1e6,
                "roofline_frac": layers * (rf + rb) / (step_ms * 1e-3),
                "roofline_frac_fwd": layers * rf / (fwd_ms * 1e-3), "roofline_frac_bwd": layers * rb / (bwd_ms * 1e-3),
                "peak_source": peak_kind, "l2": "flushed between steps" if flush is not None else "inputs larger than L2",
                "peak_memory": {"bytes": int(peak), "floor": int(floor), "ratio": peak / floor}}
        print(json.dumps(line), flush=True)
        del L, step, evsets, flush
    return None


def decode_alg_bytes(bh: int) -> int:
    """HBM bytes of one decode step: the fp32 state S read and written, z and a read and written, the
    counts, q, k, v read and o written (bf16), the fp32 normaliser written."""
    return bh * (2 * D * D * 4 + 4 * D * 4 + 2 * 4 + 4 * D * ELEM + 4)


def run_decode(args):
    """One decode step = one token for each of DEC_B sequences (all DEC_H heads) through la_decode_step,
    from the state of a 4096-token prompt.  The 268 MB state is larger than L2, so every step streams it
    from HBM."""
    import numpy as np
    import torch

    from bwd_la_fwd_gb300 import inputs, la
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    la.load_library()
    bh = DEC_B * DEC_H
    host = inputs.generate(DEC_B, DEC_H, 1, D, seed=2, dtype="bf16")
    tok = {n: torch.from_numpy(host[n].reshape(DEC_B, DEC_H, D).view(np.int16)).view(torch.bfloat16).pin_memory()
           for n in ("Q", "K", "V")}
    q, k, v = (tok[n].to(dev) for n in ("Q", "K", "V"))
    state = la.DecodeState(DEC_B, DEC_H, D, torch.bfloat16, device=dev)
    Kp = torch.randn(DEC_B, DEC_H, N, D, device=dev, dtype=torch.bfloat16) / D ** 0.5
    Vp = torch.randn(DEC_B, DEC_H, N, D, device=dev, dtype=torch.bfloat16)
    la.la_state_append(state, Kp, Vp)  # the prompt (appended once, untimed)
    del Kp, Vp
    o = torch.empty_like(q)
    g = torch.empty((DEC_B, DEC_H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.time()
    for _ in range(max(args.warmup, 3)):
        la.la_decode_step(state, q, k, v, o=o, normaliser=g)
    torch.cuda.synchronize()
    launches0 = la.la_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        la.la_decode_step(state, q, k, v, o=o, normaliser=g)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    launches = la.la_launch_count() - launches0
    ms = e0.elapsed_time(e1) / args.steps
    # end to end: this step's tokens in from pinned host memory, its outputs back, every step
    host_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    host_g = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(args.steps):
        for dst, n in ((q, "Q"), (k, "K"), (v, "V")):
            dst.copy_(tok[n], non_blocking=True)
        la.la_decode_step(state, q, k, v, o=o, normaliser=g)
        host_o.copy_(o, non_blocking=True)
        host_g.copy_(g, non_blocking=True)
    x1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    e2e_ms = x0.elapsed_time(x1) / args.steps
    hbm, _, peak_kind = measured_peaks()
    achieved = decode_alg_bytes(bh) / (ms * 1e-3) / 1e9
    clocks = sampler.summary(t0, t1)
    line = {
        "metric": f"LA decode tokens/s (one token per sequence per step) at B={DEC_B} H={DEC_H} D={D}",
        "value": DEC_B / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"LA decode step B={DEC_B} H={DEC_H} D={D} bf16 tokens, fp32 state after a "
                               f"{N}-token prompt", "l2": "state 268 MB > L2, no flush"},
        "roofline": {"bound": "hbm", "call": "la_decode_step", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic_for("decode_step"), "peak_source": peak_kind,
                     "alg_bytes_per_launch": decode_alg_bytes(bh), "avg_us": ms * 1e3},
        "e2e": {"value": DEC_B / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": 3 * q.numel() * ELEM,
                "d2h_bytes_per_step": o.numel() * ELEM + g.numel() * 4, "ms_per_step": e2e_ms},
        "gpu_launches": int(launches), "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        st = tuple(t.detach().double().cpu().numpy() if t.dtype != torch.int32 else t.cpu().numpy().astype(np.int64)
                   for t in (state.S, state.z, state.a, state.n))
        f = {n: inputs.to_f64(host[n].reshape(DEC_B, DEC_H, D), "bf16") for n in ("Q", "K", "V")}
        reps, c0 = 0, time.perf_counter()
        while reps < 2 or (time.perf_counter() - c0 < 10.0 and reps < 50):
            oracle.decode_step(*st, f["Q"], f["K"], f["V"])
            reps += 1
        sec = (time.perf_counter() - c0) / reps
        line["cpu_baseline"] = {"value": DEC_B / sec, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                                "sample": f"fp64 numpy decode_step over the whole batch, {reps} steps ({sec:.2f} s each)"}
    return line


def main():
    global B, N, D
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-heads", type=int, default=0, help="heads per reference step (default: one per core)")
    ap.add_argument("--seq-len", type=int, default=N, help="N of the attention workload (sweeps; default 4096)")
    ap.add_argument("--head-dim", type=int, default=D, help="D of the attention workload (with --profile; default 128)")
    ap.add_argument("--batch", type=int, default=B, help="B of the attention workload (with --profile; default 4)")
    ap.add_argument("--layout", choices=("bhnd", "bnhd"), default="bhnd",
                    help="attention operands contiguous [B,H,N,D] (default) or views of [B,N,H,D] tensors")
    ap.add_argument("--workload", choices=("attention", "decode", "sweep"), default="attention",
                    help="attention: the fwd+bwd hot path (default); decode: the recurrent decode step; "
                         "sweep: the head-size, sequence-length and 24-layer cases, one line each")
    ap.add_argument("--profile", action="store_true",
                    help="run only warm-up + timed steps of the hot path (for ncu); prints a reduced line")
    args = ap.parse_args()
    N = args.seq_len
    D = args.head_dim
    B = args.batch
    if args.layout != "bhnd" and not args.profile:
        ap.error("--layout bnhd times the hot path only: add --profile")
    if D != 128 and not args.profile:
        ap.error("--head-dim other than 128 times the hot path only: add --profile")
    if B != 4 and not args.profile:
        ap.error("--batch other than 4 times the hot path only: add --profile")
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.workload == "decode":
        line = run_decode(args) if args.impl == "ours" and dist_env()[0] == 0 else None
    elif args.workload == "sweep":
        line = run_sweep(args) if args.impl == "ours" else None
    else:
        line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    rank, world, _ = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
