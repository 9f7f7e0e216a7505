"""Throughput of the scaled FP8 linear layer on one GB300 (and N replicas).

Workload: the Llama-2-7B-shaped linears of one transformer block, forward +
dgrad + wgrad, per-tensor delayed scaling (amax history 16, margin 0,
"max"): tokens M = 8192, d = 4096 -> QKV 4096x12288, O 4096x4096,
gate/up 4096x11008, down 11008x4096; X ~ N(0,1) with outlier channels,
W ~ N(0, 0.02^2), dY ~ N(0, (1e-3)^2); E4M3 forward operands, E5M2
gradients, FP32 wgrad buffer.  One step = fp8_linear_fwd + fp8_linear_bwd of
all five linears (every quantiser, GEMM and scale update of the path).

value       = sum over linears of 6*M*N*K / step time (TFLOP/s), inputs
              resident in HBM, L2 flushed (256 MiB write) before each step.
e2e         = the same through the public API with pinned host buffers:
              H2D of X, W, dY and D2H of Y, dX, dW inside the timed region.
roofline    = the dominant kernel (the FP8 GEMM): GEMM FLOPs / GEMM time,
              from CUDA events around each GEMM of a component-wise pass of
              the same steps, against 2x the measured bf16 dense peak.
quantize    = the quantiser kernels' algorithmic bytes / their time against
              the measured HBM copy bandwidth.
cpu_baseline= the CPU oracle on a bounded sample of the same step.

`--impl reference` times the CPU oracle (the only reference this method has)
on the same workload; see the module docstring of oracle/.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

TOKENS = 8192
LINEARS = [("qkv", 4096, 12288), ("o", 4096, 4096), ("gate", 4096, 11008),
           ("up", 4096, 11008), ("down", 11008, 4096)]
WORKLOAD = ("llama2-7b block linears fwd+dgrad+wgrad, per-tensor delayed scaling "
            "(history 16, margin 0, max), tokens 8192")
METRIC = "FP8 linear fwd+bwd TFLOP/s and quantize GB/s, as fraction of GB300 peak"
FLUSH_BYTES = 256 << 20
LAUNCHES_PER_LINEAR = 8   # this library's kernels per linear in one fwd + bwd step


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _flops_step():
    return sum(6.0 * TOKENS * n * k for _, k, n in LINEARS)


def _gemm_alg_bytes():
    """Mean algorithmic DRAM bytes per GEMM launch of the step: both FP8
    operands read once, the output written once (FP32 accumulation: read
    and written)."""
    tot = 0.0
    for _, M, N, K, _, out, _ in step_gemms():
        tot += M * K + N * K + (2 * M * N if out == "bf16" else 8 * M * N)
    return tot / len(step_gemms())


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        out_dir = os.environ.get("FP8_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out_dir, f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- GPU arm

def run_gpu(args):
    import scaled_fp8_linear_gb300 as F

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    F.lib()
    hbm_gbs, bf16_burst, bf16_sust, peak_kind = _peaks()
    fp8_peak = 2.0 * bf16_sust   # FP8 dense = 2x bf16 dense (nominal ratio), sustained figure

    recipe = F.Recipe(F.SCALING_DELAYED, history_len=16, margin=0, amax_algo=F.AMAX_MAX)
    layers, Ws, Xs, dYs, Ys, dXs, dWs = [], [], [], [], [], [], []
    for li, (name, K, N) in enumerate(LINEARS):
        layers.append(F.Fp8Linear(TOKENS, N, K, recipe, device=dev))
        Ws.append(synthetic.normal((N, K), 0.02, seed=1000 + li, device=dev))
        n_out = 43 if K == 11008 else 16
        Xs.append([synthetic.with_outlier_channels((TOKENS, K), 1.0, n_out, 50.0,
                                                    seed=10 * li + s, device=dev) for s in range(2)])
        dYs.append([synthetic.normal((TOKENS, N), 1e-3, seed=500 + 10 * li + s, device=dev)
                    for s in range(2)])
        Ys.append(torch.empty(TOKENS, N, dtype=torch.bfloat16, device=dev))
        dXs.append(torch.empty(TOKENS, K, dtype=torch.bfloat16, device=dev))
        dWs.append(torch.zeros(N, K, dtype=torch.float32, device=dev))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(s):
        for li in range(len(LINEARS)):
            L = layers[li]
            L.forward(Xs[li][s % 2], Ws[li], Y=Ys[li])
            L.backward(dYs[li][s % 2], dX=dXs[li], dW=dWs[li], accumulate_dW=True)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for s in range(args.warmup):
        step(s)
    barrier()

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.5)                                 # let the sampler start before the region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    for s in range(args.steps):
        flush.fill_(float(s))                       # evict L2 between steps (untimed)
        ev[s][0].record(stream)
        step(args.warmup + s)
        ev[s][1].record(stream)
    barrier()
    ms = [a.elapsed_time(b) for a, b in ev]
    clk = clocks.stop()
    assert F.fp8_device_status() == 0, "a kernel reported a timeout"
    t_ms = sum(ms)
    if world > 1:
        from scaled_fp8_linear_gb300.distributed import max_over_ranks
        t_ms = max_over_ranks(t_ms, device=dev)
    flops = _flops_step() * args.steps * world
    value = flops / (t_ms * 1e-3) / 1e12

    # component-wise pass of the same steps: events around each kernel group
    comp = component_pass(F, layers, Xs, dYs, Ws, Ys, dXs, dWs, flush, args, stream)

    e2e = e2e_pass(F, recipe, dev, args, stream) if rank == 0 else None
    small = small_case_pass(F, dev, stream) if rank == 0 else None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    if rank != 0:
        return
    gemm_tflops = comp["gemm_flops"] / (comp["gemm_ms"] * 1e-3) / 1e12
    quant_gbs = comp["quant_bytes"] / (comp["quant_ms"] * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8(e4m3/e5m2)xfp8->fp32acc", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": TOKENS,
                   "linears": {n: [k, n_] for n, k, n_ in LINEARS},
                   "recipe": "HYBRID delayed, history 16, margin 0, amax max",
                   "backward_operands": "forward codes read MN-major (no transposed copies)",
                   "l2": "flushed (256 MiB write) before every timed step",
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "roofline": {"bound": "tensor", "kernel": "gemm_pair_kernel (tcgen05.mma.cta_group::2 kind::f8f6f4)",
                     "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                     "peak_source": f"{peak_kind}: 2 x bf16_tflops_sustained (FP8/BF16 nominal 2x)",
                     "traffic": _gemm_traffic(),
                     "traffic_unit": "DRAM bytes per GEMM launch (ncu, mean of the step's 15)",
                     "algorithmic_bytes_per_launch": round(_gemm_alg_bytes())},
        "quantize": {"achieved_gbs": round(quant_gbs, 1), "peak_gbs": hbm_gbs,
                     "frac": round(quant_gbs / hbm_gbs, 4), "peak_source": f"{peak_kind} hbm_gbs"},
        "kernels_ms_per_step": {k: round(v / comp["steps"], 4) for k, v in comp["by_kind"].items()},
        "component_pass_ms_per_step": round(comp["total_ms"] / comp["steps"], 4),
        # per linear and step: forward = amax zeroing, X and W cast (one launch),
        # GEMM, X/W scale update; backward = amax zeroing, dY cast, grouped
        # dgrad + wgrad GEMM, dY scale update (the ncu launch list agrees)
        "gpu_launches": LAUNCHES_PER_LINEAR * len(LINEARS) * args.steps,
        "e2e": e2e,
        "small_case": small,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(out))


def component_pass(F, layers, Xs, dYs, Ws, Ys, dXs, dWs, flush, args, stream):
    """The steps of fp8_linear_fwd/bwd issued as the individual C-ABI calls
    (same kernels, same order) with CUDA events around each call, to split
    the step time between GEMMs, quantisers and scale updates."""
    by_kind = {"gemm": 0.0, "quantize": 0.0, "update_scale": 0.0}
    gemm_flops = quant_bytes = 0.0
    total = 0.0
    pending = []

    def timed(kind, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        pending.append((kind, a, b))

    n_steps = min(args.steps, 20)
    for s in range(n_steps):
        flush.fill_(float(s))
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for li, (name, K, N) in enumerate(LINEARS):
            L = layers[li]
            M = TOKENS
            X, W, dY = Xs[li][s % 2], Ws[li], dYs[li][s % 2]
            am = L.amax
            tr = L.x_qt is not None   # transposed copies kept: K-major backward operands
            timed("quantize", lambda: F.fp8_quantize(X, F.E4M3, scale=L.scale[0:1], q=L.x_q,
                                                     q_t=L.x_qt, amax_out=am[0:1]))
            timed("quantize", lambda: F.fp8_quantize(W, F.E4M3, scale=L.scale[1:2], q=L.w_q,
                                                     q_t=L.w_qt, amax_out=am[1:2]))
            timed("gemm", lambda: F.fp8_gemm(L.x_q, F.E4M3, L.w_q, F.E4M3, L.scale_inv[0:1],
                                             L.scale_inv[1:2], D=Ys[li]))
            timed("update_scale", lambda: [F.fp8_update_scale(
                am[r:r + 1], L.history[r], L.pos[r:r + 1], 16, F.AMAX_MAX, F.E4M3, 0, False,
                L.scale[r:r + 1], L.scale_inv[r:r + 1]) for r in (0, 1)])
            dyq = L.workspace[:M * N].view(M, N)
            off = (M * N + 255) // 256 * 256          # dY_q^T follows dY_q, 256-byte aligned
            dyqt = L.workspace[off:off + M * N].view(N, M) if tr else None
            timed("quantize", lambda: F.fp8_quantize(dY, F.E5M2, scale=L.scale[2:3], q=dyq,
                                                     q_t=dyqt, amax_out=am[2:3]))
            # dgrad and wgrad in one grouped launch, as fp8_linear_bwd issues them:
            # without transposed copies they read W_q, dY_q and X_q as stored
            timed("gemm", lambda: F.fp8_gemm_group(
                dict(A=dyq, fa=F.E5M2, B=L.w_qt if tr else L.w_q, fb=F.E4M3,
                     scale_inv_a=L.scale_inv[2:3], scale_inv_b=L.scale_inv[1:2], D=dXs[li],
                     layout=F.LAYOUT_TN if tr else F.LAYOUT_B_KN),
                dict(A=dyqt if tr else dyq, fa=F.E5M2, B=L.x_qt if tr else L.x_q, fb=F.E4M3,
                     scale_inv_a=L.scale_inv[2:3], scale_inv_b=L.scale_inv[0:1], out=F.OUT_F32,
                     D=dWs[li], accumulate=True,
                     layout=F.LAYOUT_TN if tr else F.LAYOUT_KM_KN)))
            timed("update_scale", lambda: F.fp8_update_scale(
                am[2:3], L.history[2], L.pos[2:3], 16, F.AMAX_MAX, F.E5M2, 0, False,
                L.scale[2:3], L.scale_inv[2:3]))
            gemm_flops += 6.0 * M * N * K
            # quantiser bytes: bf16 read (2 B) + q write (1 B) (+ q_t write (1 B)) per element
            quant_bytes += (4.0 if tr else 3.0) * (M * K + N * K + M * N)
        t1.record(stream)
        pending.append(("__step", t0, t1))
    torch.cuda.synchronize()
    for kind, a, b in pending:
        ms = a.elapsed_time(b)
        if kind == "__step":
            total += ms
        else:
            by_kind[kind] += ms
    return {"by_kind": by_kind, "gemm_ms": by_kind["gemm"], "quant_ms": by_kind["quantize"],
            "gemm_flops": gemm_flops, "quant_bytes": quant_bytes, "total_ms": total,
            "steps": n_steps}


def small_case_pass(F, dev, stream, iters=200):
    """The small forward case (X 256 x 512 with outliers, W 512 x 512, dynamic
    scaling): latency of fp8_linear_fwd and of fwd + bwd, issued eagerly and
    replayed from a CUDA graph of the same calls.  Launch-bound at this size
    (~12 launches per fwd + bwd), so it reports microseconds, not a roofline."""
    M, K, N = 256, 512, 512
    layer = F.Fp8Linear(M, N, K, F.Recipe(F.SCALING_DYNAMIC), device=dev)
    X = synthetic.with_outlier_entries((M, K), 1.0, 0.001, 50.0, seed=0, device=dev)
    W = synthetic.normal((N, K), 0.02, seed=1, device=dev)
    dY = synthetic.normal((M, N), 1e-3, seed=2, device=dev)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    dW = torch.zeros(N, K, dtype=torch.float32, device=dev)

    def fwd():
        layer.forward(X, W, Y=Y)

    def fwd_bwd():
        layer.forward(X, W, Y=Y)
        layer.backward(dY, dX=dX, dW=dW)

    def timed(fn):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / iters

    out = {"workload": "small forward: X 256x512 (0.1% entries x50), W 512x512, dynamic scaling",
           "fwd_us": round(timed(fwd), 2), "fwd_bwd_us": round(timed(fwd_bwd), 2)}
    graphs = {}
    for name, fn in (("fwd", fwd), ("fwd_bwd", fwd_bwd)):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()                                   # warm: kernel attributes, tensor maps
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=side):
                fn()
        stream.wait_stream(side)
        graphs[name] = g
    out["graph_fwd_us"] = round(timed(graphs["fwd"].replay), 2)
    out["graph_fwd_bwd_us"] = round(timed(graphs["fwd_bwd"].replay), 2)
    out["graph_fwd_bwd_tflops"] = round(6.0 * M * N * K / (out["graph_fwd_bwd_us"] * 1e-6) / 1e12, 3)
    out["l2"] = "resident (1.3 MB of operands)"
    assert F.fp8_device_status() == 0
    return out


def e2e_pass(F, recipe, dev, args, stream):
    """Public API with host buffers.  Per step and linear: H2D of X, W, dY from
    pinned memory, fp8_linear_fwd + fp8_linear_bwd, D2H of Y, dX, dW -- all
    inside the timed region.  Copies run on their own streams so that the
    next linear's inputs arrive and the previous one's results leave while
    the current linear computes (two device buffer sets, event-ordered,
    pipelined across step boundaries as a training loop would be)."""
    nl = len(LINEARS)
    h_in, h_out, layers = [], [], []
    for li, (name, K, N) in enumerate(LINEARS):
        n_out = 43 if K == 11008 else 16
        h_in.append((synthetic.with_outlier_channels((TOKENS, K), 1.0, n_out, 50.0, seed=li).pin_memory(),
                     synthetic.normal((N, K), 0.02, seed=1000 + li).pin_memory(),
                     synthetic.normal((TOKENS, N), 1e-3, seed=500 + li).pin_memory()))
        h_out.append((torch.empty(TOKENS, N, dtype=torch.bfloat16).pin_memory(),
                      torch.empty(TOKENS, K, dtype=torch.bfloat16).pin_memory(),
                      torch.empty(N, K, dtype=torch.float32).pin_memory()))
        layers.append(F.Fp8Linear(TOKENS, N, K, recipe, device=dev))
    kmax = max(k for _, k, _ in LINEARS)
    nmax = max(n for _, _, n in LINEARS)
    nk = max(n * k for _, k, n in LINEARS)

    def dbuf():
        return {"X": torch.empty(TOKENS * kmax, dtype=torch.bfloat16, device=dev),
                "W": torch.empty(nk, dtype=torch.bfloat16, device=dev),
                "dY": torch.empty(TOKENS * nmax, dtype=torch.bfloat16, device=dev),
                "Y": torch.empty(TOKENS * nmax, dtype=torch.bfloat16, device=dev),
                "dX": torch.empty(TOKENS * kmax, dtype=torch.bfloat16, device=dev),
                "dW": torch.empty(nk, dtype=torch.float32, device=dev)}

    bufs = [dbuf(), dbuf()]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d = sum(t.numel() * t.element_size() for tr in h_in for t in tr)
    d2h = sum(t.numel() * t.element_size() for tr in h_out for t in tr)
    # Linears are numbered across steps (g = step * 5 + li) and alternate
    # between the two device buffer sets, so the loads of the next linear
    # (also across a step boundary) and the drains of the previous one run on
    # the host link while the current one computes.  Each copy waits only for
    # the last user of its own buffer set.
    computed, drained = {}, {}
    counter = [0]

    def run_linear():
        g = counter[0]
        counter[0] += 1
        li = g % nl
        _, K, N = LINEARS[li]
        b = bufs[g % 2]
        loaded = torch.cuda.Event()
        with torch.cuda.stream(h2d_s):
            if g - 2 in computed:
                h2d_s.wait_event(computed.pop(g - 2))      # last reader of this set's inputs
            hx, hw, hdy = h_in[li]
            b["X"][:TOKENS * K].view(TOKENS, K).copy_(hx, non_blocking=True)
            b["W"][:N * K].view(N, K).copy_(hw, non_blocking=True)
            b["dY"][:TOKENS * N].view(TOKENS, N).copy_(hdy, non_blocking=True)
            loaded.record(h2d_s)
        return g, li, K, N, b, loaded

    def compute_and_drain(g, li, K, N, b, loaded):
        stream.wait_event(loaded)
        if g - 2 in drained:
            stream.wait_event(drained.pop(g - 2))          # this set's outputs have left
        Y = b["Y"][:TOKENS * N].view(TOKENS, N)
        dX = b["dX"][:TOKENS * K].view(TOKENS, K)
        dW = b["dW"][:N * K].view(N, K)
        L = layers[li]
        hy, hdx, hdw = h_out[li]
        L.forward(b["X"][:TOKENS * K].view(TOKENS, K), b["W"][:N * K].view(N, K), Y=Y)
        fwd_done = torch.cuda.Event()
        fwd_done.record(stream)
        with torch.cuda.stream(d2h_s):                     # Y leaves while the backward runs
            d2h_s.wait_event(fwd_done)
            hy.copy_(Y, non_blocking=True)
        L.backward(b["dY"][:TOKENS * N].view(TOKENS, N), dX=dX, dW=dW, accumulate_dW=False)
        ev = torch.cuda.Event()
        ev.record(stream)
        computed[g] = ev
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev)
            hdx.copy_(dX, non_blocking=True)
            hdw.copy_(dW, non_blocking=True)
            dev_ev = torch.cuda.Event()
            dev_ev.record(d2h_s)
            drained[g] = dev_ev

    def steps(k):
        """k steps, issued one linear ahead on the load stream."""
        h2d_s.wait_stream(stream)                          # copies start after the start event
        d2h_s.wait_stream(stream)
        pending = run_linear()
        for i in range(k * nl):
            nxt = run_linear() if i + 1 < k * nl else None
            compute_and_drain(*pending)
            pending = nxt
        stream.wait_stream(d2h_s)                          # the last results are on the host
        stream.wait_stream(h2d_s)

    steps(max(1, min(args.warmup, 3)))
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 30))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    steps(n)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    link = _host_link(dev)
    floor_ms = _link_floor_ms(h2d, d2h, link)
    return {"value": round(_flops_step() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": n, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "copies": "pinned host <-> device on two copy streams, overlapped with compute and "
                      "with each other across linears and steps",
            "host_link": link,
            "link_floor_ms": round(floor_ms, 3),
            "link_floor_note": "the time to move h2d and d2h bytes at the link rates measured "
                               "in this run: both directions at their concurrent rates until "
                               "the smaller finishes, the rest at its one-way rate"}


def _link_floor_ms(h2d, d2h, link):
    """Least time to copy h2d bytes in and d2h bytes out over the measured
    link: both directions run at their concurrent rates until one is done,
    then the other continues at its one-way rate."""
    rh, rd = link["h2d_concurrent_gbs"] * 1e9, link["d2h_concurrent_gbs"] * 1e9
    th, td = h2d / rh, d2h / rd
    if th <= td:
        rest = d2h - rd * th
        t = th + rest / (link["d2h_gbs"] * 1e9)
    else:
        rest = h2d - rh * td
        t = td + rest / (link["h2d_gbs"] * 1e9)
    return t * 1e3


def _host_link(dev, mib=1024, reps=3):
    """Pinned host <-> device copy bandwidth of this machine, measured now: H2D
    alone, D2H alone, and both at once on two streams (GB/s, best of reps;
    for the concurrent test each direction is timed on its own stream)."""
    n = mib << 20
    hs = [torch.empty(n, dtype=torch.uint8).pin_memory() for _ in range(2)]
    ds = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(2)]
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            ds[0].copy_(hs[0], non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            hs[1].copy_(ds[1], non_blocking=True)

    def both():
        h2d()
        d2h()

    t_h, t_d, t_b = timed(h2d), timed(d2h), timed(both)
    # each direction's own duration while both run (events on each stream)
    best_h = best_d = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(s1)
        e[2].record(s2)
        h2d()
        d2h()
        e[1].record(s1)
        e[3].record(s2)
        torch.cuda.synchronize()
        best_h = min(best_h, e[0].elapsed_time(e[1]) * 1e-3)
        best_d = min(best_d, e[2].elapsed_time(e[3]) * 1e-3)
    out = {"h2d_gbs": round(n / t_h / 1e9, 1), "d2h_gbs": round(n / t_d / 1e9, 1),
           "both_gbs": round(2 * n / t_b / 1e9, 1),
           "h2d_concurrent_gbs": round(n / best_h / 1e9, 1),
           "d2h_concurrent_gbs": round(n / best_d / 1e9, 1), "bytes_per_test": n}
    del hs, ds
    return out


# ------------------------------------------------------------- CPU oracle

def _oracle_sample_step(rows_per_gemm, inputs, states, linears=None):
    """One step of the oracle on a bounded sample: whole-tensor amax, scale
    update and quantisation of X, W, dY for every linear in `linears` (all
    five by default; the oracle's linear_fwd / linear_bwd), and
    `rows_per_gemm` full output rows of each of their GEMMs.  Returns the
    FLOPs of the sampled GEMM rows."""
    import numpy as np
    import oracle
    flops = 0.0
    for li, (name, K, N) in enumerate(LINEARS):
        if linears is not None and li not in linears:
            continue
        bx, bw, bdy = inputs[li]
        st, rec = states[li]
        rows = np.arange(rows_per_gemm)
        oracle.linear_fwd(bx, bw, rec, st, rows=rows)
        oracle.linear_bwd(bdy, rec, st, rows_dx=rows, rows_dw=rows)
        flops += 2.0 * rows_per_gemm * (N * K + K * N + K * TOKENS)
    return flops


def _oracle_inputs():
    import oracle
    inputs, states = [], []
    rec = oracle.Recipe(scaling=oracle.SCALING_DELAYED, history_len=16)
    for li, (name, K, N) in enumerate(LINEARS):
        n_out = 43 if K == 11008 else 16
        X = synthetic.with_outlier_channels((TOKENS, K), 1.0, n_out, 50.0, seed=10 * li)
        W = synthetic.normal((N, K), 0.02, seed=1000 + li)
        dY = synthetic.normal((TOKENS, N), 1e-3, seed=500 + 10 * li)
        inputs.append((synthetic.bf16_bits(X), synthetic.bf16_bits(W), synthetic.bf16_bits(dY)))
        states.append((oracle.LinearState(rec), rec))
    return inputs, states


def cpu_baseline(args):
    import oracle
    inputs, states = _oracle_inputs()
    rows = args.cpu_rows
    t0 = time.perf_counter()
    flops = _oracle_sample_step(rows, inputs, states)
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": (f"one step: whole-tensor amax/scale/quantise(+transpose) of X, W, dY of the "
                       f"5 linears, and {rows} full output rows of each of the 15 GEMMs "
                       f"(fp64 accumulation); value = sampled GEMM FLOPs / wall time")}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    inputs, states = _oracle_inputs()
    rows = args.ref_rows
    # a step over all five linears takes seconds on the host cores; beyond 20
    # steps each step samples one linear, in turn, so that the whole run
    # stays within a few minutes
    per_step = len(LINEARS) if args.steps + args.warmup <= 20 else 1
    pick = lambda i: None if per_step == len(LINEARS) else {i % len(LINEARS)}
    for i in range(args.warmup):
        _oracle_sample_step(rows, inputs, states, pick(i))
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(args.steps):
        flops += _oracle_sample_step(rows, inputs, states, pick(i))
    dt = time.perf_counter() - t0
    v = flops / dt / 1e12
    which = "the 5 linears" if per_step == len(LINEARS) else "one linear (in turn)"
    sample = (f"per step: whole-tensor amax/scale/quantise(+transpose) of X, W, dY of {which} "
              f"and {rows} full output rows of each of its GEMMs; value = sampled GEMM FLOPs / "
              f"wall time")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": TOKENS,
                   "linears": {n: [k, n_] for n, k, n_ in LINEARS}},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def run_quantize_sweep(F, args, dev, flush):
    """The quantizer sweep: n = 2^20 .. 2^30 bf16 elements as [n/4096 x 4096]
    and [n/8192 x 8192], t_3-distributed, E4M3 and E5M2, with and without the
    fused transpose, in two modes:
      stale:   one cast with a fixed scale and the fused amax
               (2 + 1 (+1) bytes per element);
      dynamic: amax pass, scale update, then the cast with the new scale
               (2 + 2 + 1 (+1) bytes per element).
    One JSON line per case; L2 flushed before every timed iteration."""
    hbm_gbs = _peaks()[0]
    stream = torch.cuda.current_stream()
    for log2n in range(20, 31, 2):
        n = 1 << log2n
        for width in (4096, 8192):
            rows = n // width
            x = synthetic.student_t((rows, width), 3, 1.0, seed=log2n, device=dev)
            q = torch.empty(rows, width, dtype=torch.uint8, device=dev)
            qt = torch.empty(width, rows, dtype=torch.uint8, device=dev)
            am = torch.empty(1, dtype=torch.float32, device=dev)
            scale = torch.ones(1, dtype=torch.float32, device=dev)
            scale_inv = torch.ones(1, dtype=torch.float32, device=dev)
            hist = torch.zeros(1, dtype=torch.float32, device=dev)
            pos = torch.zeros(1, dtype=torch.int32, device=dev)
            for fname, fmt in (("e4m3", F.E4M3), ("e5m2", F.E5M2)):
                for transpose in (False, True):
                    qt_arg = qt if transpose else None
                    for mode in ("stale", "dynamic"):
                        if mode == "stale":
                            def call():
                                F.fp8_quantize(x, fmt, scale=scale, q=q, q_t=qt_arg, amax_out=am)
                            per_elem = 3 + (1 if transpose else 0)
                        else:
                            def call():
                                F.fp8_amax(x, am)
                                F.fp8_update_scale(am, hist, pos, 1, F.AMAX_MOST_RECENT, fmt, 0,
                                                   False, scale, scale_inv)
                                F.fp8_quantize(x, fmt, scale=scale, q=q, q_t=qt_arg)
                            per_elem = 5 + (1 if transpose else 0)
                        for _ in range(3):
                            call()
                        iters = args.iters
                        ev = [(torch.cuda.Event(enable_timing=True),
                               torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
                        for i in range(iters):
                            flush.fill_(float(i))
                            ev[i][0].record(stream)
                            call()
                            ev[i][1].record(stream)
                        torch.cuda.synchronize()
                        ms = sorted(a.elapsed_time(b) for a, b in ev)
                        med = ms[len(ms) // 2]
                        gbs = per_elem * n / (med * 1e-3) / 1e9
                        print(json.dumps({
                            "kernel": "quantize_sweep", "mode": mode, "log2_elements": log2n,
                            "shape": [rows, width], "format": fname, "transpose": transpose,
                            "bytes_per_element": per_elem, "median_ms": round(med, 5),
                            "achieved": round(gbs, 1), "unit": "GB/s", "peak": round(hbm_gbs, 1),
                            "frac": round(gbs / hbm_gbs, 4), "iters": iters,
                            "l2": "flushed before every launch"}), flush=True)
            del x, q, qt
            torch.cuda.empty_cache()
    assert F.fp8_device_status() == 0


def run_kernel(args):
    """Time one kernel of the path on one shape (not the headline number):
    gemm (per-tensor, E4M3 or E5M2 x E4M3, bf16 out), block_gemm (1x128 x
    128x128 scales, bf16 out), quantize (fused amax + cast + transpose,
    stale scale) or quantize_sr (the same with stochastic rounding, a new
    seed per launch).  L2 is flushed before every timed launch."""
    import scaled_fp8_linear_gb300 as F
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    F.lib()
    hbm_gbs, bf16_burst, _, peak_kind = _peaks()
    dims = [int(v) for v in args.shape.split(",")]
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    fa = F.E5M2 if args.fmt == "e5m2" else F.E4M3

    def codes(r, c):
        # random finite FP8 codes: magnitude codes 0x00..0x7B (finite in both formats) | sign
        v = torch.randint(0, 0x7C, (r, c), generator=g, device=dev, dtype=torch.int32)
        v |= torch.randint(0, 2, (r, c), generator=g, device=dev, dtype=torch.int32) << 7
        return v.to(torch.uint8)

    if args.kernel == "gemm_step":
        return run_gemm_step(F, args, dev, codes, flush)
    if args.kernel == "quantize_sweep":
        return run_quantize_sweep(F, args, dev, flush)
    if args.kernel == "block_step":
        return run_block_step(F, args, dev, flush)
    if args.kernel == "llama70b_step":
        return run_llama70b_step(F, args, dev, flush)
    if args.kernel in ("gemm", "block_gemm"):
        M, N, K = dims
        lay = {"tn": F.LAYOUT_TN, "b_kn": F.LAYOUT_B_KN, "a_km": F.LAYOUT_A_KM,
               "km_kn": F.LAYOUT_KM_KN}[args.layout] if args.kernel == "gemm" else F.LAYOUT_TN
        A = codes(K, M) if lay & F.LAYOUT_A_KM else codes(M, K)
        B = codes(K, N) if lay & F.LAYOUT_B_KN else codes(N, K)
        D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        if args.kernel == "gemm" and args.f32acc:
            # the wgrad form: FP32 output accumulated into D
            one = torch.ones(1, dtype=torch.float32, device=dev)
            D = torch.zeros(M, N, dtype=torch.float32, device=dev)
            call = lambda: F.fp8_gemm(A, fa, B, F.E4M3, one, one, D=D, out=F.OUT_F32,
                                      accumulate=True, layout=lay)
        elif args.kernel == "gemm":
            one = torch.ones(1, dtype=torch.float32, device=dev)
            call = lambda: F.fp8_gemm(A, fa, B, F.E4M3, one, one, D=D, layout=lay)
        elif args.pow2:
            # power-of-two block factors: the block-scaled MMA path
            sa = 2.0 ** torch.randint(-3, 4, (M, K // 128), generator=g, device=dev).float()
            sb = 2.0 ** torch.randint(-3, 4, (N // 128, K // 128), generator=g, device=dev).float()
            call = lambda: F.fp8_gemm(A, F.E4M3, B, F.E4M3, sa, sb, F.GRAN_1x128 | F.SCALE_POW2,
                                      F.GRAN_128x128 | F.SCALE_POW2, D=D)
        else:
            sa = torch.rand(M, K // 128, generator=g, device=dev) + 0.5
            sb = torch.rand(N // 128, K // 128, generator=g, device=dev) + 0.5
            call = lambda: F.fp8_gemm(A, F.E4M3, B, F.E4M3, sa, sb, F.GRAN_1x128,
                                      F.GRAN_128x128, D=D)
        work, unit, peak = 2.0 * M * N * K, "TFLOP/s", 2.0 * bf16_burst
    else:
        R, C = dims
        x = synthetic.student_t((R, C), 3, 1.0, seed=1, device=dev)
        q = torch.empty(R, C, dtype=torch.uint8, device=dev)
        qt = torch.empty(C, R, dtype=torch.uint8, device=dev)
        am = torch.empty(1, dtype=torch.float32, device=dev)
        one = torch.ones(1, dtype=torch.float32, device=dev)
        gran = {"tensor": F.GRAN_TENSOR, "1x128": F.GRAN_1x128, "128x128": F.GRAN_128x128,
                "row": F.GRAN_ROW}[args.gran]
        transpose = not args.no_transpose
        qt_arg = qt if transpose else None
        # algorithmic bytes: bf16 read, codes (and transposed codes), scale arrays
        work = (2.0 + (2.0 if transpose else 1.0)) * R * C
        if args.kernel == "quantize_sr":
            seed = iter(range(1, 1 << 30))
            call = lambda: F.fp8_quantize_sr(x, fa, one, next(seed), 0, q=q, q_t=qt_arg, amax_out=am)
        elif gran == F.GRAN_TENSOR:
            call = lambda: F.fp8_quantize(x, fa, scale=one, q=q, q_t=qt_arg, amax_out=am)
        else:
            s1 = torch.empty(F._scale_shape(gran, R, C), dtype=torch.float32, device=dev)
            st_ = None
            if transpose:
                st_ = torch.empty(F._scale_shape_t(gran, R, C), dtype=torch.float32, device=dev)
                work += 4.0 * st_.numel()
            work += 4.0 * s1.numel()
            call = lambda: F.fp8_quantize(x, fa, gran, q=q, q_t=qt_arg, scale_inv_blocks=s1,
                                          scale_inv_blocks_t=st_)
        unit, peak = "GB/s", hbm_gbs
    for _ in range(args.warmup):
        call()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.iters)]
    for i in range(args.iters):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    med = ms[len(ms) // 2]
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    ach = work / (med * 1e-3) / scale
    extra = {}
    if args.kernel in ("quantize", "quantize_sr"):
        extra = {"granularity": args.gran, "transpose": not args.no_transpose}
    if args.kernel == "block_gemm":
        extra = {"factors": "power of two (block-scaled MMA)" if args.pow2
                 else "fp32 (per-128-K promotion)"}
    if args.kernel == "gemm":
        extra = {"output": "fp32, accumulated" if args.f32acc else "bf16", "layout": args.layout}
    print(json.dumps({"kernel": args.kernel, "shape": dims, "format": args.fmt, **extra,
                      "median_ms": round(med, 4), "min_ms": round(ms[0], 4),
                      "achieved": round(ach, 1), "unit": unit, "peak": round(peak, 1),
                      "frac": round(ach / peak, 4),
                      "peak_source": f"{peak_kind} ({'2 x bf16 burst' if unit == 'TFLOP/s' else 'hbm_gbs'})",
                      "iters": args.iters, "l2": "flushed before every launch"}))


def step_gemms():
    """The 15 GEMMs of one layer step: (name, M, N, K, A format, output,
    layout).  The backward GEMMs read the forward's codes as stored (the
    layer's default): dgrad's B is W_q [N x K], wgrad's A and B are dY_q and
    X_q, both [tokens x ...]."""
    out = []
    for name, K, N in LINEARS:
        out.append((name + ".fwd", TOKENS, N, K, "e4m3", "bf16", 0))
        out.append((name + ".dgrad", TOKENS, K, N, "e5m2", "bf16", 1))
        out.append((name + ".wgrad", N, K, TOKENS, "e5m2", "f32acc", 3))
    return out


def run_gemm_step(F, args, dev, codes, flush):
    """The step's 15 GEMMs with their shapes, formats and output types, each on
    random codes, run once as warm-up and once timed (in that order), with
    the operands of one GEMM on the device at a time."""
    gemms = step_gemms()
    one = torch.ones(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    times = []
    for rep in range(2):
        for name, M, N, K, fa, out, layout in gemms:
            A = codes(K, M) if layout & F.LAYOUT_A_KM else codes(M, K)
            B = codes(K, N) if layout & F.LAYOUT_B_KN else codes(N, K)
            if out == "bf16":
                D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            else:
                D = torch.zeros(M, N, dtype=torch.float32, device=dev)
            flush.fill_(float(rep))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            F.fp8_gemm(A, F.E5M2 if fa == "e5m2" else F.E4M3, B, F.E4M3, one, one,
                       out=F.OUT_BF16 if out == "bf16" else F.OUT_F32, D=D,
                       accumulate=out == "f32acc", layout=layout)
            b.record(stream)
            torch.cuda.synchronize()
            if rep == 1:
                times.append(a.elapsed_time(b))
            del A, B, D
    assert F.fp8_device_status() == 0
    flops = sum(2.0 * M * N * K for _, M, N, K, _, _, _ in gemms)
    print(json.dumps({"kernel": "gemm_step", "gemms": [g[0] for g in gemms],
                      "ms": [round(t, 4) for t in times], "total_ms": round(sum(times), 4),
                      "achieved": round(flops / (sum(times) * 1e-3) / 1e12, 1),
                      "unit": "TFLOP/s"}))


def run_block_step(F, args, dev, flush):
    """One block-scaled linear layer step -- forward, dgrad and wgrad with
    their 1x128 / 128x128 casts, dW accumulated -- on the DeepSeek-style
    shapes, with fp32 or (--pow2) power-of-two block factors.  Inputs are
    seeded synthetic tensors resident on the device; L2 is flushed before
    every timed step."""
    shapes = [(16384, 18432, 7168), (16384, 7168, 18432)]
    if args.shape != "8192,12288,4096":
        shapes = [tuple(int(v) for v in args.shape.split(","))]
    stream = torch.cuda.current_stream()
    for M, N, K in shapes:
        layer = F.Fp8Linear(M, N, K, F.Recipe(F.SCALING_BLOCK, pow2=args.pow2), device=dev)
        X = synthetic.student_t_rows((M, K), 1.0, 3, seed=1, device=dev)
        W = synthetic.student_t_rows((N, K), 0.02, 3, seed=2, device=dev)
        dY = synthetic.normal((M, N), 1e-3, seed=3, device=dev)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dW = torch.zeros(N, K, dtype=torch.float32, device=dev)

        def step():
            layer.forward(X, W, Y=Y)
            layer.backward(dY, dX=dX, dW=dW, accumulate_dW=True)

        for _ in range(args.warmup):
            step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.iters)]
        for i in range(args.iters):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        assert F.fp8_device_status() == 0
        ms = sorted(a.elapsed_time(b) for a, b in ev)
        med = ms[len(ms) // 2]
        print(json.dumps({
            "kernel": "block_step", "shape": [M, N, K],
            "factors": "power of two (block-scaled MMA)" if args.pow2 else "fp32 (per-128-K promotion)",
            "median_ms": round(med, 4), "min_ms": round(ms[0], 4),
            "achieved": round(6.0 * M * N * K / (med * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "work": "6 M N K (fwd + dgrad + wgrad); casts included",
            "iters": args.iters, "l2": "flushed before every step"}), flush=True)
        del layer, X, W, dY, Y, dX, dW
        torch.cuda.empty_cache()


LINEARS_70B = [("qkv", 8192, 10240), ("o", 8192, 8192), ("gate", 8192, 28672),
               ("up", 8192, 28672), ("down", 28672, 8192)]


def run_llama70b_step(F, args, dev, flush):
    """The Llama-2-70B-shaped block linears (4096 tokens, d = 8192, GQA QKV
    8192 -> 10240, O, gate/up 8192 -> 28672, down 28672 -> 8192) through
    fp8_linear_fwd + fp8_linear_bwd with per-tensor dynamic scaling, dW
    accumulated in FP32.  Seeded synthetic inputs resident on the device
    (X with outlier channels, W ~ N(0, 0.02), dY ~ N(0, 1e-3)); L2 flushed
    before every timed step."""
    tokens = 4096
    recipe = F.Recipe(F.SCALING_DYNAMIC)
    layers, Xs, Ws, dYs, Ys, dXs, dWs = [], [], [], [], [], [], []
    for li, (name, K, N) in enumerate(LINEARS_70B):
        layers.append(F.Fp8Linear(tokens, N, K, recipe, device=dev))
        Xs.append(synthetic.with_outlier_channels((tokens, K), 1.0, max(1, K // 256), 50.0,
                                                  seed=10 * li, device=dev))
        Ws.append(synthetic.normal((N, K), 0.02, seed=1000 + li, device=dev))
        dYs.append(synthetic.normal((tokens, N), 1e-3, seed=500 + li, device=dev))
        Ys.append(torch.empty(tokens, N, dtype=torch.bfloat16, device=dev))
        dXs.append(torch.empty(tokens, K, dtype=torch.bfloat16, device=dev))
        dWs.append(torch.zeros(N, K, dtype=torch.float32, device=dev))

    def step():
        for li in range(len(LINEARS_70B)):
            layers[li].forward(Xs[li], Ws[li], Y=Ys[li])
            layers[li].backward(dYs[li], dX=dXs[li], dW=dWs[li], accumulate_dW=True)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.iters)]
    for i in range(args.iters):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    med = ms[len(ms) // 2]
    flops = sum(6.0 * tokens * N * K for _, K, N in LINEARS_70B)
    print(json.dumps({
        "kernel": "llama70b_step", "tokens": tokens,
        "linears": {n: [k, v] for n, k, v in LINEARS_70B}, "recipe": "dynamic per-tensor, HYBRID",
        "median_ms": round(med, 4), "min_ms": round(ms[0], 4),
        "achieved": round(flops / (med * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
        "work": "6 M N K per linear (fwd + dgrad + wgrad); casts, amax and scale updates included",
        "iters": args.iters, "l2": "flushed before every step"}), flush=True)


def _gemm_traffic():
    """DRAM bytes per GEMM launch of the step (mean over its 15 GEMMs), as
    measured by ncu and recorded in profiles/ together with a hash of the
    GEMM source it was measured on; None if the source has changed since."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_step_traffic.json")) as f:
            rec = json.load(f)
        with open(os.path.join(ROOT, "scaled_fp8_linear_gb300", "csrc", "gemm.cu"), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()
        return rec["bytes_per_launch"] if rec.get("gemm_cu_sha256") == h else None
    except Exception:
        return None


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=32)
    ap.add_argument("--ref-rows", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=["gemm", "block_gemm", "quantize", "quantize_sr",
                                         "quantize_sweep", "gemm_step", "block_step",
                                         "llama70b_step"],
                    help="time one kernel on --shape instead of the layer step")
    ap.add_argument("--shape", default="8192,12288,4096")
    ap.add_argument("--fmt", choices=["e4m3", "e5m2"], default="e4m3")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--gran", choices=["tensor", "1x128", "128x128", "row"], default="tensor",
                    help="--kernel quantize: scale granularity")
    ap.add_argument("--f32acc", action="store_true",
                    help="gemm: FP32 output accumulated into D (the wgrad form)")
    ap.add_argument("--layout", choices=["tn", "b_kn", "a_km", "km_kn"], default="tn",
                    help="gemm: operand storage (b_kn: B as [K x N]; a_km: A as [K x M]; km_kn: both)")
    ap.add_argument("--pow2", action="store_true",
                    help="block_gemm / block_step: power-of-two block factors (the block-scaled MMA path)")
    ap.add_argument("--no-transpose", action="store_true",
                    help="--kernel quantize / quantize_sr: no transposed copy")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.kernel:
        run_kernel(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
