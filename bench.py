"""Throughput of the scaled FP8 linear layer on one GB300 (and N replicas).

Headline workload: the Llama-2-70B-shaped linears of one transformer block,
forward + dgrad + wgrad, per-tensor dynamic scaling: tokens 4096 per
micro-batch, d = 8192 -> GQA QKV 8192x10240, O 8192x8192, gate/up
8192x28672, down 28672x8192; X ~ N(0,1) with outlier channels (1 in 256
input columns x50), W ~ N(0, 0.02^2) bf16 master weights, dY ~ N(0, 1e-3^2);
E4M3 weights and activations, E5M2 gradients.  One step = two micro-batches
through fp8_linear_fwd + fp8_linear_bwd of all five linears, the FP32 dW
buffers written by the first micro-batch and accumulated by the second (every
amax, scale update, cast and GEMM of the path).

value       = 2 x sum over linears of 6*M*N*K / step time (TFLOP/s), inputs
              resident in HBM, L2 flushed (256 MiB write) before each step.
e2e         = the same steps through the public API from pinned host
              buffers: H2D of W (once per step), X and dY (per micro-batch),
              D2H of Y and dX (per micro-batch) and dW (once per step), all
              inside the timed region.
roofline    = the dominant kernel (the FP8 GEMM): GEMM FLOPs / GEMM time,
              from CUDA events around each GEMM of a component-wise pass of
              the same steps, against 2x the measured bf16 dense burst peak
              (the FP8/BF16 nominal ratio).
quantize    = the quantiser kernels' algorithmic bytes / their time against
              the measured HBM copy bandwidth.
cpu_baseline= the CPU oracle on a bounded sample of the same step.
extra keys  = the other configurations, each timed in this run: the
              Llama-2-7B delayed-scaling step, the block-scaled GEMMs and
              layer steps on the DeepSeek-style shapes (fp32 and power-of-two
              block factors), points of the quantizer sweep, and the small
              forward case.

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

METRIC = "FP8 linear fwd+bwd TFLOP/s and quantize GB/s, as fraction of GB300 peak"
FLUSH_BYTES = 256 << 20
LAUNCHES_PER_LINEAR = 8   # this library's kernels per linear and micro-batch in fwd + bwd

# (name, K = in-features, N = out-features)
LINEARS_7B = [("qkv", 4096, 12288), ("o", 4096, 4096), ("gate", 4096, 11008),
              ("up", 4096, 11008), ("down", 11008, 4096)]
LINEARS_70B = [("qkv", 8192, 10240), ("o", 8192, 8192), ("gate", 8192, 28672),
               ("up", 8192, 28672), ("down", 28672, 8192)]


class Workload:
    """One layer-step configuration: the linears of a transformer block, the
    tokens per micro-batch, the scaling mode and the micro-batches per step
    (with more than one, the first writes dW and the rest accumulate; with
    one, two input sets alternate between steps and dW accumulates)."""

    def __init__(self, key, tokens, linears, scaling, micro_batches, label, recipe_label):
        self.key, self.tokens, self.linears = key, tokens, linears
        self.scaling, self.micro_batches = scaling, micro_batches
        self.label, self.recipe_label = label, recipe_label

    def outlier_channels(self, K):
        # 16 of 4096 input columns (43 of 11008): one in 256
        return 43 if K == 11008 else max(1, K // 256)

    def flops_step(self):
        return self.micro_batches * sum(6.0 * self.tokens * n * k for _, k, n in self.linears)

    def recipe(self, F):
        if self.scaling == "dynamic":
            return F.Recipe(F.SCALING_DYNAMIC)
        return F.Recipe(F.SCALING_DELAYED, history_len=16, margin=0, amax_algo=F.AMAX_MAX)


LLAMA70B = Workload(
    "llama2-70b", 4096, LINEARS_70B, "dynamic", 2,
    "llama2-70b block linears fwd+dgrad+wgrad, per-tensor dynamic scaling, tokens 4096 per "
    "micro-batch, dW accumulated in FP32 over 2 micro-batches",
    "HYBRID (E4M3 fwd, E5M2 grads), per-tensor dynamic (current) scaling, margin 0")
LLAMA7B = Workload(
    "llama2-7b", 8192, LINEARS_7B, "delayed", 1,
    "llama2-7b block linears fwd+dgrad+wgrad, per-tensor delayed scaling (history 16, "
    "margin 0, max), tokens 8192",
    "HYBRID delayed, history 16, margin 0, amax max")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
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
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)], stdout=self.f,
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
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "period_ms": self.period_ms, "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons)}


def _events(n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def _median_ms(ev):
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    return ms[len(ms) // 2], ms[0]


# ------------------------------------------------------------ layer steps

class LayerStep:
    """The device state of one workload: a Fp8Linear per linear, bf16 master
    weights, two sets of X and dY per linear (the two micro-batches of a
    step, or the two input sets that alternate between single-micro-batch
    steps), outputs and FP32 dW buffers."""

    def __init__(self, F, wl: Workload, dev):
        self.F, self.wl, self.dev = F, wl, dev
        self.recipe = wl.recipe(F)
        T = wl.tokens
        self.layers, self.W, self.X, self.dY, self.Y, self.dX, self.dW = [], [], [], [], [], [], []
        for li, (name, K, N) in enumerate(wl.linears):
            self.layers.append(F.Fp8Linear(T, N, K, self.recipe, device=dev))
            self.W.append(synthetic.normal((N, K), 0.02, seed=1000 + li, device=dev))
            self.X.append([synthetic.with_outlier_channels(
                (T, K), 1.0, wl.outlier_channels(K), 50.0, seed=10 * li + s, device=dev)
                for s in range(2)])
            self.dY.append([synthetic.normal((T, N), 1e-3, seed=500 + 10 * li + s, device=dev)
                            for s in range(2)])
            self.Y.append(torch.empty(T, N, dtype=torch.bfloat16, device=dev))
            self.dX.append(torch.empty(T, K, dtype=torch.bfloat16, device=dev))
            self.dW.append(torch.zeros(N, K, dtype=torch.float32, device=dev))

    def passes(self, s):
        """(input set, accumulate dW) of each micro-batch of step s."""
        if self.wl.micro_batches == 1:
            return [(s % 2, True)]
        return [(mb, mb > 0) for mb in range(self.wl.micro_batches)]

    def step(self, s):
        for mb, acc in self.passes(s):
            for li in range(len(self.wl.linears)):
                L = self.layers[li]
                L.forward(self.X[li][mb], self.W[li], Y=self.Y[li])
                L.backward(self.dY[li][mb], dX=self.dX[li], dW=self.dW[li], accumulate_dW=acc)

    def timed_steps(self, first, steps, flush, stream):
        ev = _events(steps)
        for i in range(steps):
            flush.fill_(float(i))                   # evict L2 between steps (untimed)
            ev[i][0].record(stream)
            self.step(first + i)
            ev[i][1].record(stream)
        return ev

    def component_pass(self, flush, stream, n_steps):
        """The steps of fp8_linear_fwd/bwd issued as the individual C-ABI
        calls (the same GEMM calls, the casts and scale updates as separate
        public calls) with CUDA events around each call, to split the step
        time between GEMMs, quantisers and scale updates."""
        F, wl = self.F, self.wl
        by_kind = {"gemm": 0.0, "quantize": 0.0, "update_scale": 0.0}
        gemm_flops = quant_bytes = total = 0.0
        pending = []
        dyn = wl.scaling == "dynamic"
        H = 1 if dyn else 16
        algo = F.AMAX_MOST_RECENT if dyn else F.AMAX_MAX

        def timed(kind, fn):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            pending.append((kind, a, b))

        def cast(L, x, fmt, r, q):
            """One role's cast as the layer's recipe does it: dynamic = amax
            pass, scale update, cast with the new scale (5 B per element);
            delayed = cast with the current scale and the fused amax, then the
            update (3 B per element)."""
            am = L.amax[r:r + 1]
            upd = lambda: F.fp8_update_scale(am, L.history[r], L.pos[r:r + 1], H, algo, fmt, 0,
                                             False, L.scale[r:r + 1], L.scale_inv[r:r + 1])
            if dyn:
                timed("quantize", lambda: F.fp8_amax(x, am))
                timed("update_scale", upd)
                timed("quantize", lambda: F.fp8_quantize(x, fmt, scale=L.scale[r:r + 1], q=q))
                return 5.0 * x.numel(), None
            timed("quantize", lambda: F.fp8_quantize(x, fmt, scale=L.scale[r:r + 1], q=q,
                                                     amax_out=am))
            return 3.0 * x.numel(), upd

        for s in range(n_steps):
            flush.fill_(float(s))
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for mb, acc in self.passes(s):
                for li, (name, K, N) in enumerate(wl.linears):
                    L = self.layers[li]
                    M = wl.tokens
                    X, W, dY = self.X[li][mb], self.W[li], self.dY[li][mb]
                    bx, ux = cast(L, X, F.E4M3, 0, L.x_q)
                    bw, uw = cast(L, W, F.E4M3, 1, L.w_q)
                    timed("gemm", lambda: F.fp8_gemm(L.x_q, F.E4M3, L.w_q, F.E4M3,
                                                     L.scale_inv[0:1], L.scale_inv[1:2],
                                                     D=self.Y[li]))
                    for u in (ux, uw):
                        if u is not None:
                            timed("update_scale", u)
                    dyq = L.workspace[:M * N].view(M, N)
                    bdy, udy = cast(L, dY, F.E5M2, 2, dyq)
                    # dgrad and wgrad in one grouped launch, as fp8_linear_bwd
                    # issues them: W_q, dY_q and X_q read as stored (MN-major)
                    timed("gemm", lambda: F.fp8_gemm_group(
                        dict(A=dyq, fa=F.E5M2, B=L.w_q, fb=F.E4M3, scale_inv_a=L.scale_inv[2:3],
                             scale_inv_b=L.scale_inv[1:2], D=self.dX[li], layout=F.LAYOUT_B_KN),
                        dict(A=dyq, fa=F.E5M2, B=L.x_q, fb=F.E4M3, scale_inv_a=L.scale_inv[2:3],
                             scale_inv_b=L.scale_inv[0:1], out=F.OUT_F32, D=self.dW[li],
                             accumulate=acc, layout=F.LAYOUT_KM_KN)))
                    if udy is not None:
                        timed("update_scale", udy)
                    gemm_flops += 6.0 * M * N * K
                    quant_bytes += bx + bw + bdy
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


def gemm_alg_bytes(wl: Workload):
    """Mean algorithmic DRAM bytes per GEMM launch of a step: both FP8
    operands read once, the output written once (FP32 accumulation: read and
    written)."""
    g = step_gemms(wl)
    return sum(M * K + N * K + (2 * M * N if out == "bf16" else 8 * M * N)
               for _, M, N, K, _, out, _ in g) / len(g)


def _roofline(comp, wl, bf16_burst, bf16_sust, peak_kind):
    ach = comp["gemm_flops"] / (comp["gemm_ms"] * 1e-3) / 1e12
    peak = 2.0 * bf16_burst
    return {"bound": "tensor",
            "kernel": "gemm_pair_kernel (tcgen05.mma.cta_group::2 kind::f8f6f4)",
            "achieved": round(ach, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(ach / peak, 4),
            "peak_source": f"{peak_kind}: 2 x bf16_tflops (burst; FP8/BF16 nominal ratio 2)",
            "frac_of_sustained": round(ach / (2.0 * bf16_sust), 4),
            "traffic": _gemm_traffic(wl.key),
            "traffic_unit": "DRAM bytes per GEMM launch (ncu, mean of the step's GEMM launches)",
            "algorithmic_bytes_per_launch": round(gemm_alg_bytes(wl))}


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
    wl = LLAMA70B
    run = LayerStep(F, wl, dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for s in range(args.warmup):
        run.step(s)
    barrier()

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.5)                                 # let the sampler start before the region
    barrier()
    ev = run.timed_steps(args.warmup, args.steps, flush, stream)
    barrier()
    clk = clocks.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    assert F.fp8_device_status() == 0, "a kernel reported a timeout"
    t_ms = sum(ms)
    if world > 1:
        from scaled_fp8_linear_gb300.distributed import max_over_ranks
        t_ms = max_over_ranks(t_ms, device=dev)
    flops = wl.flops_step() * args.steps * world
    value = flops / (t_ms * 1e-3) / 1e12

    # component-wise pass of the same steps: events around each kernel group
    comp = run.component_pass(flush, stream, min(args.steps, 10))
    del run
    torch.cuda.empty_cache()

    e2e = e2e_pass(F, wl, dev, args, stream) if rank == 0 else None
    e2e_all = e2e_pass(F, wl, dev, args, stream, all_tensors=True) if rank == 0 else None
    extras = {}
    if rank == 0 and not args.no_extras:
        extras["llama2_7b_delayed_step"] = extra_layer_step(F, LLAMA7B, dev, flush, stream,
                                                            bf16_burst, bf16_sust, hbm_gbs,
                                                            peak_kind)
        extras["block_scaled"] = extra_block_scaled(F, dev, flush, stream, bf16_burst)
        extras["quantize_sweep"] = extra_quantize_points(F, dev, flush, stream, hbm_gbs)
        extras["recipe_casts"] = extra_recipe_casts(F, dev, flush, stream, hbm_gbs)
        extras["small_case"] = small_case_pass(F, dev, stream)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    if rank != 0:
        return
    quant_gbs = comp["quant_bytes"] / (comp["quant_ms"] * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8(e4m3/e5m2)xfp8->fp32acc", "data": "synthetic",
        "config": {"workload": wl.label, "tokens_per_micro_batch": wl.tokens,
                   "micro_batches_per_step": wl.micro_batches,
                   "linears": {n: [k, n_] for n, k, n_ in wl.linears},
                   "recipe": wl.recipe_label,
                   "backward_operands": "forward codes read MN-major (no transposed copies)",
                   "l2": "flushed (256 MiB write) before every timed step; inputs larger than L2",
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "roofline": _roofline(comp, wl, bf16_burst, bf16_sust, peak_kind),
        "quantize": {"achieved_gbs": round(quant_gbs, 1), "peak_gbs": hbm_gbs,
                     "frac": round(quant_gbs / hbm_gbs, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_element": "5 (dynamic: amax read 2, cast read 2 + write 1)"},
        "kernels_ms_per_step": {k: round(v / comp["steps"], 4) for k, v in comp["by_kind"].items()},
        "component_pass_ms_per_step": round(comp["total_ms"] / comp["steps"], 4),
        # per linear and micro-batch: forward = amax zeroing, X and W amax (one
        # launch), X and W cast with the fused scale update (one launch), GEMM;
        # backward = amax zeroing, dY amax, dY cast with the fused update,
        # grouped dgrad + wgrad GEMM
        "gpu_launches": LAUNCHES_PER_LINEAR * len(wl.linears) * wl.micro_batches * args.steps,
        "e2e": e2e,
        "e2e_all_tensors": e2e_all,
        "clocks": clk,
        **extras,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args, run_dev=dev)
    print(json.dumps(out))


def extra_layer_step(F, wl, dev, flush, stream, bf16_burst, bf16_sust, hbm_gbs, peak_kind,
                     steps=30, warmup=3):
    """A second layer-step configuration timed like the headline (its own
    component pass for the GEMM and quantiser rates)."""
    run = LayerStep(F, wl, dev)
    for s in range(warmup):
        run.step(s)
    torch.cuda.synchronize()
    ev = run.timed_steps(warmup, steps, flush, stream)
    torch.cuda.synchronize()
    t_ms = sum(a.elapsed_time(b) for a, b in ev)
    comp = run.component_pass(flush, stream, 10)
    assert F.fp8_device_status() == 0
    del run
    torch.cuda.empty_cache()
    quant_gbs = comp["quant_bytes"] / (comp["quant_ms"] * 1e-3) / 1e9
    return {"workload": wl.label, "steps": steps, "ms_per_step": round(t_ms / steps, 4),
            "value": round(wl.flops_step() * steps / (t_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "roofline": _roofline(comp, wl, bf16_burst, bf16_sust, peak_kind),
            "quantize": {"achieved_gbs": round(quant_gbs, 1),
                         "frac": round(quant_gbs / hbm_gbs, 4),
                         "bytes_per_element": "3 (cast with fused amax: read 2 + write 1)"},
            "kernels_ms_per_step": {k: round(v / comp["steps"], 4)
                                    for k, v in comp["by_kind"].items()}}


BLOCK_SHAPES = [(16384, 18432, 7168), (16384, 7168, 18432)]


def extra_block_scaled(F, dev, flush, stream, bf16_burst, iters=10, warmup=3):
    """The block-scaled configuration (1x128 activation and 128x128 weight
    tiles) on both DeepSeek-style shapes, fp32 and power-of-two block
    factors: the forward GEMM alone on the layer's own codes and scales, and
    the whole layer step (casts, forward, dgrad, wgrad with dW accumulated).
    Inputs: rows scaled by |t_3|."""
    peak = 2.0 * bf16_burst
    out = []
    for M, N, K in BLOCK_SHAPES:
        X = synthetic.student_t_rows((M, K), 1.0, 3, seed=1, device=dev)
        W = synthetic.student_t_rows((N, K), 0.02, 3, seed=2, device=dev)
        dY = synthetic.normal((M, N), 1e-3, seed=3, device=dev)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dW = torch.zeros(N, K, dtype=torch.float32, device=dev)
        for pow2 in (False, True):
            layer = F.Fp8Linear(M, N, K, F.Recipe(F.SCALING_BLOCK, pow2=pow2), device=dev)
            p2 = F.SCALE_POW2 if pow2 else 0
            gemm = lambda: F.fp8_gemm(layer.x_q, F.E4M3, layer.w_q, F.E4M3, layer.x_sinv,
                                      layer.w_sinv, F.GRAN_1x128 | p2, F.GRAN_128x128 | p2, D=Y)

            def step():
                layer.forward(X, W, Y=Y)
                layer.backward(dY, dX=dX, dW=dW, accumulate_dW=True)

            res = {"shape": [M, N, K],
                   "factors": "power of two (block-scaled MMA)" if pow2 else
                              "fp32 (per-128-K promotion)"}
            for name, fn, work in (("step", step, 6.0 * M * N * K), ("gemm", gemm, 2.0 * M * N * K)):
                for _ in range(warmup):
                    fn()
                ev = _events(iters)
                for i in range(iters):
                    flush.fill_(float(i))
                    ev[i][0].record(stream)
                    fn()
                    ev[i][1].record(stream)
                torch.cuda.synchronize()
                med, _ = _median_ms(ev)
                ach = work / (med * 1e-3) / 1e12
                res[name] = {"median_ms": round(med, 4), "achieved": round(ach, 1),
                             "unit": "TFLOP/s"}
                if name == "gemm":
                    res[name].update({"kernel": "gemm_mx_kernel" if pow2 else "gemm_block_pair_kernel",
                                      "peak": round(peak, 1), "frac": round(ach / peak, 4)})
                else:
                    res[name]["work"] = "6 M N K; casts included"
            out.append(res)
            del layer
        del X, W, dY, Y, dX, dW
        torch.cuda.empty_cache()
    assert F.fp8_device_status() == 0
    return {"iters": iters, "l2": "flushed before every launch / step",
            "peak_source": "2 x bf16_tflops (burst)", "cases": out}


def extra_quantize_points(F, dev, flush, stream, hbm_gbs, iters=10, warmup=3):
    """Points of the quantizer sweep: n = 2^26, 2^28, 2^30 bf16 elements as
    [n/8192 x 8192], t_3-distributed values, E4M3 and E5M2, with and without
    the fused transpose; a fixed (stale) scale with the fused amax, i.e. one
    pass of 3 (4 with the transpose) algorithmic bytes per element."""
    out = []
    for log2n in (26, 28, 30):
        n = 1 << log2n
        rows, width = n // 8192, 8192
        x = synthetic.student_t((rows, width), 3, 1.0, seed=log2n, device=dev)
        q = torch.empty(rows, width, dtype=torch.uint8, device=dev)
        qt = torch.empty(width, rows, dtype=torch.uint8, device=dev)
        am = torch.empty(1, dtype=torch.float32, device=dev)
        scale = torch.ones(1, dtype=torch.float32, device=dev)
        for fname, fmt in (("e4m3", F.E4M3), ("e5m2", F.E5M2)):
            for transpose in (False, True):
                qt_arg = qt if transpose else None
                call = lambda: F.fp8_quantize(x, fmt, scale=scale, q=q, q_t=qt_arg, amax_out=am)
                for _ in range(warmup):
                    call()
                ev = _events(iters)
                for i in range(iters):
                    flush.fill_(float(i))
                    ev[i][0].record(stream)
                    call()
                    ev[i][1].record(stream)
                torch.cuda.synchronize()
                med, _ = _median_ms(ev)
                per_elem = 4 if transpose else 3
                gbs = per_elem * n / (med * 1e-3) / 1e9
                out.append({"log2_elements": log2n, "shape": [rows, width], "format": fname,
                            "transpose": transpose, "median_ms": round(med, 4),
                            "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm_gbs, 4)})
        del x, q, qt
        torch.cuda.empty_cache()
    assert F.fp8_device_status() == 0
    return {"mode": "stale scale, fused amax", "iters": iters,
            "l2": "flushed before every launch", "peak_gbs": hbm_gbs, "points": out}


def extra_recipe_casts(F, dev, flush, stream, hbm_gbs, iters=10, warmup=3):
    """The casts of the other recipes, each with its transposed output: the
    block recipe's dual 1x128 cast (activations and gradients) and 128 x 128
    cast (weights), the per-row cast with the per-column cast of x^T, the
    per-tensor cast with the fused underflow / saturation counters, and the
    stochastically rounded per-tensor cast.  Algorithmic bytes: 2 read + 1
    per code written (q and q^T) + 4 per scale."""
    out = []

    def timed(name, shape, fmt_name, work_bytes, call):
        for _ in range(warmup):
            call()
        ev = _events(iters)
        for i in range(iters):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        med, _ = _median_ms(ev)
        gbs = work_bytes / (med * 1e-3) / 1e9
        out.append({"cast": name, "shape": list(shape), "format": fmt_name,
                    "median_ms": round(med, 4), "achieved_gbs": round(gbs, 1),
                    "frac": round(gbs / hbm_gbs, 4)})

    R, C = 16384, 7168
    x = synthetic.student_t_rows((R, C), 1.0, 3, seed=7, device=dev)
    q = torch.empty(R, C, dtype=torch.uint8, device=dev)
    qt = torch.empty(C, R, dtype=torch.uint8, device=dev)
    for name, gran in (("block 1x128, with the 1x128 cast of x^T", F.GRAN_1x128),
                       ("block 128x128, with x^T", F.GRAN_128x128),
                       ("per row, with the per-row cast of x^T", F.GRAN_ROW)):
        s1 = torch.empty(F._scale_shape(gran, R, C), dtype=torch.float32, device=dev)
        s2 = torch.empty(F._scale_shape_t(gran, R, C), dtype=torch.float32, device=dev)
        timed(name, (R, C), "e4m3", 4.0 * R * C + 4.0 * (s1.numel() + s2.numel()),
              lambda: F.fp8_quantize(x, F.E4M3, gran, q=q, q_t=qt, scale_inv_blocks=s1,
                                     scale_inv_blocks_t=s2))
    del x, q, qt
    am = torch.empty(1, dtype=torch.float32, device=dev)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    counts = torch.zeros(2, dtype=torch.int64, device=dev)
    seed = iter(range(1, 1 << 30))
    for (R, C), name, fmt_name, fmt, call in (
            ((16384, 8192), "per tensor, fused counters, with x^T", "e4m3", F.E4M3,
             lambda: F.fp8_quantize_counted(x, F.E4M3, one, counts=counts, q=q, q_t=qt,
                                            amax_out=am)),
            ((65536, 8192), "per tensor, stochastic rounding, with x^T", "e5m2", F.E5M2,
             lambda: F.fp8_quantize_sr(x, F.E5M2, one, next(seed), 0, q=q, q_t=qt,
                                       amax_out=am))):
        x = synthetic.student_t((R, C), 3, 1.0, seed=R, device=dev)
        q = torch.empty(R, C, dtype=torch.uint8, device=dev)
        qt = torch.empty(C, R, dtype=torch.uint8, device=dev)
        timed(name, (R, C), fmt_name, 4.0 * R * C, call)
        del x, q, qt
    torch.cuda.empty_cache()
    assert F.fp8_device_status() == 0
    return {"iters": iters, "l2": "flushed before every launch", "peak_gbs": hbm_gbs,
            "points": out}


def small_case_pass(F, dev, stream, iters=200):
    """The small forward case (X 256 x 512 with outliers, W 512 x 512, dynamic
    scaling): latency of fp8_linear_fwd and of fwd + bwd, issued eagerly and
    replayed from a CUDA graph of the same calls.  Launch-bound at this size
    (4 launches per fwd + bwd: a small-tensor cast and a GEMM each), so it
    reports microseconds, not a roofline."""
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
    # each graph holds `reps` calls in stream order, so that the time per call
    # is the device's and not the host's cost of launching one graph
    reps = 10
    graphs = {}
    for name, fn in (("fwd", fwd), ("fwd_bwd", fwd_bwd)):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()                                   # warm: kernel attributes, tensor maps
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=side):
                for _ in range(reps):
                    fn()
        stream.wait_stream(side)
        graphs[name] = g
    out["graph_fwd_us"] = round(timed(graphs["fwd"].replay) / reps, 2)
    out["graph_fwd_bwd_us"] = round(timed(graphs["fwd_bwd"].replay) / reps, 2)
    out["graph_calls_per_replay"] = reps
    out["graph_fwd_bwd_tflops"] = round(6.0 * M * N * K / (out["graph_fwd_bwd_us"] * 1e-6) / 1e12, 3)
    out["l2"] = "resident (1.3 MB of operands)"
    assert F.fp8_device_status() == 0
    return out


def e2e_pass(F, wl: Workload, dev, args, stream, all_tensors=False):
    """Public API with host buffers, every copy inside the timed region, in the
    traffic pattern of a training loop: per micro-batch the step's data, X
    and dY of each linear, goes host -> device from pinned memory; the weights
    stay on the device (uploaded once before timing, where an optimizer keeps
    them); Y, dX and dW stay on the device (for the next layer and the
    optimizer); and after each linear's last micro-batch its scaling metrics
    (the amax and dequantisation factor of every role) come back to pinned
    host memory.  fp8_linear_fwd + fp8_linear_bwd per micro-batch and linear.
    all_tensors: every tensor crosses the host link every step as well -- W
    in, Y and dX per micro-batch and dW out -- which makes the link the bound.
    The copies run on their own streams, ordered by events, so that they
    overlap the compute and each other: X and dY of a unit (one micro-batch
    of one linear) arrive up to two units ahead (three device buffer sets);
    a linear's next W (all_tensors) is uploaded on a stream of its own once
    the step's last forward of that linear has quantised the current one (the
    backward reads the codes, not W); results leave on a third stream, before
    the next step's first use of the linear overwrites them."""
    nl, MB, T = len(wl.linears), wl.micro_batches, wl.tokens
    NB = 3
    recipe = wl.recipe(F)
    h_w, h_x, h_dy, h_y, h_dx, h_dw, h_met, layers = [], [], [], [], [], [], [], []
    for li, (name, K, N) in enumerate(wl.linears):
        h_w.append(synthetic.normal((N, K), 0.02, seed=1000 + li, device=dev).cpu().pin_memory())
        h_x.append([synthetic.with_outlier_channels((T, K), 1.0, wl.outlier_channels(K), 50.0,
                                                    seed=10 * li + mb, device=dev).cpu().pin_memory()
                    for mb in range(MB)])
        h_dy.append([synthetic.normal((T, N), 1e-3, seed=500 + 10 * li + mb,
                                      device=dev).cpu().pin_memory() for mb in range(MB)])
        if all_tensors:
            h_y.append([torch.empty(T, N, dtype=torch.bfloat16).pin_memory() for _ in range(MB)])
            h_dx.append([torch.empty(T, K, dtype=torch.bfloat16).pin_memory() for _ in range(MB)])
            h_dw.append(torch.empty(N, K, dtype=torch.float32).pin_memory())
        layers.append(F.Fp8Linear(T, N, K, recipe, device=dev))
        h_met.append(torch.empty(2, layers[-1].amax.numel(), dtype=torch.float32).pin_memory())
    kmax = max(k for _, k, _ in wl.linears)
    nmax = max(n for _, _, n in wl.linears)
    d_w = [torch.empty(n, k, dtype=torch.bfloat16, device=dev) for _, k, n in wl.linears]
    d_dw = [torch.empty(n, k, dtype=torch.float32, device=dev) for _, k, n in wl.linears]

    def dbuf():
        return {"X": torch.empty(T * kmax, dtype=torch.bfloat16, device=dev),
                "dY": torch.empty(T * nmax, dtype=torch.bfloat16, device=dev),
                "Y": torch.empty(T * nmax, dtype=torch.bfloat16, device=dev),
                "dX": torch.empty(T * kmax, dtype=torch.bfloat16, device=dev)}

    bufs = [dbuf() for _ in range(NB)]
    h2d_s, w_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nbytes = lambda t: t.numel() * t.element_size()
    h2d = sum(nbytes(t) for ts in h_x + h_dy for t in ts)
    d2h = sum(nbytes(t) for t in h_met)
    if all_tensors:
        h2d += sum(nbytes(w) for w in h_w)
        d2h += sum(nbytes(t) for ts in h_y + h_dx for t in ts) + sum(nbytes(t) for t in h_dw)
    # Units g = (step * MB + mb) * nl + li use device buffer set g % NB; each
    # copy waits only for the last user of its own buffer.
    computed, drained, w_loaded, res_drained = {}, {}, {}, {}
    counter = [0]

    def upload_w(li, after=None):
        with torch.cuda.stream(w_s):
            if after is not None:
                w_s.wait_event(after)
            d_w[li].copy_(h_w[li], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(w_s)
            w_loaded[li] = ev

    def load_unit():
        g = counter[0]
        counter[0] += 1
        li, mb = g % nl, (g // nl) % MB
        _, K, N = wl.linears[li]
        b = bufs[g % NB]
        loaded = torch.cuda.Event()
        with torch.cuda.stream(h2d_s):
            if g - NB in computed:
                h2d_s.wait_event(computed.pop(g - NB))     # last reader of this set's inputs
            b["X"][:T * K].view(T, K).copy_(h_x[li][mb], non_blocking=True)
            b["dY"][:T * N].view(T, N).copy_(h_dy[li][mb], non_blocking=True)
            loaded.record(h2d_s)
        return g, li, mb, K, N, b, loaded

    def compute_and_drain(g, li, mb, K, N, b, loaded):
        stream.wait_event(loaded)
        if mb == 0 and li in w_loaded:
            stream.wait_event(w_loaded.pop(li))            # this step's W[li] has arrived
        if g - NB in drained:
            stream.wait_event(drained.pop(g - NB))         # this set's outputs have left
        if mb == 0 and li in res_drained:
            stream.wait_event(res_drained.pop(li))         # last step's results of li have left
        Y = b["Y"][:T * N].view(T, N)
        dX = b["dX"][:T * K].view(T, K)
        L = layers[li]
        L.forward(b["X"][:T * K].view(T, K), d_w[li], Y=Y)
        fwd_done = torch.cuda.Event()
        fwd_done.record(stream)
        if all_tensors:
            if mb == MB - 1:
                upload_w(li, after=fwd_done)               # the next step's W[li]
            with torch.cuda.stream(d2h_s):                 # Y leaves while the backward runs
                d2h_s.wait_event(fwd_done)
                h_y[li][mb].copy_(Y, non_blocking=True)
        L.backward(b["dY"][:T * N].view(T, N), dX=dX, dW=d_dw[li], accumulate_dW=mb > 0)
        ev = torch.cuda.Event()
        ev.record(stream)
        computed[g] = ev
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev)
            if all_tensors:
                h_dx[li][mb].copy_(dX, non_blocking=True)
                done = torch.cuda.Event()
                done.record(d2h_s)
                drained[g] = done
            if mb == MB - 1:
                h_met[li][0].copy_(L.amax, non_blocking=True)
                h_met[li][1].copy_(L.scale_inv, non_blocking=True)
                if all_tensors:
                    h_dw[li].copy_(d_dw[li], non_blocking=True)
                rd = torch.cuda.Event()
                rd.record(d2h_s)
                res_drained[li] = rd

    def steps(k, first):
        """k steps, loads issued up to NB - 1 units ahead."""
        for st in (h2d_s, w_s, d2h_s):
            st.wait_stream(stream)                         # copies start after the start event
        if first:
            for li in range(nl):
                upload_w(li)
        units = k * MB * nl
        pending = [load_unit() for _ in range(min(NB - 1, units))]
        for i in range(units):
            if i + NB - 1 < units:
                pending.append(load_unit())
            compute_and_drain(*pending.pop(0))
        for st in (h2d_s, w_s, d2h_s):
            stream.wait_stream(st)                         # the last results are on the host

    steps(max(1, min(args.warmup, 2)), True)
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 10))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    steps(n, False)
    b.record(stream)
    torch.cuda.synchronize()
    assert F.fp8_device_status() == 0
    assert all(bool(torch.isfinite(m).all()) for m in h_met)
    ms = a.elapsed_time(b) / n
    out = {"value": round(wl.flops_step() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "ms_per_step": round(ms, 3), "steps": n, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}
    if all_tensors:
        link = _host_link(dev)
        out.update({
            "copies": "W of every linear in, X and dY per micro-batch in, Y and dX per "
                      "micro-batch and dW per step out, on three copy streams overlapped with "
                      "compute and with each other",
            "host_link": link,
            "link_floor_ms": round(_link_floor_ms(h2d, d2h, link), 3),
            "link_floor_note": "the time to move h2d and d2h bytes at the link rates measured "
                               "in this run: both directions at their concurrent rates until "
                               "the smaller finishes, the rest at its one-way rate"})
    else:
        out["copies"] = ("X and dY of every linear and micro-batch in (pinned host memory, up "
                         "to two units ahead of the compute); after each step the scaling "
                         "metrics of every linear (amax and dequantisation factor per role) "
                         "out; weights, outputs and gradients stay on the device, as in a "
                         "training loop")
        out["h2d_floor_ms"] = round(h2d / (_host_link(dev)["h2d_gbs"] * 1e9) * 1e3, 3)
    return out


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

def _oracle_inputs(wl: Workload, linears, device="cpu"):
    """Bit patterns of micro-batch 0's X, W and dY for the listed linears,
    drawn as the GPU arm draws them (same generators and seeds; on `device`,
    then copied to the host)."""
    import oracle
    inputs, states = {}, {}
    rec = (oracle.Recipe(scaling=oracle.SCALING_DYNAMIC) if wl.scaling == "dynamic"
           else oracle.Recipe(scaling=oracle.SCALING_DELAYED, history_len=16))
    for li in linears:
        _, K, N = wl.linears[li]
        X = synthetic.with_outlier_channels((wl.tokens, K), 1.0, wl.outlier_channels(K), 50.0,
                                            seed=10 * li, device=device)
        W = synthetic.normal((N, K), 0.02, seed=1000 + li, device=device)
        dY = synthetic.normal((wl.tokens, N), 1e-3, seed=500 + 10 * li, device=device)
        inputs[li] = (synthetic.bf16_bits(X), synthetic.bf16_bits(W), synthetic.bf16_bits(dY))
        states[li] = (oracle.LinearState(rec), rec)
    return inputs, states


def _oracle_unit(wl, li, rows, inputs, states, half=None):
    """The oracle's fwd + bwd of one linear (its linear_fwd / linear_bwd):
    whole-tensor amax, scale update and quantisation (with the transposed
    copies) of X, W and dY, and `rows` full output rows of each of the three
    GEMMs (fp64 accumulation).  half = "fwd" or "bwd" runs one of the two
    passes (the backward uses the state the last forward of this linear
    left).  Returns the FLOPs of the sampled rows."""
    import numpy as np
    import oracle
    _, K, N = wl.linears[li]
    bx, bw, bdy = inputs[li]
    st, rec = states[li]
    r = np.arange(rows)
    flops = 0.0
    if half in (None, "fwd"):
        oracle.linear_fwd(bx, bw, rec, st, rows=r)
        flops += 2.0 * rows * N * K
    if half in (None, "bwd"):
        oracle.linear_bwd(bdy, rec, st, rows_dx=r, rows_dw=r)
        flops += 2.0 * rows * (K * N + K * wl.tokens)
    return flops


def cpu_baseline(args, run_dev=None):
    """The oracle as it stands, on the host cores, on one bounded sample of
    the headline step: micro-batch 0 of all five linears with `--cpu-rows`
    output rows per GEMM (inputs drawn on the GPU with the GPU arm's seeds)."""
    import oracle
    wl = LLAMA70B
    lis = list(range(len(wl.linears)))
    inputs, states = _oracle_inputs(wl, lis, device=run_dev or "cpu")
    rows = args.cpu_rows
    t0 = time.perf_counter()
    flops = sum(_oracle_unit(wl, li, rows, inputs, states) for li in lis)
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": (f"micro-batch 0 of the step (half of it): whole-tensor amax/scale/"
                       f"quantise(+transpose) of X, W, dY of the 5 linears, and {rows} full "
                       f"output rows of each of their 15 GEMMs (fp64 accumulation); value = "
                       f"sampled GEMM FLOPs / wall time")}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    wl = LLAMA70B
    nl = len(wl.linears)
    rows = args.ref_rows
    # one linear's fwd + bwd takes seconds on the host cores: short runs take
    # all five linears per step; longer ones one half (the forward or the
    # backward) of one linear per step, in turn, so that the whole run stays
    # within a few minutes
    short = args.steps + args.warmup <= 10
    seq = [(li, h) for li in range(nl) for h in ("fwd", "bwd")]
    units = (lambda i: [(li, None) for li in range(nl)]) if short else (lambda i: [seq[i % len(seq)]])
    inputs, states = _oracle_inputs(wl, list(range(nl)))
    for li in range(nl):        # every linear's state exists before a backward half runs
        _oracle_unit(wl, li, 1, inputs, states, "fwd")
    for i in range(args.warmup):
        for li, h in units(i):
            _oracle_unit(wl, li, rows, inputs, states, h)
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(args.steps):
        for li, h in units(args.warmup + i):
            flops += _oracle_unit(wl, li, rows, inputs, states, h)
    dt = time.perf_counter() - t0
    v = flops / dt / 1e12
    which = ("one micro-batch of the 5 linears" if short else
             "the forward or the backward of one linear (in turn over the 5 linears)")
    sample = (f"per step: {which}: whole-tensor amax/scale/quantise(+transpose) of its "
              f"operands and {rows} full output rows of each of its GEMMs; value = sampled "
              f"GEMM FLOPs / wall time")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.label, "tokens_per_micro_batch": wl.tokens,
                   "micro_batches_per_step": wl.micro_batches,
                   "linears": {n: [k, n_] for n, k, n_ in wl.linears}},
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
            # B per 128 x 128 block, or (--colscale, the block wgrad) per column
            gb = F.GRAN_1x128 if args.colscale else F.GRAN_128x128
            sa = torch.rand(M, K // 128, generator=g, device=dev) + 0.5
            sb = torch.rand(N if args.colscale else N // 128, K // 128, generator=g,
                            device=dev) + 0.5
            call = lambda: F.fp8_gemm(A, F.E4M3, B, F.E4M3, sa, sb, F.GRAN_1x128, gb, D=D)
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
        elif gran == F.GRAN_TENSOR and args.counted:
            # the cast with the fused underflow / saturation counters
            counts = torch.zeros(2, dtype=torch.int64, device=dev)
            call = lambda: F.fp8_quantize_counted(x, fa, one, counts=counts, q=q, q_t=qt_arg,
                                                  amax_out=am)
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
        if args.counted and args.gran == "tensor" and args.kernel == "quantize":
            extra["counters"] = "underflow and saturation, fused"
    if args.kernel == "block_gemm":
        extra = {"factors": "power of two (block-scaled MMA)" if args.pow2
                 else "fp32 (per-128-K promotion)",
                 "b_factors": "per column (1x128)" if args.colscale and not args.pow2
                 else "per 128 x 128 block"}
    if args.kernel == "gemm":
        extra = {"output": "fp32, accumulated" if args.f32acc else "bf16", "layout": args.layout}
    print(json.dumps({"kernel": args.kernel, "shape": dims, "format": args.fmt, **extra,
                      "median_ms": round(med, 4), "min_ms": round(ms[0], 4),
                      "achieved": round(ach, 1), "unit": unit, "peak": round(peak, 1),
                      "frac": round(ach / peak, 4),
                      "peak_source": f"{peak_kind} ({'2 x bf16 burst' if unit == 'TFLOP/s' else 'hbm_gbs'})",
                      "iters": args.iters, "l2": "flushed before every launch"}))


def step_gemms(wl: Workload | None = None):
    """The GEMMs of one micro-batch of a layer step: (name, M, N, K, A
    format, output, layout) -- per linear the forward, the dgrad and the
    wgrad.  The backward GEMMs read the forward's codes as stored (the
    layer's default): dgrad's B is W_q [N x K], wgrad's A and B are dY_q and
    X_q, both [tokens x ...]."""
    wl = wl or LLAMA7B
    T = wl.tokens
    out = []
    for name, K, N in wl.linears:
        out.append((name + ".fwd", T, N, K, "e4m3", "bf16", 0))
        out.append((name + ".dgrad", T, K, N, "e5m2", "bf16", 1))
        out.append((name + ".wgrad", N, K, T, "e5m2", "f32acc", 3))
    return out


def run_gemm_step(F, args, dev, codes, flush):
    """The 15 GEMMs of one micro-batch of a layer step (--workload) with their
    shapes, formats and output types, each on random codes, run once as
    warm-up and once timed (in that order), with the operands of one GEMM on
    the device at a time."""
    gemms = step_gemms(WORKLOADS[args.workload])
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
    print(json.dumps({"kernel": "gemm_step", "workload": args.workload,
                      "gemms": [g[0] for g in gemms],
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


def _gemm_traffic(key):
    """DRAM bytes per GEMM launch of a workload's step (mean over its GEMM
    launches), as measured by ncu and recorded in profiles/ together with a
    hash of the GEMM source it was measured on; None if the source has
    changed since or the workload has no record."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_step_traffic.json")) as f:
            rec = json.load(f)["workloads"][key]
        with open(os.path.join(ROOT, "scaled_fp8_linear_gb300", "csrc", "gemm.cu"), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()
        return rec["bytes_per_launch"] if rec.get("gemm_cu_sha256") == h else None
    except Exception:
        return None


WORKLOADS = {"llama2-70b": LLAMA70B, "llama2-7b": LLAMA7B}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=80)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=8)
    ap.add_argument("--ref-rows", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="headline step only (skip the other configurations' keys)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama2-70b",
                    help="--kernel gemm_step: whose step GEMMs")
    ap.add_argument("--kernel", choices=["gemm", "block_gemm", "quantize", "quantize_sr",
                                         "quantize_sweep", "gemm_step", "block_step"],
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
    ap.add_argument("--counted", action="store_true",
                    help="--kernel quantize --gran tensor: the cast with the fused underflow / "
                         "saturation counters (fp8_quantize_counted)")
    ap.add_argument("--colscale", action="store_true",
                    help="--kernel block_gemm: B with 1x128 factors (one per output column and "
                         "K block, the block-wise wgrad)")
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
