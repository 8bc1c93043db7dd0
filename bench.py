"""Benchmark: GPT-2-124M training tokens/s (fwd + bwd + AdamW) on libgk, plus KV-cache decode.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--batch B]

Prints ONE JSON line (rank 0). The workload is the GPT-2-124M-shaped training step with
batch 16 x 1024 (fast mode: bf16 operands, fp32 master weights, moments, residual stream and
logits), synthetic ids and N(0, 0.02) weights. A step's working set (weights, activations,
[16384, 50304] logits) is far larger than the 129 MB L2, so consecutive steps cannot hit in
L2. `--impl reference` times the oracle (plain float64 CPU code) on a bounded sample of the
same workload on the host cores.

Multi-GPU: the path shards by sequences with no exchange in this build (replicas only): each
rank runs its own replica; value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "train tokens/s (fwd+bwd+AdamW) at GPT-2-124M shape; KV-cache decode tok/s"
UNIT = "tokens/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.idx = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------- oracle
def oracle_tokens_per_s(seconds_budget=20.0, T=1024):
    """The oracle's training step (float64, host) on one sequence of the 124M model."""
    import synth
    from oracle import gpt as ogpt

    s = synth.GPT2_124M
    ids, targets, params = synth.training_case(s, 1, 7, T=T)
    sh = ogpt.Shape(s.V, s.T, s.C, s.H, s.L)
    n, t0 = 0, time.perf_counter()
    while True:
        loss, grads, _, _ = ogpt.loss_and_grads(params, ids, targets, sh)
        ogpt.adamw_step(params, grads, {}, 1, 3e-4, wd=0.01)
        n += 1
        el = time.perf_counter() - t0
        if el > seconds_budget or n >= 3:
            break
    try:
        from threadpoolctl import threadpool_info

        cores = max((i.get("num_threads") or 1) for i in threadpool_info()) if threadpool_info() else 1
    except Exception:
        cores = os.cpu_count() or 1
    return n * T / el, cores, f"{n} oracle step(s) of 1 x {T} tokens (GPT-2-124M, float64 numpy/BLAS)"


def workload_config(B, mode, world):
    """The `config` of the training-step line (shared by both arms)."""
    return {"workload": f"gpt2-124m train step (fwd+bwd+AdamW), B={B} x T=1024, "
                        f"{'bf16 operands / fp32 master' if mode == 'bf16' else 'fp32 faithful'}",
            "l2": "inputs larger than L2 (step working set >> 129 MB)", "parallelism": f"replicas x{world}"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import synth
    from oracle import gpt as ogpt

    s = synth.GPT2_124M
    # each step: a bounded sample of the workload, the first 512 positions of one of its
    # sequences (the oracle takes seconds per sequence on the host cores)
    T = 512
    ids, targets, params = synth.training_case(s, 1, 5, T=T)
    sh = ogpt.Shape(s.V, s.T, s.C, s.H, s.L)

    def step():
        loss, grads, _, _ = ogpt.loss_and_grads(params, ids, targets, sh)
        ogpt.adamw_step(params, grads, {}, 1, 3e-4, wd=0.01)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    tps = args.steps * T / el
    try:
        from threadpoolctl import threadpool_info

        cores = max((i.get("num_threads") or 1) for i in threadpool_info())
    except Exception:
        cores = os.cpu_count() or 1
    sample = (f"each step: 1 sequence x {T} positions of the GPT-2-124M training step (fwd+bwd+AdamW), "
              f"float64 oracle on the host; tokens/s = {T} x steps / time")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.batch, args.mode, world),
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ----------------------------------------------------------------------------- ours
def time_events(fn, reps, stream=None, flush=None):
    """Median CUDA-event time (ms) of fn() on `stream` (the current stream by default); with
    `flush` (a tensor larger than L2) it is overwritten before every timed call, outside the
    events."""
    import torch

    st = stream or torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        fn()
        e1.record(st)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return sorted(ts)[len(ts) // 2]


def gemm_breakdown(m, ids, tg, lr, wd, steps=2):
    """Per-step GEMM time and algorithmic FLOPs of the training step, from CUDA events around
    every product launch: a separate, untimed pass (the events sit between launches)."""
    m.gemm_events = []
    for _ in range(steps):
        m.train_step(ids, tg, lr, wd)
    import torch

    torch.cuda.synchronize()
    gms = sum(e0.elapsed_time(e1) for (e0, e1, _) in m.gemm_events) / steps
    flops = sum(f for (_, _, f) in m.gemm_events) / steps
    m.gemm_events = None
    return gms, flops


def run_ours(args):
    import torch

    import synth
    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    s = synth.GPT2_124M
    B, T = args.batch, s.T
    stream = torch.cuda.current_stream()
    ctx = gk.Ctx(stream.cuda_stream, workspace_bytes=(256 << 20) if args.mode == "bf16" else (2 << 30))
    ids, targets, params = synth.training_case(s, B, 5 + rank)
    m = Gpt(ctx, s.V, s.T, s.C, s.H, s.L, B, mode=args.mode)
    m.load(params)
    del params
    d_ids = torch.as_tensor(ids.reshape(-1)).cuda()
    d_tg = torch.as_tensor(targets.reshape(-1)).cuda()
    lr, wd = 3e-4, 0.01

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    for _ in range(args.warmup):
        m.train_step(d_ids, d_tg, lr, wd)
    gk.gk_sync(ctx)
    # timed region: K steps, device time by CUDA events on the launching stream
    barrier()
    torch.cuda.synchronize()
    n0 = gk.gk_launch_count(ctx)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            loss = m.train_step(d_ids, d_tg, lr, wd)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    launches = gk.gk_launch_count(ctx) - n0
    gk.gk_sync(ctx)
    ms = ev0.elapsed_time(ev1) / args.steps
    if world > 1:
        import torch.distributed as dist

        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = t.item()
    tokens = B * T * world
    value = tokens / (ms / 1e3)
    # roofline of the dominant kernel class (the GEMMs), from a separate instrumented pass
    gms, flops = gemm_breakdown(m, d_ids, d_tg, lr, wd)
    hbm, bf16_burst, bf16_sus, peak_src = _peaks()
    achieved = flops / (gms / 1e3) / 1e12 if gms > 0 else 0.0
    # end to end: ids/targets from pinned host memory each step, loss read back
    h_ids = torch.as_tensor(ids.reshape(-1)).pin_memory()
    h_tg = torch.as_tensor(targets.reshape(-1)).pin_memory()
    h_loss = torch.empty(1, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 5))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        d_ids.copy_(h_ids, non_blocking=True)
        d_tg.copy_(h_tg, non_blocking=True)
        loss = m.train_step(d_ids, d_tg, lr, wd)
        h_loss.copy_(loss, non_blocking=True)
        torch.cuda.synchronize()
    e2e = tokens / ((time.perf_counter() - t0) / e2e_steps)
    loss_last = float(h_loss.item())
    extra = {}
    if rank == 0 and not args.no_decode:
        decode_params = m.params
        extra["decode"] = bench_decode(ctx, m, s)
        del decode_params
    if rank == 0 and not args.no_sweep:
        del m
        torch.cuda.empty_cache()
        extra["step_b4"] = bench_step_b4(s)
        extra["op_sweep"] = bench_op_sweep()
        extra["gemm_bf16_gpt2_b16"] = bench_gemm_shapes()
        extra["generic_ops"] = bench_generic(ctx)
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, sample = oracle_tokens_per_s()
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    tf32 = bf16_sus / 2
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.mode == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(B, args.mode, world),
        "roofline": {"bound": "tensor", "achieved": achieved,
                     "peak": bf16_sus if args.mode == "bf16" else tf32 / 3, "unit": "TFLOP/s",
                     "frac": achieved / (bf16_sus if args.mode == "bf16" else tf32 / 3),
                     "traffic": gemm_traffic_per_step(B, args.mode),
                     "kernel": "all GEMM launches of the step (timed in a separate pass)",
                     "peak_source": f"{peak_src} bf16 sustained"
                     + ("" if args.mode == "bf16" else " / 2 (tf32 nominal ratio) / 3 (3xTF32 products)"),
                     "gemm_ms_per_step": gms, "gemm_tflop_per_step": flops / 1e12},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": int(2 * B * T * 4), "d2h_bytes_per_step": 4},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "loss_last": loss_last,
    }
    out.update(extra)
    print(json.dumps(out))


def bench_step_b4(s, steps=5, warmup=2):
    """The GPT-2-124M step at batch 4 x 1024 in both modes: fp32 faithful (float32 products as
    3xTF32 on the tensor cores; attention, LayerNorm, softmax-CE and AdamW in float32) and bf16.
    For the faithful step the GEMM roofline is stated both ways: algorithmic FLOPs against the
    TF32 peak / 3, and the tensor cores' rate (three TF32 products per FLOP) against the TF32 peak."""
    import torch

    import synth
    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    hbm, _, bf16_sus, peak_src = _peaks()
    tf32 = bf16_sus / 2
    ids, targets, params = synth.training_case(s, 4, 2)
    d_ids = torch.as_tensor(ids.reshape(-1)).cuda()
    d_tg = torch.as_tensor(targets.reshape(-1)).cuda()
    res = {}
    for mode in ("fp32", "bf16"):
        ctx = gk.Ctx(torch.cuda.current_stream().cuda_stream, workspace_bytes=2 << 30)
        m = Gpt(ctx, s.V, s.T, s.C, s.H, s.L, 4, mode=mode)
        m.load(params)
        for _ in range(warmup):
            m.train_step(d_ids, d_tg, 3e-4, 0.01)
        ms = time_events(lambda: [m.train_step(d_ids, d_tg, 3e-4, 0.01) for _ in range(steps)], 1) / steps
        gms, flops = gemm_breakdown(m, d_ids, d_tg, 3e-4, 0.01, steps=1)
        gk.gk_sync(ctx)
        ach = flops / (gms / 1e3) / 1e12
        r = {"ms_per_step": ms, "tokens_s": 4 * 1024 / (ms / 1e3), "gemm_ms_per_step": gms,
             "gemm_tflop_per_step": flops / 1e12, "gemm_tflops": ach}
        if mode == "fp32":
            r.update({"math": "3xTF32", "gemm_frac_algorithmic": ach / (tf32 / 3),
                      "gemm_frac_hardware": 3 * ach / tf32, "tf32_peak_tflops": tf32,
                      "peak_source": f"{peak_src} bf16 sustained / 2 (tf32 nominal ratio)"})
        else:
            r.update({"gemm_frac": ach / bf16_sus, "peak_source": f"{peak_src} bf16 sustained"})
        res[mode] = r
        del m
        ctx.close()
        torch.cuda.empty_cache()
    return res


def bench_op_sweep(reps=5):
    """The float32 op sweep on seeded N(0, 1) inputs: MatMul / MatMulT forward and backward at
    M = N = K in {256, 1024, 4096} and (M, K, N) = (4096, 768, 3072), as 3xTF32 (TFLOP/s; the
    fraction against TF32 peak / 3) and as float32 FMA on the CUDA cores; LayerNorm, GELU and
    softmax-CE forward and backward on [4096, C], C in {768, 50257} (GB/s of the algorithmic
    bytes against the measured copy bandwidth). L2 is overwritten before every timed call."""
    import torch

    import synth
    from gpt_decoder_gb300 import gk

    hbm, _, bf16_sus, _ = _peaks()
    tf32 = bf16_sus / 2
    fma_peak = 152 * 128 * 2 * 2.07e9 / 1e12  # SMs x FP32 lanes x 2 FLOP x max clock
    flush = torch.empty(64 << 20, device="cuda")  # 256 MB, twice L2
    ctx = gk.Ctx(torch.cuda.current_stream().cuda_stream, workspace_bytes=2 << 30)
    st = synth.Stream(1)
    dn = lambda *shape: torch.as_tensor(st.normal(int(np.prod(shape))).reshape(shape)).cuda()
    res = {"gemm": {}, "rowwise": {}}
    for (M, K, N) in [(256, 256, 256), (1024, 1024, 1024), (4096, 4096, 4096), (4096, 768, 3072)]:
        x, g = dn(M, K), dn(M, N)
        for transW in (0, 1):
            w = dn(N, K) if transW else dn(K, N)
            ldw = w.shape[1]
            y, dx, dw = torch.empty(M, N, device="cuda"), torch.empty(M, K, device="cuda"), torch.zeros_like(w)
            key = f"{'matmul_t' if transW else 'matmul'}_{M}x{K}x{N}"
            r = {}
            for math, name in ((gk.GK_MATH_3XTF32, "3xtf32"), (gk.GK_MATH_FP32, "fma")):
                gk.gk_set_math(ctx, math)
                fwd = lambda: gk.gk_matmul_fwd(ctx, gk.GK_F32, x, K, w, ldw, transW, None, None, 0, y, N, gk.GK_F32,
                                               M, K, N)
                bwd = lambda: gk.gk_matmul_bwd(ctx, gk.GK_F32, x, K, w, ldw, transW, g, N, dx, K, gk.GK_F32, 0, None,
                                               0, dw, ldw, None, M, K, N)
                fwd(), bwd()
                tf = time_events(fwd, reps, flush=flush)
                tb = time_events(bwd, reps, flush=flush)
                ff, fb = 2.0 * M * N * K / (tf / 1e3) / 1e12, 4.0 * M * N * K / (tb / 1e3) / 1e12
                peak = tf32 / 3 if name == "3xtf32" else fma_peak
                r[name] = {"fwd_tflops": ff, "bwd_tflops": fb, "fwd_frac": ff / peak, "bwd_frac": fb / peak,
                           "fwd_us": tf * 1e3, "bwd_us": tb * 1e3}
            gk.gk_set_math(ctx, gk.GK_MATH_FP32)
            res["gemm"][key] = r
            del w, y, dx, dw
        del x, g
    res["gemm_peaks_tflops"] = {"3xtf32": tf32 / 3, "fma": fma_peak,
                                "note": "3xtf32: measured bf16 sustained / 2 / 3; fma: 152 SMs x 128 lanes x 2 x 2.07 GHz"}
    for C in (768, 50257):
        R = 4096
        x, gm, bt, g = dn(R, C), dn(C), dn(C), dn(R, C)
        y, dx = torch.empty(R, C, device="cuda"), torch.empty(R, C, device="cuda")
        mu, rs = torch.empty(R, device="cuda"), torch.empty(R, device="cuda")
        dgm, dbt = torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda")
        tg = torch.as_tensor(st.ints(R, C)).cuda()
        loss, lse = torch.zeros(1, device="cuda"), torch.empty(R, device="cuda")
        n = R * C
        cases = {
            "layernorm_fwd": (lambda: gk.gk_layernorm_fwd(ctx, x, gm, bt, y, gk.GK_F32, mu, rs, R, C, 1e-5), 8 * n + 8 * R),
            "layernorm_bwd": (lambda: gk.gk_layernorm_bwd(ctx, x, gm, mu, rs, g, dx, 0, None, dgm, dbt, R, C),
                              12 * n + 8 * R),
            "gelu_fwd": (lambda: gk.gk_gelu_fwd(ctx, x, y, n), 8 * n),
            "gelu_bwd": (lambda: gk.gk_gelu_bwd(ctx, x, g, dx, n), 12 * n),
            "softmax_ce_fwd": (lambda: gk.gk_softmax_ce_fwd(ctx, x, C, tg, loss, lse, R, C), 4 * n + 8 * R),
            "softmax_ce_bwd": (lambda: gk.gk_softmax_ce_bwd(ctx, x, C, tg, lse, None, dx, C, gk.GK_F32, R, C),
                               8 * n + 8 * R),
        }
        for name, (fn, nbytes) in cases.items():
            fn()
            t = time_events(fn, reps, flush=flush)
            res["rowwise"][f"{name}_{R}x{C}"] = {"gbs": nbytes / (t / 1e3) / 1e9, "frac": nbytes / (t / 1e3) / 1e9 / hbm,
                                                  "us": t * 1e3}
        del x, g, y, dx
    res["rowwise_peak_gbs"] = hbm
    gk.gk_sync(ctx)
    ctx.close()
    del flush
    torch.cuda.empty_cache()
    return res


def bench_gemm_shapes(reps=7):
    """The bf16 products of one transformer block of the GPT-2-124M step at B=16 x T=1024
    (16384 rows), called as the training step calls them (bias, residual added in place,
    GELU with its pre-activation, the GELU backward fused into dX, dW accumulated), each timed
    alone with L2 overwritten before every call: TFLOP/s against the measured bf16 peak, and
    torch.matmul (cuBLAS) on the same plain shape as a library reference."""
    import torch

    from gpt_decoder_gb300 import gk

    _, bf16, bf16_sus, _ = _peaks()
    flush = torch.empty(64 << 20, device="cuda")
    ctx = gk.Ctx(torch.cuda.current_stream().cuda_stream)
    gk.gk_set_math(ctx, gk.GK_MATH_FP32)
    N, C = 16384, 768
    BF = torch.bfloat16
    g = torch.Generator(device="cuda").manual_seed(3)
    rn = lambda *sh, dt=BF: (torch.randn(*sh, device="cuda", generator=g) * 0.5).to(dt)
    x768, x3072 = rn(N, C), rn(N, 4 * C)
    w_qkv, w_proj, w_fc, w_mp = rn(C, 3 * C), rn(C, C), rn(C, 4 * C), rn(4 * C, C)
    b3, b1, b4 = rn(3 * C, dt=torch.float32), rn(C, dt=torch.float32), rn(4 * C, dt=torch.float32)
    res = rn(N, C, dt=torch.float32)
    y2304, y3072, pre = torch.empty(N, 3 * C, dtype=BF, device="cuda"), torch.empty(N, 4 * C, dtype=BF, device="cuda"), \
        torch.empty(N, 4 * C, dtype=BF, device="cuda")
    dy768, dy2304, dy3072 = rn(N, C), rn(N, 3 * C), rn(N, 4 * C)
    dx768f, dx768b, dx3072b = torch.empty(N, C, device="cuda"), torch.empty(N, C, dtype=BF, device="cuda"), \
        torch.empty(N, 4 * C, dtype=BF, device="cuda")
    dw = torch.zeros(4 * C * C, device="cuda")
    db = torch.zeros(4 * C, device="cuda")
    fwd = lambda *a: gk.gk_matmul_fwd(ctx, gk.GK_BF16, *a)
    bwd = lambda *a: gk.gk_matmul_bwd(ctx, gk.GK_BF16, *a)
    A, NONE = gk.GK_ACT_NONE, None
    cases = {
        "qkv_fwd": (lambda: fwd(x768, C, w_qkv, 3 * C, 0, b3, NONE, 0, y2304, 3 * C, gk.GK_BF16, N, C, 3 * C, A,
                                NONE, 0, NONE, NONE), 2 * N * C * 3 * C, (x768, w_qkv)),
        "proj_fwd_residual": (lambda: fwd(x768, C, w_proj, C, 0, b1, res, C, res, C, gk.GK_F32, N, C, C, A, NONE, 0,
                                          NONE, NONE), 2 * N * C * C, (x768, w_proj)),
        "fc_fwd_gelu": (lambda: fwd(x768, C, w_fc, 4 * C, 0, b4, NONE, 0, y3072, 4 * C, gk.GK_BF16, N, C, 4 * C,
                                    gk.GK_ACT_GELU, pre, 4 * C, NONE, NONE), 2 * N * C * 4 * C, (x768, w_fc)),
        "mlpproj_fwd_residual": (lambda: fwd(x3072, 4 * C, w_mp, C, 0, b1, res, C, res, C, gk.GK_F32, N, 4 * C, C, A,
                                             NONE, 0, NONE, NONE), 2 * N * 4 * C * C, (x3072, w_mp)),
        "mlpproj_bwd_dgelu": (lambda: bwd(x3072, 4 * C, w_mp, C, 0, dy768, C, dx3072b, 4 * C, gk.GK_BF16, 0, pre,
                                          4 * C, dw, C, NONE, N, 4 * C, C), 4 * N * 4 * C * C, None),
        "fc_bwd": (lambda: bwd(x768, C, w_fc, 4 * C, 0, dy3072, 4 * C, dx768f, C, gk.GK_F32, 0, NONE, 0, dw, 4 * C,
                               db, N, C, 4 * C), 4 * N * C * 4 * C, None),
        "proj_bwd": (lambda: bwd(x768, C, w_proj, C, 0, dy768, C, dx768b, C, gk.GK_BF16, 0, NONE, 0, dw, C, NONE, N,
                                 C, C), 4 * N * C * C, None),
        "qkv_bwd": (lambda: bwd(x768, C, w_qkv, 3 * C, 0, dy2304, 3 * C, dx768f, C, gk.GK_F32, 0, NONE, 0, dw, 3 * C,
                                db, N, C, 3 * C), 4 * N * C * 3 * C, None),
    }
    out = {}
    for name, (fn, flops, plain) in cases.items():
        fn()
        t = time_events(fn, reps, flush=flush)
        r = {"tflops": flops / (t / 1e3) / 1e12, "us": t * 1e3}
        r["frac"] = r["tflops"] / bf16
        if plain is not None:
            a, b = plain
            tl = time_events(lambda: torch.matmul(a, b), reps, flush=flush)
            r["cublas_tflops"] = flops / (tl / 1e3) / 1e12
        out[name] = r
    gk.gk_sync(ctx)
    ctx.close()
    out["peak_tflops"] = bf16
    out["peak_source"] = "measured bf16 burst (each product timed alone)"
    del flush
    torch.cuda.empty_cache()
    return out


def gemm_traffic_per_step(B, mode):
    """DRAM bytes of one step's GEMM launches at batch B (bf16 mode) from the data file of the
    committed ncu capture, while every source file the capture measured is unchanged (sha256
    recorded beside the figure); else None."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "gemm_tc_traffic_gpt2.json")
    if mode != "bf16" or not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    for rel, digest in d.get("source_sha256", {}).items():
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != digest:
            return None
    return d.get("bytes_per_step", {}).get(f"B{B}")


def bench_generic(ctx, n=1 << 26, reps=10):
    """HBM bandwidth of the generic elementwise ops and the Sum reduction over n float32
    elements (256 MB per operand, larger than L2): algorithmic bytes (each operand read or
    written once) over the median CUDA-event time, against the measured copy bandwidth."""
    import torch

    from gpt_decoder_gb300 import gk

    hbm = _peaks()[0]
    a, b, y = (torch.randn(n, device="cuda") for _ in range(3))
    out = torch.empty(1, device="cuda")
    cases = {"mul_fwd": (lambda: gk.gk_mul_fwd(ctx, a, b, y, n), 12 * n),
             "add_bwd_acc": (lambda: gk.gk_add_bwd(ctx, a, y, None, n, n, 1), 12 * n),
             "tanh_bwd": (lambda: gk.gk_tanh_bwd(ctx, a, b, y, n, 0), 12 * n),
             "sum_fwd": (lambda: gk.gk_sum_fwd(ctx, a, out, n), 4 * n)}
    res = {"n": n, "peak_gbs": hbm}
    for name, (fn, nbytes) in cases.items():
        fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = sorted(ts)[len(ts) // 2]
        res[name] = {"gbs": nbytes / (ms / 1e3) / 1e9, "frac": nbytes / (ms / 1e3) / 1e9 / hbm, "us": ms * 1e3}
    gk.gk_sync(ctx)
    return res


def bench_decode(ctx, m, s, Tp=512, n_steps=256):
    """Greedy KV-cache decode tok/s (fp32 weights) at batch 1 and 16: a 512-token prompt, then
    n_steps decode steps timed (prefill excluded), each step one replay of the captured step
    graph (gk_decode_run) on a stream of its own."""
    import torch

    from gpt_decoder_gb300 import gk

    res = {}
    stream = torch.cuda.Stream()
    dctx = gk.Ctx(stream, workspace_bytes=64 << 20)
    torch.cuda.synchronize()
    warm = 8
    hbm = _peaks()[0]
    # bytes a step must move: every float32 weight once (wpe: one row) and each sequence's cache
    # (keys and values of every layer up to the current length)
    w_bytes = 4 * (gk.gk_gpt_numel(m.cfg) - (s.T - 1) * s.C)
    runs = [(1, None, "B1"), (16, None, "B16"), (1, (40, 1.0, 4, 0), "B1_topk40"), (16, (40, 1.0, 4, 0), "B16_topk40")]
    for B, samp, key in runs:
        with torch.cuda.stream(stream):
            kv = gk.KvCache(dctx, m.cfg, B, Tp + warm + n_steps)
            prompt = torch.randint(0, s.V, (B * Tp,), dtype=torch.int32, device="cuda")
            logits = torch.empty(B, s.V, device="cuda")
            tok = torch.empty(B, dtype=torch.int32, device="cuda")
            gk.gk_prefill(dctx, m.params, kv, prompt, Tp, logits)
            gk.gk_sample(dctx, kv, logits, s.V, tok, samp)
            gk.gk_decode_run(dctx, m.params, kv, tok, logits, tok, warm, samp)  # records the step graph
            l0 = gk.gk_launch_count(dctx)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            stream.synchronize()
            e0.record(stream)
            gk.gk_decode_run(dctx, m.params, kv, tok, logits, tok, n_steps, samp)
            e1.record(stream)
        stream.synchronize()
        gk.gk_sync(dctx)
        ms = e0.elapsed_time(e1)
        t_avg = Tp + warm + (n_steps + 1) / 2  # mean cache length the timed steps attend over
        step_bytes = w_bytes + B * 2 * s.L * s.C * 4 * t_avg
        gbs = step_bytes / (ms / n_steps / 1e3) / 1e9
        res[key] = {"tok_s": B * n_steps / (ms / 1e3), "ms_per_step": ms / n_steps, "prompt": Tp,
                    "steps": n_steps, "dtype": "f32", "launches_per_step": (gk.gk_launch_count(dctx) - l0) / n_steps,
                    "launch": "CUDA graph per step",
                    "selection": "greedy" if samp is None else "top-k 40, temperature 1.0, Philox seed 4",
                    "roofline": {"bound": "hbm", "bytes_per_step": step_bytes, "achieved_gbs": gbs, "peak_gbs": hbm,
                                 "frac": gbs / hbm}}
        kv.close()
    # uncached generation ([LM4] Generate: the whole sequence re-run per token) at batch 1 from
    # the same prompt length, the baseline the cached loop is compared with
    n_unc = 16
    with torch.cuda.stream(stream):
        kv = gk.KvCache(dctx, m.cfg, 1, Tp + n_unc + 1)
        ids = torch.zeros(1, Tp + n_unc + 1, dtype=torch.int32, device="cuda")
        ids[:, :Tp] = torch.randint(0, s.V, (1, Tp), dtype=torch.int32, device="cuda")
        logits = torch.empty(1, s.V, device="cuda")
        gk.gk_generate_uncached(dctx, m.params, kv, ids, Tp, 1, logits)  # warm-up
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gk.gk_generate_uncached(dctx, m.params, kv, ids, Tp, n_unc, logits)
        e1.record(stream)
    stream.synchronize()
    gk.gk_sync(dctx)
    ms = e0.elapsed_time(e1)
    res["B1_uncached"] = {"tok_s": n_unc / (ms / 1e3), "ms_per_token": ms / n_unc, "prompt": Tp, "steps": n_unc,
                          "dtype": "f32", "launch": "one full causal forward per token"}
    kv.close()
    # the pages' own generation workload: batch 1, a 5-token prompt, 40 new tokens, top-k 40 at
    # temperature 0.8, cached (prefill + selection + 39 decode steps) and uncached
    Tq, n_new, samp = 5, 40, (40, 0.8, 1234, 0)
    with torch.cuda.stream(stream):
        kv = gk.KvCache(dctx, m.cfg, 1, Tq + n_new)
        ids = torch.zeros(1, Tq + n_new, dtype=torch.int32, device="cuda")
        ids[:, :Tq] = torch.randint(0, s.V, (1, Tq), dtype=torch.int32, device="cuda")
        logits = torch.empty(1, s.V, device="cuda")
        tok = torch.empty(1, dtype=torch.int32, device="cuda")
        times = {}
        for rep in range(2):  # the first pass records the step graph and warms up
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            gk.gk_prefill(dctx, m.params, kv, ids[:, :Tq].contiguous(), Tq, logits)
            gk.gk_sample(dctx, kv, logits, s.V, tok, samp)
            gk.gk_decode_run(dctx, m.params, kv, tok, logits, tok, n_new - 1, samp)
            e1.record(stream)
            gk.gk_generate_uncached(dctx, m.params, kv, ids, Tq, n_new, logits, samp)
            e2.record(stream)
            stream.synchronize()
            times = {"cached": e0.elapsed_time(e1), "uncached": e1.elapsed_time(e2)}
    gk.gk_sync(dctx)
    res["page_workload"] = {"prompt": Tq, "new_tokens": n_new, "top_k": 40, "temperature": 0.8, "dtype": "f32",
                            "cached_tok_s": n_new / (times["cached"] / 1e3),
                            "uncached_tok_s": n_new / (times["uncached"] / 1e3)}
    kv.close()
    dctx.close()
    return res


def bench_decode_only():
    """The decode runs of bench_decode on the same random-init GPT-2-124M weights as the training
    bench (seed 5), without the training step's buffers."""
    import torch

    import synth
    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    s = synth.GPT2_124M
    ctx = gk.Ctx(torch.cuda.current_stream().cuda_stream, workspace_bytes=256 << 20)
    _, _, params = synth.training_case(s, 1, 5)
    m = Gpt(ctx, s.V, s.T, s.C, s.H, s.L, 1, mode="fp32")
    m.load(params)
    del params
    res = bench_decode(ctx, m, s)
    gk.gk_sync(ctx)
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=16)
    ap.add_argument("--mode", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--only", choices=["sweep", "gemm-shapes", "decode"],
                    help="run only the float32 op sweep, the bf16 products of one GPT-2 block at 16384 "
                         "rows, or the KV-cache decode runs, and print the result as one JSON line")
    args = ap.parse_args()
    if args.only:
        import torch

        torch.cuda.init()
        if args.only == "sweep":
            print(json.dumps({"op_sweep": bench_op_sweep()}))
        elif args.only == "decode":
            print(json.dumps({"decode": bench_decode_only()}))
        else:
            print(json.dumps({"gemm_bf16_gpt2_b16": bench_gemm_shapes()}))
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
