"""Benchmark: fused GEMM-RMSNorm-GEMM (+SwiGLU) forward + backward on GB300.

One step = one pass of the block's hot path over one batch of synthetic
input: fold g -> GEMM1 + residual + partial RMS -> rstd combine -> GEMM2 +
row scale + SwiGLU -> SwiGLU backward -> dgrad2 + RMSNorm backward -> dg
combine -> wgrad2 -> dgrad1 -> wgrad1, all through the C ABI.

Default workload: the 7B-size block (M=8192 tokens, d=4096, ffn 14336),
bf16 inputs/outputs, fp32 accumulation.  The metric counts 2*M*N*K per GEMM
for the forward, data-gradient and weight-gradient GEMMs (3x the forward).

Also reported on the same line: the unfused ablation (same GEMM kernel with
standalone add+RMSNorm / SwiGLU / SwiGLU-bwd / RMSNorm-bwd kernels), the
LM-head blocked-LSE cross-entropy forward+backward, the dominant kernel's
roofline, an end-to-end number through the public API with host buffers,
and the fp64 oracle timed on the host cores (cpu_baseline).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config 7b|70b]
       [--impl reference]
Under torchrun (N > 1) every rank runs an independent replica (the method is
single-GPU; there is no exchange step), rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from coda_inputs import B1, B7, B70, LMHEAD, BlockShape, CEShape, block_inputs, ce_inputs, down_proj_inputs  # noqa: E402

METRIC = "fused GEMM-RMSNorm-GEMM fwd+bwd TFLOP/s and % of GB300 bf16 dense peak"
UNIT = "TFLOP/s"
CONFIGS = {"7b": B7, "70b": B70, "1b": B1}  # 1b: forward only


E2E_REPEATS = 3  # timed runs of the end-to-end legs (median reported)

KERNEL_SOURCES = ["ptx.cuh", "gemm_tc.cuh", "gemm_tc2.cuh", "gemm_tc2w.cuh", "gemm_group.cuh", "gemm_launch.cuh", "gemm_fwd.cu",
                  "gemm_bwd.cu", "gemm_group.cu"]


def kernel_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "gemm_epilogue_transformer_tma_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` on `workload` from the ncu record in
    profiles/traffic.txt, or None if there is none or the kernel sources have
    changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_sources_sha256()
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == workload and parts[1] == kernel \
                    and parts[3] == sha:
                return float(parts[2])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s in sm if s > 0.5 * (max(mx) if mx else 1)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
class FusedStep:
    """The fused path's calls (stage name, call); CUDA events go between them.
    With fuse_rstd the light combine runs inside GEMM2's epilogue."""

    def __init__(self, C, b, fuse_rstd=False, g_on_activation=False):
        self.C, self.b = C, b
        s = b
        gemm2 = "gemm2_prms_rowscale_swiglu" if fuse_rstd else "gemm2_rowscale_swiglu"
        self.flops = {
            "gemm1_res_prms+fold": 2.0 * s.M * s.d * s.K1,
            gemm2: 2.0 * s.M * s.N2 * s.d,
            "dgrad2_rmsbwd": 2.0 * s.M * s.N2 * s.d,
            "wgrad2_gscale": 2.0 * s.M * s.N2 * s.d,
            # dgrad1 and wgrad1 run as one grouped launch
            "dgrad1_wgrad1": 2 * 2.0 * s.M * s.d * s.K1,
        }
        if g_on_activation:
            # g broadcast in GEMM1's epilogue (Hg), GEMM2 on the unfolded W2
            fwd = [("gemm1_res_prms_g", lambda: C.coda_gemm_res_prms_g(b.X, b.W1t, b.R, b.g, b.H, b.Hg, b.psum))]
            A2, B2 = b.Hg, b.W2t
            self.flops["gemm1_res_prms_g"] = self.flops.pop("gemm1_res_prms+fold")
        else:
            # the fold runs on a second stream beside GEMM1 (BlockBuffers.gemm1_and_fold)
            fwd = [("gemm1_res_prms+fold", b.gemm1_and_fold)]
            A2, B2 = b.H, b.W2gt
        # z is saved for the backward only: a forward-only workload has no use for it
        zs = b.z if b.with_backward else None
        if fuse_rstd:
            fwd.append((gemm2, lambda: C.coda_gemm_prms_rowscale_swiglu(A2, B2, b.psum, b.eps, b.rstd, b.out, zs,
                                                                        C.CODA_EPI_SWIGLU)))
        else:
            fwd += [
                ("rstd_combine", lambda: C.coda_rstd_combine(b.psum, b.d, b.eps, b.rstd)),
                (gemm2, lambda: C.coda_gemm_rowscale_swiglu(A2, B2, b.rstd, b.out, zs, C.CODA_EPI_SWIGLU)),
            ]
        bwd = [
            ("swiglu_bwd", lambda: C.coda_swiglu_bwd(b.dY, b.z, b.rstd, b.dP, b.c, b.d)),
            ("dgrad2_rmsbwd", lambda: C.coda_gemm_dgrad_rmsbwd(b.dP, b.W2t, b.H, b.g, b.c, b.dH, b.dgpart)),
            ("dg_combine", lambda: C.coda_dg_combine(b.dgpart, b.dg)),
            ("wgrad2_gscale", lambda: C.coda_gemm_wgrad_gscale(b.H, b.dP, b.g, b.dW2t)),
            ("dgrad1_wgrad1", lambda: C.coda_gemm_res_prms_bwd(b.dH, b.X, b.W1t, b.dX, b.dW1t, b.dH)),
        ]
        self.stages = fwd + (bwd if b.with_backward else [])
        self.n_fwd = len(fwd)
        # library kernels each stage launches (the fold + GEMM1 stage launches two)
        self.kernels = {name: (2 if name == "gemm1_res_prms+fold" else 1) for name, _ in self.stages}

    def names(self):
        return [n for n, _ in self.stages]

    def calls(self):
        return [f for _, f in self.stages]


def max_over_ranks(ms: float, dist=None, device="cpu") -> float:
    """The slowest rank's time per step (every rank calls this)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(step_flops: float, ms: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank runs one independent replica of the step
    (weak scaling), timed by the slowest rank."""
    return world * step_flops / (ms * 1e-3) / 1e12


class nvtx:
    """An NVTX range around a region of the bench (a profiler can restrict a
    capture to it, e.g. ncu --nvtx --nvtx-include "stage_pass/")."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        torch.cuda.nvtx.range_pop()


def time_steps(calls, steps, warmup, stage_events=True):
    """Run warmup + timed steps; return (total_ms, per-stage ms lists)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for f in calls:
            f()
    torch.cuda.synchronize()
    n = len(calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)] if stage_events else None
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        for i, f in enumerate(calls):
            if stage_events:
                evs[s][i].record(stream)
            f()
        if stage_events:
            evs[s][n].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1)
    per = None
    if stage_events:
        per = [[evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)] for i in range(n)]
    return total, per


def interleave(a_calls, b_calls, n, warmup, rounds=4):
    """Time two call sequences in rounds of n steps each, after warm-up of
    both: a then b, then b then a, and so on (an even number of rounds).  The
    part heats over a run, so two sequences timed one after the other would
    see different clocks, and the one timed second in every round would run
    hotter.  Returns (best a ms/step, best b ms/step, median per-round ratio
    b / a, the per-round pairs (a, b))."""
    for calls in (a_calls, b_calls):
        for _ in range(warmup):
            for f in calls:
                f()
    pairs = []
    for r in range(rounds):
        if r % 2 == 0:
            t_a = time_steps(a_calls, n, 0, stage_events=False)[0] / n
            t_b = time_steps(b_calls, n, 0, stage_events=False)[0] / n
        else:
            t_b = time_steps(b_calls, n, 0, stage_events=False)[0] / n
            t_a = time_steps(a_calls, n, 0, stage_events=False)[0] / n
        pairs.append((t_a, t_b))
    ratio = statistics.median(t_b / t_a for t_a, t_b in pairs)
    return min(p[0] for p in pairs), min(p[1] for p in pairs), ratio, pairs


def interleave_many(seqs, n, warmup, rounds=6):
    """Time several call sequences in rounds, each round running every
    sequence for n steps, the order reversed on every other round so that
    drift within a round (the part heating) falls on each sequence alike.
    Returns per-sequence lists of ms/step, one entry per round."""
    for calls in seqs:
        for _ in range(warmup):
            for f in calls:
                f()
    out = [[] for _ in seqs]
    for r in range(rounds):
        order = range(len(seqs)) if r % 2 == 0 else reversed(range(len(seqs)))
        for i in order:
            out[i].append(time_steps(seqs[i], n, 0, stage_events=False)[0] / n)
    return out


def rounds_ms(pairs):
    return [[round(a, 4), round(b, 4)] for a, b in pairs]


def cpu_oracle_baseline(shape: BlockShape, target_s: float = 12.0, max_rows: int = 4096):
    """fp64 oracle fwd+bwd of the block on a row sample of the workload (full
    weights), timed on the host cores.  Returns a cpu_baseline dict."""
    import numpy as np

    import oracle as O
    from coda_inputs import to_f64
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    full = block_inputs(BlockShape(shape.name, max_rows, shape.K1, shape.d, shape.N2), 0, "cpu")
    W = {k: to_f64(full[k]) for k in ("W1t", "g", "W2t")}
    rows = 32
    while True:
        A = {k: to_f64(full[k][:rows]) for k in ("X", "R", "dY")}
        t = time.perf_counter()
        O.block_backward(A["X"], W["W1t"], A["R"], W["g"], W["W2t"], A["dY"], shape.eps, True)
        dt = time.perf_counter() - t
        if dt >= target_s or rows >= max_rows:
            break
        rows = min(max_rows, max(rows * 2, int(rows * target_s / max(dt, 1e-3))))
        rows = max(8, (rows // 8) * 8)
    flops = 3.0 * (2.0 * rows * shape.d * shape.K1 + 2.0 * rows * shape.N2 * shape.d)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"fp64 numpy oracle block fwd+bwd on {rows} of {shape.M} token rows of the "
                      f"{shape.name} workload (full weights), {dt:.1f} s wall", "seconds": dt,
            "rows": rows}


_SINGLE_CORE = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import oracle as O
from coda_inputs import B1, TINY, BlockShape, block_inputs, to_f64
res = {}
for s, rows in ((TINY, TINY.M), (B1, 128)):
    x = block_inputs(BlockShape(s.name, rows, s.K1, s.d, s.N2, swiglu=s.swiglu, w_std=s.w_std, x_std=s.x_std,
                                backward=False), 0, "cpu")
    a = {k: to_f64(v) for k, v in x.items()}
    t = time.perf_counter()
    O.block_forward(a["X"], a["W1t"], a["R"], a["g"], a["W2t"], s.eps, s.swiglu)
    dt = time.perf_counter() - t
    fl = 2.0 * rows * s.d * s.K1 + 2.0 * rows * s.N2 * s.d
    res[s.name] = {"rows": rows, "of_rows": s.M, "seconds": dt, "gflops": fl / dt / 1e9}
print(json.dumps(res))
"""


def cpu_oracle_single_core():
    """The fp64 oracle's forward on one host core (the BLAS and OpenMP pools
    limited to one thread in a child process): the tiny configuration whole
    and a 128-row sample of the 1B one."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", _SINGLE_CORE, ROOT], env=env, capture_output=True, text=True,
                           timeout=300)
        out = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"error": str(e)[:200]}
    out["cores"] = 1
    return out


def run_reference(args, shape):
    """The oracle as the reference arm: timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = []
    res = None
    for i in range(args.warmup + args.steps):
        res = cpu_oracle_baseline(shape, target_s=max(2.0, 60.0 / (args.warmup + args.steps + 1)), max_rows=256)
        if i >= args.warmup:
            per_step.append(res)
    v = statistics.median([r["value"] for r in per_step])
    secs = statistics.median([r["seconds"] for r in per_step])
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": shape.name, "M": shape.M, "K1": shape.K1, "d": shape.d, "ffn": shape.N2 // 2,
                       "sample_rows": res["rows"]},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_block_workload(C, shape, steps, warmup, peaks, device_index, g_on_activation=False):
    """Another block workload on the same line: its fused step timed like the
    headline (events around `steps` steps after `warmup`), the dominant
    kernel's roofline from a second pass with events between stages, the
    unfused ablation and the other placement of the RMSNorm weight each in
    interleaved rounds with it, and the clocks sampled meanwhile."""
    from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers
    x = block_inputs(shape, seed=0, device="cuda")
    b = BlockBuffers(x, backward=shape.backward, g_on_activation=g_on_activation)
    fs = FusedStep(C, b, g_on_activation=g_on_activation)
    calls = fs.calls()
    for _ in range(warmup):
        for f in calls:
            f()
    torch.cuda.synchronize()
    with ClockSampler(device_index) as clk:
        total_ms, _ = time_steps(calls, steps, 0, stage_events=False)
        _, per = time_steps(calls, steps, 0, stage_events=True)
    st, bits = C.coda_sync_status()
    if st != 0:
        raise RuntimeError(f"device status {C.STATUS_NAMES.get(st)} bits={bits:#x}")
    ms = total_ms / steps
    step_flops = shape.fwdbwd_flops() if shape.backward else shape.fwd_flops()
    stage_ms = {name: statistics.mean(per[i]) for i, name in enumerate(fs.names())}
    dom = max((k for k in fs.flops if k in stage_ms), key=lambda k: stage_ms[k])
    dom_ach = fs.flops[dom] / (stage_ms[dom] * 1e-3) / 1e12
    clocks = clk.summary()
    n_cmp = max(3, steps // 2)
    out = {
        "workload": shape.name, "M": shape.M, "K1": shape.K1, "d": shape.d, "ffn": shape.N2 // 2,
        "pass": "forward+backward" if shape.backward else "forward (no z store)",
        "g": "on the activation (GEMM1 epilogue)" if g_on_activation else "folded into W2",
        "ms_per_step": ms, "value": step_flops / (ms * 1e-3) / 1e12, "unit": UNIT,
        "pct_of_peak": 100.0 * step_flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
        "steps": steps, "warmup": warmup, "stage_ms": stage_ms,
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": dom_ach, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": dom_ach / peaks["bf16_tflops"],
                     "frac_of_sustained": dom_ach / peaks["bf16_tflops_sustained"],
                     "traffic": measured_traffic(shape.name, dom),
                     "note": "peak = burst bf16 of %s: the kernel is timed inside a sub-second step loop" %
                             peaks["source"]},
        "clocks": clocks,
    }
    # this step, the other placement of the RMSNorm weight and the unfused
    # ablation, in interleaved rounds (order alternating between rounds)
    bo = BlockBuffers(x, backward=shape.backward, g_on_activation=not g_on_activation)
    ocalls = FusedStep(C, bo, g_on_activation=not g_on_activation).calls()
    bu = BlockBuffers(x, unfused=True, backward=shape.backward)
    ucalls = [bu.forward_unfused, bu.backward_unfused] if shape.backward else [bu.forward_unfused]
    t_this, t_other, t_unf = interleave_many([calls, ocalls, ucalls], n_cmp, warmup)
    med = statistics.median
    out["other_g_placement"] = {
        "g": "folded into W2" if g_on_activation else "on the activation (GEMM1 epilogue)",
        "ms_per_step": min(t_other), "time_vs_this_step": med(o / t for o, t in zip(t_other, t_this)),
        "vs_unfused_speedup": med(u / o for u, o in zip(t_unf, t_other)),
        "rounds_ms": [round(v, 4) for v in t_other]}
    out["ablation_unfused"] = {"ms_per_step": min(t_unf), "tflops": step_flops / (min(t_unf) * 1e-3) / 1e12,
                               "fused_speedup": med(u / t for u, t in zip(t_unf, t_this)),
                               "rounds_ms": [round(v, 4) for v in t_unf],
                               "fused_rounds_ms": [round(v, 4) for v in t_this],
                               "timing": "rounds of (this step, other g placement, unfused step), order reversed "
                                         "every other round; speedups = median per-round time ratios"}
    st, bits = C.coda_sync_status()
    if st != 0:
        raise RuntimeError(f"device status {C.STATUS_NAMES.get(st)} bits={bits:#x}")
    del bu, ucalls, bo, ocalls, b, fs, calls, x
    torch.cuda.empty_cache()
    return out


def host_link_gbs(nbytes: int = 256 << 20, reps: int = 3) -> dict:
    """Copy bandwidth between page-locked host memory and the device on this
    box (GB/s, best of `reps`), measured beside the end-to-end figure: the
    host-buffer step is bound by it once a step's copies outlast its kernels."""
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    best = {"h2d": 0.0, "d2h": 0.0}
    with torch.cuda.stream(s):
        dev.copy_(host, non_blocking=True)
        for _ in range(reps):
            for key, (dst, src) in (("h2d", (dev, host)), ("d2h", (host, dev))):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                dst.copy_(src, non_blocking=True)
                e1.record(s)
                e1.synchronize()
                best[key] = max(best[key], nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    torch.cuda.synchronize()
    return {k: round(v, 1) for k, v in best.items()}


def bench_memory_kernels(C, b, shape, hbm_gbs, warmup=10, iters=50):
    """The memory-bound kernels of the step, each launched alone: warmup
    untimed launches, then iters launches each preceded by a write of a
    buffer twice the L2's size (so every launch starts with a cold L2) and
    timed with CUDA events on the launching stream.  Algorithmic bytes per
    launch: what the kernel must read and write once."""
    M, d, N2, F = shape.M, shape.d, shape.N2, shape.N2 // 2
    T = C.coda_prms_num_tiles(d)
    rows = b.dgpart.shape[0] if shape.backward else 0
    kernels = [
        ("fold", 2 * N2 * d * 2, lambda: C.coda_fold_rmsnorm_weight(b.W2t, b.g, b.W2gt)),
        ("rstd_combine", M * T * 4 + M * 4, lambda: C.coda_rstd_combine(b.psum, b.d, b.eps, b.rstd)),
    ]
    if shape.backward:
        kernels += [
            ("swiglu_bwd", M * F * 2 + 2 * M * N2 * 2 + 2 * M * 4,
             lambda: C.coda_swiglu_bwd(b.dY, b.z, b.rstd, b.dP, b.c, b.d)),
            ("dg_combine", rows * d * 4 + d * 4, lambda: C.coda_dg_combine(b.dgpart, b.dg)),
        ]
    flush = torch.empty(2 * 129 * 2 ** 20, dtype=torch.uint8, device="cuda")
    out = {}
    for name, nbytes, f in kernels:
        for _ in range(warmup):
            f()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            f()
            e1.record()
        torch.cuda.synchronize()
        us = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs)
        med = statistics.median(us)
        out[name] = {"median_us": med, "min_us": us[0], "max_us": us[-1], "bytes": nbytes,
                     "gbs": nbytes / (med * 1e-6) / 1e9, "frac_of_hbm": nbytes / (med * 1e-6) / 1e9 / hbm_gbs}
    out["timing"] = (f"each kernel alone: {warmup} warm-up launches, then {iters} timed launches, each after a "
                     f"{flush.numel() >> 20} MiB write that flushes the L2; median, min and max of the CUDA-event "
                     "times; GB/s = algorithmic bytes / median (not meaningful for the latency-bound combines)")
    out["peak_gbs"] = hbm_gbs
    return out


def bench_down_proj_swiglu_bwd(C, b, shape, steps, warmup):
    """The SwiGLU backward fed by a down projection's data gradient:
    dY = dYb W3 through HBM (plain GEMM + streaming SwiGLU-backward kernel +
    dgrad2 with c) against dY kept on chip (GEMM with the SwiGLU-backward
    epilogue + dgrad2 forming c from the epilogue's partial sums)."""
    dp = down_proj_inputs(shape, 0, "cuda")
    dY = torch.empty(shape.M, shape.F, dtype=torch.bfloat16, device="cuda")
    cpart = torch.empty(shape.M, C.coda_prms_num_tiles(shape.F), device="cuda")
    through_hbm = [
        lambda: C.coda_gemm(dp["dYb"], False, dp["W3t"], True, dY, shape.M, shape.F, shape.d),
        lambda: C.coda_swiglu_bwd(dY, b.z, b.rstd, b.dP, b.c, shape.d),
        lambda: C.coda_gemm_dgrad_rmsbwd(b.dP, b.W2t, b.H, b.g, b.c, b.dH, b.dgpart),
    ]
    on_chip = [
        lambda: C.coda_gemm_dgrad_swiglu_bwd(dp["dYb"], dp["W3t"], b.z, b.rstd, b.dP, cpart),
        lambda: C.coda_gemm_dgrad_rmsbwd_cpart(b.dP, b.W2t, b.H, b.g, b.rstd, cpart, b.dH, b.dgpart),
    ]
    n = max(3, steps // 2)
    t_chip, t_hbm, ratio, pairs = interleave(on_chip, through_hbm, n, warmup)
    flops = 2.0 * shape.M * shape.F * shape.d + 2.0 * shape.M * shape.N2 * shape.d
    return {"what": "down-proj dgrad + SwiGLU bwd + dgrad2/RMSNorm bwd", "dY_through_hbm_ms": t_hbm,
            "dY_on_chip_ms": t_chip, "speedup": ratio, "on_chip_tflops": flops / (t_chip * 1e-3) / 1e12,
            "rounds_ms": rounds_ms(pairs), "timing": "rounds of (on chip, through HBM), the order reversed every other round; speedup = "
                                                   "median per-round time ratio"}


def bench_fp8_forward(C, b, shape, steps, warmup, peak_bf16):
    """The block forward with e4m3 operands (per-tensor scales; activations X
    and H quantised in the step, weights once beforehand, their cost reported
    apart) against the same forward in bf16."""
    u8 = torch.uint8
    dev = "cuda"
    Xq = torch.empty(shape.M, shape.K1, dtype=u8, device=dev)
    Hq = torch.empty(shape.M, shape.d, dtype=u8, device=dev)
    W1q = torch.empty(shape.d, shape.K1, dtype=u8, device=dev)
    W2q = torch.empty(shape.N2, shape.d, dtype=u8, device=dev)
    sc = torch.empty(4, 2, device=dev)
    weights = [lambda: C.coda_fp8_quantize(b.W1t, W1q, sc[1]),
               lambda: C.coda_fp8_quantize(b.W2t, W2q, sc[2], b.g)]
    fp8 = [
        lambda: C.coda_fp8_quantize(b.X, Xq, sc[0]),
        lambda: C.coda_gemm_res_prms_fp8(Xq, sc[0, 1:], W1q, sc[1, 1:], b.R, b.H, b.psum),
        lambda: C.coda_rstd_combine(b.psum, b.d, b.eps, b.rstd),
        lambda: C.coda_fp8_quantize(b.H, Hq, sc[3]),
        lambda: C.coda_gemm_rowscale_swiglu_fp8(Hq, sc[3, 1:], W2q, sc[2, 1:], b.rstd, b.out,
                                                b.z if b.with_backward else None),
    ]
    fs = FusedStep(C, b)
    bf16 = fs.calls()[:fs.n_fwd]  # the bf16 forward stages
    n = max(3, steps)
    t_w, _ = time_steps(weights, n, warmup, stage_events=False)
    _, per8 = time_steps(fp8, n, warmup, stage_events=True)
    t_8, t_16, ratio, pairs = interleave(fp8, bf16, n, warmup)
    fl = shape.fwd_flops()
    names = ["quantize_X", "gemm1_res_prms_fp8", "rstd_combine", "quantize_H", "gemm2_rowscale_swiglu_fp8"]
    g2 = statistics.mean(per8[4])
    return {"workload": shape.name + " forward", "fp8_fwd_ms": t_8, "bf16_fwd_ms": t_16,
            "speedup": ratio, "rounds_ms": rounds_ms(pairs), "fp8_fwd_tflops": fl / (t_8 * 1e-3) / 1e12,
            "weight_quantize_ms": t_w / n, "stage_ms": {k: statistics.mean(v) for k, v in zip(names, per8)},
            "timing": "rounds of (fp8, bf16), the order reversed every other round; speedup = median per-round time ratio; stage_ms from "
                      "a separate pass with an event between stages",
            "gemm2_fp8_tflops": 2.0 * shape.M * shape.N2 * shape.d / (g2 * 1e-3) / 1e12,
            "fp8_peak_tflops": 2 * peak_bf16,
            "gemm2_frac_of_fp8_peak": 2.0 * shape.M * shape.N2 * shape.d / (g2 * 1e-3) / 1e12 / (2 * peak_bf16),
            "peak_note": "fp8 dense peak taken as 2x the measured burst bf16 peak (nominal ratio 4.5 / 2.25 "
                         "PFLOP/s); GEMM2 timed in a stage pass inside the step loop"}


def bench_fp8_fwdbwd(C, b, shape, steps, warmup, peak_bf16):
    """The block forward + backward with FP8 operands (e4m3 activations and
    weights, e5m2 gradients; activation and gradient quantisation in the
    step, weight quantisation timed apart) against the bf16 step."""
    n = max(3, steps)
    named = b.fp8_forward_calls() + b.fp8_backward_calls()
    calls = [f for _, f in named]
    t_w, _ = time_steps([b.fp8_quantize_weights], n, warmup, stage_events=False)
    _, per8 = time_steps(calls, n, warmup, stage_events=True)
    bf16 = FusedStep(C, b).calls()
    t_8, t_16, ratio, pairs = interleave(calls, bf16, n, warmup)
    fl = shape.fwdbwd_flops()
    # delayed scaling of dP's codes (the previous step's amax; one pass of the
    # SwiGLU backward instead of two), against the exact form and bf16
    dnamed = b.fp8_forward_calls() + b.fp8_backward_calls(delayed=True)
    dcalls = [f for _, f in dnamed]
    _, perd = time_steps(dcalls, n, warmup, stage_events=True)
    t_d, _, ratio_d8, pairs_d8 = interleave(dcalls, calls, n, warmup)
    _, _, ratio_d16, pairs_d16 = interleave(dcalls, bf16, n, warmup)
    names = [k for k, _ in dnamed]
    # the FP8 step end to end through the C ABI with host buffers (the block
    # executor in FP8 mode, weights quantised once beforehand)
    from gemm_epilogue_transformer_tma_gb300.path import HostBlockStepper
    st = HostBlockStepper(b.W1t, b.g, b.W2t, shape.M, shape.eps, fp8=True)
    host = {k: getattr(b, k).cpu().pin_memory() for k in ("X", "R", "dY")}
    host.update(st.host_buffers(dX=True))
    for _ in range(3):
        st.submit(host["X"], host["R"], host["dY"], dX=host["dX"])
    st.sync()
    runs = []
    for _ in range(E2E_REPEATS):
        t0 = time.perf_counter()
        for _ in range(n):
            st.submit(host["X"], host["R"], host["dY"], dX=host["dX"])
        st.sync()
        runs.append((time.perf_counter() - t0) * 1e3 / n)
    e2e_ms = statistics.median(runs)
    st.close()
    del st, host
    e2e = {"value": fl / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms, "steps": n,
           "runs_ms_per_step": runs,
           "api": "coda_block_create(CODA_BLOCK_FP8) / coda_block_step_host / coda_block_sync (host buffers)",
           "timing": "host wall clock, synchronize at both ends, median of three runs; H2D of X, R, dY and D2H of dX "
                     "inside"}
    delayed = {"fp8_fwdbwd_ms": t_d, "fp8_fwdbwd_tflops": fl / (t_d * 1e-3) / 1e12,
               "speedup_vs_exact_fp8": ratio_d8, "speedup_vs_bf16": ratio_d16,
               "swiglu_bwd_e5m2_ms": statistics.mean(perd[names.index("swiglu_bwd_e5m2")]),
               "rounds_ms_vs_exact_fp8": rounds_ms(pairs_d8), "rounds_ms_vs_bf16": rounds_ms(pairs_d16)}
    return {"workload": shape.name, "fp8_fwdbwd_ms": t_8, "bf16_fwdbwd_ms": t_16, "speedup": ratio,
            "rounds_ms": rounds_ms(pairs), "fp8_fwdbwd_tflops": fl / (t_8 * 1e-3) / 1e12, "weight_quantize_ms": t_w / n,
            "stage_ms": {k: statistics.mean(v) for (k, _), v in zip(named, per8)},
            "timing": "rounds of (fp8, bf16), the order reversed every other round; speedup = median per-round time ratio; stage_ms from a "
                      "separate pass with an event between stages",
            "formats": "e4m3 activations and weights, e5m2 gradients (dP, dH), one fp32 scale per tensor",
            "delayed_dP_scaling": delayed, "e2e": e2e}


def bench_qkv_rope(C, steps, warmup, M=8192, S=2048, d=4096, n_heads=32):
    """QKV projection of the 7B-size block (MHA, 32 heads of 128) with RoPE
    in the epilogue, against the plain GEMM followed by a standalone RoPE
    kernel."""
    g = torch.Generator(device="cuda").manual_seed(11)
    X = torch.randn(M, d, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(3 * n_heads * 128, d, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    cos_t = torch.empty(S, 64, device="cuda")
    sin_t = torch.empty(S, 64, device="cuda")
    C.coda_rope_table(cos_t, sin_t)
    N = 3 * n_heads * 128
    qkv = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    fused = [lambda: C.coda_gemm_qkv_rope(X, W, cos_t, sin_t, qkv, n_heads, n_heads)]
    unfused = [lambda: C.coda_gemm(X, False, W, False, qkv, M, N, d),
               lambda: C.coda_rope_apply(qkv, cos_t, sin_t, n_heads, n_heads)]
    n = max(3, steps)
    t_f, t_u, ratio, pairs = interleave(fused, unfused, n, warmup)
    flops = 2.0 * M * N * d
    return {"M": M, "d": d, "heads": n_heads, "head_dim": 128, "seq": S, "fused_ms": t_f,
            "unfused_ms": t_u, "speedup": ratio, "fused_tflops": flops / (t_f * 1e-3) / 1e12,
            "rounds_ms": rounds_ms(pairs), "timing": "rounds of (fused, unfused), the order reversed every other round; speedup = median "
                                                   "per-round time ratio"}


def _vs_library(ours, lib, lib_name, flops, n, warmup, rounds=4):
    """The library's GEMM against a vendor library's on the same operands:
    rounds of n launches each, the order reversed every other round (the part
    heats over a run).  Medians over rounds; ratio = median per-round time
    ratio (vendor / ours, above 1 when ours is faster)."""
    t_o, t_l = interleave_many([ours, lib], n, warmup, rounds=rounds)
    mo, ml = statistics.median(t_o), statistics.median(t_l)
    return {"coda_ms": mo, f"{lib_name}_ms": ml, "coda_tflops": flops / mo / 1e9,
            f"{lib_name}_tflops": flops / ml / 1e9,
            "ratio": statistics.median(b / a for a, b in zip(t_o, t_l)),
            "rounds_ms": rounds_ms(zip(t_o, t_l)),
            "timing": "rounds of n launches, order alternating; medians over rounds"}


def bench_plain_vs_cublas(C, shape, steps, warmup):
    """The library's plain GEMM (K-major operands, bf16 store, no epilogue
    work) against cuBLAS (torch.matmul) on the GEMM shapes of the step, same
    operands, interleaved.  Context for the roofline: the denominator is a
    cuBLAS figure taken on its own best shape."""
    out = {}
    n = max(3, steps // 2)
    for name, (M, N, K) in {"gemm2": (shape.M, shape.N2, shape.d), "dgrad2": (shape.M, shape.d, shape.N2),
                            "gemm1": (shape.M, shape.d, shape.K1)}.items():
        g = torch.Generator(device="cuda").manual_seed(0)
        A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
        B = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
        Cd = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        ours = [lambda: C.coda_gemm(A, False, B, False, Cd, M, N, K)]
        lib = [lambda: torch.matmul(A, B.t(), out=Cd)]
        out[name] = {"M": M, "N": N, "K": K, **_vs_library(ours, lib, "cublas", 2.0 * M * N * K, n, warmup)}
        del A, B, Cd
        torch.cuda.empty_cache()
    return out


def bench_fp8_plain_vs_cublaslt(C, shape, steps, warmup):
    """The library's plain 8-bit GEMM (e4m3 K-major operands, unit scales,
    bf16 store) against cuBLASLt's (torch._scaled_mm) on the GEMM2 and dgrad2
    shapes, same codes, interleaved: a measured library figure for the FP8
    rate beside the nominal 2x of the bf16 peak."""
    if not hasattr(torch, "_scaled_mm") or not hasattr(torch, "float8_e4m3fn"):
        return {"unavailable": "torch has no float8 matmul"}
    out = {}
    n = max(3, steps // 2)
    one = torch.ones((), device="cuda")
    for name, (M, N, K) in {"gemm2": (shape.M, shape.N2, shape.d), "dgrad2": (shape.M, shape.d, shape.N2)}.items():
        g = torch.Generator(device="cuda").manual_seed(0)
        A = (torch.randn(M, K, device="cuda", generator=g) * 16).to(torch.float8_e4m3fn)
        B = (torch.randn(N, K, device="cuda", generator=g) * 16).to(torch.float8_e4m3fn)
        Cd = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        Au, Bu = A.view(torch.uint8), B.view(torch.uint8)
        ours = [lambda: C.coda_gemm_fp8(Au, False, C.E4M3, None, Bu, False, C.E4M3, None, Cd, M, N, K)]
        try:
            torch._scaled_mm(A, B.t(), one, one, out_dtype=torch.bfloat16)
        except Exception as e:  # noqa: BLE001 - report, do not fail the bench
            return {"unavailable": f"torch._scaled_mm: {str(e).splitlines()[0][:160]}"}
        lib = [lambda: torch._scaled_mm(A, B.t(), one, one, out_dtype=torch.bfloat16)]
        out[name] = {"M": M, "N": N, "K": K, **_vs_library(ours, lib, "cublaslt", 2.0 * M * N * K, n, warmup)}
        del A, B, Au, Bu, Cd
        torch.cuda.empty_cache()
    return out


def bench_lmhead(C, steps, warmup, tokens=0):
    s = LMHEAD if not tokens else CEShape(f"{LMHEAD.name}_m{tokens}", tokens, LMHEAD.d, LMHEAD.V)
    x = ce_inputs(s, 0, "cuda")
    ws = torch.empty(C.coda_lmhead_ce_workspace_bytes(s.M, s.d, s.V, True), dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(s.M, device="cuda")
    am = torch.empty(s.M, dtype=torch.int32, device="cuda")
    dH = torch.empty(s.M, s.d, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(s.V, s.d, dtype=torch.bfloat16, device="cuda")
    fwd = [lambda: C.coda_lmhead_ce(x["H"], x["Wt"], x["labels"], loss, lse, am, None, None, ws)]
    both = [lambda: C.coda_lmhead_ce(x["H"], x["Wt"], x["labels"], loss, lse, am, dH, dW, ws)]
    tf, _ = time_steps(fwd, max(1, steps // 2), 1, stage_events=False)
    tb, _ = time_steps(both, max(1, steps // 2), 1, stage_events=False)
    n = max(1, steps // 2)
    g = s.gemm_flops()
    ms_f, ms_b = tf / n, tb / n
    out = {"workload": s.name, "M": s.M, "d": s.d, "V": s.V, "fwd_ms": ms_f, "fwdbwd_ms": ms_b,
           "fwd_tflops": g / ms_f / 1e9, "fwdbwd_tflops_counted": 3 * g / ms_b / 1e9,
           "fwdbwd_tflops_executed": 4 * g / ms_b / 1e9, "loss": loss.item()}
    # the same on FP8 operands: H quantised in the step, W once (timed apart),
    # dL kept as e5m2 codes; interleaved with the bf16 form
    u8 = torch.uint8
    Hq = torch.empty(s.M, s.d, dtype=u8, device="cuda")
    Wq = torch.empty(s.V, s.d, dtype=u8, device="cuda")
    sc = torch.empty(2, 2, device="cuda")
    loss8, lse8 = torch.empty(1, device="cuda"), torch.empty(s.M, device="cuda")
    dH8 = torch.empty_like(dH)
    dW8 = torch.empty_like(dW)
    wq = [lambda: C.coda_fp8_quantize(x["Wt"], Wq, sc[1])]
    t_wq, _ = time_steps(wq, max(1, steps // 2), 1, stage_events=False)
    fp8_both = [lambda: C.coda_fp8_quantize(x["H"], Hq, sc[0]),
                lambda: C.coda_lmhead_ce_fp8(Hq, sc[0, 1:], Wq, sc[1, 1:], x["labels"], loss8, lse8, None, dH8, dW8,
                                             ws)]
    t8, t16, ratio, pairs = interleave(fp8_both, both, n, 1)
    out["fp8"] = {"fwdbwd_ms": t8, "bf16_fwdbwd_ms": t16, "speedup": ratio, "rounds_ms": rounds_ms(pairs),
                  "fwdbwd_tflops_executed": 4 * g / t8 / 1e9, "weight_quantize_ms": t_wq / max(1, steps // 2),
                  "loss": loss8.item(),
                  "formats": "e4m3 H and W (per-tensor power-of-two scales), e5m2 dL (scale fixed by |dL| <= 1/M)",
                  "timing": "rounds of (fp8, bf16), the order reversed every other round; speedup = median per-round time ratio"}
    del x, ws, dH, dW, Hq, Wq, dH8, dW8
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="7b", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="fused", choices=["fused", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip ablation, LM-head and e2e legs")
    ap.add_argument("--fuse-rstd", action="store_true",
                    help="fold the rstd combine into GEMM2's epilogue (one launch fewer)")
    ap.add_argument("--g-on-activation", action="store_true",
                    help="apply the RMSNorm weight in GEMM1's epilogue (Hg) instead of folding it into W2")
    ap.add_argument("--single-sm", action="store_true",
                    help="GEMMs on one SM per tile instead of SM pairs")
    ap.add_argument("--wide-tiles", type=int, default=0, metavar="J",
                    help="256 x 512 pair tiles with lead J for the long-K backward GEMMs (coda_set_wide_tiles)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the token count M (smaller cases for profiler captures)")
    ap.add_argument("--leg", default="", choices=["", "lmhead", "fp8"],
                    help="run only this extra leg and print its JSON (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    shape = CONFIGS[args.config]
    if args.tokens:
        shape = BlockShape(f"{shape.name}_m{args.tokens}", args.tokens, shape.K1, shape.d, shape.N2,
                           backward=shape.backward)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, shape)
    if args.leg:
        import gemm_epilogue_transformer_tma_gb300 as C
        from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        if args.leg == "lmhead":
            out = {"lmhead_ce": bench_lmhead(C, args.steps, args.warmup, args.tokens)}
        else:
            b = BlockBuffers(block_inputs(shape, seed=0, device="cuda"), backward=shape.backward)
            pk = load_peaks()["bf16_tflops"]
            out = {"next_fp8_forward": bench_fp8_forward(C, b, shape, args.steps, args.warmup, pk)}
            if shape.backward:
                out["next_fp8_fwdbwd"] = bench_fp8_fwdbwd(C, b, shape, args.steps, args.warmup, pk)
            del b
            torch.cuda.empty_cache()
            out["fp8_plain_gemm_vs_cublaslt"] = bench_fp8_plain_vs_cublaslt(C, shape, args.steps, args.warmup)
        print(json.dumps(out), flush=True)
        return

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import gemm_epilogue_transformer_tma_gb300 as C
    from gemm_epilogue_transformer_tma_gb300.path import BlockBuffers, HostBlockStepper
    peaks = load_peaks()
    C.coda_set_sm_pairing(not args.single_sm)
    C.coda_set_wide_tiles(args.wide_tiles)

    x = block_inputs(shape, seed=rank, device="cuda")
    b = BlockBuffers(x, backward=shape.backward, fuse_rstd=args.fuse_rstd, g_on_activation=args.g_on_activation)
    fs = FusedStep(C, b, fuse_rstd=args.fuse_rstd, g_on_activation=args.g_on_activation)
    calls = fs.calls()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # warmup + timed region (clock sampling during it)
    for _ in range(args.warmup):
        for f in calls:
            f()
    barrier()
    with ClockSampler(local) as clk:
        # headline: events only around the whole region, so nothing sits
        # between launches (an event between kernels would also stop the
        # next kernel's prologue from overlapping the previous one's tail)
        with nvtx("headline"):
            total_ms, _ = time_steps(calls, args.steps, 0, stage_events=False)
        # per-stage breakdown: a second pass with an event between stages
        with nvtx("stage_pass"):
            _, per = time_steps(calls, args.steps, 0, stage_events=True)
    barrier()
    st, bits = C.coda_sync_status()
    if st != 0:
        raise RuntimeError(f"device status {C.STATUS_NAMES.get(st)} bits={bits:#x}")
    ms = max_over_ranks(total_ms / args.steps, dist, "cuda")
    step_flops = shape.fwdbwd_flops() if shape.backward else shape.fwd_flops()
    value = aggregate_value(step_flops, ms, world)
    stage_ms = {name: statistics.mean(per[i]) for i, name in enumerate(fs.names())}
    dom = max((k for k in fs.flops if k in stage_ms), key=lambda k: stage_ms[k])
    dom_ach = fs.flops[dom] / (stage_ms[dom] * 1e-3) / 1e12
    clocks = clk.summary()
    # The dominant kernel is timed in the stage pass, inside a step loop of
    # well under a second: its denominator is the burst cuBLAS figure (the
    # sustained one is for kernels timed inside seconds-long runs), with its
    # fraction of the sustained figure reported beside it.
    peak = peaks["bf16_tflops"]
    peak_kind = "burst"

    launches = sum(fs.kernels.values()) * args.steps
    extras = {}
    if not args.no_extras:
        # end to end through the C ABI with host buffers: the library's block
        # executor (coda_block_*) takes each step's inputs from page-locked
        # host memory and reads its result back; every rank runs its replica
        # between barriers, the slowest rank's time counts
        ins = ("X", "R", "dY") if shape.backward else ("X", "R")
        res = "dX" if shape.backward else "out"
        host = {k: torch.empty_like(x[k], device="cpu").pin_memory() for k in ins}
        for k in host:
            host[k].copy_(x[k])
        stepper = HostBlockStepper(b.W1t, b.g, b.W2t, shape.M, shape.eps, backward=shape.backward)
        host.update(stepper.host_buffers(out=not shape.backward, dX=shape.backward))

        def e2e_steps(n):
            for _ in range(n):
                stepper.submit(host["X"], host["R"], host.get("dY"), out=host.get("out"), dX=host.get("dX"))
            stepper.sync()

        e2e_steps(3)
        # as many steps as the headline: the first step's H2D copy and the
        # last step's read-back overlap nothing and are timed in full.  The
        # run is timed three times, each beside a run of the same number of
        # device-resident steps (the order alternating), and the medians
        # taken: a host wall clock also counts any stall of the host thread,
        # and the part heats over the bench, so this leg, which runs after
        # the headline, is compared with device steps timed at the same
        # point rather than with the headline.
        n_e2e = max(3, args.steps)
        runs, dev_runs = [], []
        for r in range(E2E_REPEATS):
            for leg in (("e2e", "dev") if r % 2 == 0 else ("dev", "e2e")):
                if leg == "dev":
                    barrier()
                    dev_runs.append(max_over_ranks(time_steps(calls, n_e2e, 0, stage_events=False)[0] / n_e2e,
                                                   dist, "cuda"))
                    continue
                barrier()
                t0 = time.perf_counter()
                with nvtx("e2e"):
                    e2e_steps(n_e2e)
                barrier()
                runs.append(max_over_ranks((time.perf_counter() - t0) * 1e3 / n_e2e, dist, "cuda"))
        e2e_ms = statistics.median(runs)
        h2d = sum(host[k].numel() * host[k].element_size() for k in ins)
        d2h = host[res].numel() * host[res].element_size()
        extras["e2e"] = {"value": aggregate_value(step_flops, e2e_ms, world), "unit": UNIT, "ms_per_step": e2e_ms,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "steps": n_e2e, "runs_ms_per_step": runs,
                         "device_runs_ms_per_step": dev_runs,
                         "vs_device_same_rounds": statistics.median(d / e for d, e in zip(dev_runs, runs)),
                         "host_link_gbs": host_link_gbs(),
                         "h2d_ms_per_step_at_link_rate": None,
                         "api": "coda_block_create / coda_block_step_host / coda_block_sync (host buffers)",
                         "timing": "host wall clock over the whole run, synchronize (and barrier) at both ends, "
                                   "median of three runs, each beside a run of device-resident steps "
                                   "(vs_device_same_rounds: median per-round device / e2e time); the "
                                   "executor overlaps step i+1's H2D copies and step i-1's D2H read-back "
                                   "with step i's kernels; each step's backward waits for its dY copy, its "
                                   "forward for X and R only; the first step's X / R copy and the last step's "
                                   "D2H overlap nothing; per-rank bytes, value summed over ranks"}
        link = extras["e2e"]["host_link_gbs"]
        extras["e2e"]["h2d_ms_per_step_at_link_rate"] = h2d / (link["h2d"] * 1e9) * 1e3 if link["h2d"] else None
        stepper.close()
        del host, stepper
    if not args.no_extras and rank == 0:
        # Comparisons against the headline step are timed interleaved with it
        # (rounds of fused / other, adjacent in time): the part heats over a
        # run, and a leg timed once after the headline would see a hotter
        # part than the headline did.
        n_cmp = max(3, args.steps // 2)

        # the same step with g broadcast in GEMM1's epilogue (no fold pass over
        # W2) and the combine inside GEMM2's epilogue
        if not args.g_on_activation or not args.fuse_rstd:
            bv = BlockBuffers(x, backward=shape.backward, fuse_rstd=True, g_on_activation=True)
            vcalls = FusedStep(C, bv, fuse_rstd=True, g_on_activation=True).calls()
            _, v_ms, ratio, pairs = interleave(calls, vcalls, n_cmp, args.warmup)
            extras["variant_g_on_activation_fused_rstd"] = {
                "ms_per_step": v_ms, "value": step_flops / (v_ms * 1e-3) / 1e12,
                "time_vs_headline_step": ratio, "rounds_ms": rounds_ms(pairs),
                "timing": "rounds of (headline step, variant), the order reversed every other round; ratio = median per-round time ratio",
                "launches_per_step": len(vcalls)}
            del bv, vcalls
            torch.cuda.empty_cache()
        # the same step with 256 x 512 pair tiles for its long-K GEMMs (dgrad2):
        # the handle option is set before and cleared after each variant step
        if not args.wide_tiles and shape.backward:
            lead = 8
            wcalls = [lambda: C.coda_set_wide_tiles(lead)] + list(calls) + [lambda: C.coda_set_wide_tiles(0)]
            t_h, t_w = interleave_many([calls, wcalls], n_cmp, args.warmup, rounds=4)
            C.coda_set_wide_tiles(0)
            w_ms = statistics.median(t_w)
            extras["variant_wide_tiles"] = {
                "lead": lead, "ms_per_step": w_ms, "value": step_flops / (w_ms * 1e-3) / 1e12,
                "time_vs_headline_step": statistics.median(w / h for h, w in zip(t_h, t_w)),
                "rounds_ms": rounds_ms(zip(t_h, t_w)),
                "gemms": "dgrad2 (K = 2F) on 256 x 512 tiles; the other GEMMs as in the headline step",
                "timing": "rounds of (headline step, variant), the order reversed every other round; "
                          "ratio = median per-round time ratio"}
        # unfused ablation, same workload, interleaved the same way
        bu = BlockBuffers(x, unfused=True, backward=shape.backward)
        ucalls = [bu.forward_unfused, bu.backward_unfused] if shape.backward else [bu.forward_unfused]
        _, u_ms, ratio, pairs = interleave(calls, ucalls, n_cmp, args.warmup)
        extras["ablation_unfused"] = {"ms_per_step": u_ms, "tflops": step_flops / (u_ms * 1e-3) / 1e12,
                                      "fused_speedup": ratio, "rounds_ms": rounds_ms(pairs),
                                      "timing": "rounds of (fused step, unfused step), the order reversed every other round; speedup = median "
                                                "per-round time ratio"}
        del bu
        torch.cuda.empty_cache()
        with nvtx("memory_kernels"):
            extras["memory_kernels"] = bench_memory_kernels(C, b, shape, peaks["hbm_gbs"])
        torch.cuda.empty_cache()
        if shape.backward:
            with nvtx("next_swiglu_bwd_in_down_proj_dgrad"):
                extras["next_swiglu_bwd_in_down_proj_dgrad"] = bench_down_proj_swiglu_bwd(C, b, shape, args.steps,
                                                                                        args.warmup)
            torch.cuda.empty_cache()
        with nvtx("next_fp8_forward"):
            extras["next_fp8_forward"] = bench_fp8_forward(C, b, shape, args.steps, args.warmup, peak)
        torch.cuda.empty_cache()
        if shape.backward:
            with nvtx("next_fp8_fwdbwd"):
                extras["next_fp8_fwdbwd"] = bench_fp8_fwdbwd(C, b, shape, args.steps, args.warmup, peak)
            torch.cuda.empty_cache()
        del b, x, fs, calls
        torch.cuda.empty_cache()
        with nvtx("plain_gemm_vs_cublas"):
            extras["plain_gemm_vs_cublas"] = bench_plain_vs_cublas(C, shape, args.steps, args.warmup)
        with nvtx("fp8_plain_gemm_vs_cublaslt"):
            extras["fp8_plain_gemm_vs_cublaslt"] = bench_fp8_plain_vs_cublaslt(C, shape, args.steps, args.warmup)
        torch.cuda.empty_cache()
        with nvtx("lmhead_ce"):
            extras["lmhead_ce"] = bench_lmhead(C, args.steps, args.warmup)
        torch.cuda.empty_cache()
        with nvtx("next_qkv_rope"):
            extras["next_qkv_rope"] = bench_qkv_rope(C, args.steps, args.warmup)
        torch.cuda.empty_cache()
        # the other block workloads of the method's experiments: 70B-size
        # forward+backward (d = 8192) and 1B-size forward, each with its own
        # roofline, ablation and clocks.  Both take the RMSNorm weight on the
        # activation (broadcast in GEMM1's epilogue), which measured faster
        # than the fold at these shapes; the fold's figures are reported beside.
        for key, other in (("bench_70b", B70), ("bench_1b", B1)):
            if other.name == shape.name:
                continue
            with nvtx(key):
                extras[key] = bench_block_workload(C, other, args.steps, args.warmup, peaks, local,
                                                   g_on_activation=True)
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1)/N(0,0.02)/U(0.5,1.5))",
            "config": {"workload": shape.name, "M": shape.M, "K1": shape.K1, "d": shape.d, "ffn": shape.N2 // 2,
                       "eps": shape.eps, "parallelism": "replicas" if world > 1 else "single-gpu",
                       "gemm": "1-SM tiles" if args.single_sm else (
                           f"SM-pair tiles, 256 x 512 on the long-K backward GEMMs (lead {args.wide_tiles})"
                           if args.wide_tiles else "SM-pair tiles"),
                       "rstd": "in GEMM2's epilogue" if args.fuse_rstd else "separate combine kernel",
                       "g": "on the activation (GEMM1 epilogue)" if args.g_on_activation else "folded into W2",
                       "l2": "inputs larger than L2 (W2 alone is %d MB), no flush" % (shape.N2 * shape.d * 2 >> 20)},
            "pct_of_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "pct_of_sustained_peak": 100.0 * value / world / peaks["bf16_tflops_sustained"],
            "peak": {"used": "burst for pct_of_peak and the roofline", "bf16_tflops_burst": peaks["bf16_tflops"],
                     "bf16_tflops_sustained": peaks["bf16_tflops_sustained"], "source": peaks["source"]},
            "roofline": {"kernel": dom, "bound": "tensor", "achieved": dom_ach, "peak": peak, "unit": "TFLOP/s",
                         "frac": dom_ach / peak, "frac_of_sustained": dom_ach / peaks["bf16_tflops_sustained"],
                         "traffic": measured_traffic(shape.name, dom),
                         "note": "peak = %s bf16 of %s: the kernel is timed inside the step loop (stage pass); "
                                 "nvidia-smi SM clock %s of max %s MHz" % (
                                     peak_kind, peaks["source"], clocks.get("sm_mhz"), clocks.get("sm_max_mhz"))},
            "stage_ms": stage_ms,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if "e2e" in extras:
            line["e2e"] = extras.pop("e2e")
        line.update(extras)
        if not args.no_cpu_baseline and world == 1:
            # the oracle's host-core baseline: rank 0 of a single-GPU run only
            line["cpu_baseline"] = cpu_oracle_baseline(shape)
            line["cpu_baseline"]["single_core_fwd"] = cpu_oracle_single_core()
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
