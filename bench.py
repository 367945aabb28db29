"""Throughput of one latent-MoE layer (the prefill chunk: T=16384, d=8192, p=4096,
E=256, top-k 8, I=4096, BF16) through the C ABI on GB300s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload prefill_bf16|decode_bf16|skewed_bf16|prefill_nvfp4|decode_nvfp4|...]

A step is one moe_forward over one batch of T synthetic tokens (all eight stages:
norm, router + top-k, pooler, dispatch, gate/up + SwiGLU, down, combine, unpooler).
Inputs are resident in HBM when the timed region starts; the 24 GB of expert weights
and the 256 MB activation batch are larger than L2, so no flush is needed between
steps.  Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); the elapsed time is the max over ranks.

Prints one JSON line (rank 0).  `--impl reference` times the float64 CPU oracle on
the host cores on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "latent-MoE layer tokens/s on 1 GB300; % of BF16/FP4 tensor peak and HBM BW"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_PER_BF16 = 6.0      # nominal dense NVFP4 / BF16 tensor rate of a GB300 (13.5 / 2.25)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_bf16")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--nvfp4-kernels", default="auto", choices=["auto", "pair", "one-cta"],
                    help="NVFP4 expert GEMMs: the library's choice, both on CTA pairs "
                         "(MOE_FLAG_NVFP4_PAIR) or both on single CTAs "
                         "(MOE_FLAG_NVFP4_ONE_CTA)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--no-boundary", action="store_true",
                    help="skip the separate timing of moe_boundary on the step's output")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---- algorithmic work --------------------------------------------------------------------

def flops_per_token(s) -> dict:
    """FLOPs per token of each GEMM stage (multiply-add = 2), routed work only."""
    return {
        "router": 2.0 * s.d * s.E,
        "pool": 2.0 * s.d * s.p,
        "gemm1_gate_up_swiglu": 2.0 * s.top_k * s.p * 2 * s.I,
        "gemm2_down": 2.0 * s.top_k * s.I * s.p,
        "unpool": 2.0 * s.p * s.d,
    }


def bytes_per_token(s, act_bytes=2) -> dict:
    """Compulsory HBM bytes per token of the memory-bound stages (each operand read
    once, each result written once)."""
    k = s.top_k
    yb = 4 if s.expert == "f32" else 2          # expert outputs y: FP16 unless FP32 experts
    return {
        "norm": s.d * act_bytes + s.d * 4 + s.d * act_bytes,            # x in; h32, h16 out
        # pooled in; k rows of u out (NVFP4: codes + block scales + a per-row scale)
        "dispatch": s.p * 4 + (k * s.p * (0.5 + 1 / 16) + 4 * k if s.expert == "nvfp4"
                               else k * s.p * act_bytes) + 16 * k,
        "combine": k * s.p * yb + k * (s.p // 128) * 4 + s.p * act_bytes + 8 * k,  # y, sums in; c out
    }


def projection_bytes(s, T: int) -> dict:
    """Compulsory HBM bytes of one launch of the router, pooler and unpooler GEMMs: the
    weights once plus the rows in and out.  Router: TF32-rounded FP32 h and W_r in,
    ids and weights out.  Pooler: FP16 h and W_pool in, FP32 pooled out.  Unpooler: FP16
    c and W_unpool in, out in the activation format.  FP32 activations: FP32 operands."""
    a = 4 if s.act == "f32" else 2
    return {
        "router": s.E * s.d * 4 + T * s.d * 4 + T * s.top_k * 8,
        "pool": s.p * s.d * a + T * s.d * a + T * s.p * 4,
        "unpool": s.d * s.p * a + T * s.p * a + T * s.d * a,
    }


def expert_gemm_bytes(s, n_experts_touched: int, T: int) -> dict:
    """Compulsory HBM bytes of one launch of each expert GEMM: the weights of the experts
    the batch routes to (read once), the R = T * top_k dispatched rows in and the rows
    out.  BF16 experts: FP16 copies of W13 and W2, FP16 u and s; FP32 experts: FP32
    throughout.  NVFP4 experts: 4-bit codes plus one FP8 scale per 16 elements for the
    weights, u and s.  The down GEMM writes y (FP16; FP32 for FP32 experts) and one FP32
    sum of squares per 128 columns."""
    R = T * s.top_k
    if s.expert == "nvfp4":
        q = 0.5 + 1.0 / 16
        w13, w2, u, s_in, s_out = q, q, q, q, q
    elif s.expert == "f32":     # TF32-rounded FP32 weights and operands
        w13, w2, u, s_in, s_out = 4, 4, 4, 4, 4
    else:
        w13, w2, u, s_in, s_out = 2, 2, 2, 2, 2
    yb = 4 if s.expert == "f32" else 2
    return {
        "gemm1_gate_up_swiglu": n_experts_touched * s.p * 2 * s.I * w13 + R * s.p * u
                                + R * s.I * s_out,
        "gemm2_down": n_experts_touched * s.I * s.p * w2 + R * s.I * s_in + R * s.p * yb
                      + R * (s.p // 128) * 4,
    }


# ---- clocks --------------------------------------------------------------------------------

def parse_clock_samples(out: str):
    """Median SM clock under load, the maximum clock and the throttle reasons seen, from
    `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits` lines."""
    sm, pw, smax, reasons = [], [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in out.splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            smax = float(f[2])
        except ValueError:
            continue
        try:
            pw.append(float(f[3]))
        except ValueError:
            pw.append(float("nan"))
        for name, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(name)
    if not sm:
        return None
    # under load = the samples drawing at least half the highest power seen (the
    # idle lead-in before the timed region is left out of the median)
    top = max((w for w in pw if w == w), default=None)
    load = [c for c, w in zip(sm, pw) if top is None or (w == w and w >= 0.5 * top)]
    return {"sm_mhz": statistics.median(load or sm), "sm_max_mhz": smax,
            "samples": len(sm), "load_samples": len(load),
            "power_w_max": top, "reasons": sorted(reasons)}


class ClockSampler:
    """nvidia-smi sampling (100 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


# ---- ncu traffic record ----------------------------------------------------------------

def kernel_source_sha(files=None) -> str:
    """Hash of the kernel sources: every file under csrc/, or only `files` (the sources a
    profiled kernel and its launch are built from), in name order."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "latent_moe_layer_rmsnorm_gb300", "csrc")
    for name in sorted(os.listdir(csrc) if files is None else files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the summary
    is missing or any source it was taken on has changed since.  The summary's line
    `kernel_source_sha: <hash> (<files>)` names the csrc files the hash covers (all of
    them when no list is given)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)(?:\s*\(([^)]*)\))?", text)
    if not m or not sha:
        return None
    files = sha.group(2).split() if sha.group(2) else None
    try:
        if sha.group(1) != kernel_source_sha(files):
            return None
    except OSError:
        return None
    return float(m.group(1))


# ---- ranks ----------------------------------------------------------------------------------

def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling over independent token batches)."""
    return base + 1000 * rank


def max_over_ranks(v: float, device) -> float:
    """The job's elapsed time is the slowest rank's (no-op for one process)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- roofline ---------------------------------------------------------------------------

# A kernel timed inside a short region runs at the boost clock: its tensor peak is the
# burst figure.  Only a timed region of at least this many seconds of back-to-back GEMMs
# runs at the power-capped clock the sustained figure was measured at.
SUSTAINED_MIN_S = 2.0
# The FP4 MMA issue rate measured on a GB300 (a 128 x 128 x 64 block-scaled MMA every 64
# cycles per SM = 16384 MAC/clk, 4x the BF16 kind's 4096): reported beside the nominal
# 6x ratio, which sets the peak.
FP4_MEASURED_ISSUE_PER_BF16 = 4.0


def tensor_peak(peaks: dict, peak_src: str, timed_s: float, nvfp4: bool):
    """(peak TFLOP/s, description) for a contraction timed inside a region of timed_s
    seconds: burst BF16 below SUSTAINED_MIN_S, sustained at or above it; NVFP4 GEMMs
    take FP4_PER_BF16 times that (the nominal dense ratio)."""
    if timed_s >= SUSTAINED_MIN_S:
        key, why = "bf16_tflops_sustained", f"timed region {timed_s:.2f} s >= {SUSTAINED_MIN_S:g} s"
    else:
        key, why = "bf16_tflops", f"timed region {timed_s:.2f} s < {SUSTAINED_MIN_S:g} s (boost clock)"
    bf16 = float(peaks.get(key, FALLBACK_PEAKS[key]))
    if nvfp4:
        return bf16 * FP4_PER_BF16, (f"nvfp4 = {FP4_PER_BF16:g} x {key} ({peak_src}; nominal "
                                     f"13.5 / 2.25 PFLOP/s ratio; measured FP4 MMA issue rate "
                                     f"{FP4_MEASURED_ISSUE_PER_BF16:g} x bf16); {why}")
    return bf16, f"{key} ({peak_src}); {why}"


def roofline_of(shape, T, stage_ms, n_touched, timed_s, peaks, peak_src, workload):
    """Roofline of the dominant GEMM stage, plus every stage's TFLOP/s and GB/s."""
    fl = flops_per_token(shape)
    by = bytes_per_token(shape)
    stage_tflops = {n: fl[n] * T / (stage_ms[n] / 1e3) / 1e12 for n in fl if stage_ms.get(n)}
    stage_gbs = {n: by[n] * T / (stage_ms[n] / 1e3) / 1e9 for n in by if stage_ms.get(n)}
    gb = expert_gemm_bytes(shape, n_touched, T)
    for n, b in projection_bytes(shape, T).items():   # weight streams at decode sizes
        if stage_ms.get(n):
            stage_gbs[n] = b / (stage_ms[n] / 1e3) / 1e9
    for n, b in gb.items():
        if stage_ms.get(n):
            stage_gbs[n] = b / (stage_ms[n] / 1e3) / 1e9
    dominant = max(fl, key=lambda n: stage_ms.get(n, 0.0))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    nv = shape.expert == "nvfp4" and dominant.startswith("gemm")
    peak, kind = tensor_peak(peaks, peak_src, timed_s, nv)
    traffic = recorded_traffic(workload, dominant)
    flops_launch = fl[dominant] * T
    bytes_launch = gb.get(dominant)
    ridge = peak * 1e12 / (hbm_peak * 1e9)          # FLOP per byte where the bounds meet
    intensity = flops_launch / bytes_launch if bytes_launch else None
    if intensity is not None and intensity < ridge:
        # too few rows per expert to reuse a weight tile: the launch streams the weights
        achieved = stage_gbs[dominant]
        roof = {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                "peak": round(hbm_peak, 1), "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                "peak_kind": f"hbm_gbs ({peak_src}, copy bandwidth)",
                "bytes_per_launch": bytes_launch, "flops_per_launch": flops_launch,
                "experts_touched": n_touched,
                "intensity_flop_per_byte": round(intensity, 2), "ridge": round(ridge, 1),
                "tensor_tflops": round(stage_tflops[dominant], 1)}
    else:
        achieved = stage_tflops[dominant]
        roof = {"bound": "tensor", "kernel": dominant, "achieved": round(achieved, 1),
                "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": traffic, "peak_kind": kind, "flops_per_launch": flops_launch,
                "bytes_per_launch": bytes_launch, "experts_touched": n_touched,
                "intensity_flop_per_byte": round(intensity, 1) if intensity else None,
                "ridge": round(ridge, 1)}
        if nv:
            meas = peak / FP4_PER_BF16 * FP4_MEASURED_ISSUE_PER_BF16
            roof["frac_of_measured_fp4_issue_rate"] = round(achieved / meas, 4)
    return roof, stage_tflops, stage_gbs


# ---- our arm -----------------------------------------------------------------------------

class Runner:
    """One latent-MoE layer of a workload, with its inputs resident on the device."""

    def __init__(self, shape, seed, experts=None, flags=0):
        import torch

        from latent_moe_layer_rmsnorm_gb300 import synth
        from latent_moe_layer_rmsnorm_gb300 import _lib as nst
        from latent_moe_layer_rmsnorm_gb300.layer import LatentMoE
        self.shape = shape
        inp = synth.make_dense(shape, seed, "cuda")
        if experts is None:
            experts = make_experts(shape, seed)
        inp.update(experts)
        if shape.expert == "nvfp4":
            inp["gs_act2"] = synth.nvfp4_act2_scales(shape, "cuda")
        self.out_kind = "bf16" if shape.act == "bf16" else "f32"
        self.layer = LatentMoE(shape, inp, out=self.out_kind, keep_canonical=False)
        self.x = inp["x"]
        self.out = torch.empty((shape.T, shape.d), dtype=self.layer.out_dtype(), device="cuda")
        self.stream = torch.cuda.current_stream()
        self.stage_names = [nst.moe_stage_name(i) for i in range(nst.moe_num_stages())]
        self.flags = flags

    def forward(self, ids=None, w=None, events=None):
        return self.layer.forward(self.x, ids=ids, w=w, out=self.out, events=events,
                                  flags=self.flags)

    def touched(self):
        import torch
        ids, _ = self.layer.route(self.x)
        return int(torch.unique(ids).numel())

    def time(self, steps, warmup, world, replay=False):
        """K steps bracketed by a barrier and synchronisations (plain calls: the kernels
        of consecutive steps overlap their launches); then the same steps again with
        CUDA events between the stages for the per-stage times.  Events between kernels
        stop each kernel from starting before the previous one ends, so the stage times
        come from that second pass and sum to a little more than a timed step.  Returns
        (elapsed ms of the timed pass, mean ms per stage)."""
        import torch
        import torch.distributed as dist
        ids = w = None
        if replay:
            ids, w = self.layer.route(self.x)
        for _ in range(warmup):
            self.forward(ids, w)
        torch.cuda.synchronize()
        st = self.layer.read_status()
        if st != (0, 0):
            raise SystemExit(f"device status after warm-up: {st}")
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        for _ in range(steps):
            self.forward(ids, w)
        t1.record(self.stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        elapsed = max_over_ranks(t0.elapsed_time(t1), "cuda")
        st = self.layer.read_status()
        if st != (0, 0):
            raise SystemExit(f"device status after the timed steps: {st}")
        n = len(self.stage_names)
        np_ = min(steps, PROFILED_STEPS)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(np_)]
        for row in evs:
            for e in row:
                e.record(self.stream)       # create the handles; re-recorded by the library
        torch.cuda.synchronize()
        for k in range(np_):
            self.forward(ids, w, events=[e.cuda_event for e in evs[k]])
        torch.cuda.synchronize()
        stage_ms = {nm: 0.0 for nm in self.stage_names}
        for row in evs:
            for i, nm in enumerate(self.stage_names):
                stage_ms[nm] += row[i].elapsed_time(row[i + 1]) / np_
        if replay:
            stage_ms.pop("router", None)
        return elapsed, stage_ms


# steps of the second, event-bracketed pass that gives the per-stage times
PROFILED_STEPS = 20


def make_experts(shape, seed):
    """Expert matrices of a workload, drawn on the device."""
    import torch

    from latent_moe_layer_rmsnorm_gb300 import synth
    dt = synth.storage_dtype(shape.expert)
    E, p, I = shape.E, shape.p, shape.I
    out = {"w_gate": torch.empty((E, I, p), dtype=dt, device="cuda"),
           "w_up": torch.empty((E, I, p), dtype=dt, device="cuda"),
           "w_down": torch.empty((E, p, I), dtype=dt, device="cuda")}
    for e in range(E):
        m = synth.make_expert(shape, seed, e, "cuda")
        for k in out:
            out[k][e].copy_(m[k])
    return out


def workload_line(shape, runner, steps, warmup, world, peaks, peak_src, local, replay=False):
    """Throughput, stage times and roofline of one more workload (not the headline)."""
    import torch
    t0 = time.perf_counter()
    for _ in range(2):
        runner.forward()
    torch.cuda.synchronize()
    est_ms = (time.perf_counter() - t0) * 1e3 / 2
    steps = max(steps, min(2000, int(WORKLOAD_MIN_MS / max(est_ms, 1e-3)) + 1))
    sampler = ClockSampler(local)
    time.sleep(0.3)
    elapsed, stage_ms = runner.time(steps, warmup, world, replay=replay)
    clocks = sampler.stop()
    T = shape.T
    roof, tfl, gbs = roofline_of(shape, T, stage_ms, runner.touched(), elapsed / 1e3, peaks,
                                 peak_src, shape.name)
    return {"workload": describe(shape, runner.out_kind) + (" (routing replayed: ids and "
                                                            "weights passed in)" if replay else ""),
            "tokens_per_s": round(T * steps * world / (elapsed / 1e3), 1),
            "ms_per_step": round(elapsed / steps, 4), "steps": steps, "warmup": warmup,
            "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "stages_tflops": {k: round(v, 1) for k, v in tfl.items()},
            "stages_gbs": {k: round(v, 1) for k, v in gbs.items()},
            "roofline": roof, "gpu_launches": runner.layer.launches(T, not replay) * steps,
            "clocks": clocks}


def describe(shape, out_kind):
    return (f"{shape.name}: T={shape.T} d={shape.d} p={shape.p} E={shape.E} "
            f"top_k={shape.top_k} I={shape.I} act={shape.act} expert={shape.expert} "
            f"out={out_kind}")


# the other workloads reported beside the headline (BF16 prefill chunk), in order; the
# replay entry runs the prefill chunk with routing passed in
EXTRA_WORKLOADS = ("decode_bf16", "skewed_bf16", "prefill_nvfp4", "decode_nvfp4", "replay")
# each extra workload's timed region is at least this long (more steps for short ones),
# so the clock sampler sees it under load
WORKLOAD_MIN_MS = 500.0


def run_ours(args):
    import torch
    import torch.distributed as dist

    from latent_moe_layer_rmsnorm_gb300 import build, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    shape = synth.WORKLOADS[args.workload]
    seed = rank_seed(args.seed, rank)
    experts = make_experts(shape, seed)
    from latent_moe_layer_rmsnorm_gb300 import _lib as nst
    run_flags = {"auto": 0, "pair": nst.MOE_FLAG_NVFP4_PAIR,
                 "one-cta": nst.MOE_FLAG_NVFP4_ONE_CTA}[args.nvfp4_kernels]
    run = Runner(shape, seed, experts, run_flags)
    layer, x, out, stream = run.layer, run.x, run.out, run.stream
    T = shape.T
    n_touched = run.touched()

    # ---- timed region: K steps, stage events recorded between the kernels ---------------
    sampler = ClockSampler(local)
    time.sleep(0.3)
    elapsed_ms, stage_ms = run.time(args.steps, args.warmup, world)
    ms_per_step = elapsed_ms / args.steps
    tokens = T * args.steps * world
    value = tokens / (elapsed_ms / 1e3)

    # ---- end to end from pinned host buffers ------------------------------------------
    # Every step copies its tokens host -> device, runs the layer and copies its output
    # back.  Two device slots let the copies of neighbouring steps run on their own
    # streams (one per direction) under the current step's kernels; events order each
    # slot's copy-in -> forward -> copy-out, and the timed region spans the first
    # copy-in to the last copy-out.
    e2e = None
    if not args.no_e2e:
        hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        hx.copy_(x)
        ho = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        dx = [torch.empty_like(x) for _ in range(2)]
        dout = [torch.empty_like(out) for _ in range(2)]
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

        def pipelined(n, start_event=None):
            fwd_done = [None, None]
            out_done = [None, None]
            if start_event is not None:
                h2d.wait_event(start_event)
            for i in range(n):
                j = i & 1
                if fwd_done[j] is not None:
                    h2d.wait_event(fwd_done[j])     # slot j's previous forward has read dx[j]
                with torch.cuda.stream(h2d):
                    dx[j].copy_(hx, non_blocking=True)
                    in_done = torch.cuda.Event()
                    in_done.record(h2d)
                stream.wait_event(in_done)
                if out_done[j] is not None:
                    stream.wait_event(out_done[j])  # slot j's previous output has left
                layer.forward(dx[j], out=dout[j])
                fwd_done[j] = torch.cuda.Event()
                fwd_done[j].record(stream)
                d2h.wait_event(fwd_done[j])
                with torch.cuda.stream(d2h):
                    ho[j].copy_(dout[j], non_blocking=True)
                    out_done[j] = torch.cuda.Event()
                    out_done[j].record(d2h)
            for ev in out_done:
                if ev is not None:
                    stream.wait_event(ev)

        pipelined(3)
        torch.cuda.synchronize()
        if layer.read_status() != (0, 0):
            raise SystemExit(f"device status after the end-to-end warm-up: {layer.read_status()}")
        if not torch.equal(ho[0].to(out.device), out) or not torch.equal(ho[1].to(out.device), out):
            raise SystemExit("end-to-end output differs from the device-resident run")
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(4, args.steps)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        pipelined(n_e2e, start_event=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), "cuda")
        e2e = {"value": T * n_e2e * world / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": x.numel() * x.element_size(),
               "d2h_bytes_per_step": out.numel() * out.element_size(),
               "ms_per_step": e2e_ms / n_e2e,
               "copies": "pinned host buffers; copy-in and copy-out on their own streams, "
                         "overlapping the neighbouring steps' kernels (two device slots)"}

    clocks = sampler.stop()           # samples cover both timed regions

    # ---- the block boundary (post-norm, residual add, next pre-norm), timed on its own ----
    boundary = None
    if not args.no_boundary:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed + 17)
        g_post = torch.rand(shape.d, generator=gen, device="cuda") + 0.5
        g_next = torch.rand(shape.d, generator=gen, device="cuda") + 0.5
        xo, hn = torch.empty_like(x), torch.empty_like(x)
        for _ in range(3):
            layer.boundary(x, out, g_post, g_next, x_out=xo, h_next=hn)
        torch.cuda.synchronize()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(args.steps):
            layer.boundary(x, out, g_post, g_next, x_out=xo, h_next=hn)
        b1.record(stream)
        torch.cuda.synchronize()
        b_ms = max_over_ranks(b0.elapsed_time(b1), "cuda") / args.steps
        b_bytes = 3 * x.numel() * x.element_size() + out.numel() * out.element_size()
        boundary = {"ms": round(b_ms, 4), "gbs": round(b_bytes / (b_ms / 1e3) / 1e9, 1),
                    "bytes": b_bytes}
        # the block followed by that pass, against the block with the row pass inside its
        # unpooler (moe_forward_boundary): same results, one pass over [T, d] fewer
        yb = torch.empty_like(out)

        def block_then_pass():
            layer.forward(x, out=yb)
            layer.boundary(x, yb, g_post, g_next, x_out=xo, h_next=hn)

        def block_fused():
            layer.forward_boundary(x, g_post, g_next, y=yb, x_out=xo, h_next=hn)

        # interleaved repetitions, so that drift of the clock under the power cap falls on
        # both arms alike
        arms = (("block_then_pass_ms", block_then_pass), ("fused_ms", block_fused))
        for _, fn in arms:
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        reps, per = 4, max(1, args.steps // 4)
        acc = {name: 0.0 for name, _ in arms}
        for _ in range(reps):
            for name, fn in arms:
                b0.record(stream)
                for _ in range(per):
                    fn()
                b1.record(stream)
                torch.cuda.synchronize()
                acc[name] += max_over_ranks(b0.elapsed_time(b1), "cuda")
        for name, _ in arms:
            boundary[name] = round(acc[name] / (reps * per), 4)
        boundary["fused_saves_ms"] = round(boundary["block_then_pass_ms"] - boundary["fused_ms"], 4)
        del xo, hn, yb

    # ---- roofline of the dominant kernel -------------------------------------------------
    peaks, peak_src = load_peaks()
    roofline, stage_tflops, stage_gbs = roofline_of(shape, T, stage_ms, n_touched,
                                                    elapsed_ms / 1e3, peaks, peak_src,
                                                    args.workload)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    out_kind = run.out_kind

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_from_gpu_inputs(shape, layer, x, seed)

    # ---- the other workloads, each on its own layer (the headline's is freed first) ------
    workloads = {}
    if not args.no_workloads and shape.name == "prefill_bf16":
        workloads["replay_prefill_bf16"] = workload_line(shape, run, args.steps, args.warmup,
                                                         world, peaks, peak_src, local,
                                                         replay=True)
    launches = layer.launches(T) * args.steps
    if workloads:
        del run, layer, x, out
        torch.cuda.empty_cache()
        for name in EXTRA_WORKLOADS:
            if name == "replay":
                continue
            sh = synth.WORKLOADS[name]
            r = Runner(sh, seed, experts, run_flags)
            workloads[name] = workload_line(sh, r, args.steps, args.warmup, world, peaks,
                                            peak_src, local)
            del r
            torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    dtype = "bf16+fp16" if shape.act == "bf16" else "f32(tf32)"
    if shape.expert == "nvfp4":
        dtype = "nvfp4 experts, bf16+fp16 projections"
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights, U(0.5,1.5) gains)",
        "config": {"workload": f"{shape.name}: T={T} d={shape.d} p={shape.p} E={shape.E} "
                               f"top_k={shape.top_k} I={shape.I} act={shape.act} "
                               f"expert={shape.expert} out={out_kind}",
                   "global_batch": T * world, "parallelism": f"replicas x{world} (token batches)",
                   "l2": "inputs larger than L2 (24 GB expert weights, 256 MB x per step)"},
        "roofline": roofline,
        "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "stages_tflops": {k: round(v, 1) for k, v in stage_tflops.items()},
        "stages_gbs": {k: round(v, 1) for k, v in stage_gbs.items()},
        "hbm_peak_gbs": hbm_peak,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    if shape.expert == "nvfp4":
        line["config"]["nvfp4_kernels"] = args.nvfp4_kernels
    if workloads:
        line["workloads"] = workloads
    if boundary is not None:
        # not part of the step: the pass that follows the block (moe_boundary), timed alone
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        boundary["frac_of_hbm"] = round(boundary["gbs"] / hbm, 3)
        line["boundary"] = boundary
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ---- CPU oracle baselines ------------------------------------------------------------------

def _oracle_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_from_gpu_inputs(shape, layer, x, seed, n_groups=6, group=4):
    """Time the oracle, as it stands, on n_groups x group tokens of the benchmark's own
    batch.  Each group's inputs (dense weights and its routed experts' matrices) are
    staged on the host before its clock starts, so host memory holds one group's
    experts at a time; the oracle's float64 work (conversion included) is timed."""
    import numpy as np
    import torch

    import oracle
    from latent_moe_layer_rmsnorm_gb300 import synth

    n_tok = n_groups * group
    toks = [int(t) for t in np.linspace(0, shape.T - 1, n_tok).round()]
    dense = synth.make_dense(shape, seed=seed, device="cuda")
    view = {k: v.float().cpu().numpy() for k, v in dense.items()}
    del dense
    total, n_exp = 0.0, 0
    for g0 in range(0, n_tok, group):
        tg = toks[g0: g0 + group]
        view["x"] = x[tg].float().cpu().numpy()
        ids, _ = layer.route(x[tg].contiguous())
        need = sorted(set(ids.cpu().numpy().reshape(-1).tolist()))
        n_exp += len(need)
        experts = {e: {k: v.float().cpu().numpy() for k, v in
                       synth.make_expert(shape, seed, e, device="cuda").items()} for e in need}

        class Sparse:
            def __init__(self, key):
                self.key = key

            def __getitem__(self, e):
                e = int(e)
                if e not in experts:     # the oracle routed a token elsewhere than the GPU
                    experts[e] = {k: v.float().cpu().numpy() for k, v in
                                  synth.make_expert(shape, seed, e, device="cuda").items()}
                return experts[e][self.key]

        for key in ("w_gate", "w_up", "w_down"):
            view[key] = Sparse(key)
        t0 = time.perf_counter()
        oracle.moe_forward(view, top_k=shape.top_k, eps=shape.eps, act=shape.act,
                           expert=shape.expert, out="bf16", chain=True)
        total += time.perf_counter() - t0
        del experts
    del np, torch
    return {"value": round(n_tok / total, 4), "unit": "tokens/s", "cores": _oracle_cores(),
            "kind": "oracle",
            "sample": f"{n_tok} tokens of the {shape.name} batch in groups of {group} "
                      f"({n_exp} routed expert matrices staged per group), float64 numpy, "
                      f"{total:.1f} s of oracle time"}


def run_reference(args):
    """The oracle on the host cores: each step is one token of the workload with its
    routed experts (drawn on the CPU from the same generator recipe)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from latent_moe_layer_rmsnorm_gb300 import synth

    shape = synth.WORKLOADS[args.workload]
    n_tok = max(args.steps + args.warmup, 1)
    small = shape.replace(T=n_tok)
    # inputs are only drawn on the GPU when one is present (faster); the timed work is
    # the oracle on the host cores either way
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    dense = synth.make_dense(small, seed=args.seed, device=gen_dev)
    view = {k: v.float().cpu().numpy() for k, v in dense.items()}
    ids, _, _ = oracle.route(view, top_k=shape.top_k, eps=shape.eps)
    cache = {}

    def experts_for(t):
        out = {}
        for e in ids[t]:
            e = int(e)
            if e not in cache:
                cache[e] = {k: v.float().cpu().numpy()
                            for k, v in synth.make_expert(shape, args.seed, e, gen_dev).items()}
            out[e] = cache[e]
        return out

    class Sparse:
        def __init__(self, key, ex):
            self.key, self.ex = key, ex

        def __getitem__(self, e):
            return self.ex[int(e)][self.key]

    times = []
    for t in range(n_tok):
        ex = experts_for(t)
        v = dict(view)
        for key in ("w_gate", "w_up", "w_down"):
            v[key] = Sparse(key, ex)
        t0 = time.perf_counter()
        oracle.moe_forward(v, top_k=shape.top_k, eps=shape.eps, act=shape.act,
                           expert=shape.expert, out="bf16", chain=True, tokens=[t])
        times.append(time.perf_counter() - t0)
        if len(cache) > 64:
            cache.clear()
    timed = times[args.warmup:] if len(times) > args.warmup else times
    total = sum(timed)
    value = len(timed) / total
    cores = _oracle_cores()
    sample = (f"{len(timed)} tokens of {shape.name}, one per step, float64 numpy oracle "
              f"with its routed experts")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
            "n_gpus": world, "steps": len(timed), "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / len(timed), 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{shape.name}: T={shape.T} d={shape.d} p={shape.p} "
                                   f"E={shape.E} top_k={shape.top_k} I={shape.I}",
                       "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    del np, torch
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
