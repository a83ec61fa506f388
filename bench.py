#!/usr/bin/env python3
"""Encoder throughput on GB300: tokens/s and TFLOP/s of the shared ViT encoder forward.

Workload: V-JEPA 2 ViT-L/16 on 16 x 256 x 256 clips (2048 tokens each), eight clips per GPU per
step by default (--batch), bf16 weights and activations with fp32 accumulation, synthetic seeded
weights and pixels. A step is one jepa_encode of the batch (patchify, patch GEMM, 24 blocks,
final norm) on inputs resident in HBM. The line also carries the same clip at batch 1 ("batch1"),
timed the same way.

--workload vjepa2_vitl16_ssv2_head times the V-JEPA 2 SSv2 attentive-pool head + 174-way classifier
over the 2048 encoder tokens of each clip (3 pooler layers, the cross attention of one query,
the MLP and the classifier), eight clips per step. --workload vjepa2_vitl16_predictor times the
V-JEPA 2 masked predictor instead (12 layers of
width 384 over the 2048 tokens of each clip: the first 1024 as context, the last 1024 as
targets, the split of the pages' predictor example), eight clips per step, on encoder tokens
resident in HBM. --workload also picks one of the fixed-table families: V-JEPA ViT-L/16 16 x 256 x 256 clips
whose 3-D sin-cos table is baked for 16 x 224 x 224 and resized (trilinear), or I-JEPA-style
ViT-L/16 256 x 256 images whose 2-D table is baked for 224 x 224 and resized (bicubic). Their
lines add the one-off table kernels' times ("pos_table").

--workload also times the other encoder workloads, one line each: hfvit_ti14_224 (ViT-Ti/14 224^2
image, fp32 SIMT path, roofline against the fp32 FFMA peak), vjepa2_1_vitl16_16x384 (4608 tokens,
interleaved RoPE rescaled 15/23, modality vector), levjepa_vitl16_16x256 (4097 tokens, CLS,
block-causal, two clips; the line adds the same clips with full attention, which shows what
skipping the masked key tiles saves) and vjepa2_vitg16_64x256 (ViT-g/16, 8192 tokens).

    python bench.py [--gpus N --steps K --warmup W] [--batch B] [--workload NAME] [--impl reference]

Timing: W untimed steps, then K steps replaying one CUDA graph of the encode, each bracketed by
CUDA events on the context stream, with a 256 MiB write between steps to flush L2 (outside the
events); barrier + synchronize around the timed region; the max over ranks of the device time.
Per-kernel durations (the roofline and the kernel table) come from a second pass of K steps with
the library's event hook (events captured inside the graph), since those events lengthen the
step. One JSON line on rank 0.

--impl reference times the oracle (the plain fp64 CPU encoder) on the host cores instead.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "encoder tokens/s and TFLOP/s (fraction of bf16 peak), ViT-L 16×256² video"
BENCH_WORKLOADS = {
    "vjepa2_vitl16_16x256": dict(preset="vjepa2_vitl16", T=16, H=256, W=256, batch=8, metric=METRIC,
                                 label="V-JEPA 2 ViT-L/16 16x256x256 clip"),
    "vjepa_vitl16_16x256": dict(preset="vjepa_vitl16", T=16, H=256, W=256, batch=8,
                                metric="encoder tokens/s and TFLOP/s, V-JEPA ViT-L/16 16×256² video, 3-D sin-cos table",
                                label="V-JEPA ViT-L/16 16x256x256 clip (3-D sin-cos table baked for 16x224x224, "
                                      "resized trilinear)"),
    "ijepa_vitl16_256": dict(preset="ijepa_vitl16", T=1, H=256, W=256, batch=64,
                             metric="encoder tokens/s and TFLOP/s, I-JEPA-style ViT-L/16 256² image, 2-D sin-cos table",
                             label="I-JEPA-style ViT-L/16 256x256 image (2-D [w|h] sin-cos table baked for 224x224, "
                                   "resized bicubic)"),
}
PREDICTOR = "vjepa2_vitl16_predictor"
HEADW = "vjepa2_vitl16_ssv2_head"
HEAD_METRIC = "attentive-pool head tokens/s and TFLOP/s, V-JEPA 2 ViT-L SSv2 classifier head over 16×256² clips"
PRED_METRIC = "masked predictor tokens/s and TFLOP/s, V-JEPA 2 ViT-L predictor over 16×256² clips"
BENCH_WORKLOADS.update({
    "hfvit_ti14_224": dict(preset="hfvit_ti14", T=1, H=224, W=224, batch=1, dtype="fp32",
                           metric="encoder tokens/s and fraction of fp32 FFMA peak, hfvit ViT-Ti/14 224² image (fp32)",
                           label="hfvit ViT-Ti/14 224x224 image (CLS, learned positions), fp32 SIMT path"),
    "vjepa2_1_vitl16_16x384": dict(preset="vjepa2_1_vitl16", T=16, H=384, W=384, batch=1,
                                   metric="encoder tokens/s and TFLOP/s, V-JEPA 2.1 ViT-L/16 16×384² video",
                                   label="V-JEPA 2.1 ViT-L/16 16x384x384 clip (interleaved RoPE rescaled 15/23, "
                                         "modality vector)"),
    "levjepa_vitl16_16x256": dict(preset="levjepa_vitl16", T=16, H=256, W=256, batch=2, full_attention_control=True,
                                  metric="encoder tokens/s and TFLOP/s, LeVJEPA ViT-L/16 16×256² video, block-causal",
                                  label="LeVJEPA ViT-L/16 16x256x256 clip (tubelet 1, CLS, block-causal attention)"),
    "vjepa2_vitg16_64x256": dict(preset="vjepa2_vitg16", T=64, H=256, W=256, batch=1,
                                 metric="encoder tokens/s and TFLOP/s, V-JEPA 2 ViT-g/16 64×256² video",
                                 label="V-JEPA 2 ViT-g/16 64x256x256 clip"),
})
HEADLINE = "vjepa2_vitl16_16x256"
FLUSH_BYTES = 256 << 20  # > 129 MB of L2

# Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel class, from ncu
# captures; `sha1` is the hash of the class's source files when the counters were taken (a changed
# kernel reports traffic null until it is captured again). The 8-clip attention figure is a 4-clip
# launch of the two-half encode (50.39 MB read + 0.29 MB written) times two: attention reads each
# clip's q, k, v once, so its traffic grows with the clips.
NCU_TRAFFIC = {  # (workload, kernel class, clips per GPU): bytes per launch, source hash at capture
    (HEADLINE, "attention", 8): {"bytes_per_launch": 2 * 50.747392e6, "sha1": "eee1d6dcabdd5ee9aa18316715cbd18682d75a57"},
    ("levjepa_vitl16_16x256", "attention", 2): {"bytes_per_launch": 50.655232e6,
                                                "sha1": "eee1d6dcabdd5ee9aa18316715cbd18682d75a57"},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--batch", type=int, default=None, help="clips per GPU per step (default: the workload's)")
    p.add_argument("--workload", choices=sorted(BENCH_WORKLOADS) + [PREDICTOR, HEADW], default=HEADLINE)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float, device=None) -> float:
    """Max of a scalar over ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


# ------------------------------------------------------------------ measured peaks and clocks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, device_index: int, interval_ms: int = 50):
        self.cmd = ["nvidia-smi", "-i", str(device_index), "--query-gpu=" + ",".join(CLOCK_FIELDS),
                    "--format=csv,noheader,nounits", "-lms", str(interval_ms)]
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land before the timed region starts
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle timing (host cores)
def oracle_layer_times(workload=HEADLINE, layers=(0, 1)):
    """Time the oracle on one item of the workload with each depth in `layers`; returns
    (times, tokens, threads, full depth)."""
    from dataclasses import replace
    import oracle
    import synth
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from configs import WORKLOADS
    cfg, dtype, _, (T, H, W) = WORKLOADS[workload]
    pix = synth.pixels(0, (1, T, 3, H, W))
    times = []
    for nl in layers:
        t0 = time.perf_counter()
        oracle.encode(replace(cfg, n_layer=nl), 0, dtype == "bf16", pix)
        times.append(time.perf_counter() - t0)
    return times, oracle.n_tokens(cfg, T, H, W), oracle.num_threads(), cfg.n_layer


def cpu_baseline(workload=HEADLINE, full_depth_budget_s=20.0):
    """The oracle on the host cores: the embedding + final norm alone (0 layers) and with one
    layer; the full depth is then measured directly when it should take under the budget, else
    extrapolated linearly per layer (the layers are identical in cost)."""
    (t0, t1), N, threads, L = oracle_layer_times(workload)
    per_layer = max(t1 - t0, 1e-9)
    est = t0 + L * per_layer
    if est <= full_depth_budget_s:
        reps = max(1, min(9, int(5.0 / max(est, 1e-3))))   # short runs: the median of several
        (*fulls,), _, _, _ = oracle_layer_times(workload, layers=(L,) * reps)
        full = statistics.median(fulls)
        how = f"measured at full depth ({full:.2f} s, median of {reps})"
    else:
        full = est
        how = f"full-depth time {full:.1f} s extrapolated linearly per layer"
    return {"value": N / full, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle on one {N}-token item with 0 and 1 of the {L} layers ({t0:.2f} s, {t1:.2f} s); "
                      + how}


def pred_inputs(B, seed=0):
    """Encoder tokens N(0, 1) from the shared generator and the pages' half / half split."""
    import numpy as np
    import synth
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from configs import PRED_VJEPA2_L16, PRED_WORKLOAD
    grid, n_ctx, n_tgt = PRED_WORKLOAD["grid"], PRED_WORKLOAD["n_ctx"], PRED_WORKLOAD["n_tgt"]
    n_pos = grid[0] * grid[1] * grid[2]
    enc = synth.fill(seed, "input.enc_tokens", synth.NORMAL, 0.0, 1.0, (B, n_pos, PRED_VJEPA2_L16.enc_dim))
    ctx = np.tile(np.arange(n_ctx, dtype=np.int32), (B, 1))
    tgt = np.tile(np.arange(n_ctx, n_ctx + n_tgt, dtype=np.int32), (B, 1))
    return enc, ctx, tgt, grid, PRED_VJEPA2_L16


def pred_oracle_layer_times():
    """The oracle predictor on one clip's tokens with 1 and 2 layers: (t1, t2, tokens, threads, L)."""
    from dataclasses import replace
    import oracle
    enc, ctx, tgt, grid, cfg = pred_inputs(1)
    times = []
    for nl in (1, 2):
        t0 = time.perf_counter()
        oracle.predict(replace(cfg, n_layer=nl), 0, True, enc, ctx, tgt, grid[1:])
        times.append(time.perf_counter() - t0)
    return times[0], times[1], ctx.shape[1] + tgt.shape[1], oracle.num_threads(), cfg.n_layer


def pred_cpu_baseline():
    t1, t2, N, threads, L = pred_oracle_layer_times()
    per_layer = max(t2 - t1, 1e-9)
    full = t1 + (L - 1) * per_layer
    return {"value": N / full, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle predictor on one clip's {N} tokens with 1 and 2 of the {L} layers "
                      f"({t1:.2f} s, {t2:.2f} s); full-depth time {full:.1f} s extrapolated linearly per layer"}


def head_inputs(B, seed=0):
    """Encoder tokens N(0, 1) from the shared generator for the head workload."""
    import synth
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from configs import HEAD_VJEPA2_L16_SSV2, HEAD_WORKLOAD
    N = HEAD_WORKLOAD["tokens"]
    return synth.fill(seed, "input.enc_tokens", synth.NORMAL, 0.0, 1.0, (B, N, HEAD_VJEPA2_L16_SSV2.embed_dim)), \
        HEAD_VJEPA2_L16_SSV2


def head_oracle_layer_times():
    """The oracle head on one clip's tokens with 1 and 2 pooler layers: (t1, t2, tokens, threads, L)."""
    from dataclasses import replace
    import oracle
    tok, cfg = head_inputs(1)
    times = []
    for nl in (1, 2):
        t0 = time.perf_counter()
        oracle.attentive_head(replace(cfg, n_pool_layers=nl), 0, True, tok)
        times.append(time.perf_counter() - t0)
    return times[0], times[1], tok.shape[1], oracle.num_threads(), cfg.n_pool_layers


def head_cpu_baseline():
    t1, t2, N, threads, L = head_oracle_layer_times()
    full = t1 + (L - 1) * max(t2 - t1, 1e-9)
    return {"value": N / full, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle head on one clip's {N} tokens with 1 and 2 of the {L} pooler layers "
                      f"({t1:.2f} s, {t2:.2f} s); full-depth time {full:.1f} s extrapolated linearly per layer"}


def run_reference_layers(args, times, one_layer, metric, label):
    """The reference arm of a head-side workload: the oracle with one layer per step, the other
    layers added at the per-layer time calibrated from the 1- and 2-layer runs."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    t1, t2, N, threads, L = times
    per_layer = max(t2 - t1, 1e-9)
    for _ in range(args.warmup):
        one_layer()
    full_times = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one_layer()
        full_times.append((time.perf_counter() - t0) + (L - 1) * per_layer)
    wall = time.perf_counter() - t_start
    mean_full = statistics.mean(full_times)
    value = N / mean_full
    B = args.batch or 8
    sample = (f"each step: the fp64 oracle on one clip's {N} tokens with 1 of the {L} layers; the other {L - 1} "
              f"layers added at the calibrated per-layer time {per_layer:.2f} s; the {B} clips of a step are "
              f"independent, so a step costs {B} such clips")
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean_full * B, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{label} x {B} per GPU", "tokens_per_step": B * N, "global_batch": B,
                       "seq_len": N, "wall_s_sampled_steps": wall},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_reference_predictor(args):
    from dataclasses import replace
    import oracle
    enc, ctx, tgt, grid, cfg = pred_inputs(1)
    one = replace(cfg, n_layer=1)
    return run_reference_layers(args, pred_oracle_layer_times(),
                                lambda: oracle.predict(one, 0, True, enc, ctx, tgt, grid[1:]), PRED_METRIC,
                                f"V-JEPA 2 ViT-L masked predictor, {ctx.shape[1] + tgt.shape[1]} tokens per clip "
                                f"({ctx.shape[1]} context + {tgt.shape[1]} targets)")


def run_reference_head(args):
    from dataclasses import replace
    import oracle
    tok, cfg = head_inputs(1)
    one = replace(cfg, n_pool_layers=1)
    return run_reference_layers(args, head_oracle_layer_times(), lambda: oracle.attentive_head(one, 0, True, tok),
                                HEAD_METRIC, f"V-JEPA 2 ViT-L SSv2 attentive-pool head + classifier, {tok.shape[1]} "
                                             f"tokens per clip")


class SeqBench:
    """What run_sequence needs of a head-side workload (predictor, attentive-pool head)."""
    metric = label = ""
    tokens_per_step = launches = h2d_bytes = d2h_bytes = 0
    stream = None

    def step(self):               # one step on inputs resident in HBM, issued on self.stream
        raise NotImplementedError

    def e2e_step(self):           # host inputs in, host results out, synchronous
        raise NotImplementedError


def run_sequence(args, wl, make):
    """Time a head-side workload the way run_ours times the encoder: W warm-up steps, K steps of
    graph replay bracketed by CUDA events (L2 flushed between steps), then K eager steps with the
    context's per-kernel events (roofline and kernel table), then K' end-to-end steps."""
    import torch
    import torch.distributed as dist

    rank, world, local = init_ranks()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    import jepa_vision_encoder_gb300 as jv

    B = args.batch or wl["batch"]
    w = make(jv, B, rank, local)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = w.stream
    peaks = measured_peaks()
    with torch.cuda.stream(stream):
        w.ctx.set_graph(True)
        for _ in range(args.warmup):
            flush.zero_()
            w.step()
        w.ctx.sync()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        barrier(local)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            for i in range(args.steps):
                flush.zero_()
                starts[i].record(stream)
                w.step()
                ends[i].record(stream)
            torch.cuda.synchronize()
        barrier(local)
        torch.cuda.synchronize()
        w.ctx.sync()
        step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        w.ctx.set_profiling(True)
        for _ in range(2):
            w.step()
        w.ctx.profile(reset=True)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(args.steps):
            flush.zero_()
            w.step()
        p1.record(stream)
        torch.cuda.synchronize()
        prof = w.ctx.profile(reset=True)
        w.ctx.set_profiling(False)
    total_ms = reduce_max(sum(step_ms), device="cuda" if world > 1 else None)
    ms_per_step = total_ms / args.steps
    tokens_per_step = world * w.tokens_per_step
    value = tokens_per_step * args.steps / (total_ms / 1e3)
    flops_per_step = sum(v["flops"] for v in prof.values()) / args.steps
    tflops = world * flops_per_step * args.steps / (total_ms / 1e3) / 1e12
    name, st = max(prof.items(), key=lambda kv: kv[1]["total_ms"])
    avg_ms = st["total_ms"] / st["launches"]
    if st["flops"] > 0:
        achieved = st["flops"] / st["launches"] / (avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "kernel": name,
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = st["bytes"] / st["launches"] / (avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "kernel": name}
    rec = NCU_TRAFFIC.get((args.workload, name, B))
    roof["traffic"] = rec["bytes_per_launch"] if rec and rec.get("sha1") == source_sha1(name) else None
    roof["peak_source"] = peaks["source"]
    tot = max(sum(x["total_ms"] for x in prof.values()), 1e-9)
    kernels = {k: {"launches": v["launches"], "avg_us": 1e3 * v["total_ms"] / v["launches"], "share": v["total_ms"] / tot,
                   **({"tflops": v["flops"] / (v["total_ms"] / 1e3) / 1e12} if v["flops"] else {}),
                   **({"gbs": v["bytes"] / (v["total_ms"] / 1e3) / 1e9} if v["bytes"] else {})}
               for k, v in prof.items()}
    e2e_steps = min(args.steps, 20)
    w.e2e_step()
    barrier(local)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        w.e2e_step()
    e2e_s = reduce_max(time.perf_counter() - t0, device="cuda" if world > 1 else None)
    e2e = {"value": tokens_per_step * e2e_steps / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": w.h2d_bytes,
           "d2h_bytes_per_step": w.d2h_bytes}
    if rank == 0:
        line = {"metric": w.metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w.label, "tokens_per_step": tokens_per_step, "global_batch": world * B,
                           "seq_len": w.seq_len, "parallelism": f"replicas x{world} (independent clips, no collective)",
                           "l2": "flushed (256 MiB write) between steps", "weights": "seeded synthetic"},
                "tflops": tflops, "frac_of_bf16_peak": tflops / (world * peaks["bf16_tflops"]),
                "launch_mode": "CUDA graph replay", "roofline": roof, "kernels": kernels, "e2e": e2e,
                "gpu_launches": w.launches * args.steps, "clocks": clk.summary(),
                "profiled_pass": {"ms_per_step": p0.elapsed_time(p1) / args.steps}}
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = w.cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def make_predictor(jv, B, rank, local):
    """The V-JEPA 2 masked predictor over B clips' tokens (the pages' half / half split)."""
    import torch
    enc_h, ctx_h, tgt_h, grid, cfg = pred_inputs(B, seed=rank)
    w = SeqBench()
    pred = jv.Predictor.preset("vjepa2_vitl16", seed=0, device=local)
    n_ctx, n_tgt = ctx_h.shape[1], tgt_h.shape[1]
    w.ctx = jv.PredContext(pred, B, n_ctx, n_tgt)
    w.stream = w.ctx.stream
    enc, ctx, tgt = (torch.from_numpy(a).cuda() for a in (enc_h, ctx_h, tgt_h))
    out = torch.empty((B, n_tgt, cfg.out_dim), dtype=torch.float32, device="cuda")
    pin = [torch.from_numpy(a).pin_memory() for a in (enc_h, ctx_h, tgt_h)]
    pin_out = torch.empty((B, n_tgt, cfg.out_dim), dtype=torch.float32).pin_memory()
    w.step = lambda: w.ctx.predict(enc, ctx, tgt, grid, out)

    def e2e_step():
        with torch.cuda.stream(w.stream):
            enc.copy_(pin[0], non_blocking=True)
            ctx.copy_(pin[1], non_blocking=True)
            tgt.copy_(pin[2], non_blocking=True)
            w.ctx.predict(enc, ctx, tgt, grid, out)
            pin_out.copy_(out, non_blocking=True)
        w.ctx.sync()
    w.e2e_step = e2e_step
    w.h2d_bytes = sum(t.numel() * t.element_size() for t in pin)
    w.d2h_bytes = pin_out.numel() * 4
    w.seq_len = n_ctx + n_tgt
    w.tokens_per_step = B * w.seq_len
    w.launches = w.ctx.launches(n_ctx)
    w.metric = PRED_METRIC
    w.label = (f"V-JEPA 2 ViT-L masked predictor, {w.seq_len} tokens per clip ({n_ctx} context + {n_tgt} targets) "
               f"x {B} per GPU")
    w.cpu_baseline = pred_cpu_baseline
    w.keep = (pred, enc, ctx, tgt, out, pin, pin_out)
    return w


def make_head(jv, B, rank, local):
    """The V-JEPA 2 ViT-L SSv2 attentive-pool head + classifier over B clips' encoder tokens."""
    import torch
    tok_h, cfg = head_inputs(B, seed=rank)
    w = SeqBench()
    head = jv.Head.preset("vjepa2_vitl16_ssv2", seed=0, device=local)
    N = tok_h.shape[1]
    w.ctx = jv.HeadContext(head, B, N)
    w.stream = w.ctx.stream
    tok = torch.from_numpy(tok_h).cuda()
    pooled = torch.empty((B, cfg.embed_dim), dtype=torch.float32, device="cuda")
    logits = torch.empty((B, cfg.n_classes), dtype=torch.float32, device="cuda")
    pin = torch.from_numpy(tok_h).pin_memory()
    pin_logits = torch.empty((B, cfg.n_classes), dtype=torch.float32).pin_memory()
    w.step = lambda: w.ctx.forward(tok, pooled, logits)

    def e2e_step():
        with torch.cuda.stream(w.stream):
            tok.copy_(pin, non_blocking=True)
            w.ctx.forward(tok, pooled, logits)
            pin_logits.copy_(logits, non_blocking=True)
        w.ctx.sync()
    w.e2e_step = e2e_step
    w.h2d_bytes = pin.numel() * 4
    w.d2h_bytes = pin_logits.numel() * 4
    w.seq_len = N
    w.tokens_per_step = B * N
    w.launches = w.ctx.launches(True)
    w.metric = HEAD_METRIC
    w.label = f"V-JEPA 2 ViT-L SSv2 attentive-pool head + 174-way classifier, {N} tokens per clip x {B} per GPU"
    w.cpu_baseline = head_cpu_baseline
    w.keep = (head, tok, pooled, logits, pin, pin_logits)
    return w


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    if args.workload == PREDICTOR:
        return run_reference_predictor(args)
    if args.workload == HEADW:
        return run_reference_head(args)
    import oracle
    from dataclasses import replace
    import synth
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from configs import WORKLOADS
    wl = BENCH_WORKLOADS[args.workload]
    cfg, dtype, _, (T, H, W) = WORKLOADS[args.workload]
    bf16 = dtype == "bf16"
    pix = synth.pixels(0, (1, T, 3, H, W))
    one = replace(cfg, n_layer=1)
    # calibration: the per-layer cost (1 layer minus the embedding and final norm alone)
    (t0_, t1_), N, threads, L = oracle_layer_times(args.workload)
    per_layer = max(t1_ - t0_, 1e-9)
    for _ in range(args.warmup):
        oracle.encode(one, 0, bf16, pix)
    full_times = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.encode(one, 0, bf16, pix)
        full_times.append((time.perf_counter() - t0) + (L - 1) * per_layer)
    wall = time.perf_counter() - t_start
    mean_full = statistics.mean(full_times)
    value = N / mean_full
    B = args.batch or wl["batch"]
    sample = (f"each step: the fp64 oracle on one {N}-token item with 1 of the {L} layers; the other {L - 1} "
              f"layers added at the calibrated per-layer time {per_layer:.2f} s; the {B} items of a step are "
              f"independent, so a step costs {B} such items")
    line = {"impl": "reference", "metric": wl["metric"], "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean_full * B, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl['label']} ({N} tokens) x {B} per GPU",
                       "tokens_per_step": B * N, "global_batch": B, "seq_len": N,
                       "wall_s_sampled_steps": wall},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
KERNEL_SOURCES = {
    "attention": ("attention_tc.cu", "ptx.cuh"),
    "layernorm": ("rowops.cu", "ptx.cuh"), "layernorm_final": ("rowops.cu", "ptx.cuh"),
    "patchify": ("rowops.cu", "ptx.cuh"),
}
GEMM_SOURCES = ("gemm_tc.cu", "gemm_tc2.cu", "epilogue.cuh", "ptx.cuh")


def source_sha1(kernel_class: str):
    """sha1 over the source files the kernel class is built from."""
    h = hashlib.sha1()
    for name in KERNEL_SOURCES.get(kernel_class, GEMM_SOURCES):
        with open(os.path.join(ROOT, "jepa_vision_encoder_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def time_graph_steps(jv, model, wl, B, steps, warmup, flush, rank):
    """ms per step of graph-replayed encodes of B clips (L2 flushed between steps)."""
    import torch
    import synth
    T, H, W = wl["T"], wl["H"], wl["W"]
    ctx = jv.Context(model, B, T, H, W, graph=True)
    pix = torch.from_numpy(synth.pixels(rank, (B, T, 3, H, W))).cuda()
    out = torch.empty((B, model.n_tokens(T, H, W), model.hp.embed_dim), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(ctx.stream):
        for _ in range(warmup):
            flush.zero_()
            ctx.encode(pix, out)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(ctx.stream)
            ctx.encode(pix, out)
            e1.record(ctx.stream)
        torch.cuda.synchronize()
    ctx.sync()
    ctx.close()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def time_pos_tables(jv, model, T, H, W, reps=20):
    """The one-off table kernels of a fixed-table model: the training-grid table (at load) and its
    resize to the clip grid (once per clip shape), each timed alone with CUDA events."""
    import torch
    hp = model.hp
    three = hp.pos_type == jv.POS_SINCOS3D
    grid0 = ((hp.n_frames // hp.tubelet_size) if three else 1, hp.img_size // hp.patch_size, hp.img_size // hp.patch_size)
    grid1 = (T // hp.tubelet_size, H // hp.patch_size, W // hp.patch_size)
    D = hp.embed_dim
    mode = jv.RESIZE_TRILINEAR if three else jv.RESIZE_BICUBIC

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return 1e3 * e0.elapsed_time(e1) / reps

    base = jv.ops.sincos_table(hp.pos_type, *grid0, D, bool(hp.sincos_w_first), bool(hp.sincos_uniform_power))
    us_table = timed(lambda: jv.ops.sincos_table(hp.pos_type, *grid0, D, bool(hp.sincos_w_first),
                                                 bool(hp.sincos_uniform_power)))
    us_resize = timed(lambda: jv.ops.pos_resize(base, grid0, grid1, mode))
    rows0, rows1 = grid0[0] * grid0[1] * grid0[2], grid1[0] * grid1[1] * grid1[2]
    resize_bytes = 4.0 * D * (rows0 + rows1)   # the source table once, the resized table once
    return {"train_grid": list(grid0), "clip_grid": list(grid1),
            "table_us": us_table, "table_bytes": 4.0 * D * rows0,
            "resize_us": us_resize, "resize_mode": "trilinear" if three else "bicubic",
            "resize_bytes": resize_bytes, "resize_gbs": resize_bytes / (us_resize * 1e-6) / 1e9,
            "note": "outside the step: the table is baked at load, the resize runs once per clip shape; "
                    "both tables fit in L2, timed back to back without a flush"}


def fp32_ffma_peak_tflops():
    """Dense fp32 FFMA peak of this GPU: SMs x 128 FP32 lanes x 2 flops per FMA x the maximum SM
    clock (the measured-peaks file's, else 2070 MHz)."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", 2070.0))
    except (OSError, ValueError):
        mhz = 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12, sms, mhz


def profile_classes(jv, ctx, pix, out, flush, steps, warmup, stream):
    """Per-kernel-class durations: `steps` encodes with the library's event hook (events captured
    inside the graph; eager launches if the driver cannot time those). Returns (classes, ms per
    step of the profiled pass, launch mode, clock summary)."""
    import torch
    ctx.set_profiling(True)
    launch_mode = "CUDA graph replay of the encode"
    try:
        for _ in range(2):
            ctx.encode(pix, out)
        ctx.sync()
        ctx.profile(reset=True)
    except jv.JepaError:
        ctx.set_graph(False)
        launch_mode = "CUDA graph replay of the encode (per-kernel events: eager launches)"
    for _ in range(warmup):
        flush.zero_()
        ctx.encode(pix, out)
    ctx.sync()
    ctx.profile(reset=True)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        p0.record(stream)
        for _ in range(steps):
            flush.zero_()
            ctx.encode(pix, out)
        p1.record(stream)
        torch.cuda.synchronize()
    ctx.sync()
    prof = ctx.profile(reset=True)
    ctx.set_profiling(False)
    return prof, p0.elapsed_time(p1) / steps, launch_mode, clk.summary()


def full_attention_control(jv, wl, B, steps, warmup, flush, rank, local):
    """The same clips through the same encoder with full attention instead of the block-causal
    mask: what skipping the masked key tiles saves (step time and attention kernel time)."""
    import torch
    import synth
    T, H, W = wl["T"], wl["H"], wl["W"]
    model = jv.Model.preset(wl["preset"], seed=0, dtype="bf16", device=local, attn_mode=jv.ATTN_FULL)
    ms = time_graph_steps(jv, model, wl, B, steps, warmup, flush, rank)
    ctx = jv.Context(model, B, T, H, W, graph=True)
    pix = torch.from_numpy(synth.pixels(rank, (B, T, 3, H, W))).cuda()
    out = torch.empty((B, model.n_tokens(T, H, W), model.hp.embed_dim), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(ctx.stream):
        prof, _, _, _ = profile_classes(jv, ctx, pix, out, flush, min(steps, 10), warmup, ctx.stream)
    ctx.close()
    att = prof["attention"]
    return {"ms_per_step": ms, "attention_avg_us": 1e3 * att["total_ms"] / att["launches"],
            "attention_tflops_all_pairs": att["flops"] / (att["total_ms"] / 1e3) / 1e12}


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = init_ranks()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    import jepa_vision_encoder_gb300 as jv
    import synth

    wl = BENCH_WORKLOADS[args.workload]
    B, T, H, W = args.batch or wl["batch"], wl["T"], wl["H"], wl["W"]
    dtype = wl.get("dtype", "bf16")
    model = jv.Model.preset(wl["preset"], seed=0, dtype=dtype, device=local)
    ctx = jv.Context(model, B, T, H, W)
    N = model.n_tokens(T, H, W)
    D = model.hp.embed_dim
    pix_h = torch.from_numpy(synth.pixels(rank, (B, T, 3, H, W)))
    pix = pix_h.cuda()
    out = torch.empty((B, N, D), dtype=torch.float32, device="cuda")
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = ctx.stream
    peaks = measured_peaks()

    with torch.cuda.stream(stream):
        # headline: the timed steps replay one CUDA graph of the encode, nothing else inside it
        ctx.set_graph(True)
        for _ in range(args.warmup):
            flush.zero_()
            ctx.encode(pix, out)
        ctx.sync()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        barrier(local)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            for i in range(args.steps):
                flush.zero_()
                starts[i].record(stream)
                ctx.encode(pix, out)
                ends[i].record(stream)
            torch.cuda.synchronize()
        barrier(local)
        torch.cuda.synchronize()
        ctx.sync()
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

        # per-kernel durations: the same K steps again with the library's event hook (events
        # captured inside the graph; eager launches if the driver cannot time those). The events
        # between kernels lengthen the step, so the headline above is taken without them.
        prof, prof_ms, launch_mode, clk_prof = profile_classes(jv, ctx, pix, out, flush, args.steps, args.warmup,
                                                               stream)

        # the same step with eager launches, for comparison (not the headline)
        ctx.set_graph(False)
        for _ in range(2):
            ctx.encode(pix, out)
        e_ms = []
        for _ in range(min(args.steps, 20)):
            flush.zero_()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            ctx.encode(pix, out)
            s1.record(stream)
            e_ms.append((s0, s1))
        torch.cuda.synchronize()
        eager_ms = statistics.mean(a.elapsed_time(b) for a, b in e_ms)
        ctx.set_graph(True)

    total_ms = reduce_max(sum(step_ms), device="cuda" if world > 1 else None)
    ms_per_step = total_ms / args.steps
    tokens_per_step = world * B * N
    value = tokens_per_step * args.steps / (total_ms / 1e3)
    flops_per_step = sum(v["flops"] for v in prof.values()) / args.steps  # per GPU
    tflops = world * flops_per_step * args.steps / (total_ms / 1e3) / 1e12

    # dominant kernel class of the timed region
    name, st = max(prof.items(), key=lambda kv: kv[1]["total_ms"])
    avg_ms = st["total_ms"] / st["launches"]
    fp32_peak, n_sms, max_mhz = fp32_ffma_peak_tflops()
    if st["flops"] > 0 and dtype == "fp32":
        achieved = st["flops"] / st["launches"] / (avg_ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": fp32_peak, "unit": "TFLOP/s",
                "frac": achieved / fp32_peak, "kernel": name,
                "peak_derivation": f"{n_sms} SMs x 128 fp32 FMA lanes x 2 flops x {max_mhz:.0f} MHz"}
    elif st["flops"] > 0:
        achieved = st["flops"] / st["launches"] / (avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "kernel": name,
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
    else:
        achieved = st["bytes"] / st["launches"] / (avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "kernel": name}
    rec = NCU_TRAFFIC.get((args.workload, name, B))  # null for other workloads, batches or changed sources
    roof["traffic"] = rec["bytes_per_launch"] if rec and rec.get("sha1") == source_sha1(name) else None
    roof["peak_source"] = peaks["source"]
    kernels = {k: {"launches": v["launches"], "avg_us": 1e3 * v["total_ms"] / v["launches"],
                   "share": v["total_ms"] / max(sum(x["total_ms"] for x in prof.values()), 1e-9),
                   **({"tflops": v["flops"] / (v["total_ms"] / 1e3) / 1e12} if v["flops"] else {}),
                   **({"gbs": v["bytes"] / (v["total_ms"] / 1e3) / 1e9} if v["bytes"] else {})}
               for k, v in prof.items()}

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region: a
    # stream of clips through the pipelined host call (every step uploads its pixels and downloads
    # its tokens; the copies overlap the neighbouring steps' encodes), one sync closing the region
    pin_in = pix_h.pin_memory()
    pin_out = torch.empty((B, N, D), dtype=torch.float32).pin_memory()
    ctx.encode_host_async(pin_in, pin_out)
    ctx.sync()
    e2e_steps = min(args.steps, 20)
    barrier(local)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ctx.encode_host_async(pin_in, pin_out)
    ctx.sync()
    e2e_s = reduce_max(time.perf_counter() - t0, device="cuda" if world > 1 else None)
    ctx.encode_host(pin_in, pin_out)  # the synchronous call, one clip batch at a time, for comparison
    e2e_sync_steps = min(args.steps, 5)
    t1 = time.perf_counter()
    for _ in range(e2e_sync_steps):
        ctx.encode_host(pin_in, pin_out)
    e2e_sync_s = time.perf_counter() - t1
    e2e = {"value": tokens_per_step * e2e_steps / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": pin_in.numel() * 4, "d2h_bytes_per_step": pin_out.numel() * 4,
           "api": "jepa_encode_host_async x steps, then jepa_context_sync",
           "synchronous_value": tokens_per_step * e2e_sync_steps / e2e_sync_s}

    launches = ctx.launches(B, T, H, W)
    # the same clip at batch 1 (latency case of the workload), measured the same way
    b1 = None
    if B != 1:
        ms1 = reduce_max(time_graph_steps(jv, model, wl, 1, min(args.steps, 50), args.warmup, flush, rank),
                         device="cuda" if world > 1 else None)
        fl1 = flops_per_step / B
        b1 = {"ms_per_step": ms1, "value": world * N / (ms1 / 1e3), "unit": "tokens/s",
              "tflops": world * fl1 / (ms1 / 1e3) / 1e12,
              "frac_of_bf16_peak": fl1 / (ms1 / 1e3) / 1e12 / peaks["bf16_tflops"]}
    control = None
    if wl.get("full_attention_control"):
        control = full_attention_control(jv, wl, B, min(args.steps, 20), args.warmup, flush, rank, local)
        att = prof["attention"]
        att_us = 1e3 * att["total_ms"] / att["launches"]
        control.update({"block_causal_ms_per_step": ms_per_step, "block_causal_attention_avg_us": att_us,
                        "step_speedup": control["ms_per_step"] / ms_per_step,
                        "attention_speedup": control["attention_avg_us"] / att_us,
                        "note": "same weights and clips, attn_mode full: every key tile visited; the "
                                "block-causal run visits only tiles with a visible pair"})
    pos_table = time_pos_tables(jv, model, T, H, W) if model.hp.pos_type in (jv.POS_SINCOS2D, jv.POS_SINCOS3D) else None
    line = None
    if rank == 0:
        line = {"metric": wl["metric"], "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": f"{wl['label']} ({N} tokens) x {B} per GPU",
                           "tokens_per_step": tokens_per_step, "global_batch": world * B, "seq_len": N,
                           "parallelism": f"replicas x{world} (independent clips, no collective)",
                           "l2": "flushed (256 MiB write) between steps", "weights": "seeded synthetic"},
                "tflops": tflops, "eager_ms_per_step": eager_ms, "launch_mode": launch_mode,
                "roofline": roof, "kernels": kernels,
                "e2e": e2e, "gpu_launches": launches * args.steps, "batch1": b1,
                "clocks": {k: v for k, v in clk.summary().items()},
                "profiled_pass": {"ms_per_step": prof_ms, "clocks": clk_prof}}
        if dtype == "fp32":
            line["dtype"] = "f32"
            line["frac_of_fp32_peak"] = tflops / (world * fp32_peak)
        else:
            line["frac_of_bf16_peak"] = tflops / (world * peaks["bf16_tflops"])
        if control:
            line["full_attention_control"] = control
        if pos_table:
            line["pos_table"] = pos_table
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def spawn_ranks(n: int, argv) -> int:
    """`python bench.py --gpus N` without torchrun: start N ranks, one process per GPU, through
    torch.distributed.run on 127.0.0.1 with the same arguments, and return their exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def init_ranks():
    """Process group of a multi-rank run (NCCL on GPUs, gloo on a CPU-only host); returns the
    (rank, world, local rank) triple and reports it on stderr."""
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
        print(f"bench.py: rank {rank} of {world} (local GPU {local})", file=sys.stderr, flush=True)
    return rank, world, local


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if args.gpus < 1:
        raise SystemExit(f"bench.py: --gpus {args.gpus} must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return spawn_ranks(args.gpus, argv)
    if dist_env()[1] != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but the launcher started {dist_env()[1]} ranks")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == PREDICTOR:
        return run_sequence(args, {"batch": 8}, make_predictor)
    if args.workload == HEADW:
        return run_sequence(args, {"batch": 8}, make_head)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
