#!/usr/bin/env python
"""Benchmark of the Wan DiT guided denoising step on B300 (libwan, sm_103a).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload wan1.3b-30blk-guided-step | wan1.3b-block | wan14b-i2v-block |
                                wan1.3b-20step-sampler]

One step = one pass of the whole hot path over the 30-block 1.3B-shaped DiT at 480p
(21x60x104 latent -> 32760 tokens), batch 2 (cond + uncond): text projection, time
embedding, patchify, 30 blocks (AdaLN, QKV + 3D RoPE, self-attention, cross-attention,
GELU FFN, gated residuals), head + depatchify, fused CFG + Euler update.  Synthetic
seeded inputs, random-init weights ~N(0, 0.02).  Rank 0 prints one JSON line.

The 20-step sampler workload times one whole generation per bench step (text projection,
every block's cross-attention keys/values once, 20 guided steps on the uniform schedule).

--impl reference times the CPU fp64 oracle (the method's plain definition) on the
host cores, on a bounded sample of the same workload, and extrapolates to one step.
Multi-GPU: the step does not shard (self-attention couples every token); N ranks run
N independent replicas (weak scaling, no collective on the data path).
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

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "DiT step latent tokens/s and bf16 TFLOP/s on 1 B300; % of BF16 tensor peak"
UNIT = "latent tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def step_macs(s) -> dict:
    """Algorithmic multiply-accumulates of one guided step, by role (for the sampler: one
    whole generation, whose text projection and cross-attention keys/values are computed
    once and reused by every step)."""
    B, L, D, F, Lt, Li = s.batch, s.tokens, s.dim, s.ffn, s.text_len, s.img_len
    m = {
        "text": B * Lt * (s.text_dim * D + D * D) if s.text_dim else 0,
        "time": B * (s.freq_dim * D + D * D + 6 * D * D + 2 * D * D),
        "patchify": B * L * s.c_in * 4 * D,
        "qkv": s.blocks * B * L * 3 * D * D,
        "self_attn": s.blocks * B * 2 * L * L * D,
        "o": s.blocks * B * L * D * D,
        "cross_q_o": s.blocks * B * L * 2 * D * D,
        "cross_kv": s.blocks * B * (Lt + Li) * 2 * D * D,
        "cross_attn": s.blocks * B * 2 * L * (Lt + Li) * D,
        "ffn": s.blocks * B * L * 2 * D * F,
        "head": B * L * D * s.c_out * 4,
    }
    if s.steps > 1:
        for k in m:
            if k not in ("text", "cross_kv"):
                m[k] *= s.steps
    return m


# ---------------------------------------------------------------- clocks during the timed region

class Clocks:
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[3:7]):
                if flag.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle baseline

def blas_threads() -> int:
    """Threads numpy's BLAS runs the oracle's matrix products on."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def oracle_step_estimate(s, seed=0, rows_small=1, rows_large=513):
    """Time the fp64 oracle on a bounded sample of one block and extrapolate to a step.

    Sample: one 1.3B-shaped block on batch entry 0, run twice: with `rows_small` query
    rows (the row-independent part: LN and the key/value projections over all L tokens)
    and with `rows_large` rows (plus that many rows through attention over all keys,
    cross-attention and the FFN).  per_row = the difference / (rows_large - rows_small),
    measured over thousands of rows so it is not lost in the fixed part's noise; block =
    fixed + L * per_row; step = batch * blocks * block.
    """
    from oracle import wan_oracle as O
    one = s.replace(blocks=1)
    w = synth.make_weights(one, seed)
    inp = synth.make_inputs(one, seed)
    hp = O.Hyper.of(one)
    blk = w["blocks"][0]
    x = O.patchify(inp["latent"], w["patch_w"], w["patch_b"])[0]
    ctx = O.text_projection(inp["text"][:1], w)[0] if one.text_dim else inp["ctx_txt"][0]
    mods = np.zeros((6, one.dim))
    times = {}
    for n in (rows_small, rows_large):
        rows = np.arange(n)
        t0 = time.perf_counter()
        O.dit_block(x, mods, blk, ctx, None, hp, rows=rows)
        times[n] = time.perf_counter() - t0
    per_row = max((times[rows_large] - times[rows_small]) / (rows_large - rows_small), 1e-12)
    fixed = max(times[rows_small] - rows_small * per_row, 0.0)
    block = fixed + one.tokens * per_row
    step = block * s.batch * s.blocks * max(s.steps, 1)
    threads = blas_threads()
    sample = (f"one {one.dim}-wide block, batch entry 0: full LN+QKV over {one.tokens} tokens plus "
              f"{rows_small} and {rows_large} query rows end to end ({sum(times.values()):.1f} s of CPU); "
              f"extrapolated x{s.batch} batch x{s.blocks} blocks" + (f" x{s.steps} steps" if s.steps > 1 else ""))
    return step, threads, sample, sum(times.values())


def oracle_baseline(s, repeats=3):
    """The oracle's rate on this host: `repeats` all-core samples (mean and spread) and one
    single-threaded sample, the same sampling method as the reference arm."""
    units = s.batch * s.tokens * max(s.steps, 1)
    runs, sample, threads, spent = [], "", 1, 0.0
    for _ in range(repeats):
        step_s, threads, sample, cpu_s = oracle_step_estimate(s)
        runs.append(units / step_s)
        spent += cpu_s
    # Single-threaded: a child process whose BLAS starts with one thread.
    single = None
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, bench, synth; s = synth.WORKLOADS[%r].replace(batch=%d); "
            "r = bench.oracle_step_estimate(s); print(json.dumps([r[0], r[1], r[3]]))" % (s.name, s.batch))
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                             timeout=600)
        step_s, th, cpu_s = json.loads(out.stdout.strip().splitlines()[-1])
        if th == 1:
            single = units / step_s
        spent += cpu_s
    except (subprocess.SubprocessError, ValueError, IndexError):
        pass
    return {"value": round(statistics.mean(runs), 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": sample, "repeats": [round(r, 3) for r in runs],
            "spread": round((max(runs) - min(runs)) / statistics.mean(runs), 4),
            "single_thread_value": None if single is None else round(single, 3),
            "cpu_model": cpu_model(), "nproc": os.cpu_count(), "affinity": len(os.sched_getaffinity(0)),
            "cpu_seconds": round(spent, 1)}


# ---------------------------------------------------------------- multi-rank bookkeeping

def max_over_ranks(value: float, device="cpu") -> float:
    """The slowest rank's value (every rank gets it); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank_step: float, steps: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank_step * steps * world / (ms_max / 1e3)


# ---------------------------------------------------------------- our arm

def run_ours(a, s):
    import torch
    import torch.distributed as dist

    from video_diffusion_transformer_04_b300 import wan

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    w = synth.make_weights(s, 0)
    inp = synth.make_inputs(s, 0)
    m = wan.DiT(s, w, device=dev)
    del w
    bf = torch.bfloat16
    text_h = torch.from_numpy(inp["text"]).to(bf).pin_memory() if s.text_dim else None
    lat_h = torch.from_numpy(inp["latent"]).pin_memory()
    t0 = float(inp["t"][0])
    t_pair_h = torch.tensor([t0, t0 + s.dt], dtype=torch.float32).pin_memory()
    text = text_h.to(dev) if s.text_dim else None
    ctx_fixed = None if s.text_dim else torch.from_numpy(inp["ctx_txt"]).to(dev, bf)
    ctx_img = torch.from_numpy(inp["ctx_img"]).to(dev, bf) if s.img_len else None
    x = lat_h.to(dev)
    t_pair = t_pair_h.to(dev)
    v_ws = torch.empty(2, s.c_out, s.frames, s.height, s.width, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sampler = s.steps > 1
    noise = x.clone() if sampler else None

    def step():
        ctx = m.text_embed(text) if s.text_dim else ctx_fixed
        if sampler:  # one whole generation from the same noise
            x.copy_(noise)
            m.sample(x, s.steps, s.guide_scale, ctx, ctx_img)
        else:
            m.guided_step(x, t_pair, s.guide_scale, ctx, ctx_img, v_ws=v_ws)

    for _ in range(a.warmup):
        step()
    wan.wan_sync_status()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) == 36:
        gpu_id = "GPU-" + gpu_id
    clocks = Clocks(gpu_id)
    clocks.start()
    time.sleep(0.3)
    launches0 = wan.wan_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    launches = wan.wan_launch_count() - launches0
    clk = clocks.stop()
    wan.wan_sync_status()
    ms = max_over_ranks(e0.elapsed_time(e1), dev)

    # ---- the per-kernel split: a separate pass with CUDA events around every launch
    # (not the timed region above), sampled clocks alongside.
    prof_steps = 1 if sampler else a.steps
    pclocks = Clocks(gpu_id)
    pclocks.start()
    time.sleep(0.3)
    wan.wan_profile_begin(1 << 17)
    for _ in range(prof_steps):
        step()
    torch.cuda.synchronize(dev)
    prof = wan.wan_profile_end()
    pclk = pclocks.stop()
    wan.wan_sync_status()

    # ---- end to end through the public API with host buffers (copies inside the timed region)
    x_out_h = torch.empty_like(lat_h).pin_memory()
    h2d = lat_h.numel() * 4 + t_pair_h.numel() * 4 + (text_h.numel() * 2 if s.text_dim else 0)
    d2h = x_out_h.numel() * 4

    def step_host():
        (noise if sampler else x).copy_(lat_h, non_blocking=True)
        t_pair.copy_(t_pair_h, non_blocking=True)
        if s.text_dim:
            text.copy_(text_h, non_blocking=True)
        step()
        x_out_h.copy_(x, non_blocking=True)

    step_host()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    eclocks = Clocks(gpu_id)  # the e2e pass runs last: its own clock record shows any drift
    eclocks.start()
    time.sleep(0.3)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(a.steps):
        step_host()
    f1.record(stream)
    torch.cuda.synchronize(dev)
    eclk = eclocks.stop()
    ms_e2e = max_over_ranks(f0.elapsed_time(f1), dev)

    tokens_per_step = s.batch * s.tokens * max(s.steps, 1)
    weight_gb = sum(t.numel() * t.element_size() for bt in m.block_tensors for t in bt.values()) / 1e9
    ws_gb = m.ws.numel() / 1e9
    value = aggregate_rate(tokens_per_step, a.steps, world, ms)
    macs = step_macs(s)
    flop_step = 2 * sum(macs.values())
    pk, pk_kind = peaks()
    tflops = flop_step * a.steps / (ms / 1e3) / 1e12

    total_prof = sum(v[0] for v in prof.values()) or 1.0
    kernels = {k: {"ms_per_step": round(v[0] / prof_steps, 3), "launches_per_step": v[1] / prof_steps,
                   "share": round(v[0] / total_prof, 4)} for k, v in sorted(prof.items(), key=lambda kv: -kv[1][0])}
    fp8_attn = bool(s.fp8 & 1)
    dom = "attn_self_e4m3" if fp8_attn else "attn_self"
    roof = None
    if dom in prof:
        per_launch_flop = 2 * macs["self_attn"] / (s.blocks * max(s.steps, 1))  # one launch = one block, whole batch
        avg_ms = prof[dom][0] / prof[dom][1]
        achieved = per_launch_flop / (avg_ms / 1e3) / 1e12
        mhz = pclk.get("sm_mhz")
        clock_scaled = achieved / (mhz / pk["sm_max_mhz"]) if mhz and pk.get("sm_max_mhz") else None
        # E4M3 tensor peak: the measured bf16 figure times the nominal dense ratio 4.5 / 2.25
        peak = pk["bf16_tflops_sustained"] * (2.0 if fp8_attn else 1.0)
        kind = "e4m3 sustained = 2 x measured bf16 sustained (nominal ratio)" if fp8_attn else "bf16 sustained"
        burst = pk["bf16_tflops"] * (2.0 if fp8_attn else 1.0)
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "peak_kind": f"{kind} ({pk_kind})",
                "frac_of_burst": round(achieved / burst, 4),
                "achieved_at_max_clock": None if clock_scaled is None else round(clock_scaled, 1),
                "frac_of_burst_at_max_clock": None if clock_scaled is None else round(clock_scaled / burst, 4),
                "profiled_sm_mhz": mhz,
                "flop_per_launch": per_launch_flop, "avg_launch_ms": round(avg_ms, 4),
                "traffic": traffic_record(dom)}

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "per_guided_latent_tokens_per_s": round(value / s.batch, 1),
        "warmup": a.warmup, "ms_per_step": round(ms / a.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if not s.fp8 else "bf16 + e4m3", "data": "synthetic (seeded N(0,1) latent and text, N(0,0.02) weights)",
        "config": {"workload": s.name, "blocks": s.blocks, "batch": s.batch,
                   "latent": [s.c_in, s.frames, s.height, s.width], "tokens": s.tokens, "dim": s.dim,
                   "heads": s.heads, "head_dim": s.head_dim, "ffn": s.ffn, "text_len": s.text_len,
                   "img_len": s.img_len, "guide_scale": s.guide_scale,
                   "variant": {"qk_norm": s.qk_norm, "gelu_tanh": s.gelu_tanh, "fp8": s.fp8},
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "units": ("latent tokens of both CFG branches (batch 2) per DiT step"
                             + (f", {s.steps} steps per generation" if sampler else "")),
                   "l2": (f"inputs larger than L2 (126 MB): {weight_gb:.2f} GB of weights and {ws_gb:.1f} GB of "
                          "workspace stream through every step, so no flush is needed between steps")},
        "tflops": round(tflops, 1), "bf16_peak_frac": round(tflops / pk["bf16_tflops"], 4),
        "bf16_sustained_frac": round(tflops / pk["bf16_tflops_sustained"], 4),
        "flop_per_step": flop_step,
        "roofline": roof,
        "e2e": {"value": round(aggregate_rate(tokens_per_step, a.steps, world, ms_e2e), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "sm_mhz": eclk.get("sm_mhz")},
        "gpu_launches": launches,
        "clocks": clk,
        "kernels": kernels,
    }
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        print(json.dumps({"partial": out}), file=sys.stderr, flush=True)
        out["cpu_baseline"] = oracle_baseline(s)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def traffic_record(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/<kernel>_traffic.txt), or None when the kernel source changed since the
    counters were taken (the summary records the source's sha256 prefix)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.txt")
    if not os.path.exists(path):
        return None
    try:
        import hashlib
        rec = {}
        for line in open(path):
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
        src = os.path.join(ROOT, "video_diffusion_transformer_04_b300", "csrc", rec["source"])
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["source_sha256_16"]:
            return None
        return int(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(a, s):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    est = []
    threads, sample = 1, ""
    for i in range(a.warmup + a.steps):
        step_s, threads, sample, _ = oracle_step_estimate(s)
        if i >= a.warmup:
            est.append(step_s)
    step_s = statistics.mean(est)
    units = s.batch * s.tokens * max(s.steps, 1)
    value = units / step_s
    rates = [units / e for e in est]
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
           "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(step_s * 1e3, 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": s.name, "tokens": s.tokens, "blocks": s.blocks,
                      "batch": s.batch},
           "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": sample, "repeats": [round(r, 3) for r in rates],
                            "spread": round((max(rates) - min(rates)) / statistics.mean(rates), 4),
                            "cpu_model": cpu_model(), "nproc": os.cpu_count()},
           "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="wan1.3b-30blk-guided-step",
                    choices=["wan1.3b-30blk-guided-step", "wan1.3b-block", "wan14b-i2v-block",
                             "wan1.3b-20step-sampler"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--qk-norm", action="store_true", help="variant: RMSNorm on q and k before RoPE")
    ap.add_argument("--gelu-tanh", action="store_true", help="variant: tanh-form GELU in the FFN")
    ap.add_argument("--fp8", type=int, default=0, choices=[0, 1, 2, 3],
                    help="8-bit variant: 1 = 8-bit self-attention, 2 = FP8 QKV / FFN-up GEMMs, 3 = both")
    a = ap.parse_args()
    s = synth.WORKLOADS[a.workload].replace(qk_norm=a.qk_norm, gelu_tanh=a.gelu_tanh, fp8=a.fp8)
    if s.blocks == 1:
        s = s.replace(batch=2)  # guided step over a single block: cond + uncond
    if a.impl == "reference":
        run_reference(a, s)
    else:
        run_ours(a, s)


if __name__ == "__main__":
    main()
