"""Benchmark of the chunked gated delta rule on GB300: one step = forward + backward of the
whole path (gdn_fwd in save mode, then gdn_bwd on the saved chunk intermediates) over one
batch of synthetic inputs. Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent
replicas, no collective on the data path); the reported value is all ranks' tokens divided
by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN/KDA fwd+bwd tokens/s and TFLOP/s on 1 GB300; % of bf16 TC peak"
DEFAULT_WORKLOAD = "gdn_b2_t4096_h16"
# Algorithmic tensor-core work of the chunked form per (token, head), C=64, K=V=128:
# forward 6CK + 4CV + 6KV, backward 12CK + 8CV + 12KV + 4C^2 (FLOP; recomputation excluded).
FWD_FLOP_PER_TOKEN_HEAD = 180_224
BWD_FLOP_PER_TOKEN_HEAD = 376_832
# Useful MMA FLOP per (chunk, head) of each kernel (C=64, K=V=128) and its operand kind.
KERNEL_FLOP_PER_CHUNK_HEAD = {
    "prepare": (4 * 2 * 64 * 64 * 128, "bf16"),            # K K^T, Q K^T, A K1, A V1
    "chain_fwd": (3 * 2 * 64 * 128 * 128 + 2 * 64 * 64 * 128, "tf32"),   # W S, Qt S, k~^T v_new; Aqk v_new
    "chain_bwd": (3 * 2 * 64 * 128 * 128 + 2 * 64 * 64 * 128, "tf32"),   # Kt dS', Qt^T dO, W^T dv; Aqk^T dO
    "bwd_feat": (3 * 2 * 64 * 128 * 128 + 2 * 2 * 64 * 64 * 128, "tf32"),
    "bwd_tok": (2 * 64 * 64 * 128 * 3 + 2 * 64 * 64 * 256 + 2 * 2 * 64 * 64 * 64 + 4 * 2 * 64 * 64 * 128, "tf32"),
    "tables": (0, "none"),
    "compose": (0, "none"),     # segmented-chain overhead: no algorithmic work of its own
    "group_sum": (0, "none"),   # grouped q/k heads only
}
TF32_OVER_BF16 = 1.1 / 2.25    # nominal dense tf32 / bf16 tensor rates of a GB300
# DRAM bytes (read + write) of one step's launches of a kernel, from an ncu capture of
# dram__bytes_read.sum and dram__bytes_write.sum on the same kernel build and workload
# (profiles/kernels_gdn_b2_t4096_h16.md); None elsewhere, and None for a kernel changed since.
NCU_TRAFFIC_BYTES = {
    ("prepare", "gdn_b2_t4096_h16"): (104.790272 + 511.031040) * 1e6,
    ("chain_fwd", "gdn_b2_t4096_h16"): (186.442752 + 35.709184 + 249.326592 + 136.108032) * 1e6,
    ("compose", "gdn_b2_t4096_h16"): (21.011200 + 21.011200) * 1e6,
    ("chain_bwd", "gdn_b2_t4096_h16"): (215.708160 + 31.632640 + 230.861568 + 115.156992) * 1e6,
    ("bwd_feat", "gdn_b2_t4096_h16"): (479.928576 + 288.795392) * 1e6,
    ("bwd_tok", "gdn_b2_t4096_h16"): (644.071168 + 88.860416) * 1e6,
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the slowest rank's time); x itself on a single rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / (ms * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            val = d.get(key)
            if isinstance(val, dict):
                val = val.get("value")
            if val is not None:
                out[key] = float(val)
        if "bf16_tflops" in out:
            out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
            out.setdefault("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
            return out, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample_tokens_per_s(w, d, seconds_hint: str):
    """Time the CPU oracle (fp64 recurrence, forward + backward) on the workload's inputs."""
    import oracle
    f = lambda t: None if t is None else t.double().numpy()
    t0 = time.time()
    oracle.gdr_fwd(f(d["q"]), f(d["k"]), f(d["v"]), f(d["g"]), f(d["beta"]), initial_state=f(d["h0"]),
                   use_qk_l2norm=w.use_qk_l2norm, use_beta_sigmoid=w.beta_logits, cu_seqlens=d["cu_seqlens"])
    oracle.gdr_bwd(f(d["q"]), f(d["k"]), f(d["v"]), f(d["g"]), f(d["beta"]), f(d["dO"]), dht=f(d["dht"]),
                   initial_state=f(d["h0"]), use_qk_l2norm=w.use_qk_l2norm, use_beta_sigmoid=w.beta_logits,
                   cu_seqlens=d["cu_seqlens"])
    dt = time.time() - t0
    tokens = d["q"].shape[0] * d["q"].shape[1]
    return tokens / dt, dt


def sample_inputs(w, tokens: int):
    """The first `tokens` tokens of batch row 0 of workload `w` (same draws, sliced)."""
    from chunked_gated_delta_05_gb300 import synth
    d = synth.make_inputs(w)
    out = {}
    for key in ("q", "k", "v", "g", "beta", "dO"):
        out[key] = d[key][:1, :tokens].contiguous()
    out["h0"] = None if d["h0"] is None else d["h0"][:1].contiguous()
    out["dht"] = None if d["dht"] is None else d["dht"][:1].contiguous()
    out["cu_seqlens"] = None
    return out


def run_reference(args, rank):
    """The oracle as it stands, timed on the host cores: each step = fwd+bwd on a sample."""
    if rank != 0:
        return
    from chunked_gated_delta_05_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    sample_tokens = min(w.T, args.reference_tokens)
    d = sample_inputs(w, sample_tokens)
    for _ in range(args.warmup):
        oracle_sample_tokens_per_s(w, d, "")
    times = []
    for _ in range(args.steps):
        _, dt = oracle_sample_tokens_per_s(w, d, "")
        times.append(dt)
    total = sum(times)
    value = sample_tokens * args.steps / total
    cores = os.cpu_count()
    sample = f"batch row 0, first {sample_tokens} tokens, all {w.H} heads of {w.name}; fwd+bwd per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": 1, "T": sample_tokens, "H": w.H,
                                             "K": w.K, "V": w.V, "chunk": 64},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_short_conv(w, dev, peaks, iters=10):
    """HBM roofline of the short convolution ahead of the path (causal depthwise Conv1d + SiLU,
    W = 4) on the mixed q/k/v channels of the workload (3 H 128 channels, B*T rows). Two input
    sets larger than L2 together alternate between launches. Algorithmic bytes: forward reads
    x and writes y (4 B per element); backward reads x and dy and writes dx (6 B per element)."""
    import torch
    from chunked_gated_delta_05_gb300 import _lib, causal_conv1d_bwd, causal_conv1d_fwd
    C, Wt = 3 * w.H * w.K, 4
    gen = torch.Generator(device="cpu")
    gen.manual_seed(7)
    sets = []
    for _ in range(2):
        x = torch.randn(w.B, w.T, C, generator=gen).to(torch.bfloat16).to(dev)
        dy = torch.randn(w.B, w.T, C, generator=gen).to(torch.bfloat16).to(dev)
        sets.append((x, dy))
    weight = (torch.randn(C, Wt, generator=gen) * 0.5).to(dev)
    bias = (torch.randn(C, generator=gen) * 0.1).to(dev)
    elems = w.B * w.T * C
    out = {}
    for name, fn, nbytes in (("fwd", lambda x, dy: causal_conv1d_fwd(x, weight, bias), 4 * elems),
                             ("bwd", lambda x, dy: causal_conv1d_bwd(x, weight, bias, dy), 6 * elems)):
        for i in range(3):
            fn(*sets[i % 2])
        torch.cuda.synchronize(dev)
        # device time of the library's launches (CUDA events on the launching stream around each
        # call's kernels), so the wrapper's host work between calls is not counted
        _lib.timing_enable(True)
        for i in range(iters):
            fn(*sets[i % 2])
        torch.cuda.synchronize(dev)
        t = _lib.timing_read()
        _lib.timing_enable(False)
        ms = t["conv_" + name][0] / iters
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
                     "frac_of_hbm": gbs / peaks["hbm_gbs"], "timing": "CUDA events around the kernels"}
    return {"shape": {"rows": w.B * w.T, "channels": C, "taps": Wt, "activation": "silu"}, "bound": "hbm", **out}


def measure_forward_target(dev, peaks, iters=10):
    """Forward alone (inference: no saves) at T = 8192, H = 16, the shape of the forward
    target: chunked-form FLOP / device time of the forward's kernels, against the bf16 peak.
    Inputs larger than L2 (67 MB of q/k/v plus the workspace tiles) are rewritten each call."""
    import torch
    from chunked_gated_delta_05_gb300 import _lib, gdn_fwd, synth
    w = synth.WORKLOADS["gdn_b1_t8192_h16"]
    d = synth.make_inputs(w)
    dc = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    fwd = lambda: gdn_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], output_final_state=True)
    for _ in range(3):
        fwd()
    torch.cuda.synchronize(dev)
    _lib.timing_enable(True)
    for _ in range(iters):
        fwd()
    torch.cuda.synchronize(dev)
    t = _lib.timing_read()
    _lib.timing_enable(False)
    ms = sum(v[0] for v in t.values()) / iters
    flop = FWD_FLOP_PER_TOKEN_HEAD * w.B * w.T * w.H
    tflops = flop / (ms * 1e-3) / 1e12
    return {"workload": w.name, "ms": ms, "tflops": tflops, "pct_of_bf16_peak": tflops / peaks["bf16_tflops"],
            "peak_kind": "bf16 burst", "kernels_ms": {k: v[0] / iters for k, v in t.items() if v[1]},
            "timing": "CUDA events around the forward's kernels"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--reference-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    from chunked_gated_delta_05_gb300 import _lib, gdn_bwd, gdn_fwd, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    w = synth.WORKLOADS[args.workload]
    host = synth.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    kw = dict(use_qk_l2norm=w.use_qk_l2norm, use_beta_sigmoid=w.beta_logits, cu_seqlens=d["cu_seqlens"])
    fwd_fn, bwd_fn = gdn_fwd, gdn_bwd
    if w.per_channel:
        from chunked_gated_delta_05_gb300 import kda_bwd, kda_fwd
        fwd_fn, bwd_fn = kda_fwd, kda_bwd
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(inp):
        # training step: the forward saves its chunk intermediates, the backward consumes them
        o, hT, saved = fwd_fn(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], initial_state=inp["h0"],
                              output_final_state=True, status=status, save=True, **kw)
        grads = bwd_fn(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["dO"], dht=inp["dht"],
                       initial_state=inp["h0"], status=status, saved=saved, **kw)
        return (o, hT) + tuple(grads)

    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")

    stream = torch.cuda.current_stream(dev)
    _lib.timing_enable(True)
    sampler = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(d)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    per_kernel = _lib.timing_read()
    _lib.timing_enable(False)
    ms = max_over_ranks(ms, dev)

    tokens = w.B * w.T
    value = job_throughput(tokens, world, ms)
    flop = (FWD_FLOP_PER_TOKEN_HEAD + BWD_FLOP_PER_TOKEN_HEAD) * tokens * w.H
    tflops = flop * world / (ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    bf16_sus = peaks["bf16_tflops_sustained"]

    # roofline of the dominant kernel (largest device time in the timed region)
    n_chunk_heads = sum((min(64, w.T - 64 * j) > 0) for j in range((w.T + 63) // 64)) * w.B * w.H
    if d["cu_seqlens"] is not None:
        cu = d["cu_seqlens"]
        n_chunk_heads = sum((cu[i + 1] - cu[i] + 63) // 64 for i in range(len(cu) - 1)) * w.H
    name, (tot_ms, launches) = max(per_kernel.items(), key=lambda kv: kv[1][0])
    flop_chunk, kind = KERNEL_FLOP_PER_CHUNK_HEAD[name]
    avg_ms = tot_ms / max(launches, 1)
    # the kernel's device time per step (the chains launch twice per step when segmented)
    step_ms = tot_ms / args.steps
    achieved = flop_chunk * n_chunk_heads / (step_ms * 1e-3) / 1e12
    peak = bf16_sus * (TF32_OVER_BF16 if kind == "tf32" else 1.0)
    kernel_share = {k: round(v[0] / max(1e-9, sum(x[0] for x in per_kernel.values())), 4) for k, v in per_kernel.items()}
    traffic = NCU_TRAFFIC_BYTES.get((name, w.name))
    roofline = {"bound": "tensor", "kernel": name, "operands": kind, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "traffic_gbs": None if traffic is None else traffic / (step_ms * 1e-3) / 1e9,
                "traffic_frac_of_hbm": None if traffic is None else traffic / (step_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "peak_source": f"{peak_src} bf16 sustained" + (" x nominal tf32/bf16 ratio" if kind == "tf32" else ""),
                "avg_launch_ms": avg_ms, "launches_per_step": launches / args.steps, "kernel_ms_per_step": step_ms,
                "kernel_time_share": kernel_share}
    gpu_launches = sum(v[1] for v in per_kernel.values())

    # End to end through the public API with host buffers (pinned), every copy inside the timed
    # region: step i's inputs go host -> device on a copy stream while step i-1 computes, and
    # step i's outputs (every gradient, o and the final state) go device -> host on a second copy
    # stream while step i+1 computes. Two input slots; a slot is refilled only after the step
    # that read it has finished.
    pinned_in = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    slots = [{k: (torch.empty_like(v, device=dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
             for _ in range(2)]
    outs_dev = step(d)
    pinned_out = [[None if x is None else torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs_dev]
                  for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pinned_in.values() if isinstance(v, torch.Tensor))
    d2h = sum(x.numel() * x.element_size() for x in outs_dev if x is not None)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    slot_free = [torch.cuda.Event(), torch.cuda.Event()]
    for ev in slot_free:
        ev.record(stream)

    def e2e_run(n):
        # no copy starts before this point of the compute stream (the timed region's start)
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        last_out = None
        for i in range(n):
            sl = i % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(slot_free[sl])
                for k, v in pinned_in.items():
                    if isinstance(v, torch.Tensor):
                        slots[sl][k].copy_(v, non_blocking=True)
                loaded = torch.cuda.Event()
                loaded.record(s_in)
            stream.wait_event(loaded)
            outs = step(slots[sl])
            done = torch.cuda.Event()
            done.record(stream)
            slot_free[sl] = done
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for src, dst in zip(outs, pinned_out[sl]):
                    if src is not None:
                        src.record_stream(s_out)
                        dst.copy_(src, non_blocking=True)
                last_out = torch.cuda.Event()
                last_out.record(s_out)
        stream.wait_event(last_out)   # the timed region ends after the last result is on the host

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / args.steps
    e_ms = max_over_ranks(e_ms, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the timed region")

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 io, bf16/tf32 mma, fp32 accumulate", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Hk": w.num_k_heads or w.H, "K": w.K,
                       "V": w.V, "chunk": 64,
                       "gate": "per-channel" if w.per_channel else "scalar", "l2norm": w.use_qk_l2norm,
                       "parallelism": f"replicas x{world}",
                       "l2": "per-step working set (67 MB inputs + ~1 GB workspace) exceeds the 129 MB L2"},
            "tflops": tflops, "pct_of_bf16_peak": tflops / bf16_sus,
            "roofline": roofline, "clocks": clocks, "gpu_launches": gpu_launches,
            "e2e": {"value": job_throughput(tokens, world, e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                    "copies": "pinned host buffers; inputs of step i+1 and outputs of step i-1 copied on two "
                              "streams while step i computes"}}
    if rank == 0:
        line["next_rows"] = {"short_conv": measure_short_conv(w, dev, peaks)}
        line["forward_target"] = measure_forward_target(dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_tps, dt = oracle_sample_tokens_per_s(w, host, "")
        line["cpu_baseline"] = {"value": cpu_tps, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"the full {w.name} batch once (fwd+bwd), {dt:.1f} s wall"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
