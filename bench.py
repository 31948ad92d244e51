"""Benchmark of the chunked gated delta rule on GB300: one step = forward + backward of the
whole path (the forward in save mode, then the backward on its saved chunk intermediates) over
one batch of synthetic input. Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

The headline is the largest single-GPU workload of the benchmark plan (GDN, B=1, T=32768,
H=16); the other forward+backward workloads of the plan (the B=2 T=4096 training shape, packed
documents, KDA, grouped q/k heads) are measured the same way and reported under `workloads`.

Timing. Every timed region is exactly K steps between CUDA events on the launching stream,
with a synchronize (and a barrier across ranks) on both sides. The region is repeated until
the repeats span at least --min-seconds, and `ms_per_step` is the median over the repeats
(all repeat times are reported). The library's per-launch timing hook is off in these regions;
per-kernel device times come from a separate pass afterwards. Inputs are larger than L2.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent
replicas, no collective on the data path); the reported value is all ranks' tokens divided
by the slowest rank's time.
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

METRIC = "GDN/KDA fwd+bwd tokens/s and TFLOP/s on 1 GB300; % of bf16 TC peak"
DEFAULT_WORKLOAD = "gdn_b1_t32768_h16"
SECONDARY_WORKLOADS = ("gdn_b2_t4096_h16", "gdn_varlen_t16384_12docs_h16", "kda_b1_t8192_h32",
                       "gdn_gqa_b2_t4096_h16_hk4", "gdn_b1_t8192_h16")
# Algorithmic tensor-core work of the chunked form per (token, head), C=64, K=V=128:
# forward 6CK + 4CV + 6KV, backward 12CK + 8CV + 12KV + 4C^2 (FLOP; recomputation excluded).
FWD_FLOP_PER_TOKEN_HEAD = 180_224
BWD_FLOP_PER_TOKEN_HEAD = 376_832
# Minimal HBM bytes per (token, head): the inputs read and the outputs written once
# (GDN: q, k, v, o 256 B each, g 4 B, beta 2 B; the backward adds dO and the gradients).
IO_BYTES_PER_TOKEN_HEAD = {("gdn", "fwd"): 1030, ("gdn", "bwd"): 1804, ("kda", "fwd"): 1538,
                           ("kda", "bwd"): 2820}
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
# Kernel name of the timing hook -> source file of that kernel.
KERNEL_SOURCES = {"prepare": "k_prep.cu", "chain_fwd": "k_chain.cu", "chain_bwd": "k_chain_bwd.cu",
                  "bwd_feat": "k_bwd_feat.cu", "bwd_tok": "k_bwd_tok.cu", "compose": "k_scan.cu"}
KERNEL_SOURCES_KDA = {**KERNEL_SOURCES, "prepare": "k_prep_kda.cu", "bwd_tok": "k_bwd_tok_kda.cu"}
# DRAM bytes (read + write) of one step's launches of a kernel from an ncu capture of
# dram__bytes_read.sum and dram__bytes_write.sum: (kernel, workload) -> (bytes, source_hash()
# of the kernel when captured). Reported only while the source is unchanged; null otherwise.
# Captured on the B=2 T=4096 H=16 GDN step and the B=1 T=4096 H=32 KDA step (2048 chunk-heads
# each, all heads in one group). The chunk kernels' traffic is per chunk-head, so the
# B=1 T=32768 H=16 entries are those bytes x 4 (8192 chunk-heads) and the B=1 T=8192 H=32 KDA
# entries x 2 (4096); the chains' traffic depends on the segment plan and is not scaled.
_GDN_T4096 = {"prepare": 611_470_336, "chain_fwd": 545_798_400, "compose": 29_376_000,
              "chain_bwd": 532_253_440, "bwd_feat": 526_161_920, "bwd_tok": 623_438_592}
_KDA_T4096 = {"prepare": 748_809_984, "chain_fwd": 548_044_800, "compose": 29_377_024,
              "chain_bwd": 533_810_176, "bwd_feat": 526_905_344, "bwd_tok": 749_082_368}
_HASHES = {("prepare", False): "9f4bd99a328245fe", ("prepare", True): "ef796d48524c2ad1",
           ("chain_fwd", False): "ede9cdea014a4770", ("chain_fwd", True): "ede9cdea014a4770",
           ("compose", False): "aee154a000cfde9f", ("compose", True): "aee154a000cfde9f",
           ("chain_bwd", False): "9a792f73725d839b", ("chain_bwd", True): "9a792f73725d839b",
           ("bwd_feat", False): "ca6dc5d5b6a21f11", ("bwd_feat", True): "ca6dc5d5b6a21f11",
           ("bwd_tok", False): "e3d84be8a81a7d84", ("bwd_tok", True): "674c8996578b69be"}
NCU_TRAFFIC_BYTES = {}
for _k, _v in _GDN_T4096.items():
    NCU_TRAFFIC_BYTES[(_k, "gdn_b2_t4096_h16")] = (_v, _HASHES[(_k, False)])
    if _k in ("prepare", "bwd_feat", "bwd_tok"):
        NCU_TRAFFIC_BYTES[(_k, "gdn_b1_t32768_h16")] = (4 * _v, _HASHES[(_k, False)])
for _k, _v in _KDA_T4096.items():
    NCU_TRAFFIC_BYTES[(_k, "kda_b1_t4096_h32")] = (_v, _HASHES[(_k, True)])
    if _k in ("prepare", "bwd_feat", "bwd_tok"):
        NCU_TRAFFIC_BYTES[(_k, "kda_b1_t8192_h32")] = (2 * _v, _HASHES[(_k, True)])
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


def source_hash(kernel: str, per_channel: bool = False):
    """First 16 hex digits of the SHA-256 of the kernel's source file (the per-channel gate's
    own file where it has one) and the headers it includes (common.cuh, umma.cuh, and the
    inverse's tri_inverse.cuh for the prepare kernels), or None."""
    name = (KERNEL_SOURCES_KDA if per_channel else KERNEL_SOURCES).get(kernel)
    if name is None:
        return None
    h = hashlib.sha256()
    parts = (name, "common.cuh", "umma.cuh") + (("tri_inverse.cuh",) if kernel == "prepare" else ())
    for part in parts:
        try:
            with open(os.path.join(ROOT, "chunked_gated_delta_05_gb300", "csrc", part), "rb") as f:
                h.update(f.read())
        except OSError:
            return None
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, per_channel: bool = False):
    """Per-step DRAM bytes of `kernel` on `workload` from the ncu table, or None when the table
    has no entry or the kernel's source has changed since the capture."""
    entry = NCU_TRAFFIC_BYTES.get((kernel, workload))
    if entry is None:
        return None
    nbytes, digest = entry
    return nbytes if digest == source_hash(kernel, per_channel) else None


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
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm), "interval_ms": 100}


def oracle_sample_tokens_per_s(w, d):
    """Time the CPU oracle (fp64 recurrence, forward + backward) on the given inputs."""
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


def sample_inputs(w, tokens: int, d=None):
    """The first `tokens` tokens of batch row 0 of workload `w` (same draws, sliced)."""
    from chunked_gated_delta_05_gb300 import synth
    if d is None:
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
        oracle_sample_tokens_per_s(w, d)
    times = []
    for _ in range(args.steps):
        _, dt = oracle_sample_tokens_per_s(w, d)
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


def n_chunk_heads(w, cu):
    if cu is not None:
        return sum((cu[i + 1] - cu[i] + 63) // 64 for i in range(len(cu) - 1)) * w.H
    return w.B * ((w.T + 63) // 64) * w.H


class Runner:
    """One workload on one GPU: device inputs, the training step, and its timers."""

    def __init__(self, w, dev, world, barrier):
        import torch
        from chunked_gated_delta_05_gb300 import gdn_bwd, gdn_fwd, kda_bwd, kda_fwd, synth
        self.torch = torch
        self.w, self.dev, self.world, self.barrier = w, dev, world, barrier
        self.host = synth.make_inputs(w)
        self.d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in self.host.items()}
        self.kw = dict(use_qk_l2norm=w.use_qk_l2norm, use_beta_sigmoid=w.beta_logits,
                       cu_seqlens=self.d["cu_seqlens"])
        self.fwd_fn, self.bwd_fn = (kda_fwd, kda_bwd) if w.per_channel else (gdn_fwd, gdn_bwd)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.tokens = w.B * w.T
        self.head_groups = 0  # the library's setting for the timed steps (0: automatic)

    # inputs that only the backward reads (the end-to-end region copies them behind the rest)
    BWD_ONLY_INPUTS = ("dO", "dht")

    def forward(self, inp):
        # training forward: saves its chunk intermediates for the backward
        return self.fwd_fn(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], initial_state=inp["h0"],
                           output_final_state=True, status=self.status, save=True, **self.kw)

    def backward(self, inp, saved):
        return tuple(self.bwd_fn(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["dO"], dht=inp["dht"],
                                 initial_state=inp["h0"], status=self.status, saved=saved, **self.kw))

    def step(self, inp):
        o, hT, saved = self.forward(inp)
        return (o, hT) + self.backward(inp, saved)

    def check_status(self, where):
        if int(self.status.item()) != 0:
            raise RuntimeError(f"device status {int(self.status.item())} {where} ({self.w.name})")

    def warmup(self, n):
        for _ in range(n):
            self.step(self.d)
        self.torch.cuda.synchronize(self.dev)
        self.check_status("during warm-up")

    def timed_regions(self, steps, min_seconds, run=None):
        """Repeats of an exactly-`steps`-step region until they span `min_seconds`; returns the
        per-step time of each repeat (ms, slowest rank)."""
        torch = self.torch
        run = run or (lambda n: [self.step(self.d) for _ in range(n)])
        per_step = []
        spent = 0.0
        while not per_step or spent < min_seconds:
            self.barrier()
            torch.cuda.synchronize(self.dev)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(self.stream)
            run(steps)
            t1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            self.barrier()
            ms = max_over_ranks(t0.elapsed_time(t1), self.dev)
            per_step.append(ms / steps)
            spent += ms * 1e-3
            if len(per_step) >= 1000:
                break
        return per_step

    def kernel_pass(self, steps, groups=1):
        """Per-kernel device times of `steps` steps with the library's timing hook on. With
        groups=1 all heads run in one group (one stream), so no launch overlaps another and
        each event pair brackets one kernel alone; groups=0 keeps the automatic choice of the
        timed steps (for counting their launches)."""
        from chunked_gated_delta_05_gb300 import _lib, set_head_groups
        torch = self.torch
        torch.cuda.synchronize(self.dev)
        set_head_groups(groups)
        try:
            _lib.timing_enable(True)
            for _ in range(steps):
                self.step(self.d)
            torch.cuda.synchronize(self.dev)
            t = _lib.timing_read()
            _lib.timing_enable(False)
        finally:
            set_head_groups(self.head_groups)
        return t

    def e2e(self, steps, min_seconds):
        """End to end through the public API with host buffers (pinned), every copy inside the
        timed region: step i's inputs go host -> device on a copy stream while step i-1 computes,
        and step i's outputs (every gradient, o and the final state) go device -> host on a second
        copy stream while step i+1 computes. Each step's forward waits only for the inputs it
        reads; dO and dht, which only the backward reads, are copied behind them and waited for
        before the backward. o and the final state leave as soon as the forward has written them.
        Two input slots; a slot is refilled only after the step that read it has finished. No copy
        starts before the region's first event."""
        torch, dev, stream = self.torch, self.dev, self.stream
        host = self.host
        pinned_in = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        slots = [{k: (torch.empty_like(v, device=dev) if isinstance(v, torch.Tensor) else v)
                  for k, v in host.items()} for _ in range(2)]
        outs_dev = self.step(self.d)
        pinned_out = [[None if x is None else torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
                       for x in outs_dev] for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in pinned_in.values() if isinstance(v, torch.Tensor))
        d2h = sum(x.numel() * x.element_size() for x in outs_dev if x is not None)
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        slot_free = [torch.cuda.Event(), torch.cuda.Event()]
        for ev in slot_free:
            ev.record(stream)

        def run(n):
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)
            s_out.wait_event(start)
            last_out = None
            def copy_out(ev, srcs, dsts):
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev)
                    for src, dst in zip(srcs, dsts):
                        if src is not None:
                            src.record_stream(s_out)
                            dst.copy_(src, non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(s_out)
                return e

            for i in range(n):
                sl = i % 2
                loaded = []
                with torch.cuda.stream(s_in):
                    s_in.wait_event(slot_free[sl])
                    for part in (False, True):   # the forward's inputs, then the backward's own
                        for k, v in pinned_in.items():
                            if isinstance(v, torch.Tensor) and (k in self.BWD_ONLY_INPUTS) == part:
                                slots[sl][k].copy_(v, non_blocking=True)
                        loaded.append(torch.cuda.Event())
                        loaded[-1].record(s_in)
                stream.wait_event(loaded[0])
                o, hT, saved = self.forward(slots[sl])
                fwd_done = torch.cuda.Event()
                fwd_done.record(stream)
                copy_out(fwd_done, (o, hT), pinned_out[sl][:2])
                stream.wait_event(loaded[1])
                grads = self.backward(slots[sl], saved)
                done = torch.cuda.Event()
                done.record(stream)
                slot_free[sl] = done
                last_out = copy_out(done, grads, pinned_out[sl][2:])
            stream.wait_event(last_out)   # the region ends after the last result is on the host

        run(2)
        torch.cuda.synchronize(dev)
        per_step = self.timed_regions(steps, min_seconds, run)
        self.check_status("during the end-to-end region")
        ms = statistics.median(per_step)

        # The same copies with no compute: one step's inputs in and outputs out, concurrently on
        # the two copy streams (the host link's floor for this region's per-step time).
        def copies_only():
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            evs = []
            for s, pairs in ((s_in, [(slots[0][k], v) for k, v in pinned_in.items() if isinstance(v, torch.Tensor)]),
                             (s_out, [(dst, src) for src, dst in zip(outs_dev, pinned_out[0]) if src is not None])):
                s.wait_event(start)
                with torch.cuda.stream(s):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
                    evs.append(torch.cuda.Event())
                    evs[-1].record(s)
            for ev in evs:
                stream.wait_event(ev)
            end.record(stream)
            torch.cuda.synchronize(dev)
            return start.elapsed_time(end)

        copies_only()
        copy_ms = statistics.median([copies_only() for _ in range(5)])
        return {"value": job_throughput(self.tokens, self.world, ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
                "repeats": len(per_step),
                "copies": "pinned host buffers; inputs of step i+1 and outputs of step i-1 copied on two "
                          "streams while step i computes",
                "copies_only_ms_per_step": copy_ms,
                "copies_only": "one step's host-to-device and device-to-host copies alone, both directions "
                               "at once, no compute: the host link's floor for ms_per_step"}


def roofline_of(runner, per_kernel, steps, peaks, peak_src):
    """Roofline of the kernel with the largest device time in the kernel pass: algorithmic MMA
    FLOP per step / that kernel's device time per step, against the sustained bf16 peak (x the
    nominal tf32/bf16 ratio for tf32 operands)."""
    w = runner.w
    nch = n_chunk_heads(w, runner.d["cu_seqlens"])
    name, (tot_ms, launches) = max(per_kernel.items(), key=lambda kv: kv[1][0])
    flop_chunk, kind = KERNEL_FLOP_PER_CHUNK_HEAD.get(name, (0, "none"))
    step_ms = tot_ms / steps
    achieved = flop_chunk * nch / (step_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"] * (TF32_OVER_BF16 if kind == "tf32" else 1.0)
    total = max(1e-9, sum(x[0] for x in per_kernel.values()))
    traffic = ncu_traffic(name, w.name, w.per_channel)
    return {"bound": "tensor", "kernel": name, "operands": kind, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
            "traffic_gbs": None if traffic is None else traffic / (step_ms * 1e-3) / 1e9,
            "traffic_frac_of_hbm": None if traffic is None else traffic / (step_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, same kernel source"
                              if traffic is not None else "no capture of the current kernel source",
            "peak_source": f"{peak_src} bf16 sustained" + (" x nominal tf32/bf16 ratio" if kind == "tf32" else ""),
            "algorithmic_flop_per_chunk_head": flop_chunk, "chunk_heads": nch,
            "avg_launch_ms": tot_ms / max(launches, 1), "launches_per_step": launches / steps,
            "kernel_ms_per_step": step_ms,
            "kernel_time_share": {k: round(v[0] / total, 4) for k, v in per_kernel.items() if v[1]},
            "kernel_ms_per_step_all": {k: round(v[0] / steps, 5) for k, v in per_kernel.items() if v[1]}}


def measure_workload(runner, args, peaks, with_e2e=True):
    w = runner.w
    runner.warmup(args.warmup)
    per_step = runner.timed_regions(args.steps, args.min_seconds)
    runner.check_status("during the timed region")
    ms = statistics.median(per_step)
    flop = (FWD_FLOP_PER_TOKEN_HEAD + BWD_FLOP_PER_TOKEN_HEAD) * runner.tokens * w.H
    tflops_gpu = flop / (ms * 1e-3) / 1e12
    gate = "kda" if w.per_channel else "gdn"
    io = (IO_BYTES_PER_TOKEN_HEAD[(gate, "fwd")] + IO_BYTES_PER_TOKEN_HEAD[(gate, "bwd")]) * runner.tokens * w.H
    out = {"ms_per_step": ms, "tokens_per_s": job_throughput(runner.tokens, runner.world, ms),
           "tflops": tflops_gpu * runner.world, "pct_of_bf16_peak": tflops_gpu / peaks["bf16_tflops_sustained"],
           "io_gbs": io / (ms * 1e-3) / 1e9, "pct_of_hbm_io": io / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "timing": {"steps_per_region": args.steps, "repeats": len(per_step),
                      "region_ms_per_step": [round(x, 5) for x in per_step],
                      "mean_ms_per_step": statistics.fmean(per_step), "min_ms_per_step": min(per_step)}}
    if with_e2e:
        out["e2e"] = runner.e2e(args.steps, args.min_seconds)
    return out


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


def measure_forward_target(dev, peaks, iters=20):
    """Forward alone (inference: no saves) at T = 8192, H = 16, the shape of the forward
    target: chunked-form FLOP / wall time of the whole call (CUDA events around each call, so
    launch gaps and the wrapper's host work count), against the bf16 burst peak. Two input sets
    (q, k, v, g, beta: 2 x 100 MB, together larger than L2) alternate between calls."""
    import torch
    from chunked_gated_delta_05_gb300 import _lib, gdn_fwd, synth
    w = synth.WORKLOADS["gdn_b1_t8192_h16"]
    sets = []
    for seed in (w.seed, w.seed + 100):
        d = synth.make_inputs(w, seed=seed)
        sets.append({k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()})
    fwd = lambda d: gdn_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], output_final_state=True)
    stream = torch.cuda.current_stream(dev)
    for i in range(4):
        fwd(sets[i % 2])
    torch.cuda.synchronize(dev)
    times = []
    for i in range(iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fwd(sets[i % 2])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    # the same calls captured in CUDA graphs (one per input set) and replayed: the device time of
    # the forward without the call's host work
    graphs = []
    for dset in sets:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fwd(dset)
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fwd(dset)
        graphs.append(graph)
    for i in range(4):
        graphs[i % 2].replay()
    torch.cuda.synchronize(dev)
    gtimes = []
    for i in range(iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graphs[i % 2].replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        gtimes.append(e0.elapsed_time(e1))
    graph_ms = statistics.median(gtimes)
    del graphs
    _lib.timing_enable(True)
    for i in range(iters):
        fwd(sets[i % 2])
    torch.cuda.synchronize(dev)
    t = _lib.timing_read()
    _lib.timing_enable(False)
    flop = FWD_FLOP_PER_TOKEN_HEAD * w.B * w.T * w.H
    tflops = flop / (ms * 1e-3) / 1e12
    io = IO_BYTES_PER_TOKEN_HEAD[("gdn", "fwd")] * w.B * w.T * w.H
    gtflops = flop / (graph_ms * 1e-3) / 1e12
    return {"workload": w.name, "ms": ms, "tflops": tflops, "pct_of_bf16_peak": tflops / peaks["bf16_tflops"],
            "graph_replay": {"ms": graph_ms, "tflops": gtflops, "pct_of_bf16_peak": gtflops / peaks["bf16_tflops"],
                             "timing": "median of CUDA-event times around replays of the call captured in a "
                                       "CUDA graph (no host work)"},
            "peak_kind": "bf16 burst (measured)", "io_gbs": io / (ms * 1e-3) / 1e9,
            "pct_of_hbm_io": io / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "kernels_ms": {k: v[0] / iters for k, v in t.items() if v[1]},
            "timing": "median of CUDA-event times around each whole call; kernels_ms from a separate pass "
                      "with the library's timing hook"}


def run_forward_only(runner, args, peaks, rank):
    """The inference forward alone (no saves): K calls per timed region, repeated as in the
    training-step measurement; prints one JSON line."""
    w = runner.w
    d = runner.d

    def fwd_steps(n):
        for _ in range(n):
            runner.fwd_fn(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["h0"],
                          output_final_state=True, status=runner.status, **runner.kw)

    fwd_steps(args.warmup)
    runner.torch.cuda.synchronize(runner.dev)
    per_step = runner.timed_regions(args.steps, args.min_seconds, fwd_steps)
    runner.check_status("during the forward-only region")
    ms = statistics.median(per_step)
    flop = FWD_FLOP_PER_TOKEN_HEAD * runner.tokens * w.H
    gate = "kda" if w.per_channel else "gdn"
    io = IO_BYTES_PER_TOKEN_HEAD[(gate, "fwd")] * runner.tokens * w.H
    line = {"metric": "forward (inference) tokens/s", "value": job_throughput(runner.tokens, runner.world, ms),
            "unit": "tokens/s", "n_gpus": runner.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 io, bf16/tf32 mma, fp32 accumulate", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "mode": "inference forward"},
            "tflops": flop / (ms * 1e-3) / 1e12 * runner.world,
            "pct_of_bf16_burst_peak": flop / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "io_gbs": io / (ms * 1e-3) / 1e9, "timing": {"repeats": len(per_step)}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the K-step timed region until the repeats span this long")
    ap.add_argument("--reference-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="headline workload only")
    ap.add_argument("--head-groups", type=int, default=0,
                    help="force 1 or 2 head groups (0: the library's automatic choice)")
    ap.add_argument("--forward-only", action="store_true",
                    help="time the inference forward (no saves, no backward) of the workload instead")
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
    from chunked_gated_delta_05_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    peaks, peak_src = load_peaks()
    if args.head_groups:
        from chunked_gated_delta_05_gb300 import set_head_groups
        set_head_groups(args.head_groups)
    w = synth.WORKLOADS[args.workload]
    runner = Runner(w, dev, world, barrier)
    runner.head_groups = args.head_groups
    if args.forward_only:
        run_forward_only(runner, args, peaks, rank)
        if world > 1:
            dist.destroy_process_group()
        return
    sampler = ClockSampler(local_rank)
    runner.warmup(args.warmup)
    sampler.start()
    head = measure_workload(runner, args, peaks, with_e2e=False)
    clocks = sampler.stop()
    head_e2e = runner.e2e(args.steps, args.min_seconds)
    per_kernel = runner.kernel_pass(args.steps)
    roofline = roofline_of(runner, per_kernel, args.steps, peaks, peak_src)
    gpu_launches = sum(v[1] for v in runner.kernel_pass(args.steps, groups=args.head_groups).values())
    ms = head["ms_per_step"]
    if clocks.get("sm_mhz"):
        clocks["ms_x_median_sm_mhz"] = ms * clocks["sm_mhz"]

    line = {"metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 io, bf16/tf32 mma, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Hk": w.num_k_heads or w.H, "K": w.K,
                       "V": w.V, "chunk": 64, "gate": "per-channel" if w.per_channel else "scalar",
                       "l2norm": w.use_qk_l2norm, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (q/k/v/dO alone exceed the 129 MB L2), no flush",
                       "timing": "median over repeats of an exactly-K-step region (>= "
                                 f"{args.min_seconds:g} s of repeats); timing hook off"},
            "tflops": head["tflops"], "pct_of_bf16_peak": head["pct_of_bf16_peak"],
            "pct_of_hbm_io": head["pct_of_hbm_io"], "timing": head["timing"],
            "roofline": roofline, "clocks": clocks, "gpu_launches": gpu_launches,
            "gpu_launches_note": "library kernel launches in one K-step region as the timed steps run "
                                 "them (the timing hook counts them in a separate pass of K steps); "
                                 "the roofline's per-kernel times come from another pass with all "
                                 "heads in one group",
            "e2e": head_e2e}
    del runner
    torch.cuda.empty_cache()
    if not args.no_extras:
        # every rank runs the secondary workloads (their regions are bracketed by barriers)
        works = {}
        for name in SECONDARY_WORKLOADS:
            if name == w.name:
                continue
            r = Runner(synth.WORKLOADS[name], dev, world, barrier)
            r.head_groups = args.head_groups
            works[name] = measure_workload(r, args, peaks)
            del r
            torch.cuda.empty_cache()
        line["workloads"] = works
    if rank == 0 and not args.no_extras:
        line["next_rows"] = {"short_conv": measure_short_conv(synth.WORKLOADS["gdn_b2_t4096_h16"], dev, peaks)}
        line["forward_target"] = measure_forward_target(dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_tps, dt = oracle_sample_tokens_per_s(w, synth.make_inputs(w))
        line["cpu_baseline"] = {"value": cpu_tps, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"the full {w.name} batch once (fwd+bwd), {dt:.1f} s wall"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
