"""Benchmark of the KDA operator on one GB300 (or N, one process each).

Headline: prefill tokens/s of one 96-head KDA layer (B=1, T=8192, H=96,
d=128; bf16 q/k/v/o, fp32 g/beta/state) -- one step is one kda_prefill call
over the whole layer, every row of the hot path (decay prefix, decay-weighted
operands, Gram matrices, triangular solve, inter-chunk readout, state carry,
epilogue).  The decode workload (256 sequences x 64 single-token steps) is
measured in the same run and reported under "decode".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload (weak
scaling, no collective on the data path); rank 0 prints one JSON line with the
aggregate over ranks timed as the max over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA tokens/s per layer (96 heads, d=128) prefill & decode; % of roofline"
UNIT = "tokens/s"

# Algorithmic bytes per token of one 96-head layer (prefill): q, k, v, o bf16
# (4 x 96 x 128 x 2) + g fp32 (96 x 128 x 4) + beta fp32 (96 x 4).
PREFILL_BYTES_PER_TOKEN = 4 * 96 * 128 * 2 + 96 * 128 * 4 + 96 * 4  # 147840
# the gated call reads bf16 decay logits z instead of fp32 g, and beta logits
GATED_BYTES_PER_TOKEN = 5 * 96 * 128 * 2 + 96 * 4  # 123264
# the output-gated call also reads the bf16 gate logits [T, H, d_v]
OGATED_BYTES_PER_TOKEN = 147840 + 96 * 128 * 2  # 172416
# the scalar-decay call (Gated DeltaNet) reads one fp32 log-decay per (token, head) instead of g
SDECAY_BYTES_PER_TOKEN = 4 * 96 * 128 * 2 + 2 * 96 * 4  # 99072
# the q, k, v prologue (ShortConv, Swish, L2Norm): three bf16 projections read and
# three bf16 results written per (token, head, channel); its fp32 conv weights
# [3, 96, 128, 4] are read once per launch
PROLOGUE_BYTES_PER_TOKEN = 6 * 96 * 128 * 2  # 147456
PROLOGUE_WEIGHT_BYTES = 3 * 96 * 128 * 4 * 4  # 589824
# the end-to-end leg streams the layer from host memory in this many segments
E2E_SEGMENTS = 8
# backward: algorithmic fp32 flops per (chunk, head) of the chunked backward (C = 32,
# d = 128), counted as 2 per multiply-add over the products it forms:
#   G, P (pairwise, C(C+1)/2 pairs x 2 d)      135,168 MACs
#   Y = V - Kt S0, dU's Kb dS, dQt, dKt, dKb, the two products of dS0   7 C d^2
#   P^T dO, T B, T^T dU, dP, dT (triangular, C^2 d / 2 each)            5/2 C^2 d
#   dA = -T^T dT T^T (2 C^3 / 3), the pairwise gradient terms (3 C^2 d)
BWD_C, BWD_D = 32, 128
BWD_MACS_PER_CHUNK_HEAD = (BWD_C * (BWD_C + 1) // 2 * 2 * BWD_D + 7 * BWD_C * BWD_D * BWD_D
                           + 5 * BWD_C * BWD_C * BWD_D // 2 + 2 * BWD_C ** 3 // 3
                           + 3 * BWD_C * BWD_C * BWD_D)
# fp32 CUDA-core peak of the part: SMs (read from the device) x 128 fp32 lanes x 2 flops
# per FMA x SM clock (the backward of fp32 inputs or d = 64 runs on the CUDA cores)
FP32_LANES_PER_SM = 128
# The tensor-core backward (bf16 inputs, d = 128) multiplies in tf32: its peak is the
# measured bf16 dense rate times the nominal tf32 / bf16 ratio of the part (1.1 / 2.25
# PFLOP/s dense)
TF32_PER_BF16 = 1.1 / 2.25
# Decode, per (sequence, head) step: fp32 state read + write (2 x 65536),
# q/k/v bf16 (768), g fp32 (512), beta (4), o bf16 (256).
DECODE_BYTES_PER_HEAD_STEP = 2 * 128 * 128 * 4 + 3 * 128 * 2 + 128 * 4 + 4 + 128 * 2  # 132612
L2_BYTES = 129 * 2 ** 20


# ----------------------------------------------------------------------------
# distributed plumbing (host side; no collective on the data path)
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (the slowest rank sets the
    job's time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampled every 20 ms in the background; samples are tagged
    with wall time so that those inside the timed region can be picked."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)
        return self

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

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = None
        if not inside:  # region shorter than the sampling period: take the nearest
            near = min(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))
            inside, note = [near[1]], "nearest sample (timed region shorter than the sampling period)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i] == "Active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def source_digest(relpath: str) -> str:
    with open(os.path.join(ROOT, relpath), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:12]


def profiled_traffic(kernel: str, source: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(source)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[2] == digest:
                return float(parts[3])
    return None


def time_steps(fn, steps: int, warmup: int, world: int, stream):
    """W untimed steps, then exactly K steps between CUDA events on `stream`,
    bracketed by a barrier and a device synchronize.  Returns
    (ms_per_step max over ranks, t_wall_start, t_wall_end)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(stream)
    for _ in range(steps):
        fn()
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    ms = ev0.elapsed_time(ev1) / steps
    return reduce_max(ms, world, device="cuda"), t0, t1


# ----------------------------------------------------------------------------
# CPU baseline: the fp64 oracle as it stands, on this host's cores
# ----------------------------------------------------------------------------

def cpu_baseline_prefill(heads: int = 96, tokens: int = 8192, seed: int = 1):
    """Time the oracle on a sample of the prefill workload (the first
    `tokens` tokens of `heads` heads, the same recipe), scaled to layer
    tokens/s (96 heads)."""
    import torch
    import oracle
    from linear_attention_sequence_gb300 import synth
    w = synth.WORKLOADS["prefill_8k"]
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q, k, v, g, beta = synth.draw_tokens(tokens, heads, w.d, w.d, w.dtype, w.mu, gen, "cpu")
    args = [x.to(torch.float64).numpy() for x in (q, k, v, g, beta)]
    cores = oracle.num_cpus()
    t0 = time.perf_counter()
    oracle.prefill(*args, num_threads=cores)
    dt = time.perf_counter() - t0
    layer_tokens = tokens * heads / 96.0
    return {"value": layer_tokens / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{heads} heads x {tokens} tokens of the prefill_8k recipe "
                      f"(fp64 token loop, {cores} threads), {dt:.2f} s wall"}


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------

def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    heads, tokens = 24, 8192
    # warm-up and timed steps, each one bounded sample of the workload
    import torch
    import oracle
    from linear_attention_sequence_gb300 import synth
    w = synth.WORKLOADS["prefill_8k"]
    gen = torch.Generator(device="cpu")
    gen.manual_seed(1)
    q, k, v, g, beta = synth.draw_tokens(tokens, heads, w.d, w.d, w.dtype, w.mu, gen, "cpu")
    a = [x.to(torch.float64).numpy() for x in (q, k, v, g, beta)]
    cores = oracle.num_cpus()
    for _ in range(args.warmup):
        oracle.prefill(*a, num_threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.prefill(*a, num_threads=cores)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = tokens * heads / 96.0 / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "prefill_8k sample: 24 of 96 heads x 8192 tokens (B=1, d=128, "
                               "bf16 q/k/v widened to fp64), scaled to 96-head layer tokens/s"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{heads} heads x {tokens} tokens per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def leg_summary(ms, units, nbytes, hbm_gbs, steps, kernel, extra=None):
    """A compact record of one secondary leg: time per step, units/s, and the
    HBM roofline fraction over its algorithmic bytes (of the measured peak)."""
    ach = nbytes / (ms * 1e-3) / 1e9
    d = {"ms": round(ms, 4), "tok_s": round(units / (ms * 1e-3)), "frac": round(ach / hbm_gbs, 4),
         "gbs": round(ach, 1), "bytes": int(nbytes), "steps": steps, "kernel": kernel}
    if extra:
        d.update(extra)
    return d


def check_device_status(kda, stream, leg: str):
    """A bounded device-side wait that gave up ends its kernel early: a step
    that stopped would look faster.  Any nonzero status ends the run."""
    st = kda.kda_get_last_device_error(stream)
    if st != 0:
        print(json.dumps({"error": f"device status {st} ({kda.kda_status_string(st)}) after the "
                                   f"{leg} leg: a bounded wait gave up; no result is reported"}),
              flush=True)
        sys.exit(3)


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from linear_attention_sequence_gb300 import _build
    _build.build()
    import linear_attention_sequence_gb300 as kda
    from linear_attention_sequence_gb300 import synth

    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, peak_src = measured_peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    if args.profile:
        return run_profile_case(args, kda, synth, dev, stream)
    check_device_status(kda, stream, "start")

    # ---------------- prefill (headline) ----------------
    w = synth.WORKLOADS["prefill_8k"]
    inp = synth.prefill_inputs(w, dev)
    T = w.total_tokens
    out = torch.empty((T, w.heads, w.d), dtype=w.dtype, device=dev)
    fin = torch.empty((1, w.heads, w.d, w.d), dtype=torch.float32, device=dev)
    in_bytes = sum(inp[x].numel() * inp[x].element_size() for x in ("q", "k", "v", "g", "beta"))

    def prefill_step():
        kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                        cu_seqlens=inp["cu_seqlens"], out=out, final_state=fin, stream=stream)

    sampler = ClockSampler(local).start() if rank == 0 else None
    ms, t0, t1 = time_steps(prefill_step, args.steps, args.warmup, world, stream)
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler and clocks.get("samples", 0) < 5:
        # A short timed region holds few samples: the same step, untimed, for about
        # 0.25 s right after it shows the clocks under that load as well.
        tl0 = time.time()
        while time.time() - tl0 < 0.25:
            for _ in range(20):
                prefill_step()
            stream.synchronize()
        clocks["same_load_after"] = {k: v for k, v in sampler.summary(tl0, time.time()).items()
                                     if k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")}
    check_device_status(kda, stream, "prefill_8k")
    value = T * world / (ms * 1e-3)
    achieved = PREFILL_BYTES_PER_TOKEN * T / (ms * 1e-3) / 1e9
    kernel_src = "linear_attention_sequence_gb300/csrc/kda_prefill_tc.cu"
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "peak_source": peak_src,
                "kernel": "kda_prefill_tc_kernel",
                "traffic": profiled_traffic("kda_prefill_tc_kernel", kernel_src, "prefill_8k"),
                "algorithmic_bytes_per_launch": PREFILL_BYTES_PER_TOKEN * T}
    legs = {}
    short = max(3, min(args.steps, 20))

    # ---------------- the same layer through the split kernel (state chain / intra-chunk SMs) ----
    def split_step():
        kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                        cu_seqlens=inp["cu_seqlens"], out=out, final_state=fin,
                        variant=kda.PREFILL_TC_SPLIT, stream=stream)

    ms_sp, _, _ = time_steps(split_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "split")
    legs["split"] = leg_summary(
        ms_sp, T * world, PREFILL_BYTES_PER_TOKEN * T, hbm_gbs, short, "kda_prefill_chain_kernel",
        {"traffic": profiled_traffic("kda_prefill_chain_kernel",
                                     "linear_attention_sequence_gb300/csrc/kda_prefill_chain.cu",
                                     "prefill_8k")})

    # ---------------- the same layer in two passes (intra-chunk products, then the chain) ----
    def two_pass_step():
        kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                        cu_seqlens=inp["cu_seqlens"], out=out, final_state=fin,
                        variant=kda.PREFILL_TC_2PASS, stream=stream)

    ms_tp, _, _ = time_steps(two_pass_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "two_pass")
    # DRAM traffic of both passes: the 8 KB a chunk and head of intra-chunk products
    # is written by the first and read by the second, on top of the algorithmic bytes
    tp_src = "linear_attention_sequence_gb300/csrc/kda_prefill_2pass.cu"
    tp_a = profiled_traffic("kda_intra_kernel", tp_src, "prefill_8k")
    tp_b = profiled_traffic("kda_chain2_kernel", tp_src, "prefill_8k")
    legs["two_pass"] = leg_summary(
        ms_tp, T * world, PREFILL_BYTES_PER_TOKEN * T, hbm_gbs, short,
        "kda_intra_kernel + kda_chain2_kernel",
        {"traffic": tp_a + tp_b if tp_a is not None and tp_b is not None else None})

    # ---------------- the same layer with state checkpoints every 1024 tokens ----------------
    interval = 1024
    ck = torch.empty((kda.checkpoint_count(T, interval, inp["cu_seqlens"]), w.heads, w.d, w.d),
                     dtype=torch.float32, device=dev)

    def checkpointed_step():
        kda.kda_prefill_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     cu_seqlens=inp["cu_seqlens"], interval=interval,
                                     checkpoints=ck, out=out, final_state=fin, stream=stream)

    ms_ck, _, _ = time_steps(checkpointed_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "checkpointed")
    ck_bytes = ck.numel() * ck.element_size()
    legs["checkpointed"] = leg_summary(ms_ck, T * world, PREFILL_BYTES_PER_TOKEN * T + ck_bytes,
                                       hbm_gbs, short, "kda_prefill_tc_kernel")
    del ck

    # ---------------- the same layer through the fused gate prologue ----------------
    gl = synth.gate_logits(T, w.heads, w.d, dtype=w.dtype, seed=81, device=dev)

    def gated_step():
        kda.kda_prefill_gated(inp["q"], inp["k"], inp["v"], gl["z"], gl["a_log"],
                              gl["beta_logit"], cu_seqlens=inp["cu_seqlens"], out=out,
                              final_state=fin, stream=stream)

    ms_gt, _, _ = time_steps(gated_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "gated")
    legs["gated"] = leg_summary(ms_gt, T * world, GATED_BYTES_PER_TOKEN * T, hbm_gbs, short,
                                "kda_prefill_tc_kernel")
    del gl

    # ---------------- the output gate: the entry point, and the unfused pair ----------------
    og = synth.output_gate_inputs(T, w.heads, w.d, dtype=w.dtype, seed=83, device=dev)

    def ogated_step():
        kda.kda_prefill_output_gated(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     og["gate"], og["norm_weight"], 1e-6,
                                     cu_seqlens=inp["cu_seqlens"], out=out, final_state=fin,
                                     stream=stream)

    def ogate_pair_step():
        prefill_step()
        kda.kda_output_gate(out, og["gate"], og["norm_weight"], 1e-6, stream=stream)

    ms_og, _, _ = time_steps(ogated_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "output_gated")
    ms_op, _, _ = time_steps(ogate_pair_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "output_gate_pair")
    legs["output_gated"] = leg_summary(ms_og, T * world, OGATED_BYTES_PER_TOKEN * T, hbm_gbs,
                                       short, "kda_prefill_tc_kernel + kda_output_gate_kernel")
    legs["output_gate_pair"] = leg_summary(
        ms_op, T * world, OGATED_BYTES_PER_TOKEN * T, hbm_gbs, short,
        "kda_prefill then kda_output_gate (two calls)")
    del og

    # ---------------- Gated DeltaNet: one decay per head and step ----------------
    gh = synth.scalar_decay(T, w.heads, seed=85, device=dev)

    def sdecay_step():
        kda.kda_prefill_scalar_decay(inp["q"], inp["k"], inp["v"], gh, inp["beta"],
                                     cu_seqlens=inp["cu_seqlens"], out=out, final_state=fin,
                                     stream=stream)

    ms_sd, _, _ = time_steps(sdecay_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "scalar_decay")
    legs["scalar_decay"] = leg_summary(ms_sd, T * world, SDECAY_BYTES_PER_TOKEN * T, hbm_gbs,
                                       short, "kda_prefill_tc_kernel")
    del gh

    # ---------------- the q, k, v prologue of the same layer ----------------
    pj = synth.qkv_projections(T, w.heads, w.d, dtype=w.dtype, seed=89, device=dev)
    pq, pk, pv = (torch.empty_like(pj["x_q"]) for _ in range(3))

    def prologue_step():
        kda.kda_qkv_prologue(pj["x_q"], pj["x_k"], pj["x_v"], pj["conv_weight"],
                             cu_seqlens=inp["cu_seqlens"], q=pq, k=pk, v=pv,
                             return_conv_state=False, stream=stream)

    ms_pr, _, _ = time_steps(prologue_step, short, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "qkv_prologue")
    pr_bytes = PROLOGUE_BYTES_PER_TOKEN * T + PROLOGUE_WEIGHT_BYTES
    legs["qkv_prologue"] = leg_summary(
        ms_pr, T * world, pr_bytes, hbm_gbs, short, "kda_qkv_prologue_kernel",
        {"traffic": profiled_traffic("kda_qkv_prologue_kernel",
                                     "linear_attention_sequence_gb300/csrc/kda_qkv_prologue.cu",
                                     "prologue_8k")})
    del pj, pq, pk, pv

    # ---------------- the backward pass (gradients of the same layer) ----------------
    gen = torch.Generator(device=dev).manual_seed(87)
    d_out = torch.randn((T, w.heads, w.d), generator=gen, device=dev).to(w.dtype)
    _, _, cstates = kda.kda_prefill_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"],
                                                 inp["beta"], cu_seqlens=inp["cu_seqlens"],
                                                 interval=kda.CHUNK, stream=stream)

    def backward_step():
        kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out,
                         cu_seqlens=inp["cu_seqlens"], chunk_states=cstates, stream=stream)

    bw_steps = 3
    ms_bw, _, _ = time_steps(backward_step, bw_steps, 2, world, stream)
    check_device_status(kda, stream, "backward")
    bw_flops = 2.0 * BWD_MACS_PER_CHUNK_HEAD * ((T + BWD_C - 1) // BWD_C) * w.heads
    sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    fp32_peak = sm_count * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    tf32_peak = bf16_tf * TF32_PER_BF16
    bw_ach = bw_flops / (ms_bw * 1e-3) / 1e12
    legs["backward"] = {"ms": round(ms_bw, 3), "tok_s": round(T * world / (ms_bw * 1e-3)),
                        "bound": "tensor", "tflops": round(bw_ach, 2),
                        "peak_tflops": round(tf32_peak, 1),
                        "peak_source": f"tf32 = {peak_src} bf16 x {TF32_PER_BF16:.3f} (nominal ratio)",
                        "frac": round(bw_ach / tf32_peak, 4),
                        "frac_of_fp32_alu": round(bw_ach / fp32_peak, 4), "steps": bw_steps,
                        "kernel": "kda_backward_tc_kernel"}
    del cstates, d_out

    # ---------------- e2e through the public API, host buffers ----------------
    # A step streams the layer from pinned host memory in E2E_SEGMENTS segments of
    # whole chunks: segment s is copied in on one stream while segment s-1 runs
    # (kda_prefill with init_state = the previous segment's final_state, which the
    # API allows to alias), and each segment's output is copied out on another
    # stream as soon as it is written.  Every input byte, the output and the final
    # state cross the host link inside the timed region.
    host = {x: inp[x].cpu().pin_memory() for x in ("q", "k", "v", "g", "beta")}
    dbuf = {x: torch.empty_like(inp[x]) for x in host}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    fin_h = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    nseg = E2E_SEGMENTS
    seg_len = (T // nseg + kda.CHUNK - 1) // kda.CHUNK * kda.CHUNK
    bounds = [(s0, min(T, s0 + seg_len)) for s0 in range(0, T, seg_len)]

    def e2e_step():
        ev_in = [torch.cuda.Event() for _ in bounds]
        ev_out = [torch.cuda.Event() for _ in bounds]
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        with torch.cuda.stream(h2d_stream):
            for i, (a0, b0) in enumerate(bounds):
                for x in host:
                    dbuf[x][a0:b0].copy_(host[x][a0:b0], non_blocking=True)
                ev_in[i].record(h2d_stream)
        for i, (a0, b0) in enumerate(bounds):
            stream.wait_event(ev_in[i])
            kda.kda_prefill(dbuf["q"][a0:b0], dbuf["k"][a0:b0], dbuf["v"][a0:b0],
                            dbuf["g"][a0:b0], dbuf["beta"][a0:b0],
                            init_state=None if i == 0 else fin, out=out[a0:b0],
                            final_state=fin, stream=stream)
            ev_out[i].record(stream)
            d2h_stream.wait_event(ev_out[i])
            with torch.cuda.stream(d2h_stream):
                out_h[a0:b0].copy_(out[a0:b0], non_blocking=True)
        with torch.cuda.stream(d2h_stream):
            fin_h.copy_(fin, non_blocking=True)
        stream.wait_stream(d2h_stream)
        stream.wait_stream(h2d_stream)

    e2e_steps = short
    ms_e2e, _, _ = time_steps(e2e_step, e2e_steps, max(args.warmup, 3), world, stream)
    check_device_status(kda, stream, "e2e")
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * fin_h.element_size()
    e2e = {"value": T * world / (ms_e2e * 1e-3), "unit": UNIT, "h2d_bytes_per_step": in_bytes,
           "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "pipeline": f"{len(bounds)} segments of {seg_len} tokens, state carried through "
                       "final_state; copies on their own streams, overlapping the kernels"}
    del host, dbuf, out_h, fin_h, inp, out, fin, h2d_stream, d2h_stream
    torch.cuda.empty_cache()

    # ---------------- packed variable-length batch (8 sequences, 1K-32K tokens) ----------------
    wv = synth.WORKLOADS["varlen_8seq"]
    vi = synth.prefill_inputs(wv, dev)
    Tv = wv.total_tokens
    vout = torch.empty((Tv, wv.heads, wv.d), dtype=wv.dtype, device=dev)
    vfin = torch.empty((wv.num_seqs, wv.heads, wv.d, wv.d), dtype=torch.float32, device=dev)

    def varlen_step():
        kda.kda_prefill(vi["q"], vi["k"], vi["v"], vi["g"], vi["beta"],
                        init_state=vi["init_state"], cu_seqlens=vi["cu_seqlens"], out=vout,
                        final_state=vfin, stream=stream)

    v_steps = max(3, min(args.steps, 10))
    ms_v, _, _ = time_steps(varlen_step, v_steps, 3, world, stream)
    check_device_status(kda, stream, "varlen_8seq")
    st_bytes = 2 * vfin.numel() * vfin.element_size()   # initial states read, final written
    legs["varlen_8seq"] = leg_summary(
        ms_v, Tv * world, PREFILL_BYTES_PER_TOKEN * Tv + st_bytes, hbm_gbs, v_steps,
        "kda_prefill_tc_kernel",
        {"tokens": Tv, "longest": max(wv.lengths),
         "longest_seq_ms_at_8k_rate": round(ms * max(wv.lengths) / T, 3)})
    del vi, vout, vfin
    torch.cuda.empty_cache()

    # ---------------- long context: one 262,144-token sequence ----------------
    wl = synth.WORKLOADS["prefill_256k"]
    li = synth.prefill_inputs(wl, dev)
    Tl = wl.total_tokens
    lout = torch.empty((Tl, wl.heads, wl.d), dtype=wl.dtype, device=dev)
    lfin = torch.empty((1, wl.heads, wl.d, wl.d), dtype=torch.float32, device=dev)

    def long_step():
        kda.kda_prefill(li["q"], li["k"], li["v"], li["g"], li["beta"],
                        cu_seqlens=li["cu_seqlens"], out=lout, final_state=lfin, stream=stream)

    l_steps = 3
    ms_l, _, _ = time_steps(long_step, l_steps, 3, world, stream)
    check_device_status(kda, stream, "prefill_256k")
    legs["prefill_256k"] = leg_summary(ms_l, Tl * world, PREFILL_BYTES_PER_TOKEN * Tl, hbm_gbs,
                                       l_steps, "kda_prefill_tc_kernel", {"tokens": Tl})
    del li, lout, lfin
    torch.cuda.empty_cache()

    # ---------------- decode ----------------
    wd = synth.WORKLOADS["decode_256x64"]
    dx = synth.decode_inputs(wd, dev)
    state = dx["state"]
    dout = torch.empty((wd.num_seqs, wd.heads, wd.d), dtype=wd.dtype, device=dev)

    def decode_round():
        for s in range(wd.steps):
            kda.kda_decode(dx["q"][s], dx["k"][s], dx["v"][s], dx["g"][s], dx["beta"][s], state,
                           out=dout, stream=stream)

    # one warm-up round and one timed round of 64 steps: the decode leg is a
    # secondary figure, and the prefill (the headline step) stays the kernel
    # that dominates the run's GPU time
    d_rounds = 1
    ms_round, dt0, dt1 = time_steps(decode_round, d_rounds, 1, world, stream)
    check_device_status(kda, stream, "decode")
    dclocks = sampler.summary(dt0, dt1) if sampler else None
    ms_dstep = ms_round / wd.steps
    d_tokens = wd.num_seqs
    d_bytes = DECODE_BYTES_PER_HEAD_STEP * wd.num_seqs * wd.heads
    d_ach = d_bytes / (ms_dstep * 1e-3) / 1e9
    decode = {"tok_s": round(d_tokens * world / (ms_dstep * 1e-3)), "ms_per_step": round(ms_dstep, 5),
              "frac": round(d_ach / hbm_gbs, 4), "gbs": round(d_ach, 1), "bytes": d_bytes,
              "peak_gbs": hbm_gbs, "steps": wd.steps * d_rounds, "kernel": "kda_decode_kernel",
              "traffic": profiled_traffic("kda_decode_kernel",
                                          "linear_attention_sequence_gb300/csrc/kda_decode.cu",
                                          "decode_256x64"),
              "sm_mhz": (dclocks or {}).get("sm_mhz")}
    if sampler:
        sampler.stop()

    if rank == 0:
        cpu = None if world > 1 else cpu_baseline_prefill()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "tf32", "data": "synthetic",
            "config": {"workload": "prefill_8k: B=1, T=8192, H=96, d_k=d_v=128, bf16 q/k/v/o, "
                                   "fp32 g/beta/state, zero initial state",
                       "l2": f"inputs {in_bytes / 1e9:.2f} GB > L2 {L2_BYTES / 2**20:.0f} MiB; "
                             "no flush between steps",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "sms": sm_count},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": clocks,
            "legs": legs,
            "decode_tokens_per_s": decode["tok_s"], "decode_roofline_frac": decode["frac"],
            "decode": decode,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_profile_case(args, kda, synth, dev, stream):
    """A reduced run for profilers: only one kernel family, a smaller prefill
    (same recipe, --tokens tokens, all 96 heads) or fewer decode sequences;
    W warm-up launches, then K launches.  Prints one short JSON line (not a
    benchmark result)."""
    import torch
    if args.profile == "prefill":
        w = synth.WORKLOADS["prefill_8k"]
        inp = synth.prefill_inputs(w, dev, lengths=(args.tokens,))
        out = torch.empty((args.tokens, w.heads, w.d), dtype=w.dtype, device=dev)
        fin = torch.empty((1, w.heads, w.d, w.d), dtype=torch.float32, device=dev)

        def step():
            kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                            cu_seqlens=inp["cu_seqlens"], out=out, final_state=fin,
                            variant=args.variant, stream=stream)
        units = args.tokens
    elif args.profile == "prologue":
        w = synth.WORKLOADS["prefill_8k"]
        pj = synth.qkv_projections(args.tokens, w.heads, w.d, dtype=w.dtype, seed=89, device=dev)

        def step():
            kda.kda_qkv_prologue(pj["x_q"], pj["x_k"], pj["x_v"], pj["conv_weight"],
                                 return_conv_state=False, stream=stream)
        units = args.tokens
    elif args.profile == "backward":
        w = synth.WORKLOADS["prefill_8k"]
        inp = synth.prefill_inputs(w, dev, lengths=(args.tokens,))
        gen = torch.Generator(device=dev).manual_seed(87)
        d_out = torch.randn((args.tokens, w.heads, w.d), generator=gen, device=dev).to(w.dtype)
        _, _, cstates = kda.kda_prefill_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"],
                                                     inp["beta"], cu_seqlens=inp["cu_seqlens"],
                                                     interval=kda.CHUNK, stream=stream)

        def step():
            kda.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], d_out,
                             cu_seqlens=inp["cu_seqlens"], chunk_states=cstates, stream=stream)
        units = args.tokens
    else:
        wd = synth.WORKLOADS["decode_256x64"]
        dx = synth.decode_inputs(wd, dev, num_seqs=args.seqs, steps=1)
        state = dx["state"]
        dout = torch.empty((args.seqs, wd.heads, wd.d), dtype=wd.dtype, device=dev)

        def step():
            kda.kda_decode(dx["q"][0], dx["k"][0], dx["v"][0], dx["g"][0], dx["beta"][0], state,
                           out=dout, stream=stream)
        units = args.seqs
    ms, _, _ = time_steps(step, args.steps, args.warmup, 1, stream)
    print(json.dumps({"profile_case": args.profile, "units": units, "ms_per_launch": ms,
                      "note": "profiling run, not a benchmark result"}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--profile", choices=["prefill", "decode", "backward", "prologue"],
                    default=None,
                    help="run only one kernel family on a reduced case (for ncu)")
    ap.add_argument("--tokens", type=int, default=2048, help="--profile prefill: tokens")
    ap.add_argument("--seqs", type=int, default=64, help="--profile decode: sequences")
    ap.add_argument("--variant", type=int, default=0, help="prefill kernel variant (0 default)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
