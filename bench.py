#!/usr/bin/env python3
"""Benchmark of the LoRA MoE expert layer on GB300.

One step = one batch through the whole hot path: moe_lora_batch_info (once per
batch) and fused_moe_lora_forward (align, LoRA shrinks, gate_up GEMM with the
fused LoRA expand and SiLU*up, down GEMM with the fused LoRA expand and the
top-k combine).  Inputs are seeded synthetic tensors resident in HBM.  The
headline workload is the DeepSeek-V3-like prefill (8192 tokens, hidden 7168,
intermediate 2048, 256 experts top-8, 4 LoRA slots ranks {16,32,64,64}, 22.5 GB
of bf16 expert weights), the largest of the layer's workloads.  Each step
streams far more than the 129 MB L2, so no explicit L2 flush is done between
steps.  The Qwen-MoE-like prefill, decode and the metadata-only stress batch
(batch_info + align on 1,048,576 tokens, inputs rotated over four copies so
that they do not sit in L2) are measured in the same run, each with its own
roofline fractions, under "workloads".

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded token sample of the same workload instead.
Multi-GPU (torchrun): each rank runs its own batch (data-parallel replicas,
no collective on the data path); value = all ranks' tokens / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-LoRA layer tokens/s and % of roofline (bf16, 1×GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Tensor peak for the fractions: the burst figure.  Every timed region here is
# at most a few seconds of back-to-back steps, and the burst peak is the
# stricter (larger) denominator.
PEAK_KIND = "bf16_tflops"
DEFAULT_EXTRAS = "qwen_moe_prefill,decode,metadata_stress"
COMBINE_NAME = {False: "atomic (fp32 reductions)", True: "deterministic (per-pair rows, summed in k order)"}
METADATA_METRIC = "MoE-LoRA metadata (batch_info + align) tokens/s and % of HBM roofline (int32, 1×GB300)"
STAGE_KERNELS = {"gate_up": "moe_gemm_kernel<1>", "down": "moe_gemm_kernel<3>",
                 "shrink_gate_up": "moe_gemm_kernel<0>", "shrink_down": "moe_gemm_kernel<2>"}


# ----------------------------------------------------------------- helpers --
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of the translation unit that holds the GEMM kernels (forward.cu and
    the headers); a recorded DRAM capture applies only while it is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lora_moe_expert_info_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name == "forward.cu" or name.endswith(".cuh"):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(stage: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for r in rec.get("captures", []):
        if r.get("stage") == stage and r.get("workload") == workload and \
                r.get("source_hash") == kernel_source_hash():
            return r.get("dram_bytes_per_launch")
    return None


def stage_profile(lib, step, n_calls):
    """Average ms per stage over n_calls untimed steps, every stage marked."""
    import torch
    lib.moe_lora_profile_stages(all_stages(lib))
    lib.moe_lora_profile_begin(n_calls)
    for _ in range(n_calls):
        step()
    torch.cuda.synchronize()
    return read_stage_profile(lib)


def read_stage_profile(lib):
    """End the library's recording; average ms per stage over the recorded calls."""
    import ctypes
    stage_ms = (ctypes.c_double * 16)()
    n_st, n_calls = ctypes.c_int32(0), ctypes.c_int32(0)
    lib.moe_lora_profile_end(stage_ms, 16, ctypes.byref(n_st), ctypes.byref(n_calls))
    return {lib.moe_lora_profile_stage_name(i).decode(): stage_ms[i] / max(1, n_calls.value)
            for i in range(n_st.value)}


def all_stages(lib):
    n = 0
    while lib.moe_lora_profile_stage_name(n) is not None:
        n += 1
    return (1 << n) - 1


def stage_index(lib, name):
    i = 0
    while True:
        n = lib.moe_lora_profile_stage_name(i)
        if n is None:
            raise KeyError(name)
        if n.decode() == name:
            return i
        i += 1


def capture_steps(step, n, stream):
    """A CUDA graph of n steps, captured on a side stream: replaying it runs the
    same launches (same kernels, same arguments) without the host's per-launch
    cost.  One warm replay uploads it."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.graph(g, stream=side):
        for _ in range(n):
            step()
    stream.wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    return g


def timed_region(lib, args, step, stream, dist, local, dom):
    """The timed steps: barrier and synchronise on both sides, CUDA events on the
    launching stream, clocks sampled throughout.  Only the two events that bound
    stage `dom` are recorded inside the forward, so its launch time is measured
    live at the cost of two events per step instead of eight.

    Returns (ms over all steps, dom's average ms, kernels launched, clock sampler).
    """
    import torch
    lib.moe_lora_profile_stages(1 << stage_index(lib, dom))
    if dist is not None:
        dist.barrier()
    n_launch0 = lib.moe_lora_launch_count()
    lib.moe_lora_profile_begin(min(args.steps, 4096))
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
    live = read_stage_profile(lib)
    lib.moe_lora_profile_stages(all_stages(lib))
    n_launch = lib.moe_lora_launch_count() - n_launch0
    return e0.elapsed_time(e1), live[dom], n_launch, clk


def graph_region(args, step, stream, dist):
    """The same steps as one CUDA graph replay (captured after the eager timed
    region, no profiling events inside): ms over all steps, barriers and
    synchronisation on both sides, CUDA events on the stream."""
    import torch
    g = capture_steps(step, args.steps, stream)
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1)


def pipelined_e2e(n_steps, upload, compute, download, stream):
    """Milliseconds per step with two steps in flight, as a serving loop runs.

    Step i uploads its inputs into buffer slot i % 2 on an upload stream, runs on
    `stream` (the library's launch stream), and its result is read back on a
    download stream.  Slot reuse is ordered by events: step i's upload waits for
    step i - 2's compute (which read the slot's inputs), and its compute waits
    for step i - 2's download (which read the slot's result).  So step i + 1's
    upload and step i - 1's download overlap step i's compute, while every step
    still copies its own inputs in and its own result out.  Timed from the
    first upload to the last download with CUDA events.
    """
    import torch
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    f0.record(s_in)
    for i in range(n_steps):
        sl = i % 2
        if i >= 2:
            s_in.wait_event(done[sl])
        with torch.cuda.stream(s_in):
            upload(sl)
        ready[sl].record(s_in)
        stream.wait_event(ready[sl])
        if i >= 2:
            stream.wait_event(read[sl])
        with torch.cuda.stream(stream):
            compute(sl)
        done[sl].record(stream)
        s_out.wait_event(done[sl])
        with torch.cuda.stream(s_out):
            download(sl)
        read[sl].record(s_out)
    f1.record(s_out)  # every earlier step precedes the last download
    torch.cuda.synchronize()
    return f0.elapsed_time(f1) / n_steps


def measure_e2e(args, upload, compute, download, stream, dist, dev):
    """End-to-end ms per step: two steps in flight (the reported figure), and
    one step at a time on one stream (reported beside it).  Max over ranks."""
    import torch
    n = max(3, min(args.steps, 200))

    def serial_step():
        with torch.cuda.stream(stream):
            upload(0)
            compute(0)
            download(0)

    for _ in range(3):
        serial_step()
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(n):
        serial_step()
    f1.record(stream)
    torch.cuda.synchronize()
    serial = f0.elapsed_time(f1) / n
    pipelined_e2e(4, upload, compute, download, stream)  # warm-up of the streams and events
    piped = pipelined_e2e(n, upload, compute, download, stream)
    return reduce_max(piped, dist, dev), reduce_max(serial, dist, dev)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "50"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


def reduce_max(value, dist, device):
    """The largest of a per-rank float over all ranks (the slowest rank sets the time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_rate(units_per_rank, world, ms_per_step_max):
    """Whole-job throughput: every rank processes units_per_rank per step, timed by the slowest."""
    return world * units_per_rank / (ms_per_step_max * 1e-3)


def layer_work(cfg, batch, mapping, fp8=False, fmt=None):
    """Algorithmic FLOPs and bytes of the layer and of each stage (from the routing).

    fmt (or fp8=True for "fp8"): the base expert weights' format.  "fp8" and
    "int8": one byte per weight plus a float32 scale per 128 x 128 block;
    "w4a16": half a byte per weight plus a float32 scale and a one-byte zero
    point per row and 128-column group; "w8a8": one byte per weight plus a
    one-byte exponent per 128 x 128 block.  LoRA operands and the layer's
    input and output stay bf16 (the quantised activation copies are
    implementation traffic, not counted).
    """
    fmt = fmt or ("fp8" if fp8 else "bf16")
    import torch
    T, K, E, H, I, L = cfg.num_tokens, cfg.topk, cfg.num_experts, cfg.hidden, cfg.intermediate, cfg.num_loras
    ids = batch.topk_ids.long().cpu()
    mp = mapping.long().cpu()
    ranks = batch.lora_ranks.long().cpu()
    P = T * K
    touched_e = torch.unique(ids).numel()
    tok_r = torch.where(mp >= 0, ranks[mp.clamp_min(0)], torch.zeros_like(mp))
    pair_r = tok_r.repeat_interleave(K)
    sum_r_pairs = float(pair_r.sum())
    pair_l = mp.repeat_interleave(K)
    sel = pair_r > 0
    keys = torch.unique(pair_l[sel] * E + ids.reshape(-1)[sel])
    sum_r_le = float(ranks[keys // E].sum()) if keys.numel() else 0.0
    W = 2  # bf16 bytes
    nb = lambda n: (n + 127) // 128  # noqa: E731
    # base expert bytes per touched expert: gate_up and down matrices
    if fmt in ("fp8", "int8"):
        wgu = 2 * H * I + 4 * nb(2 * I) * nb(H)
        wdn = H * I + 4 * nb(H) * nb(I)
    elif fmt == "w8a8":
        wgu = 2 * H * I + nb(2 * I) * nb(H)
        wdn = H * I + nb(H) * nb(I)
    elif fmt == "w4a16":
        wgu = H * I + 5 * 2 * I * nb(H)
        wdn = H * I // 2 + 5 * H * nb(I)
    else:
        wgu, wdn = 2 * H * I * W, H * I * W
    st = {
        "shrink_gate_up": (4 * H * sum_r_pairs, 2 * H * sum_r_le * W + T * H * W),
        "gate_up": (4 * H * I * P + 4 * I * sum_r_pairs, wgu * touched_e + 2 * I * sum_r_le * W + T * H * W),
        "shrink_down": (2 * I * sum_r_pairs, I * sum_r_le * W),
        "down": (2 * H * I * P + 2 * H * sum_r_pairs, wdn * touched_e + H * sum_r_le * W + T * H * W + P * 4),
    }
    flops = 6 * H * I * P + 6 * (H + I) * sum_r_pairs
    byts = (wgu + wdn) * touched_e + (3 * H + 3 * I) * sum_r_le * W + 2 * T * H * W + P * 8 + T * 4
    return flops, byts, st


def roofline_entry(flops, byts, ms, peaks, peak_kind):
    t_f = flops / (peaks[peak_kind] * 1e12)
    t_b = byts / (peaks["hbm_gbs"] * 1e9)
    s = ms * 1e-3
    if t_b >= t_f:
        ach = byts / s / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4)}
    ach = flops / s / 1e12
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": peaks[peak_kind], "unit": "TFLOP/s",
            "frac": round(ach / peaks[peak_kind], 4)}


# ------------------------------------------------------------ the two arms --
def make_inputs(cfg_name, device, seed, fmt="bf16"):
    """Batch, bf16 weights and x; for a quantised format also its experts (else None)."""
    from lora_moe_expert_info_gb300 import workloads
    cfg = workloads.CONFIGS[cfg_name]
    b = workloads.make_batch(cfg, device=device, seed=seed)
    w = workloads.make_weights(cfg, b.lora_ranks, device=device, seed=seed)
    x = workloads.make_x(cfg, device=device, seed=seed)
    make = {"fp8": workloads.make_fp8_experts, "int8": workloads.make_int8_experts,
            "w4a16": workloads.make_w4a16_experts, "w8a8": workloads.make_fp8_w8a8_experts}.get(fmt)
    q = make(cfg, device=device, seed=seed) if make else None
    return cfg, b, w, x, q


QUANT_KEYS = {"fp8": ("w_gate_up_q", "w_gate_up_scale", "w_down_q", "w_down_scale"),
              "int8": ("w_gate_up_q", "w_gate_up_scale", "w_down_q", "w_down_scale"),
              "w4a16": ("w_gate_up_q", "w_gate_up_scale", "w_gate_up_zero", "w_down_q", "w_down_scale",
                        "w_down_zero"),
              "w8a8": ("w_gate_up_q", "w_gate_up_exp", "w_down_q", "w_down_exp")}
# The FP8 tensor cores' dense peak: the measured bf16 peak times the nominal
# FP8 / bf16 ratio (4.5 / 2.25 PFLOP/s).
FP8_OVER_BF16 = 2.0


def peak_kind_of(fmt):
    """The tensor peak a format's base GEMMs run against."""
    return "fp8_tflops" if fmt == "w8a8" else PEAK_KIND


def oracle_sample_rate(cfg, b, w, x, mapping_np, target_s=10.0, max_tokens=None, seed=0, q=None, fmt="bf16"):
    """Oracle tokens/s on a bounded seeded token sample; returns (rate, n_tokens, secs, threads).
    With q (quantised experts of format fmt) the oracle's matching forward runs."""
    import numpy as np
    import torch

    import oracle
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    lora = [bits(getattr(w, k)) for k in ("lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")]
    if q is None:
        fwd = oracle.forward
        host = [bits(w.w_gate_up), bits(w.w_down)] + lora
    else:
        fwd = {"fp8": oracle.forward_fp8, "int8": oracle.forward_int8, "w4a16": oracle.forward_w4a16,
               "w8a8": oracle.forward_fp8_w8a8}[fmt]
        host = [getattr(q, k).cpu().numpy() for k in QUANT_KEYS[fmt]] + lora
    xb = bits(x)
    ids = b.topk_ids.cpu().numpy()
    wts = b.topk_weights.cpu().numpy()
    ranks = b.lora_ranks.cpu().numpy()
    scal = b.scalings.cpu().numpy()
    rng = np.random.default_rng(seed)
    T = cfg.num_tokens
    # calibrate on a few tokens, then size the sample to ~target_s of CPU work
    n0 = min(T, 8)
    t0 = time.perf_counter()
    fwd(xb, ids, wts, mapping_np, ranks, scal, *host, tokens=rng.choice(T, n0, replace=False))
    per_tok = (time.perf_counter() - t0) / n0
    n = int(max(n0, min(T, target_s / max(per_tok, 1e-9))))
    if max_tokens:
        n = min(n, max_tokens)
    toks = np.sort(rng.choice(T, n, replace=False))
    t0 = time.perf_counter()
    st, _ = fwd(xb, ids, wts, mapping_np, ranks, scal, *host, tokens=toks)
    secs = time.perf_counter() - t0
    assert st == 0
    return n / secs, n, secs, oracle.max_threads()


def run_reference(args, rank, world):
    """The oracle as it stands, timed on host cores (rank 0 only)."""
    import numpy as np
    import torch

    import oracle
    if rank != 0:
        return None
    oracle.build()
    dev = "cpu"
    fmt = args.weights
    cfg, b, w, x, q = make_inputs(args.config, dev, args.seed, fmt)
    st, mp, _ = oracle.batch_info(b.seg_indptr.numpy(), b.weight_indices.numpy(), b.lora_ranks.numpy(),
                                  cfg.num_tokens)
    # each step a bounded sample: the whole run takes about 90 s of oracle time
    per_step_target = max(0.25, 90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_rate(cfg, b, w, x, mp, target_s=per_step_target, max_tokens=args.ref_tokens, q=q, fmt=fmt)
    rates, ns, secs = [], 0, 0.0
    thr = 1
    for i in range(args.steps):
        r, n, s, thr = oracle_sample_rate(cfg, b, w, x, mp, target_s=per_step_target,
                                          max_tokens=args.ref_tokens, seed=i, q=q, fmt=fmt)
        rates.append(r)
        ns += n
        secs += s
    value = ns / secs
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "tokens": cfg.num_tokens, "hidden": cfg.hidden,
                       "intermediate": cfg.intermediate, "experts": cfg.num_experts, "topk": cfg.topk,
                       "loras": cfg.num_loras, "max_rank": cfg.max_rank, "seed": args.seed,
                       "weights": WEIGHT_LABEL[args.weights]},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                             "sample": f"{ns} tokens over {args.steps} steps (seeded samples of the "
                                       f"{cfg.num_tokens}-token batch), fp64 C oracle, OpenMP over tokens"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


def measure_moe(name, args, rank, world, dist, lib, with_e2e, with_cpu):
    """One MoE workload: the timed steps, the live-timed dominant stage, the
    stage breakdown, and optionally the end-to-end loop and the oracle's rate.
    Returns the workload's entry (rank 0) or None (other ranks)."""
    import torch

    import lora_moe_expert_info_gb300 as mlr

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    fmt = args.weights
    cfg, b, w, x, q = make_inputs(name, dev, args.seed + rank, fmt)
    T, K, E, H, I, L, R = (cfg.num_tokens, cfg.topk, cfg.num_experts, cfg.hidden, cfg.intermediate,
                           cfg.num_loras, cfg.max_rank)
    max_len = int(b.seg_lens.max())
    enabled = torch.empty(L, dtype=torch.int32, device=dev)
    mapping = torch.empty(T, dtype=torch.int32, device=dev)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    wsb = (mlr.fused_moe_lora_workspace_bytes_fp8_w8a8 if fmt == "w8a8" else mlr.fused_moe_lora_workspace_bytes)
    ws = torch.empty(wsb(T, K, E, H, I, L, R), dtype=torch.uint8, device=dev)
    lk = {k: getattr(w, k) for k in ("lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")}
    if q is not None:
        forward = {"fp8": mlr.fused_moe_lora_forward_fp8, "int8": mlr.fused_moe_lora_forward_int8,
                   "w4a16": mlr.fused_moe_lora_forward_w4a16,
                   "w8a8": mlr.fused_moe_lora_forward_fp8_w8a8}[fmt]
        wk = dict({k: getattr(q, k) for k in QUANT_KEYS[fmt]}, **lk)
    else:
        forward = mlr.fused_moe_lora_forward
        wk = dict(w_gate_up=w.w_gate_up, w_down=w.w_down, **lk)

    def step():
        mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, T, max_len,
                                adapter_enabled=enabled, token_lora_mapping=mapping, check=False)
        forward(x, b.topk_ids, b.topk_weights, mapping, b.lora_ranks, b.scalings, **wk, y=y, workspace=ws,
                check=False)

    # correctness gate before timing: the status word of a checked call
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, T, max_len,
                            adapter_enabled=enabled, token_lora_mapping=mapping)
    forward(x, b.topk_ids, b.topk_weights, mapping, b.lora_ranks, b.scalings, **wk, y=y, workspace=ws,
            status=status)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    # per-stage breakdown from untimed steps; the dominant GEMM stage is then
    # timed live inside the timed region
    stages = stage_profile(lib, step, max(3, min(args.steps, 50)))
    dom = max((s for s in STAGE_KERNELS if s in stages), key=lambda s: stages[s])
    ms_total, dom_ms, n_launch, clk = timed_region(lib, args, step, stream, dist, local, dom)
    ms_max = reduce_max(ms_total, dist, dev)
    graph_ms = reduce_max(graph_region(args, step, stream, dist), dist, dev) / args.steps if args.graph else None
    # the other top-k combine, timed the same way (events around the steps)
    mode = mlr.deterministic()
    mlr.set_deterministic(not mode)
    try:
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(args.steps):
            step()
        a1.record(stream)
        torch.cuda.synchronize()
        alt_ms = reduce_max(a0.elapsed_time(a1), dist, dev) / args.steps
    finally:
        mlr.set_deterministic(mode)
    combine = {"mode": COMBINE_NAME[mode], "alternative": {"mode": COMBINE_NAME[not mode],
                                                           "ms_per_step": round(alt_ms, 4)}}

    e2e = None
    if with_e2e:
        # end to end through the public API from pinned host buffers
        host_in = {"x": x.cpu().pin_memory(), "topk_ids": b.topk_ids.cpu().pin_memory(),
                   "topk_weights": b.topk_weights.cpu().pin_memory(),
                   "seg_indptr": b.seg_indptr.cpu().pin_memory(),
                   "weight_indices": b.weight_indices.cpu().pin_memory(),
                   "lora_ranks": b.lora_ranks.cpu().pin_memory(), "scalings": b.scalings.cpu().pin_memory()}
        dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()} for _ in range(2)]
        y_dev = [y, torch.empty_like(y)]
        y_host = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = y_host[0].numel() * y_host[0].element_size()

        def upload(sl):
            for k, v in host_in.items():
                dev_in[sl][k].copy_(v, non_blocking=True)

        def compute(sl):
            d = dev_in[sl]
            mlr.moe_lora_batch_info(d["seg_indptr"], d["weight_indices"], d["lora_ranks"], T,
                                    max_len, adapter_enabled=enabled, token_lora_mapping=mapping, check=False)
            forward(d["x"], d["topk_ids"], d["topk_weights"], mapping, d["lora_ranks"], d["scalings"], **wk,
                    y=y_dev[sl], workspace=ws, check=False)

        def download(sl):
            y_host[sl].copy_(y_dev[sl], non_blocking=True)

        e2e_ms, e2e_serial_ms = measure_e2e(args, upload, compute, download, stream, dist, dev)
        e2e = {"value": round(weak_scaling_rate(T, world, e2e_ms), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_ms, 4), "steps_in_flight": 2,
               "serial_ms_per_step": round(e2e_serial_ms, 4)}

    # check the status of the gated call only now (it synchronised long ago)
    if int(status.item()) != 0:
        raise RuntimeError(f"{name}: forward reported device status {int(status.item())}")
    if rank != 0:
        return None

    mp_np = mapping.cpu().numpy()
    flops, byts, st_work = layer_work(cfg, b, mapping, fmt=fmt)
    cpu = None
    if with_cpu:
        import oracle
        oracle.build()
        rate, n, secs, thr = oracle_sample_rate(cfg, b, w, x, mp_np, target_s=args.cpu_seconds, q=q, fmt=fmt)
        cpu = {"value": round(rate, 3), "unit": "tokens/s", "cores": thr, "kind": "oracle",
               "sample": f"{n} seeded tokens of the {T}-token batch ({secs:.1f} s), fp64 C oracle, "
                         f"OpenMP over tokens"}

    peaks, peak_src = load_peaks()
    peaks["fp8_tflops"] = peaks[PEAK_KIND] * FP8_OVER_BF16
    pk = peak_kind_of(fmt)
    ms_step = ms_max / args.steps
    rf = roofline_entry(st_work[dom][0], st_work[dom][1], dom_ms, peaks, pk)
    rf["kernel"] = STAGE_KERNELS.get(dom, dom)
    rf["stage"] = dom
    rf["peak_source"] = peak_label(peak_src, pk)
    rf["traffic"] = recorded_traffic(dom, cfg.name + ("" if fmt == "bf16" else "_" + fmt))
    rf["algorithmic_bytes"] = int(st_work[dom][1])
    rf["algorithmic_flops"] = int(st_work[dom][0])
    rf["launch_ms"] = round(dom_ms, 4)
    layer = layer_fractions(flops, byts, ms_step, peaks, pk)
    entry = {"value": round(weak_scaling_rate(T, world, ms_step), 1), "unit": "tokens/s",
             "ms_per_step": round(ms_step, 4),
             "config": {"workload": cfg.name, "tokens": T, "hidden": H, "intermediate": I, "experts": E,
                        "topk": K, "loras": L, "max_rank": R, "seed": args.seed,
                        "weights": WEIGHT_LABEL[args.weights],
                        "l2": f"no flush: each step streams {byts / 1e9:.2f} GB of algorithmic bytes "
                              f"(> 129 MB L2)"},
             "roofline": rf, "layer_roofline": layer,
             "graph": None if graph_ms is None else {
                 "ms_per_step": round(graph_ms, 4), "value": round(weak_scaling_rate(T, world, graph_ms), 1),
                 "note": "the same steps as one CUDA graph replay (captured after the timed region)"},
             "stages_ms": {k: round(v, 4) for k, v in stages.items()},
             "combine": combine,
             "gpu_launches": int(n_launch), "clocks": clk.summary()}
    if cpu is not None:
        entry["cpu_baseline"] = cpu
    if e2e is not None:
        entry["e2e"] = e2e
    return entry


def layer_fractions(flops, byts, ms_step, peaks, peak_kind=PEAK_KIND):
    """The layer's roofline entry with both fractions: HBM (bytes) and the
    dense tensor peak of the base GEMMs' type (FLOPs), the latter being the
    prefill bar."""
    layer = roofline_entry(flops, byts, ms_step, peaks, peak_kind)
    s = ms_step * 1e-3
    layer["hbm_frac"] = round(byts / s / 1e9 / peaks["hbm_gbs"], 4)
    layer["tensor_frac"] = round(flops / s / 1e12 / peaks[peak_kind], 4)
    layer["roofline_ms"] = round(1e3 * max(byts / (peaks["hbm_gbs"] * 1e9),
                                           flops / (peaks[peak_kind] * 1e12)), 4)
    layer["algorithmic_bytes"] = int(byts)
    layer["algorithmic_flops"] = int(flops)
    return layer


def peak_label(src, kind=PEAK_KIND):
    base = f"{src} {PEAK_KIND} (MEASURED_PEAKS.json)" if src == "measured" else f"fallback {PEAK_KIND}"
    return base if kind == PEAK_KIND else f"{base} x {FP8_OVER_BF16:g} (nominal FP8 / bf16 ratio)"


def metadata_bytes(bs, L, T, P, npad, block_size):
    """Algorithmic bytes of the metadata calls: batch_info reads seg_indptr,
    weight_indices and lora_ranks and writes the mapping and the enabled mask;
    align reads topk_ids and the mapping and writes the padded sorted ids, the
    two block label arrays and the padded count."""
    bi = 4 * (2 * bs + 1 + 2 * L + T)
    al = 4 * (P + T) + 4 * (npad + 2 * (npad // block_size) + 1)
    return bi, al


def measure_metadata(args, rank, world, dist, n_copies=4):
    """The metadata-only stress workload: moe_lora_batch_info + moe_lora_align
    on 1,048,576 tokens.  Its inputs and outputs (about 80 MB per step) would
    sit in the 129 MB L2, so every step uses the next of n_copies copies of
    them (rotated, about 320 MB in all)."""
    import torch

    import lora_moe_expert_info_gb300 as mlr
    from lora_moe_expert_info_gb300 import workloads
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    cfg = workloads.CONFIGS["metadata_stress"]
    T, K, E, L, bsz = cfg.num_tokens, cfg.topk, cfg.num_experts, cfg.num_loras, cfg.block_size
    b = workloads.make_batch(cfg, device=dev, seed=args.seed + rank)
    bs = b.weight_indices.numel()
    P = T * K
    cap = mlr.moe_lora_align_capacity(T, K, E, L, bsz)
    nblk = cap // bsz
    ws = torch.empty(max(256, mlr.moe_lora_align_workspace_bytes(T, K, E, L, bsz)), dtype=torch.uint8,
                     device=dev)
    copies = []
    for _ in range(n_copies):
        copies.append({
            "indptr": b.seg_indptr.clone(), "wi": b.weight_indices.clone(), "ranks": b.lora_ranks.clone(),
            "ids": b.topk_ids.clone(), "mapping": torch.empty(T, dtype=torch.int32, device=dev),
            "enabled": torch.empty(L, dtype=torch.int32, device=dev),
            "out": (torch.empty(cap, dtype=torch.int32, device=dev),
                    torch.empty(nblk, dtype=torch.int32, device=dev),
                    torch.empty(nblk, dtype=torch.int32, device=dev),
                    torch.empty(1, dtype=torch.int32, device=dev))})

    # The timed calls go straight through the C ABI with their pointer
    # arguments prepared once, so that the host's per-call cost stays below the
    # kernels' time (the checked wrapper calls above validated every buffer).
    import ctypes
    lib = mlr.library()
    vp = ctypes.c_void_p
    sp = vp(torch.cuda.current_stream().cuda_stream)
    for c in copies:
        o = c["out"]
        c["bi_args"] = (vp(c["indptr"].data_ptr()), vp(c["wi"].data_ptr()), vp(c["ranks"].data_ptr()), bs, L, T, 0,
                        vp(c["mapping"].data_ptr()), vp(c["enabled"].data_ptr()), None, sp)
        c["al_args"] = (vp(c["ids"].data_ptr()), vp(c["mapping"].data_ptr()), T, K, E, L, bsz, vp(o[0].data_ptr()),
                        vp(o[1].data_ptr()), vp(o[2].data_ptr()), vp(o[3].data_ptr()), cap, vp(ws.data_ptr()),
                        ws.numel(), None, sp)

    def batch_info(c):
        if lib.moe_lora_batch_info(*c["bi_args"]) != 0:
            raise RuntimeError("moe_lora_batch_info failed")

    def align(c):
        if lib.moe_lora_align(*c["al_args"]) != 0:
            raise RuntimeError("moe_lora_align failed")

    # checked calls first (status words), then warm-up
    for c in copies:
        mlr.moe_lora_batch_info(c["indptr"], c["wi"], c["ranks"], T, 0, adapter_enabled=c["enabled"],
                                token_lora_mapping=c["mapping"])
        mlr.moe_lora_align(c["ids"], c["mapping"], E, L, bsz, out=c["out"], workspace=ws)
    npad = int(copies[0]["out"][3].item())
    stream = torch.cuda.current_stream()
    n = max(4 * n_copies, args.steps)

    def timed(fn):
        for i in range(max(3, args.warmup)):
            fn(copies[i % n_copies])
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            fn(copies[i % n_copies])
        e1.record(stream)
        torch.cuda.synchronize()
        return reduce_max(e0.elapsed_time(e1) / n, dist, dev)

    with ClockSampler(local) as clk:
        ms_bi = timed(batch_info)
        ms_al = timed(align)
        l0 = mlr.library().moe_lora_launch_count()
        ms_step = timed(lambda c: (batch_info(c), align(c)))
        launches_per_step = (mlr.library().moe_lora_launch_count() - l0) // (n + max(3, args.warmup))
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    bi_bytes, al_bytes = metadata_bytes(bs, L, T, P, npad, bsz)

    def rl(byts, ms):
        ach = byts / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "algorithmic_bytes": int(byts),
                "launch_ms": round(ms, 5), "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)"}

    return {"value": round(weak_scaling_rate(T, world, ms_step), 1), "unit": "tokens/s",
            "ms_per_step": round(ms_step, 5),
            "config": {"workload": cfg.name, "tokens": T, "segments": bs, "experts": E, "topk": K, "loras": L,
                       "block_size": bsz, "pairs": P, "num_tokens_post_pad": npad, "seed": args.seed,
                       "l2": f"{n_copies} rotated copies of every input and output "
                             f"({n_copies * (bi_bytes + al_bytes) / 1e6:.0f} MB > 129 MB L2)"},
            "roofline": dict(rl(bi_bytes + al_bytes, ms_step), kernel="batch_info + align (one step)"),
            "calls": {"moe_lora_batch_info": rl(bi_bytes, ms_bi), "moe_lora_align": rl(al_bytes, ms_al)},
            "gpu_launches_per_step": int(launches_per_step), "clocks": clk.summary()}


def run_ours(args, rank, world, dist):
    """The headline workload (its JSON line), with the other workloads of the
    same north-star table measured in the same run under "workloads"."""
    import torch

    import lora_moe_expert_info_gb300 as mlr

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(torch.device("cuda", local))
    lib = mlr.library()
    mlr.set_deterministic(args.combine == "deterministic")
    if args.config == "metadata_stress":
        head = measure_metadata(args, rank, world, dist)
        if rank != 0:
            return None
        return {"metric": METADATA_METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
                "data": "synthetic", "config": head["config"], "roofline": head["roofline"],
                "calls": head["calls"], "cpu_baseline": None, "e2e": None,
                "gpu_launches": head["gpu_launches_per_step"] * max(4 * 4, args.steps),
                "clocks": head["clocks"]}
    head = measure_moe(args.config, args, rank, world, dist, lib, with_e2e=True,
                       with_cpu=not args.no_cpu_baseline)
    extras = {}
    for name in [n for n in args.extras.split(",") if n and n != args.config]:
        torch.cuda.empty_cache()
        if name == "metadata_stress":
            extras[name] = measure_metadata(args, rank, world, dist)
        else:
            extras[name] = measure_moe(name, args, rank, world, dist, lib, with_e2e=False, with_cpu=False)
    if rank != 0:
        return None
    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8" if args.weights == "w8a8" else "bf16",
            "data": "synthetic",
            "config": dict(head["config"],
                           parallelism=f"dp{world} (replicas)" if world > 1 else "single GPU"),
            "roofline": head["roofline"], "layer_roofline": head["layer_roofline"], "graph": head["graph"],
            "stages_ms": head["stages_ms"], "combine": head["combine"], "cpu_baseline": head.get("cpu_baseline"),
            "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "clocks": head["clocks"]}
    if extras:
        line["workloads"] = extras
    return line


# --------------------------------------- dense projection with split-B LoRA --
# The MLA fused q_a_proj + kv_a_proj projection of a DeepSeek-V3-like prefill
# batch: hidden 7168 -> 1536 + 576 output rows in two parts, 4 adapter slots.
LINEAR_CONFIGS = {
    "mla_fused_proj": {"tokens": 8192, "in": 7168, "offsets": (0, 1536, 2112), "loras": 4, "max_rank": 64,
                       "ranks": (16, 32, 64, 64), "segments": 8},
}
WEIGHT_LABEL = {"bf16": "bf16", "fp8": "fp8 e4m3, fp32 scale per 128x128 block (bf16 LoRA)",
                "int8": "int8, fp32 scale per 128x128 block (bf16 LoRA)",
                "w4a16": "uint4 two per byte, fp32 scale and uint8 zero point per row and 128 columns (bf16 LoRA)",
                "w8a8": "fp8 e4m3 weights and activations on the FP8 tensor cores, power-of-two scales per "
                        "128x128 weight block and per token and 128 channels (bf16 LoRA)"}
LINEAR_METRIC = "MLA fused-projection LoRA tokens/s and % of roofline (bf16, 1×GB300)"


def make_linear_inputs(cfg, device, seed):
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    gc = torch.Generator().manual_seed(seed)
    T, D_in, offs, L, R = cfg["tokens"], cfg["in"], cfg["offsets"], cfg["loras"], cfg["max_rank"]
    D_out, S = offs[-1], len(offs) - 1
    bf = torch.bfloat16
    x = torch.randn(T, D_in, generator=g, device=device, dtype=bf)
    w = torch.randn(D_out, D_in, generator=g, device=device, dtype=bf).mul_(D_in ** -0.5)
    a = torch.randn(L, S, R, D_in, generator=g, device=device, dtype=bf).mul_(D_in ** -0.5)
    b = torch.randn(L, D_out, R, generator=g, device=device, dtype=bf).mul_(R ** -0.5)
    ranks = torch.tensor(cfg["ranks"], dtype=torch.int32, device=device)
    scal = torch.full((L,), 2.0, dtype=torch.float32, device=device)
    seg = T // cfg["segments"]
    adapters = torch.randint(0, L, (cfg["segments"],), generator=gc)
    mapping = adapters.repeat_interleave(seg).to(torch.int32).to(device)
    return x, w, a, b, ranks, scal, mapping, list(offs)


def linear_work(cfg, ranks_np, mapping_np):
    """(flops, algorithmic bytes) of one projection call: base GEMM, shrink and
    expand per token, the weights, every used adapter's factors, x and y."""
    import numpy as np
    T, D_in, offs, R = cfg["tokens"], cfg["in"], cfg["offsets"], cfg["max_rank"]
    D_out, S = offs[-1], len(offs) - 1
    r_tok = np.where(mapping_np >= 0, ranks_np[np.clip(mapping_np, 0, None)], 0).astype(np.float64)
    flops = 2.0 * T * D_out * D_in + float((2.0 * S * D_in + 2.0 * D_out) * r_tok.sum())
    used = np.unique(mapping_np[mapping_np >= 0])
    lora_bytes = float(sum((S * D_in + D_out) * int(ranks_np[l]) * 2 for l in used))
    byts = 2.0 * D_out * D_in + lora_bytes + 2.0 * T * D_in + 2.0 * T * D_out + 4.0 * T
    return flops, byts


def linear_oracle_rate(x, w, a, b, ranks, scal, mapping_np, offs, target_s, seed=0, max_tokens=None):
    import numpy as np
    import torch

    import oracle
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    xb, wb, ab, bb = bits(x), bits(w), bits(a), bits(b)
    rk, sc = ranks.cpu().numpy(), scal.cpu().numpy()
    T = x.shape[0]
    rng = np.random.default_rng(seed)
    n0 = min(T, 8)
    t0 = time.perf_counter()
    oracle.lora_linear(xb, mapping_np, rk, sc, wb, ab, bb, offs, tokens=rng.choice(T, n0, replace=False))
    per_tok = (time.perf_counter() - t0) / n0
    n = int(max(n0, min(T, target_s / max(per_tok, 1e-9))))
    if max_tokens:
        n = min(n, max_tokens)
    toks = np.sort(rng.choice(T, n, replace=False))
    t0 = time.perf_counter()
    st, _ = oracle.lora_linear(xb, mapping_np, rk, sc, wb, ab, bb, offs, tokens=toks)
    secs = time.perf_counter() - t0
    assert st == 0
    return n / secs, n, secs, oracle.max_threads()


def linear_config_entry(cfg, args, world):
    return {"workload": args.config, "tokens": cfg["tokens"], "in_features": cfg["in"],
            "out_parts": list(cfg["offsets"]), "loras": cfg["loras"], "max_rank": cfg["max_rank"],
            "seed": args.seed, "parallelism": f"dp{world} (replicas)" if world > 1 else "single GPU"}


def run_linear_reference(args, rank, world):
    """The oracle's dense projection as it stands, timed on host cores (rank 0 only)."""
    import oracle
    if rank != 0:
        return None
    oracle.build()
    cfg = LINEAR_CONFIGS[args.config]
    x, w, a, b, ranks, scal, mapping, offs = make_linear_inputs(cfg, "cpu", args.seed)
    mp = mapping.numpy()
    per_step_target = max(0.25, 90.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup):
        linear_oracle_rate(x, w, a, b, ranks, scal, mp, offs, per_step_target, seed=1000 + i, max_tokens=args.ref_tokens)
    ns, secs, thr = 0, 0.0, 1
    for i in range(args.steps):
        r, n, s_, thr = linear_oracle_rate(x, w, a, b, ranks, scal, mp, offs, per_step_target, seed=i,
                                           max_tokens=args.ref_tokens)
        ns += n
        secs += s_
    value = ns / secs
    return {"impl": "reference", "metric": LINEAR_METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": linear_config_entry(cfg, args, world),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                             "sample": f"{ns} tokens over {args.steps} steps (seeded samples of the "
                                       f"{cfg['tokens']}-token batch), fp64 C oracle, OpenMP over tokens"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_linear(args, rank, world, dist):
    import ctypes

    import numpy as np
    import torch

    import lora_moe_expert_info_gb300 as mlr
    import oracle
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = mlr.library()
    cfg = LINEAR_CONFIGS[args.config]
    x, w, a, b, ranks, scal, mapping, offs = make_linear_inputs(cfg, dev, args.seed + rank)
    T, D_in, D_out, L, R, S = cfg["tokens"], cfg["in"], offs[-1], cfg["loras"], cfg["max_rank"], len(offs) - 1
    y = torch.empty(T, D_out, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(int(lib.lora_linear_workspace_bytes(T, D_in, D_out, L, R, S)), dtype=torch.uint8, device=dev)

    def step():
        mlr.lora_linear_forward(x, w, mapping, ranks, scal, a, b, offs, y=y, workspace=ws, check=False)

    # correctness gate before timing: status word and a sampled oracle check
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mlr.lora_linear_forward(x, w, mapping, ranks, scal, a, b, offs, y=y, workspace=ws, status=status)
    mp_np = mapping.cpu().numpy()
    toks = np.sort(np.random.default_rng(7).choice(T, 16, replace=False))
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    st, yref = oracle.lora_linear(bits(x), mp_np, ranks.cpu().numpy(), scal.cpu().numpy(), bits(w), bits(a),
                                  bits(b), offs, tokens=toks)
    yg = y.float().cpu().numpy()[toks]
    if st != 0 or (np.abs(yg - yref) - (2e-2 + 2e-2 * np.abs(yref))).max() > 0:
        raise RuntimeError("projection differs from the oracle on the sampled tokens")
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # per-stage breakdown from untimed steps; the projection GEMM (profile stage
    # "down") is timed live inside the timed region
    stages = stage_profile(lib, step, max(3, min(args.steps, 50)))
    ms_total, proj_ms, n_launch, clk = timed_region(lib, args, step, stream, dist, local, "down")
    ms_max = reduce_max(ms_total, dist, dev)

    # end to end through the public API from pinned host buffers
    host_in = {"x": x.cpu().pin_memory(), "mapping": mapping.cpu().pin_memory(),
               "ranks": ranks.cpu().pin_memory(), "scal": scal.cpu().pin_memory()}
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()} for _ in range(2)]
    y_dev = [y, torch.empty_like(y)]
    y_host = [torch.empty(T, D_out, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = y_host[0].numel() * y_host[0].element_size()

    def upload(sl):
        for k, v in host_in.items():
            dev_in[sl][k].copy_(v, non_blocking=True)

    def compute(sl):
        d = dev_in[sl]
        mlr.lora_linear_forward(d["x"], w, d["mapping"], d["ranks"], d["scal"], a, b, offs,
                                y=y_dev[sl], workspace=ws, check=False)

    def download(sl):
        y_host[sl].copy_(y_dev[sl], non_blocking=True)

    e2e_ms, e2e_serial_ms = measure_e2e(args, upload, compute, download, stream, dist, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"projection reported device status {int(status.item())}")
    if rank != 0:
        return None

    cpu = None
    if not args.no_cpu_baseline:
        oracle.build()
        rate, n, secs, thr = linear_oracle_rate(x, w, a, b, ranks, scal, mp_np, offs, args.cpu_seconds)
        cpu = {"value": round(rate, 3), "unit": "tokens/s", "cores": thr, "kind": "oracle",
               "sample": f"{n} seeded tokens of the {T}-token batch ({secs:.1f} s), fp64 C oracle, "
                         f"OpenMP over tokens"}
    peaks, peak_src = load_peaks()
    ms_step = ms_max / args.steps
    flops, byts = linear_work(cfg, ranks.cpu().numpy(), mp_np)
    # the projection GEMM (profile stage "down") carries the base GEMM and the expand
    r_tok = np.where(mp_np >= 0, ranks.cpu().numpy()[np.clip(mp_np, 0, None)], 0).astype(np.float64)
    proj_flops = 2.0 * T * D_out * D_in + float(2.0 * D_out * r_tok.sum())
    proj_bytes = 2.0 * D_out * D_in + 2.0 * T * D_in + 4.0 * T * D_out
    rf = roofline_entry(proj_flops, proj_bytes, proj_ms, peaks, PEAK_KIND)
    rf.update({"kernel": "moe_gemm_kernel<3>", "stage": "down (the projection GEMM)",
               "peak_source": peak_label(peak_src),
               "traffic": recorded_traffic("down", args.config), "algorithmic_bytes": int(proj_bytes),
               "algorithmic_flops": int(proj_flops), "launch_ms": round(proj_ms, 4)})
    layer = layer_fractions(flops, byts, ms_step, peaks)
    layer.update({"algorithmic_bytes": int(byts), "algorithmic_flops": int(flops)})
    return {"metric": LINEAR_METRIC, "value": round(weak_scaling_rate(T, world, ms_step), 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": linear_config_entry(cfg, args, world),
            "roofline": rf, "layer_roofline": layer,
            "stages_ms": linear_stage_times(stages),
            "cpu_baseline": cpu,
            "e2e": {"value": round(weak_scaling_rate(T, world, e2e_ms), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 4), "steps_in_flight": 2,
                    "serial_ms_per_step": round(e2e_serial_ms, 4)},
            "gpu_launches": int(n_launch), "clocks": clk.summary()}


def linear_stage_times(stages):
    """The profile's stage times under the projection's own stage names.

    The projection records its launches on the forward's stage markers: the
    shrink on "shrink_gate_up", the projection GEMM on "down". The markers
    between them enclose no launch; their small gap is reported as such.
    """
    names = {"align_plan": "align_plan", "gather": "gather", "shrink_gate_up": "shrink",
             "down": "projection_gemm", "convert": "convert"}
    out = {names[k]: round(v, 4) for k, v in stages.items() if k in names}
    gap = sum(v for k, v in stages.items() if k not in names)
    out["marker_gaps"] = round(gap, 4)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="deepseek_v3_prefill",
                    help="headline workload (default: the DeepSeek-V3-like prefill, the largest that fits one GPU)")
    ap.add_argument("--extras", default=DEFAULT_EXTRAS,
                    help="comma-separated workloads measured after the headline and reported under "
                         "'workloads' ('' for none)")
    ap.add_argument("--weights", choices=["bf16", "fp8", "int8", "w4a16", "w8a8"], default="bf16",
                    help="base expert weights of the MoE workloads: bf16; FP8 E4M3, INT8 or UINT4 codes "
                         "dequantised on chip; or w8a8: FP8 weights and activations on the FP8 tensor cores")
    ap.add_argument("--combine", choices=["atomic", "deterministic"], default="deterministic",
                    help="top-k combine of the MoE forward (the other one is timed beside it)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-tokens", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="skip the extra measurement of the steps as one CUDA graph replay")
    args = ap.parse_args(argv)
    if args.config in LINEAR_CONFIGS and args.weights != "bf16":
        ap.error("--weights applies to the MoE workloads only")
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    linear = args.config in LINEAR_CONFIGS
    if args.impl == "reference":
        line = run_linear_reference(args, rank, world) if linear else run_reference(args, rank, world)
    else:
        line = run_linear(args, rank, world, dist) if linear else run_ours(args, rank, world, dist)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
