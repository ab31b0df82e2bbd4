"""bench.py's multi-process plumbing on CPU (gloo, world size 2).

The GPU arm runs one replica per GPU with no data-path collective; what crosses
ranks is the timing: the slowest rank's time sets the job's, and the job's
throughput is every rank's work over that time.  The reference arm runs on
rank 0 only; other ranks exit 0 without output.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]  # rank 1 is the slower one
        ms_max = bench.reduce_max(ms, dist, "cpu")
        out[rank] = (ms_max, bench.weak_scaling_rate(4096, world, ms_max))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_rate():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of a multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    for rank in range(world):
        ms_max, rate = got[rank]
        assert ms_max == 5.0
        assert rate == pytest.approx(2 * 4096 / 5e-3)


def test_single_process_needs_no_group():
    assert bench.reduce_max(2.5, None, "cpu") == 2.5
    assert bench.weak_scaling_rate(10, 1, 1.0) == pytest.approx(1e4)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_linear_stage_names():
    stages = {"align_plan": 0.05, "gather": 0.04, "shrink_gate_up": 0.03, "gate_up": 0.002,
              "shrink_down": 0.001, "down": 0.16, "convert": 0.02}
    out = bench.linear_stage_times(stages)
    assert out == {"align_plan": 0.05, "gather": 0.04, "shrink": 0.03, "projection_gemm": 0.16,
                   "convert": 0.02, "marker_gaps": 0.003}
    assert abs(sum(out.values()) - sum(stages.values())) < 1e-9


def test_layer_work_fp8_weights_are_one_byte_plus_block_scales():
    import math

    from lora_moe_expert_info_gb300 import workloads
    cfg = workloads.CONFIGS["tiny"]
    b = workloads.make_batch(cfg, device="cpu", seed=0)
    # any mapping with valid adapters serves the byte count
    mapping = torch.zeros(cfg.num_tokens, dtype=torch.int32)
    f16, b16, s16 = bench.layer_work(cfg, b, mapping)
    f8, b8, s8 = bench.layer_work(cfg, b, mapping, fp8=True)
    assert f16 == f8 and {k: v[0] for k, v in s16.items()} == {k: v[0] for k, v in s8.items()}
    H, I = cfg.hidden, cfg.intermediate
    touched = torch.unique(b.topk_ids).numel()
    nb = lambda n: math.ceil(n / 128)  # noqa: E731
    per_expert_bf16 = 3 * H * I * 2
    per_expert_fp8 = 3 * H * I + 4 * (nb(2 * I) * nb(H) + nb(H) * nb(I))
    assert b16 - b8 == touched * (per_expert_bf16 - per_expert_fp8)
    # the shrinks do not read base weights
    assert s16["shrink_gate_up"] == s8["shrink_gate_up"] and s16["shrink_down"] == s8["shrink_down"]
