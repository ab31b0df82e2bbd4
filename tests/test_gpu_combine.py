"""The deterministic top-k combine of the MoE forward against the oracle.

With moe_lora_set_deterministic(1) (the default) the down GEMM writes each pair's weighted
output w * d as a bf16 row of its own and a combine kernel sums a token's K
rows in increasing k, so y is bit-identical from run to run.  The extra bf16
rounding of each w * d (relative 2^-9) stays far inside the layer's tolerance
|y - y_ref| <= 2e-2 + 2e-2 |y_ref|.  Checked on the workloads, on the LoRA
delta with O(1) adapters, on the FP8 experts and with a dropped pair.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import workloads
from test_gpu_forward import WKEYS, bits, custom_case, within, workload_case

pytestmark = pytest.mark.gpu


@pytest.fixture
def deterministic():
    assert mlr.deterministic()  # the default
    mlr.set_deterministic(True)
    try:
        yield
    finally:
        mlr.set_deterministic(True)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_workload_all_tokens_bit_identical_runs(cuda_device, deterministic, name):
    c = workload_case(name, cuda_device)
    y1, y2 = c.gpu(), c.gpu()
    assert np.array_equal(y1, y2)
    assert within(y1, c.ref()) <= 0


def test_qwen_prefill_sampled(cuda_device, deterministic):
    c = workload_case("qwen_moe_prefill", cuda_device)
    y1, y2 = c.gpu(), c.gpu()
    assert np.array_equal(y1, y2)
    toks = np.sort(np.random.default_rng(3).choice(c.cfg.num_tokens, 64, replace=False))
    toks = np.concatenate([[0, c.cfg.num_tokens - 1], toks])
    assert within(y1[toks], c.ref(tokens=toks)) <= 0


def test_lora_delta_and_ragged_shapes(cuda_device, deterministic):
    c = custom_case(cuda_device, T=203, K=3, E=5, H=200, I=136, L=4, R=32, ranks=[12, 0, 24, 5],
                    seg_lens=[17, 60, 1, 90, 35], adapters=[0, 3, -1, 2, 1], seed=1,
                    lora_std="fan_in", expert_bias=1.0)
    none = np.full_like(c.mapping, -1)
    y, y0 = c.gpu(), c.gpu(mapping=none)
    r, r0 = c.ref(), c.ref(mapping=none)
    assert np.abs(r - r0).max() > 0.5
    assert within(y, r) <= 0 and within(y0, r0) <= 0


def test_matches_the_atomic_combine(cuda_device):
    c = custom_case(cuda_device, T=900, K=2, E=3, H=128, I=192, L=6, R=32,
                    ranks=[8, 16, 32, 0, 24, 8], seg_lens=[100, 200, 50, 300, 150, 100],
                    adapters=[0, 1, 2, 3, 4, 5], lora_std="fan_in", expert_bias=3.0)
    yd = c.gpu()
    mlr.set_deterministic(False)
    try:
        ya = c.gpu()
        assert within(ya, c.ref()) <= 0
    finally:
        mlr.set_deterministic(True)
    r = c.ref()
    assert within(ya, r) <= 0 and within(yd, r) <= 0
    # the two combines differ only by roundings of the sum
    assert np.abs(ya - yd).max() <= 2e-2 * max(1.0, float(np.abs(r).max()))


def test_fp8_experts(cuda_device, deterministic):
    cfg = workloads.CONFIGS["tiny"]
    dev = cuda_device
    b = workloads.make_batch(cfg, device=dev, seed=0)
    w = workloads.make_weights(cfg, b.lora_ranks, device=dev, seed=0)
    x = workloads.make_x(cfg, device=dev, seed=0)
    q = workloads.make_fp8_experts(cfg, device=dev, seed=0)
    _, mp = mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, cfg.num_tokens)
    lo = {k: getattr(w, k) for k in WKEYS[2:]}
    args = (x, b.topk_ids, b.topk_weights, mp, b.lora_ranks, b.scalings, q.w_gate_up_q, q.w_gate_up_scale,
            q.w_down_q, q.w_down_scale)
    y1 = mlr.fused_moe_lora_forward_fp8(*args, **lo).float().cpu().numpy()
    y2 = mlr.fused_moe_lora_forward_fp8(*args, **lo).float().cpu().numpy()
    assert np.array_equal(y1, y2)
    st, yref = oracle.forward_fp8(bits(x), b.topk_ids.cpu().numpy(), b.topk_weights.cpu().numpy(),
                                  mp.cpu().numpy(), b.lora_ranks.cpu().numpy(), b.scalings.cpu().numpy(),
                                  q.w_gate_up_q.cpu().numpy(), q.w_gate_up_scale.cpu().numpy(),
                                  q.w_down_q.cpu().numpy(), q.w_down_scale.cpu().numpy(),
                                  *[bits(getattr(w, k)) for k in WKEYS[2:]])
    assert st == 0 and within(y1, yref) <= 0


def test_dropped_pair_adds_nothing(cuda_device, deterministic):
    # an out-of-range expert id: the call reports it, the pair is dropped, and
    # every other output still equals the oracle's layer without that pair
    c = custom_case(cuda_device, T=40, K=2, E=4, H=128, I=128, L=2, R=16, ranks=[16, 8],
                    seg_lens=[20, 20], adapters=[0, 1])
    ids = c.b.topk_ids.clone()
    ids[3, 1] = 4  # E = 4
    args = dict(x=c.x, topk_ids=ids, topk_weights=c.b.topk_weights,
                token_lora_mapping=torch.from_numpy(np.ascontiguousarray(c.mapping)).to(cuda_device),
                lora_ranks=c.b.lora_ranks, scalings=c.scal, **{k: getattr(c.w, k) for k in WKEYS})
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    y = mlr.fused_moe_lora_forward(**args, check=False, status=status).float().cpu().numpy()
    assert int(status.item()) & 0x04
    wts = c.b.topk_weights.clone()
    wts[3, 1] = 0.0
    ids_ok = ids.clone()
    ids_ok[3, 1] = 0
    st, r = oracle.forward(bits(c.x), ids_ok.cpu().numpy(), wts.cpu().numpy(), c.mapping,
                           c.b.lora_ranks.cpu().numpy(), c.scal.cpu().numpy(),
                           *[bits(getattr(c.w, k)) for k in WKEYS])
    assert st == 0 and within(y, r) <= 0
