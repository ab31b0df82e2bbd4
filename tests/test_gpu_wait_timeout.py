"""Failure detection on the GPU: the bounded pipeline waits give up.

Every mbarrier wait of the GEMM kernels (operands landing, an accumulator
filling or draining, the FP8 converters' raw tiles) gives up after a limit that
the host sets (moe_lora_set_wait_limit_ns, 2 s by default) and reports
MLR_STATUS_TIMEOUT instead of spinning.  These tests set the limit to 1 ns, so
that the first wait of every GEMM launch that is not already satisfied gives up:
the single-CTA shrinks, the CTA-pair gate_up and down GEMMs, the FP8 converter
warps and the block-scaled W8A8 GEMMs (their scale-factor warps included).  The call must still return normally with the timeout bit set,
and after the limit is put back the next call on the same context must match
the oracle, which shows that every role left, freed its TMEM and kept the
context usable.  No fault, trap or endless wait is involved: the waits are
made to run out by their own limit.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import workloads

pytestmark = pytest.mark.gpu
ATOL = RTOL = 2e-2
WKEYS = ("w_gate_up", "w_down", "lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")
TIMEOUT = 0x10
DEFAULT_NS = 2_000_000_000


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def within(y, yref):
    return float((np.abs(y - yref) - (ATOL + RTOL * np.abs(yref))).max())


@pytest.fixture
def short_waits():
    assert mlr.wait_limit_ns() == DEFAULT_NS
    mlr.set_wait_limit_ns(0)
    assert mlr.wait_limit_ns() == 1
    try:
        yield
    finally:
        mlr.set_wait_limit_ns(DEFAULT_NS)
    assert mlr.wait_limit_ns() == DEFAULT_NS


def _tiny(dev):
    cfg = workloads.CONFIGS["tiny"]
    b = workloads.make_batch(cfg, device=dev, seed=0)
    w = workloads.make_weights(cfg, b.lora_ranks, device=dev, seed=0)
    x = workloads.make_x(cfg, device=dev, seed=0)
    _, mp = mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, cfg.num_tokens)
    return cfg, b, w, x, mp


def _ref(b, w, x, mp):
    st, y = oracle.forward(bits(x), b.topk_ids.cpu().numpy(), b.topk_weights.cpu().numpy(),
                           mp.cpu().numpy(), b.lora_ranks.cpu().numpy(), b.scalings.cpu().numpy(),
                           *[bits(getattr(w, k)) for k in WKEYS])
    assert st == 0
    return y


def test_limit_setter_rejects_more_than_a_minute():
    with pytest.raises(ValueError):
        mlr.set_wait_limit_ns(61_000_000_000)
    assert mlr.wait_limit_ns() == DEFAULT_NS


def test_bf16_layer_waits_give_up_then_recover(cuda_device):
    cfg, b, w, x, mp = _tiny(cuda_device)
    args = dict(x=x, topk_ids=b.topk_ids, topk_weights=b.topk_weights, token_lora_mapping=mp,
                lora_ranks=b.lora_ranks, scalings=b.scalings, **{k: getattr(w, k) for k in WKEYS})
    mlr.set_wait_limit_ns(0)
    try:
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        mlr.fused_moe_lora_forward(**args, check=False, status=status)   # returns normally
        torch.cuda.synchronize()
        assert int(status.item()) & TIMEOUT
        # the checked wrapper turns the bit into an error
        with pytest.raises(mlr.MoeLoraError) as ei:
            mlr.fused_moe_lora_forward(**args)
        assert ei.value.code == mlr.MLR_ERR_TIMEOUT
    finally:
        mlr.set_wait_limit_ns(DEFAULT_NS)
    y = mlr.fused_moe_lora_forward(**args).float().cpu().numpy()   # same context, default limit
    assert within(y, _ref(b, w, x, mp)) <= 0


def test_fp8_converter_waits_give_up_then_recover(cuda_device, short_waits):
    cfg, b, w, x, mp = _tiny(cuda_device)
    q = workloads.make_fp8_experts(cfg, device=cuda_device, seed=0)
    args = dict(x=x, topk_ids=b.topk_ids, topk_weights=b.topk_weights, token_lora_mapping=mp,
                lora_ranks=b.lora_ranks, scalings=b.scalings, w_gate_up_q=q.w_gate_up_q,
                w_gate_up_scale=q.w_gate_up_scale, w_down_q=q.w_down_q, w_down_scale=q.w_down_scale,
                **{k: getattr(w, k) for k in WKEYS[2:]})
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mlr.fused_moe_lora_forward_fp8(**args, check=False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & TIMEOUT
    mlr.set_wait_limit_ns(DEFAULT_NS)
    y = mlr.fused_moe_lora_forward_fp8(**args).float().cpu().numpy()
    st, yref = oracle.forward_fp8(bits(x), b.topk_ids.cpu().numpy(), b.topk_weights.cpu().numpy(),
                                  mp.cpu().numpy(), b.lora_ranks.cpu().numpy(), b.scalings.cpu().numpy(),
                                  q.w_gate_up_q.cpu().numpy(), q.w_gate_up_scale.cpu().numpy(),
                                  q.w_down_q.cpu().numpy(), q.w_down_scale.cpu().numpy(),
                                  *[bits(getattr(w, k)) for k in WKEYS[2:]])
    assert st == 0 and within(y, yref) <= 0


def test_w8a8_waits_give_up_then_recover(cuda_device, short_waits):
    cfg, b, w, x, mp = _tiny(cuda_device)
    q = workloads.make_fp8_w8a8_experts(cfg, device=cuda_device, seed=0)
    args = dict(x=x, topk_ids=b.topk_ids, topk_weights=b.topk_weights, token_lora_mapping=mp,
                lora_ranks=b.lora_ranks, scalings=b.scalings, w_gate_up_q=q.w_gate_up_q,
                w_gate_up_exp=q.w_gate_up_exp, w_down_q=q.w_down_q, w_down_exp=q.w_down_exp,
                **{k: getattr(w, k) for k in WKEYS[2:]})
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mlr.fused_moe_lora_forward_fp8_w8a8(**args, check=False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & TIMEOUT
    mlr.set_wait_limit_ns(DEFAULT_NS)
    y = mlr.fused_moe_lora_forward_fp8_w8a8(**args).float().cpu().numpy()
    st, yref = oracle.forward_fp8_w8a8(bits(x), b.topk_ids.cpu().numpy(), b.topk_weights.cpu().numpy(),
                                       mp.cpu().numpy(), b.lora_ranks.cpu().numpy(), b.scalings.cpu().numpy(),
                                       q.w_gate_up_q.cpu().numpy(), q.w_gate_up_exp.cpu().numpy(),
                                       q.w_down_q.cpu().numpy(), q.w_down_exp.cpu().numpy(),
                                       *[bits(getattr(w, k)) for k in WKEYS[2:]])
    assert st == 0 and within(y, yref) <= 0


def test_projection_pair_waits_give_up_then_recover(cuda_device, short_waits):
    # the split-B projection runs the down-shape GEMM on CTA pairs
    g = torch.Generator(device=cuda_device).manual_seed(5)
    T, D_in, offs, L, R = 300, 256, [0, 256, 320], 2, 16
    D_out = offs[-1]
    bf = torch.bfloat16
    x = torch.randn(T, D_in, generator=g, device=cuda_device, dtype=bf)
    wt = torch.randn(D_out, D_in, generator=g, device=cuda_device, dtype=bf).mul_(D_in ** -0.5)
    a = torch.randn(L, 2, R, D_in, generator=g, device=cuda_device, dtype=bf).mul_(D_in ** -0.5)
    bb = torch.randn(L, D_out, R, generator=g, device=cuda_device, dtype=bf).mul_(R ** -0.5)
    ranks = torch.tensor([16, 8], dtype=torch.int32, device=cuda_device)
    scal = torch.tensor([0.5, 0.5], dtype=torch.float32, device=cuda_device)
    mapping = torch.randint(-1, L, (T,), generator=g, device=cuda_device).to(torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mlr.lora_linear_forward(x, wt, mapping, ranks, scal, a, bb, offs, check=False, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & TIMEOUT
    mlr.set_wait_limit_ns(DEFAULT_NS)
    y = mlr.lora_linear_forward(x, wt, mapping, ranks, scal, a, bb, offs).float().cpu().numpy()
    st, yref = oracle.lora_linear(bits(x), mapping.cpu().numpy(), ranks.cpu().numpy(), scal.cpu().numpy(),
                                  bits(wt), bits(a), bits(bb), offs)
    assert st == 0 and within(y, yref) <= 0
