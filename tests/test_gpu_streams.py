"""The binding on a caller's side stream.

When a call is given stream=s other than torch's current stream, the outputs,
workspace and status word it allocates are zeroed on s, the caching allocator
records them on s, and the status read synchronises s: the device checks still
see the kernels' status bits, and results equal those of the same call on the
current stream.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
from lora_moe_expert_info_gb300 import workloads

pytestmark = pytest.mark.gpu
WKEYS = ("w_gate_up", "w_down", "lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")


def _tiny(dev):
    cfg = workloads.CONFIGS["tiny"]
    b = workloads.make_batch(cfg, device=dev, seed=0)
    w = workloads.make_weights(cfg, b.lora_ranks, device=dev, seed=0)
    x = workloads.make_x(cfg, device=dev, seed=0)
    return cfg, b, w, x


def test_side_stream_out_of_range_id_still_raises(cuda_device):
    cfg, b, w, x = _tiny(cuda_device)
    _, mp = mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, cfg.num_tokens)
    ids = b.topk_ids.clone()
    ids[5, 1] = cfg.num_experts + 3
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with pytest.raises(mlr.MoeLoraError) as ei:
        mlr.fused_moe_lora_forward(x, ids, b.topk_weights, mp, b.lora_ranks, b.scalings,
                                   *[getattr(w, k) for k in WKEYS], stream=s)
    assert ei.value.code == mlr.MLR_ERR_INDEX
    with pytest.raises(mlr.MoeLoraError):
        mlr.moe_lora_align(ids, mp, cfg.num_experts, cfg.num_loras, cfg.block_size, stream=s)
    bad = b.seg_indptr.clone()
    bad[2] = bad[3] + 1  # decreasing offsets
    with pytest.raises(mlr.MoeLoraError):
        mlr.moe_lora_batch_info(bad, b.weight_indices, b.lora_ranks, cfg.num_tokens, stream=s)


def test_side_stream_results_equal_current_stream(cuda_device):
    cfg, b, w, x = _tiny(cuda_device)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    en0, mp0 = mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, cfg.num_tokens)
    en1, mp1 = mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, cfg.num_tokens, stream=s)
    assert torch.equal(en0, en1) and torch.equal(mp0, mp1)
    a0 = mlr.moe_lora_align(b.topk_ids, mp0, cfg.num_experts, cfg.num_loras, cfg.block_size)
    a1 = mlr.moe_lora_align(b.topk_ids, mp0, cfg.num_experts, cfg.num_loras, cfg.block_size, stream=s)
    n = int(a0[3].item())
    assert int(a1[3].item()) == n and torch.equal(a0[0][:n], a1[0][:n])
    args = [x, b.topk_ids, b.topk_weights, mp0, b.lora_ranks, b.scalings] + [getattr(w, k) for k in WKEYS]
    y0 = mlr.fused_moe_lora_forward(*args)
    y1 = mlr.fused_moe_lora_forward(*args, stream=s)
    torch.cuda.synchronize()
    # the top-k combine adds in any order, so compare within a few bf16 ulps
    assert torch.allclose(y0.float(), y1.float(), atol=1e-2, rtol=1e-2)
