"""The layer captured in a CUDA graph: the calls make no host-side decision on
device data and never synchronise, so a captured step (batch info + forward)
replays the same launches.  With the default (deterministic) top-k combine the
replayed y equals the eagerly computed one bit for bit, for the bf16 and the
W8A8 layers, and a replay after new inputs were copied in reflects them."""
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
from lora_moe_expert_info_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(name, dev, w8a8=False):
    cfg = workloads.CONFIGS[name]
    b = workloads.make_batch(cfg, device=dev, seed=0)
    w = workloads.make_weights(cfg, b.lora_ranks, device=dev, seed=0)
    x = workloads.make_x(cfg, device=dev, seed=0)
    q = workloads.make_fp8_w8a8_experts(cfg, device=dev, seed=0) if w8a8 else None
    return cfg, b, w, x, q


@pytest.mark.parametrize("name,w8a8", [("decode", False), ("qwen_moe_prefill", False), ("decode", True)])
def test_graph_replay_matches_eager(cuda_device, name, w8a8):
    cfg, b, w, x, q = _inputs(name, cuda_device, w8a8)
    T, K, E, H, I, L, R = (cfg.num_tokens, cfg.topk, cfg.num_experts, cfg.hidden, cfg.intermediate,
                           cfg.num_loras, cfg.max_rank)
    wsb = mlr.fused_moe_lora_workspace_bytes_fp8_w8a8 if w8a8 else mlr.fused_moe_lora_workspace_bytes
    ws = torch.empty(wsb(T, K, E, H, I, L, R), dtype=torch.uint8, device=cuda_device)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=cuda_device)
    en = torch.empty(L, dtype=torch.int32, device=cuda_device)
    mp = torch.empty(T, dtype=torch.int32, device=cuda_device)
    xin = x.clone()
    max_len = int(b.seg_lens.max())  # read once on the host, outside the captured step
    lo = dict(lora_a_gu=w.lora_a_gu, lora_b_gu=w.lora_b_gu, lora_a_down=w.lora_a_down, lora_b_down=w.lora_b_down)

    def step():
        mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, T, max_len,
                                adapter_enabled=en, token_lora_mapping=mp, check=False)
        if w8a8:
            mlr.fused_moe_lora_forward_fp8_w8a8(xin, b.topk_ids, b.topk_weights, mp, b.lora_ranks, b.scalings,
                                                q.w_gate_up_q, q.w_gate_up_exp, q.w_down_q, q.w_down_exp, **lo,
                                                y=y, workspace=ws, check=False)
        else:
            mlr.fused_moe_lora_forward(xin, b.topk_ids, b.topk_weights, mp, b.lora_ranks, b.scalings,
                                       w.w_gate_up, w.w_down, **lo, y=y, workspace=ws, check=False)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    y_eager = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)
    # new inputs in the captured buffer: the replay computes with them
    xin.copy_(torch.flip(x, dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    y_new = y.clone()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    assert torch.equal(y, y_new)
    assert not torch.equal(y_new, y_eager)
