"""GPU parity of fused_moe_lora_forward_fp8 (FP8 E4M3 base experts, 128 x 128
block scales, bf16 LoRA) against the oracle's forward_fp8.

The oracle dequantises each weight exactly (code x scale in fp64); the kernels
round code x scale to bf16 once before the tensor cores, a relative error of
at most 2^-9 per weight, well inside the layer's tolerance
|y - y_ref| <= 2e-2 + 2e-2 |y_ref|.  The shapes cover ragged 128-blocks (H,
I not multiples of 128, a W_gate_up scale block shared by gate and up rows),
adapters -1 and rank 0, the CUDA-core shrink (decode), the CTA-pair down
kernel's partial row blocks, and a LoRA delta large enough that a dropped term
fails.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import workloads
from test_gpu_forward import bits, custom_case, within, workload_case

pytestmark = pytest.mark.gpu


def fp8_of(case, seed=0):
    return workloads.make_fp8_experts(case.cfg, device=case.dev, seed=seed)


def gpu_fp8(case, q, mapping=None):
    m = case.mapping if mapping is None else mapping
    return mlr.fused_moe_lora_forward_fp8(
        case.x, case.b.topk_ids, case.b.topk_weights,
        torch.from_numpy(np.ascontiguousarray(m)).to(case.dev), case.b.lora_ranks, case.scal,
        q.w_gate_up_q, q.w_gate_up_scale, q.w_down_q, q.w_down_scale,
        case.w.lora_a_gu, case.w.lora_b_gu, case.w.lora_a_down, case.w.lora_b_down).float().cpu().numpy()


def ref_fp8(case, q, tokens=None, mapping=None):
    m = case.mapping if mapping is None else mapping
    st, y = oracle.forward_fp8(
        bits(case.x), case.b.topk_ids.cpu().numpy(), case.b.topk_weights.cpu().numpy(), m,
        case.b.lora_ranks.cpu().numpy(), case.scal.cpu().numpy(),
        q.w_gate_up_q.cpu().numpy(), q.w_gate_up_scale.cpu().numpy(),
        q.w_down_q.cpu().numpy(), q.w_down_scale.cpu().numpy(),
        bits(case.w.lora_a_gu), bits(case.w.lora_b_gu), bits(case.w.lora_a_down), bits(case.w.lora_b_down),
        tokens=tokens)
    assert st == 0
    return y


def test_fp8_tiny_all_tokens(cuda_device):
    c = workload_case("tiny", cuda_device)
    q = fp8_of(c)
    assert within(gpu_fp8(c, q), ref_fp8(c, q)) <= 0


@pytest.mark.parametrize("H,I", [(144, 80), (272, 208), (128, 64)])
def test_fp8_ragged_blocks(cuda_device, H, I):
    # I = 80: gate rows and up rows share W_gate_up's first scale block; H, I
    # not multiples of 128 leave partial row and column blocks in both GEMMs
    c = custom_case(cuda_device, T=96, K=2, E=5, H=H, I=I, L=3, R=32, ranks=(16, 0, 32),
                    seg_lens=[30, 10, 40, 16], adapters=[0, -1, 2, 1], seed=7)
    q = fp8_of(c, seed=7)
    assert within(gpu_fp8(c, q), ref_fp8(c, q)) <= 0


def test_fp8_no_adapters(cuda_device):
    c = custom_case(cuda_device, T=64, K=2, E=4, H=256, I=128, L=0, R=0, ranks=(),
                    seg_lens=[64], adapters=[-1], seed=3)
    q = fp8_of(c, seed=3)
    assert within(gpu_fp8(c, q), ref_fp8(c, q)) <= 0


def test_fp8_lora_delta(cuda_device):
    # A, B ~ N(0, 1/fan_in): the adapters move y by O(1); compare the delta itself
    c = custom_case(cuda_device, T=80, K=2, E=4, H=256, I=256, L=2, R=32, ranks=(32, 16),
                    seg_lens=[40, 40], adapters=[0, 1], seed=5, lora_std="fan_in")
    q = fp8_of(c, seed=5)
    off = np.full_like(c.mapping, -1)
    d_gpu = gpu_fp8(c, q) - gpu_fp8(c, q, mapping=off)
    d_ref = ref_fp8(c, q) - ref_fp8(c, q, mapping=off)
    assert np.abs(d_ref).max() > 0.5
    assert within(d_gpu, d_ref) <= 0


def test_fp8_qwen_prefill_sampled(cuda_device):
    c = workload_case("qwen_moe_prefill", cuda_device)
    q = fp8_of(c)
    toks = np.sort(np.random.default_rng(11).choice(c.cfg.num_tokens, 48, replace=False))
    y = gpu_fp8(c, q)[toks]
    assert within(y, ref_fp8(c, q, tokens=toks)) <= 0


def test_fp8_decode_all_tokens(cuda_device):
    c = workload_case("decode", cuda_device)
    q = fp8_of(c)
    assert within(gpu_fp8(c, q), ref_fp8(c, q)) <= 0


def test_fp8_deterministic(cuda_device):
    c = workload_case("tiny", cuda_device)
    q = fp8_of(c)
    a, b = gpu_fp8(c, q), gpu_fp8(c, q)
    # the combine's fp32 reductions may land in any order: equal up to rounding
    np.testing.assert_allclose(a, b, rtol=1e-2, atol=1e-2)
