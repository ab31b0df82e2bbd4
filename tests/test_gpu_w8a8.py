"""GPU parity of the FP8 W8A8 layer (block-scaled MMAs on the FP8 tensor
cores) against the oracle's forward_fp8_w8a8.

The oracle takes the activations' quantisation decisions from the same bf16
values the kernels see for x (so those agree exactly) and from its fp64
SiLU(g)*u rounded to bf16 for the intermediate, which differs from the
kernel's fp32 value by accumulation order only; a code one E4M3 step apart is
rare and well inside the layer's tolerance |y - y_ref| <= 2e-2 + 2e-2 |y_ref|.
Shapes cover partial 128-groups and blocks (hidden 144 / 272, intermediate
80 / 208: a weight block shared by gate and up rows), adapters -1 and rank 0,
tiles split at 224 rows, the CUDA-core shrink (decode), a LoRA delta large
enough that a dropped term fails, and the Qwen-like and DeepSeek-V3-like
prefills on sampled tokens.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import workloads
from test_gpu_forward import bits, custom_case, joint_expand_case, within, workload_case
from test_gpu_quant import LORA, _common, _ref_common

pytestmark = pytest.mark.gpu


def gpu(case, q, mapping=None):
    lo = [getattr(case.w, k) for k in LORA]
    y = mlr.fused_moe_lora_forward_fp8_w8a8(*_common(case, mapping), q.w_gate_up_q, q.w_gate_up_exp, q.w_down_q,
                                            q.w_down_exp, *lo)
    return y.float().cpu().numpy()


def ref(case, q, tokens=None, mapping=None):
    lo = [bits(getattr(case.w, k)) for k in LORA]
    np_ = lambda t: t.cpu().numpy()  # noqa: E731
    st, y = oracle.forward_fp8_w8a8(*_ref_common(case, mapping), np_(q.w_gate_up_q), np_(q.w_gate_up_exp),
                                    np_(q.w_down_q), np_(q.w_down_exp), *lo, tokens=tokens)
    assert st == 0
    return y


def quant_of(case, seed=0):
    return workloads.make_fp8_w8a8_experts(case.cfg, device=case.dev, seed=seed)


def test_tiny_all_tokens(cuda_device):
    c = workload_case("tiny", cuda_device)
    q = quant_of(c)
    assert within(gpu(c, q), ref(c, q)) <= 0


@pytest.mark.parametrize("H,I", [(144, 80), (272, 208), (256, 128)])
def test_ragged_groups_and_blocks(cuda_device, H, I):
    c = custom_case(cuda_device, T=150, K=3, E=5, H=H, I=I, L=4, R=32, ranks=[12, 0, 24, 5],
                    seg_lens=[40, 30, 50, 30], adapters=[0, 3, -1, 2], lora_std="fan_in", seed=2, expert_bias=1.0)
    q = quant_of(c, seed=1)
    assert within(gpu(c, q), ref(c, q)) <= 0


def test_tiles_split_at_224_rows(cuda_device):
    # one expert takes every pair: 600 dense rows split into three tiles of at
    # most 224 rows, each with LoRA pieces of several adapters
    c = custom_case(cuda_device, T=600, K=1, E=1, H=256, I=128, L=3, R=16, ranks=[16, 8, 4],
                    seg_lens=[250, 200, 150], adapters=[0, 1, 2], lora_std="fan_in", seed=4)
    q = quant_of(c, seed=2)
    assert within(gpu(c, q), ref(c, q)) <= 0


def test_lora_delta(cuda_device):
    c = workload_case("tiny", cuda_device, lora_std="fan_in")
    q = quant_of(c)
    none = np.full_like(c.mapping, -1)
    y, y0 = gpu(c, q), gpu(c, q, mapping=none)
    r, r0 = ref(c, q), ref(c, q, mapping=none)
    assert np.abs(r - r0).max() > 0.5
    assert within(y, r) <= 0 and within(y0, r0) <= 0


def test_gate_up_joint_and_split_expand_steps(cuda_device):
    c = joint_expand_case(cuda_device)
    q = quant_of(c, seed=5)
    none = np.full_like(c.mapping, -1)
    y, r = gpu(c, q), ref(c, q)
    assert np.abs(r - ref(c, q, mapping=none)).max() > 0.5
    assert within(y, r) <= 0


def test_decode_all_tokens(cuda_device):
    c = workload_case("decode", cuda_device)
    q = quant_of(c)
    assert within(gpu(c, q), ref(c, q)) <= 0


@pytest.mark.parametrize("name,n", [("qwen_moe_prefill", 48), ("deepseek_v3_prefill", 10)])
def test_prefill_sampled(cuda_device, name, n):
    c = workload_case(name, cuda_device)
    q = quant_of(c)
    y = gpu(c, q)
    toks = np.sort(np.random.default_rng(5).choice(c.cfg.num_tokens, n, replace=False))
    toks = np.concatenate([[0, c.cfg.num_tokens - 1], toks])
    assert within(y[toks], ref(c, q, tokens=toks)) <= 0


def test_repeatable(cuda_device):
    # the default combine is deterministic: two calls give identical bits
    c = workload_case("qwen_moe_prefill", cuda_device)
    q = quant_of(c)
    assert (gpu(c, q) == gpu(c, q)).all()


def test_empty_batch(cuda_device):
    # T = 0: nothing to do, an empty y
    c = custom_case(cuda_device, T=8, K=2, E=4, H=128, I=128, L=2, R=16, ranks=[16, 8], seg_lens=[8],
                    adapters=[0])
    q = quant_of(c)
    lo = [getattr(c.w, k) for k in LORA]
    y = mlr.fused_moe_lora_forward_fp8_w8a8(c.x[:0], c.b.topk_ids[:0], c.b.topk_weights[:0],
                                            torch.zeros(0, dtype=torch.int32, device=cuda_device),
                                            c.b.lora_ranks, c.scal, q.w_gate_up_q, q.w_gate_up_exp, q.w_down_q,
                                            q.w_down_exp, *lo)
    assert tuple(y.shape) == (0, 128)


def test_no_adapter_slots(cuda_device):
    # L = 0: the base layer only, nothing of the LoRA path runs
    c = custom_case(cuda_device, T=70, K=2, E=6, H=192, I=256, L=0, R=0, ranks=[], seg_lens=[70],
                    adapters=[-1])
    q = quant_of(c, seed=3)
    assert within(gpu(c, q), ref(c, q)) <= 0


def test_all_ranks_zero_equals_base(cuda_device):
    c = custom_case(cuda_device, T=64, K=2, E=4, H=128, I=128, L=3, R=16, ranks=[0, 0, 0],
                    seg_lens=[30, 34], adapters=[0, 2], lora_std="fan_in")
    q = quant_of(c, seed=4)
    y, y0 = gpu(c, q), gpu(c, q, mapping=np.full_like(c.mapping, -1))
    assert within(y, ref(c, q)) <= 0
    assert np.array_equal(y, y0)


def test_hidden_not_multiple_of_16_refused(cuda_device):
    c = custom_case(cuda_device, T=20, K=2, E=4, H=136, I=64, L=2, R=16, ranks=[16, 8], seg_lens=[20],
                    adapters=[0])
    q = quant_of(c)
    with pytest.raises(mlr.MoeLoraError):
        gpu(c, q)
