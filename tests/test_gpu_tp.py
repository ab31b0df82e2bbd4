"""GPU parity of one tensor-parallel rank's fused q/k/v projection with LoRA.

A column-parallel rank holds the rows lora_tp_qkv_b_rows gives of the base
weight and of LoRA B (sglang PR #24420 page: q split by rank, k and v by
rank // replicas once the KV heads are replicated).  Its projection is
lora_linear_forward on those rows, with the unsplit LoRA A.  Every rank is
run here, one after another on the one GPU (no rank waits on another: the
column-parallel projection has no exchange step), and each output is compared
with the same columns of the oracle's full, unsplit projection, within the
layer's tolerance.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from test_gpu_linear import bits, within

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_every_rank_is_its_column_block(cuda_device, tp):
    # 16 q heads, 2 KV heads of 32: tp 1-2 split the KV heads, tp 4-8 replicate them
    nh, nkv, hd, D_in, T, L, R = 16, 2, 32, 256, 120, 3, 16
    D = (nh + 2 * nkv) * hd
    dev = cuda_device
    g = torch.Generator(device=dev).manual_seed(tp)
    bf = torch.bfloat16
    x = torch.randn(T, D_in, generator=g, device=dev, dtype=bf)
    w = torch.randn(D, D_in, generator=g, device=dev, dtype=bf).mul_(D_in ** -0.5)
    a = torch.randn(L, 1, R, D_in, generator=g, device=dev, dtype=bf).mul_(D_in ** -0.5)
    b = torch.randn(L, D, R, generator=g, device=dev, dtype=bf).mul_(R ** -0.5)
    ranks = torch.tensor([16, 8, 0], dtype=torch.int32, device=dev)
    scal = torch.tensor([0.5, 0.5, 0.0], dtype=torch.float32, device=dev)
    mp = np.repeat(np.array([0, 1, -1, 2, 0], np.int32), [30, 20, 10, 25, 35])
    mapping = torch.from_numpy(mp).to(dev)
    st, y_full = oracle.lora_linear(bits(x), mp, ranks.cpu().numpy(), scal.cpu().numpy(), bits(w), bits(a),
                                    bits(b), [0, D])
    assert st == 0
    for r in range(tp):
        ranges, n = mlr.lora_tp_qkv_b_rows(nh, nkv, hd, tp, r)
        w_r = mlr.tp_take_rows(w, ranges, dim=0)
        b_r = mlr.tp_take_rows(b, ranges, dim=1)
        assert w_r.shape == (n, D_in) and b_r.shape == (L, n, R)
        y_r = mlr.lora_linear_forward(x, w_r, mapping, ranks, scal, a, b_r, [0, n]).float().cpu().numpy()
        cols = [i for lo, hi in ranges for i in range(lo, hi)]
        assert within(y_r, y_full[:, cols]) <= 0, f"rank {r} of {tp}"
