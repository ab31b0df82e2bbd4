"""GPU parity of moe_lora_align against the oracle (bit-exact int32).

Every valid-prefix entry (sorted pair ids, per-block expert and adapter ids)
and num_tokens_post_pad must equal the oracle's stable counting sort, on
random cases, ragged and degenerate shapes and the five workloads' routings.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import workloads

pytestmark = pytest.mark.gpu


def _compare(dev, topk, mapping, E, L, bs):
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    mapping = np.ascontiguousarray(mapping, dtype=np.int32)
    st, s, be, bl, n = oracle.align(topk, mapping, E, L, bs)
    assert st == oracle.OK
    ts, tbe, tbl, tn = mlr.moe_lora_align(torch.from_numpy(topk).to(dev),
                                          torch.from_numpy(mapping).to(dev), E, L, bs)
    gn = int(tn.item())
    assert gn == n
    assert np.array_equal(ts[:n].cpu().numpy(), s)
    assert np.array_equal(tbe[:n // bs].cpu().numpy(), be)
    assert np.array_equal(tbl[:n // bs].cpu().numpy(), bl)
    return n


def _random(seed, T, K, E, L, p_none=0.1, distinct=True):
    rng = np.random.default_rng(seed)
    if distinct and K <= E:
        topk = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)
    else:
        topk = rng.integers(0, E, (T, K)).astype(np.int32)
    mapping = rng.integers(0, L, T).astype(np.int32) if L > 0 else np.full(T, -1, np.int32)
    mapping[rng.random(T) < p_none] = -1
    return topk, mapping


@pytest.mark.parametrize("seed,T,K,E,L,bs", [
    (0, 1, 1, 1, 0, 1), (1, 7, 2, 4, 2, 4), (2, 33, 3, 5, 3, 16), (3, 64, 2, 8, 4, 16),
    (4, 50, 4, 3, 1, 1), (5, 20, 8, 16, 6, 8), (7, 40, 2, 2, 0, 5), (8, 25, 6, 3, 7, 64),
    (9, 5000, 8, 64, 8, 16), (10, 4097, 8, 256, 4, 64), (11, 1000, 1, 1, 0, 16),
    (12, 30000, 2, 2, 1, 16), (13, 3, 4, 100, 399, 4096),
    # the limits of the single-block path: 16384 pairs, 8192 buckets (and one past each)
    (14, 2048, 8, 64, 7, 16), (15, 2049, 8, 64, 7, 16), (16, 100, 4, 128, 63, 16),
    (17, 100, 4, 128, 64, 16), (18, 4096, 8, 64, 7, 16),
])
def test_random_cases(cuda_device, seed, T, K, E, L, bs):
    topk, mapping = _random(seed, T, K, E, L, distinct=(seed % 2 == 0))
    _compare(cuda_device, topk, mapping, E, L, bs)


def test_empty_batch(cuda_device):
    topk = np.zeros((0, 8), np.int32)
    assert _compare(cuda_device, topk, np.zeros(0, np.int32), 16, 4, 16) == 0


def test_single_bucket_long_runs(cuda_device):
    # every pair in one bucket: the longest possible runs inside a chunk
    T, K = 40000, 2
    topk = np.zeros((T, K), np.int32)
    _compare(cuda_device, topk, np.full(T, 1, np.int32), 1, 2, 16)


def test_single_bucket_long_runs_one_block(cuda_device):
    # 16384 pairs in one bucket: every round of the single-block path is one run
    T, K = 8192, 2
    topk = np.zeros((T, K), np.int32)
    _compare(cuda_device, topk, np.full(T, 0, np.int32), 1, 1, 16)


def test_all_minus_one(cuda_device):
    topk, _ = _random(21, 3000, 8, 32, 4)
    _compare(cuda_device, topk, np.full(3000, -1, np.int32), 32, 4, 16)


@pytest.mark.parametrize("name", ["tiny", "qwen_moe_prefill", "decode", "deepseek_v3_prefill",
                                  "metadata_stress"])
def test_workload_routings(cuda_device, name):
    cfg = workloads.CONFIGS[name]
    b = workloads.make_batch(cfg, device=cuda_device, seed=0)
    st, mapping, _ = oracle.batch_info(b.seg_indptr.cpu().numpy(), b.weight_indices.cpu().numpy(),
                                       b.lora_ranks.cpu().numpy(), cfg.num_tokens)
    assert st == oracle.OK
    _compare(cuda_device, b.topk_ids.cpu().numpy(), mapping, cfg.num_experts, cfg.num_loras,
             cfg.block_size)


def test_out_of_range_ids_raise(cuda_device):
    topk = torch.tensor([[0, 1], [9, 2]], dtype=torch.int32, device=cuda_device)
    mp = torch.tensor([0, 1], dtype=torch.int32, device=cuda_device)
    with pytest.raises(mlr.MoeLoraError, match="id out of range"):
        mlr.moe_lora_align(topk, mp, 8, 4, 4)
    topk = torch.tensor([[0, 1], [3, 2]], dtype=torch.int32, device=cuda_device)
    mp = torch.tensor([0, 4], dtype=torch.int32, device=cuda_device)
    with pytest.raises(mlr.MoeLoraError, match="id out of range"):
        mlr.moe_lora_align(topk, mp, 8, 4, 4)


def test_capacity_too_small_is_reported_and_bounded(cuda_device):
    topk, mapping = _random(3, 64, 2, 8, 4)
    st, s, *_, n = oracle.align(topk, mapping, 8, 4, 16)
    small = n - 16
    out = (torch.full((small + 64,), -7, dtype=torch.int32, device=cuda_device),
           torch.full((small // 16 + 8,), -7, dtype=torch.int32, device=cuda_device),
           torch.full((small // 16 + 8,), -7, dtype=torch.int32, device=cuda_device),
           torch.zeros(1, dtype=torch.int32, device=cuda_device))
    lib = mlr.library()
    import ctypes
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ws = torch.empty(mlr.moe_lora_align_workspace_bytes(64, 2, 8, 4, 16), dtype=torch.uint8,
                     device=cuda_device)
    t_topk = torch.from_numpy(topk).to(cuda_device)
    t_map = torch.from_numpy(mapping).to(cuda_device)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = lib.moe_lora_align(p(t_topk), p(t_map), 64, 2, 8, 4, 16, p(out[0]), p(out[1]), p(out[2]),
                              p(out[3]), small, p(ws), ws.numel(), p(status),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    assert status.item() & 0x08
    assert torch.all(out[0][small:] == -7)          # nothing written at or past capacity
    assert torch.all(out[1][small // 16:] == -7)
