"""GPU parity of moe_lora_batch_info against the oracle (bit-exact int32).

Covers the sglang PR #24160 page's worked example (fresh and preallocated
buffers with its 123/456 canaries and aliasing), its under-coverage case, the
-1 adapter, empty segments, unaligned outputs and the 1,048,576-token
metadata-stress batch.
"""
import json
import os

import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import workloads

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden", "batch_info_worked_example.json")


def _indptr(lens):
    return torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)


def _check(dev, ip, wi, ranks, T, max_len=0):
    st, ref_map, ref_en = oracle.batch_info(ip.numpy(), wi.numpy(), ranks.numpy(), T, max_len)
    assert st == oracle.OK
    en, mp = mlr.moe_lora_batch_info(ip.to(dev), wi.to(dev), ranks.to(dev), T, max_len)
    assert np.array_equal(mp.cpu().numpy(), ref_map)
    assert np.array_equal(en.cpu().numpy(), ref_en)


@pytest.mark.parametrize("prealloc", [False, True])
def test_worked_example(cuda_device, prealloc):
    g = json.load(open(GOLD))
    ip = _indptr(g["seg_lens"]).to(cuda_device)
    wi = torch.tensor(g["weight_indices"], dtype=torch.int32, device=cuda_device)
    ranks = torch.tensor(g["lora_ranks"], dtype=torch.int32, device=cuda_device)
    T = int(ip[-1])
    en_buf = mp_buf = None
    if prealloc:
        pre = g["preallocated"]
        en_buf = torch.full_like(ranks, pre["adapter_enabled_fill"])
        mp_buf = torch.full((T + pre["token_lora_mapping_extra"],), pre["token_lora_mapping_fill"],
                            dtype=torch.int32, device=cuda_device)
    en, mp = mlr.moe_lora_batch_info(ip, wi, ranks, T, max_len=max(g["seg_lens"]),
                                     adapter_enabled=en_buf, token_lora_mapping=mp_buf)
    assert mp.cpu().tolist() == g["expected_token_lora_mapping"]
    assert en.cpu().tolist() == g["expected_adapter_enabled"]
    if prealloc:
        assert mp.data_ptr() == mp_buf.data_ptr() and en.data_ptr() == en_buf.data_ptr()
        tail = mp_buf[T:].cpu()
        assert torch.all(tail == g["preallocated"]["token_lora_mapping_fill"])


def test_undercovered_launch_raises(cuda_device):
    u = json.load(open(GOLD))["undercovered"]
    d = lambda v: torch.tensor(v, dtype=torch.int32, device=cuda_device)
    with pytest.raises(AssertionError, match=u["error_match"]):
        mlr.moe_lora_batch_info(d(u["seg_indptr"]), d(u["weight_indices"]), d(u["lora_ranks"]),
                                u["num_tokens"], max_len=u["max_len"])


def test_segment_longer_than_hint_raises(cuda_device):
    d = lambda v: torch.tensor(v, dtype=torch.int32, device=cuda_device)
    with pytest.raises(AssertionError, match="under-covers tokens"):
        mlr.moe_lora_batch_info(d([0, 1, 5]), d([0, 0]), d([8]), 5, max_len=3)


@pytest.mark.parametrize("seed", range(8))
def test_random_vs_oracle(cuda_device, seed):
    g = torch.Generator().manual_seed(seed)
    bs = int(torch.randint(1, 3000, (1,), generator=g))
    L = int(torch.randint(1, 70, (1,), generator=g))
    lens = torch.randint(0, 60, (bs,), generator=g).int()
    lens[torch.rand(bs, generator=g) < 0.2] = 0          # empty segments
    wi = torch.randint(-1, L, (bs,), generator=g).int()  # includes -1
    ranks = (torch.randint(0, 4, (L,), generator=g) * 8).int()
    ip = _indptr(lens.numpy())
    _check(cuda_device, ip, wi, ranks, int(ip[-1]))


def test_long_segments_and_many_segments_per_tile(cuda_device):
    lens = np.array([5000, 1, 1, 3, 70000, 2] + [1] * 5000, dtype=np.int64)
    L = 16
    wi = torch.tensor(np.random.default_rng(0).integers(-1, L, lens.size), dtype=torch.int32)
    ranks = torch.arange(L, dtype=torch.int32) % 3 * 8
    ip = _indptr(lens)
    _check(cuda_device, ip, wi, ranks, int(ip[-1]))


def test_unaligned_mapping_buffer(cuda_device):
    lens = np.array([3, 9, 1, 20])
    ip = _indptr(lens).to(cuda_device)
    wi = torch.tensor([1, -1, 0, 2], dtype=torch.int32, device=cuda_device)
    ranks = torch.tensor([8, 0, 16], dtype=torch.int32, device=cuda_device)
    buf = torch.full((40,), 777, dtype=torch.int32, device=cuda_device)
    view = buf[1:34]   # 4-byte aligned, not 16-byte aligned
    en, mp = mlr.moe_lora_batch_info(ip, wi, ranks, 33, token_lora_mapping=view)
    assert mp.cpu().tolist() == [1] * 3 + [-1] * 9 + [0] + [2] * 20
    assert buf[0].item() == 777 and torch.all(buf[34:] == 777)
    assert en.cpu().tolist() == [1, 0, 1]


def test_empty(cuda_device):
    d = lambda v: torch.tensor(v, dtype=torch.int32, device=cuda_device)
    en, mp = mlr.moe_lora_batch_info(d([0]), d([]), d([4, 0]), 0)
    assert mp.numel() == 0 and en.cpu().tolist() == [0, 0]


def test_out_of_range_adapter_raises(cuda_device):
    d = lambda v: torch.tensor(v, dtype=torch.int32, device=cuda_device)
    with pytest.raises(mlr.MoeLoraError, match="id out of range"):
        mlr.moe_lora_batch_info(d([0, 2, 4]), d([0, 5]), d([8, 8]), 4)


def test_bad_indptr_raises(cuda_device):
    d = lambda v: torch.tensor(v, dtype=torch.int32, device=cuda_device)
    with pytest.raises(mlr.MoeLoraError, match="bad seg_indptr"):
        mlr.moe_lora_batch_info(d([0, 3, 2]), d([0, 0]), d([8]), 2)


def test_metadata_stress_batch(cuda_device):
    cfg = workloads.CONFIGS["metadata_stress"]
    b = workloads.make_batch(cfg, device=cuda_device, seed=0)
    _check(cuda_device, b.seg_indptr.cpu(), b.weight_indices.cpu(), b.lora_ranks.cpu(),
           cfg.num_tokens, max_len=int(b.seg_lens.max()))
