"""GPU parity of lora_linear_forward (dense projection with per-segment LoRA and
split B, the MLA fused q_a_proj + kv_a_proj projection) against the oracle.

Tolerance as for the layer: |y - y_ref| <= 2e-2 + 2e-2*|y_ref| elementwise,
y_ref from the fp64 oracle.  The LoRA factors are drawn at fan-in scale with
scaling 0.5, so that the LoRA delta is O(1) and a part reading the wrong rank
block, a dropped scaling or a lost segment exceeds the tolerance.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle

pytestmark = pytest.mark.gpu
ATOL = RTOL = 2e-2


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def within(y, yref):
    err = np.abs(y - yref) - (ATOL + RTOL * np.abs(yref))
    return float(err.max()) if err.size else -1.0


class Lin:
    def __init__(self, dev, T, D_in, offs, L, R, ranks, seg_lens, adapters, seed=0):
        g = torch.Generator(device=dev).manual_seed(seed)
        D_out, S = offs[-1], len(offs) - 1
        bf = torch.bfloat16
        self.x = torch.randn(T, D_in, generator=g, device=dev, dtype=bf)
        self.w = torch.randn(D_out, D_in, generator=g, device=dev, dtype=bf).mul_(D_in ** -0.5)
        self.a = torch.randn(L, S, R, D_in, generator=g, device=dev, dtype=bf).mul_(D_in ** -0.5)
        self.b = torch.randn(L, D_out, R, generator=g, device=dev, dtype=bf).mul_(max(R, 1) ** -0.5)
        self.ranks = torch.tensor(ranks, dtype=torch.int32, device=dev)
        self.scal = torch.tensor([0.0 if r == 0 else 0.5 for r in ranks], dtype=torch.float32, device=dev)
        mp = np.repeat(np.asarray(adapters, np.int32), np.asarray(seg_lens))
        assert mp.shape == (T,)
        self.mapping_np = mp
        self.mapping = torch.from_numpy(mp).to(dev)
        self.offs = list(offs)

    def gpu(self, mapping=None):
        m = self.mapping if mapping is None else torch.from_numpy(np.ascontiguousarray(mapping)).to(self.x.device)
        return mlr.lora_linear_forward(self.x, self.w, m, self.ranks, self.scal, self.a, self.b,
                                       self.offs).float().cpu().numpy()

    def ref(self, mapping=None, tokens=None):
        m = self.mapping_np if mapping is None else mapping
        st, y = oracle.lora_linear(bits(self.x), m, self.ranks.cpu().numpy(), self.scal.cpu().numpy(),
                                   bits(self.w), bits(self.a), bits(self.b), self.offs, tokens=tokens)
        assert st == 0
        return y


def test_mla_shaped_two_parts(cuda_device):
    c = Lin(cuda_device, T=150, D_in=256, offs=[0, 256, 576], L=3, R=32, ranks=[32, 8, 0],
            seg_lens=[40, 25, 60, 25], adapters=[0, -1, 1, 2])
    none = np.full(150, -1, np.int32)
    y, y0 = c.gpu(), c.gpu(mapping=none)
    r, r0 = c.ref(), c.ref(mapping=none)
    assert np.abs(r - r0).max() > 0.5  # the LoRA delta is large enough to be seen
    assert within(y, r) <= 0 and within(y0, r0) <= 0


def test_one_part_ragged_sizes(cuda_device):
    c = Lin(cuda_device, T=203, D_in=200, offs=[0, 136], L=2, R=16, ranks=[16, 5],
            seg_lens=[17, 90, 96], adapters=[1, 0, -1], seed=1)
    assert within(c.gpu(), c.ref()) <= 0


def test_second_part_reads_its_own_A(cuda_device):
    c = Lin(cuda_device, T=64, D_in=128, offs=[0, 256, 384], L=1, R=16, ranks=[16],
            seg_lens=[64], adapters=[0], seed=2)
    y0 = c.gpu()
    c.a[0, 1] += 0.25  # part 1's A only
    y1 = c.gpu()
    assert np.abs(y1[:, 256:] - y0[:, 256:]).max() > 0.1
    assert np.array_equal(y1[:, :256], y0[:, :256])
    assert within(y1, c.ref()) <= 0


def test_mla_projection_full_size_sampled(cuda_device):
    # DeepSeek-V3 MLA: hidden 7168 -> q_a 1536 + kv_a (with the rope part) 576
    c = Lin(cuda_device, T=512, D_in=7168, offs=[0, 1536, 2112], L=4, R=64, ranks=[16, 32, 64, 64],
            seg_lens=[128, 128, 128, 128], adapters=[0, 1, 2, 3], seed=3)
    y = c.gpu()
    toks = np.sort(np.random.default_rng(3).choice(512, 48, replace=False))
    assert within(y[toks], c.ref(tokens=toks)) <= 0
    assert np.isfinite(y).all()


def test_chunked_align_path(cuda_device):
    # more than 16,384 tokens: the align runs in chunks instead of one block
    T = 36000
    c = Lin(cuda_device, T=T, D_in=128, offs=[0, 256], L=3, R=16, ranks=[16, 8, 16],
            seg_lens=[9000, 12600, 5400, 9000], adapters=[2, -1, 0, 1], seed=4)
    y = c.gpu()
    toks = np.sort(np.random.default_rng(4).choice(T, 64, replace=False))
    toks = np.concatenate([[0, T - 1], toks])
    assert within(y[toks], c.ref(tokens=toks)) <= 0


def test_no_adapters_and_empty_batch(cuda_device):
    c = Lin(cuda_device, T=40, D_in=128, offs=[0, 128], L=0, R=0, ranks=[], seg_lens=[40], adapters=[-1], seed=5)
    assert within(c.gpu(), c.ref()) <= 0
    e = Lin(cuda_device, T=0, D_in=128, offs=[0, 128], L=1, R=16, ranks=[8], seg_lens=[0], adapters=[0], seed=6)
    assert e.gpu().shape == (0, 128)
