"""Expert parallelism on one GPU by rank emulation, against the oracle.

moe_lora_ep_dispatch is compared bit for bit with the oracle's dispatch order
(send counts, pair positions and every packed row, including dropped pairs).
The whole expert-parallel step is then run for n emulated ranks on one GPU:
each rank has its own batch and only its experts' weights and LoRA stacks; the
all-to-all is emulated by slicing and concatenating the ranks' send buffers
(the ranks never wait on one another), each owner runs fused_moe_lora_forward
with top-1 routing over its local experts, the rows go back the same way and
moe_lora_ep_combine sums them.  Every rank's y must match the oracle's layer
over all experts within |y - y_ref| <= 2e-2 + 2e-2 |y_ref|.
"""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import ep, workloads
from oracle import ep as oep

pytestmark = pytest.mark.gpu
KEYS = ("w_gate_up", "w_down", "lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")
DIMS = (0, 0, 1, 1, 1, 1)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def within(y, yref):
    return float((np.abs(y - yref) - (2e-2 + 2e-2 * np.abs(yref))).max())


@pytest.mark.parametrize("T,K,E,n,H,seed", [(300, 4, 16, 4, 128, 0), (1500, 8, 64, 8, 256, 1), (7, 2, 8, 2, 64, 2),
                                            (0, 2, 8, 2, 64, 3), (5000, 8, 256, 64, 64, 4)])
def test_dispatch_matches_oracle(cuda_device, T, K, E, n, H, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    ids = torch.randint(0, E, (T, K), generator=g, dtype=torch.int32)
    if T > 4:
        ids[1, 0] = E + 2   # dropped
        ids[3, K - 1] = -1  # dropped
    wts = torch.rand(T, K, generator=g)
    mapping = torch.randint(-1, 3, (T,), generator=g, dtype=torch.int32)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    d = cuda_device
    if T > 4:
        with pytest.raises(mlr.MoeLoraError):
            ep.ep_dispatch(x.to(d), ids.to(d), wts.to(d), mapping.to(d), E, n)
    out = ep.ep_dispatch(x.to(d), ids.to(d), wts.to(d), mapping.to(d), E, n, check=False)
    st, order, counts, pos = oep.ep_dispatch(ids.numpy(), E, n)
    assert np.array_equal(out["send_counts"].cpu().numpy(), counts)
    assert np.array_equal(out["pair_pos"].cpu().numpy(), pos)
    m = order.size
    per = E // n
    o = torch.from_numpy(order).long()
    assert torch.equal(out["send_x"][:m].cpu(), x[o // K])
    assert np.array_equal(out["send_expert"][:m].cpu().numpy(), ids.reshape(-1)[o].numpy() % per)
    assert np.array_equal(out["send_weight"][:m].cpu().numpy(), wts.reshape(-1)[o].numpy())
    assert np.array_equal(out["send_lora"][:m].cpu().numpy(), mapping[o // K].numpy())


def _emulated_step(batches, w, E, n, lora_ranks, scalings):
    """The expert-parallel step of n ranks, each batch = (x, ids, wts, mapping)."""
    K = batches[0][1].shape[1]
    disp = [ep.ep_dispatch(x, i, wt, mp, E, n) for x, i, wt, mp in batches]
    counts = [dd["send_counts"].cpu().tolist() for dd in disp]
    starts = [np.concatenate([[0], np.cumsum(c)]).tolist() for c in counts]

    def gather(key, dst):
        return torch.cat([disp[s][key][starts[s][dst]:starts[s][dst] + counts[s][dst]] for s in range(n)])

    rows_back = [[None] * n for _ in range(n)]
    for dst in range(n):
        rx, re, rw, rl = (gather(k, dst) for k in ("send_x", "send_expert", "send_weight", "send_lora"))
        local = {k: ep.local_expert_slice(getattr(w, k), dst, n, dim) for k, dim in zip(KEYS, DIMS)}
        m = rx.shape[0]
        y = mlr.fused_moe_lora_forward(rx, re.view(m, 1), rw.view(m, 1), rl, lora_ranks, scalings, **local)
        off = 0
        for s in range(n):
            rows_back[s][dst] = y[off:off + counts[s][dst]]
            off += counts[s][dst]
    ys = []
    for s, (x, i, wt, mp) in enumerate(batches):
        back = torch.cat(rows_back[s])
        ys.append(ep.ep_combine(back, disp[s]["pair_pos"], x.shape[0], K))
    return ys


@pytest.mark.parametrize("n", [2, 4, 8])
def test_tiny_layer_over_emulated_ranks(cuda_device, n):
    cfg = workloads.CONFIGS["tiny"]
    dev = cuda_device
    b0 = workloads.make_batch(cfg, device=dev, seed=0)
    w = workloads.make_weights(cfg, b0.lora_ranks, device=dev, seed=0, lora_std="fan_in")
    scal = b0.scalings * 0.25
    batches, refs = [], []
    for r in range(n):
        b = workloads.make_batch(cfg, device=dev, seed=r)
        x = workloads.make_x(cfg, device=dev, seed=r)
        _, mp = mlr.moe_lora_batch_info(b.seg_indptr, b.weight_indices, b.lora_ranks, cfg.num_tokens)
        batches.append((x, b.topk_ids, b.topk_weights, mp))
        st, yr = oracle.forward(bits(x), b.topk_ids.cpu().numpy(), b.topk_weights.cpu().numpy(), mp.cpu().numpy(),
                                b.lora_ranks.cpu().numpy(), scal.cpu().numpy(), *[bits(getattr(w, k)) for k in KEYS])
        assert st == 0
        refs.append(yr)
    ys = _emulated_step(batches, w, cfg.num_experts, n, b0.lora_ranks, scal)
    for y, yr in zip(ys, refs):
        assert within(y.float().cpu().numpy(), yr) <= 0


def test_qwen_like_shapes_over_four_ranks(cuda_device):
    # Qwen-MoE-like layer shapes (hidden 2048, intermediate 768, 128 experts
    # top-8, 8 adapters) with 512 tokens per rank
    dev = cuda_device
    cfg = workloads.custom_config(hidden=2048, intermediate=768, num_experts=128, topk=8, num_loras=8,
                                  max_rank=64, num_tokens=512)
    ranks = torch.tensor([8, 16, 32, 64, 8, 16, 32, 64], dtype=torch.int32, device=dev)
    scal = torch.full((8,), 2.0, dtype=torch.float32, device=dev)
    w = workloads.make_weights(cfg, ranks.cpu(), device=dev, seed=5)
    n = 4
    batches, refs, samples = [], [], []
    for r in range(n):
        g = torch.Generator(device=dev).manual_seed(50 + r)
        x = torch.randn(512, 2048, generator=g, device=dev, dtype=torch.bfloat16)
        ids, wts = workloads.route(512, 128, 8, g, dev)
        mp = torch.randint(-1, 8, (512,), generator=g, device=dev, dtype=torch.int32)
        batches.append((x, ids, wts, mp))
        toks = np.sort(np.random.default_rng(r).choice(512, 24, replace=False))
        st, yr = oracle.forward(bits(x), ids.cpu().numpy(), wts.cpu().numpy(), mp.cpu().numpy(), ranks.cpu().numpy(),
                                scal.cpu().numpy(), *[bits(getattr(w, k)) for k in KEYS], tokens=toks)
        assert st == 0
        refs.append(yr)
        samples.append(toks)
    ys = _emulated_step(batches, w, 128, n, ranks, scal)
    for y, yr, toks in zip(ys, refs, samples):
        assert within(y.float().cpu().numpy()[toks], yr) <= 0


def test_ep_host_checks(cuda_device):
    lib = ep._lib()
    assert lib.moe_lora_ep_workspace_bytes(10, 2, 65) == 0
    assert lib.moe_lora_ep_workspace_bytes(10, 2, 4) > 0
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device=cuda_device)
    ids = torch.zeros(4, 2, dtype=torch.int32, device=cuda_device)
    with pytest.raises(ValueError):
        ep.ep_dispatch(x, ids, torch.zeros(4, 2, device=cuda_device), torch.zeros(4, dtype=torch.int32,
                                                                                    device=cuda_device), 10, 4)
