"""x_sorted for batches whose dense rows stream more than twice the L2
(P x H x 2 bytes > 256 MB): the forward first finds each pair's dense row and
then writes x_sorted token by token, each row of x read once for its K pairs.
Checked against the oracle on sampled tokens, with top-k above one warp's 32
lanes (a token's pairs in two tasks) and with a pair whose expert id is out of
range (reported, dropped, and its token's other pair still computed), for the
bf16 and the W8A8 layers."""
import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle
from lora_moe_expert_info_gb300 import workloads
from test_gpu_forward import WKEYS, bits, custom_case, within

pytestmark = pytest.mark.gpu

CASES = {
    # T, K, E: P * H * 2 = 268 MB and 335 MB with H = 4096
    "k8": dict(T=4096, K=8, E=8),
    "k40": dict(T=1024, K=40, E=48),
}


def _case(dev, T, K, E, seed=11):
    return custom_case(dev, T=T, K=K, E=E, H=4096, I=128, L=2, R=16, ranks=[16, 8],
                       seg_lens=[T // 2, T - T // 2], adapters=[0, 1], lora_std="fan_in", seed=seed)


def _run(c, ids, w8a8, status):
    args = dict(topk_ids=ids, topk_weights=c.b.topk_weights,
                token_lora_mapping=torch.from_numpy(np.ascontiguousarray(c.mapping)).to(c.dev),
                lora_ranks=c.b.lora_ranks, scalings=c.scal)
    lo = {k: getattr(c.w, k) for k in ("lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")}
    if w8a8:
        q = workloads.make_fp8_w8a8_experts(c.cfg, device=c.dev, seed=3)
        y = mlr.fused_moe_lora_forward_fp8_w8a8(c.x, args["topk_ids"], args["topk_weights"],
                                                args["token_lora_mapping"], args["lora_ranks"], args["scalings"],
                                                q.w_gate_up_q, q.w_gate_up_exp, q.w_down_q, q.w_down_exp, **lo,
                                                check=False, status=status)
        return y.float().cpu().numpy(), q
    y = mlr.fused_moe_lora_forward(x=c.x, **args, w_gate_up=c.w.w_gate_up, w_down=c.w.w_down, **lo, check=False,
                                   status=status)
    return y.float().cpu().numpy(), None


def _ref(c, ids, wts, toks, q):
    common = (bits(c.x), ids.cpu().numpy(), wts.cpu().numpy(), c.mapping, c.b.lora_ranks.cpu().numpy(),
              c.scal.cpu().numpy())
    if q is None:
        st, r = oracle.forward(*common, *[bits(getattr(c.w, k)) for k in WKEYS], tokens=toks)
    else:
        np_ = lambda t: t.cpu().numpy()  # noqa: E731
        lo = [bits(getattr(c.w, k)) for k in ("lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")]
        st, r = oracle.forward_fp8_w8a8(*common, np_(q.w_gate_up_q), np_(q.w_gate_up_exp), np_(q.w_down_q),
                                        np_(q.w_down_exp), *lo, tokens=toks)
    assert st == 0
    return r


@pytest.mark.parametrize("w8a8", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_token_major_gather(cuda_device, name, w8a8):
    c = _case(cuda_device, **CASES[name])
    T, K = c.cfg.num_tokens, c.cfg.topk
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    y, q = _run(c, c.b.topk_ids, w8a8, status)
    assert int(status.item()) == 0
    toks = np.sort(np.random.default_rng(2).choice(T, 24, replace=False))
    toks = np.concatenate([[0, T - 1], toks])
    assert within(y[toks], _ref(c, c.b.topk_ids, c.b.topk_weights, toks, q)) <= 0


@pytest.mark.parametrize("w8a8", [False, True])
def test_token_major_gather_dropped_pair(cuda_device, w8a8):
    c = _case(cuda_device, **CASES["k40"])
    E = c.cfg.num_experts
    ids = c.b.topk_ids.clone()
    ids[5, 33] = E  # out of range: reported and dropped
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    y, q = _run(c, ids, w8a8, status)
    assert int(status.item()) & 0x04
    ids_ok, wts = ids.clone(), c.b.topk_weights.clone()
    ids_ok[5, 33], wts[5, 33] = 0, 0.0
    toks = np.array([0, 4, 5, 6, c.cfg.num_tokens - 1])
    assert within(y[toks], _ref(c, ids_ok, wts, toks, q)) <= 0
