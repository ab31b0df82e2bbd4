"""Pins of the expert-parallel oracle (oracle/ep.py) on CPU.

The dispatch order is checked against a brute-force enumeration (for each rank,
the pairs it owns listed in increasing index), pair_pos against the order it
inverts, and the combine against the per-token sum of a reshaped array.  The
whole protocol (dispatch, per-owner forward over its own experts with top-1
routing, combine) is checked against the oracle's single-process layer.
"""
import numpy as np
import pytest

import oracle
from oracle import ep as oep


def _brute_order(ids, E, n):
    per = E // n
    flat = np.asarray(ids).reshape(-1)
    order = []
    for d in range(n):
        order += [p for p in range(flat.size) if 0 <= flat[p] < E and flat[p] // per == d]
    return order


@pytest.mark.parametrize("T,K,E,n,seed", [(50, 2, 8, 2, 0), (37, 4, 16, 4, 1), (5, 8, 64, 8, 2), (0, 2, 4, 2, 3),
                                          (64, 1, 6, 3, 4), (20, 3, 8, 1, 5)])
def test_dispatch_order_matches_brute_force(T, K, E, n, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, (T, K)).astype(np.int32)
    st, order, counts, pos = oep.ep_dispatch(ids, E, n)
    assert st == oep.OK
    assert order.tolist() == _brute_order(ids, E, n)
    per = E // n
    assert counts.tolist() == [int(np.sum(ids // per == d)) for d in range(n)]
    for q, p in enumerate(order):
        assert pos[p] == q
    assert np.all(pos >= 0)


def test_dropped_pairs():
    ids = np.array([[0, 9], [-1, 3], [5, 2]], dtype=np.int32)
    st, order, counts, pos = oep.ep_dispatch(ids, 8, 2)
    assert st == oep.INDEX
    # rank 0 owns experts 0-3: pairs 0 (e 0), 3 (e 3), 5 (e 2); rank 1 owns 4-7: pair 4 (e 5)
    assert order.tolist() == [0, 3, 5, 4]
    assert counts.tolist() == [3, 1]
    assert pos.tolist() == [0, -1, -1, 1, 3, 2]


def test_uneven_split_is_refused():
    st, *_ = oep.ep_dispatch(np.zeros((2, 2), np.int32), 10, 4)
    assert st != oep.OK


def test_combine_identity_order_is_the_token_sum():
    rng = np.random.default_rng(7)
    T, K, H = 6, 3, 5
    rows = rng.standard_normal((T * K, H))
    y = oep.ep_combine(rows, np.arange(T * K), T, K)
    assert np.allclose(y, rows.reshape(T, K, H).sum(1), rtol=0, atol=1e-14)
    pos = np.arange(T * K)
    pos[4] = -1
    y2 = oep.ep_combine(rows, pos, T, K)
    assert np.allclose(y2[1], rows[3] + rows[5])


def _bits(a):
    import torch
    return a.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("n", [2, 4])
def test_protocol_equals_the_layer(n):
    """Every owner runs the oracle layer on its received rows with top-1 routing
    over its experts; the combined rows equal the layer over all experts."""
    import torch
    from lora_moe_expert_info_gb300 import workloads
    cfg = workloads.custom_config(hidden=64, intermediate=32, num_experts=8, topk=2, num_loras=3, max_rank=16,
                                  num_tokens=30)
    ranks = np.array([8, 0, 16], dtype=np.int32)
    scal = np.array([0.5, 0.0, 0.5], dtype=np.float32)
    w = workloads.make_weights(cfg, torch.from_numpy(ranks), seed=3, lora_std="fan_in")
    g = torch.Generator().manual_seed(4)
    x = torch.randn(30, 64, generator=g).to(torch.bfloat16)
    ids, wts = workloads.route(30, 8, 2, g, "cpu")
    mapping = torch.randint(-1, 3, (30,), generator=g).int().numpy()
    keys = ("w_gate_up", "w_down", "lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")
    dims = (0, 0, 1, 1, 1, 1)
    st, y_ref = oracle.forward(_bits(x), ids.numpy(), wts.numpy(), mapping, ranks, scal,
                               *[_bits(getattr(w, k)) for k in keys])
    assert st == 0
    st, order, counts, pos = oep.ep_dispatch(ids.numpy(), 8, n)
    assert st == oep.OK
    per = 8 // n
    flat_ids, flat_w = ids.numpy().reshape(-1), wts.numpy().reshape(-1)
    rows = np.zeros((order.size, 64))
    start = 0
    for d in range(n):
        sel = order[start:start + counts[d]]
        local = [_bits(getattr(w, k).narrow(dim, d * per, per)) for k, dim in zip(keys, dims)]
        st, yr = oracle.forward(_bits(x)[sel // 2], (flat_ids[sel] - d * per).reshape(-1, 1),
                                flat_w[sel].reshape(-1, 1), mapping[sel // 2], ranks, scal, *local)
        assert st == 0
        rows[start:start + counts[d]] = yr
        start += counts[d]
    y = oep.ep_combine(rows, pos, 30, 2)
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12)
