"""Pins for the column-parallel LoRA B rows of a fused q/k/v projection (CPU).

The sglang PR #24420 page fixes two things: the per-rank B output size
(an even split, or 1/tp of q plus one whole head of k and v once tp exceeds
the KV heads) and the rows a rank takes (q shard by rank; k and v shard by
rank // replicas, offset by the full q and k sizes).  Pinned here against:
  * the page's stated sizes for both regimes;
  * an independent head-ownership model (which q heads and which KV head each
    rank owns, turned into rows);
  * coverage: over all ranks every q row is held once and every KV head by
    exactly `replicas` ranks;
  * the projection: for every rank, the projection on its rows of W and B
    equals those columns of the full projection (oracle.lora_linear);
and the library's host function against the oracle, with its argument checks.
"""
import ctypes

import numpy as np
import pytest

import lora_moe_expert_info_gb300 as mlr
import oracle

CASES = [(32, 8, 128, tp) for tp in (1, 2, 4, 8, 16, 32)] + \
        [(8, 2, 64, tp) for tp in (1, 2, 4, 8)] + [(28, 4, 128, tp) for tp in (1, 2, 4)] + \
        [(64, 1, 64, tp) for tp in (1, 2, 8, 64)] + [(12, 12, 16, tp) for tp in (1, 2, 3, 4, 6, 12)]


def heads_model(nh, nkv, hd, tp, r):
    """Rows from head ownership: rank r owns q heads [r*nh/tp, (r+1)*nh/tp) and
    KV heads [r*nkv/tp, ...) when tp <= nkv, else KV head r // (tp / nkv)."""
    q_heads = range(r * nh // tp, (r + 1) * nh // tp)
    if tp <= nkv:
        kv_heads = range(r * nkv // tp, (r + 1) * nkv // tp)
    else:
        kv_heads = [r // (tp // nkv)]
    q_rows = [h * hd + i for h in q_heads for i in range(hd)]
    k_rows = [nh * hd + j * hd + i for j in kv_heads for i in range(hd)]
    v_rows = [nh * hd + nkv * hd + j * hd + i for j in kv_heads for i in range(hd)]
    return q_rows + k_rows + v_rows


def rows_of(ranges):
    return [i for a, b in ranges for i in range(a, b)]


@pytest.mark.parametrize("nh,nkv,hd,tp", CASES)
def test_rows_match_head_ownership(nh, nkv, hd, tp):
    for r in range(tp):
        ranges, n = oracle.tp_qkv_b_rows(nh, nkv, hd, tp, r)
        assert rows_of(ranges) == heads_model(nh, nkv, hd, tp, r)
        assert n == len(rows_of(ranges))


@pytest.mark.parametrize("nh,nkv,hd,tp", CASES)
def test_page_sizes_and_coverage(nh, nkv, hd, tp):
    total = (nh + 2 * nkv) * hd
    count = np.zeros(total, np.int64)
    for r in range(tp):
        ranges, n = oracle.tp_qkv_b_rows(nh, nkv, hd, tp, r)
        assert n == (total // tp if tp <= nkv else nh * hd // tp + 2 * hd)
        count[rows_of(ranges)] += 1
    q = nh * hd
    assert (count[:q] == 1).all()
    assert (count[q:] == max(1, tp // nkv)).all()


def test_invalid_splits():
    assert oracle.tp_qkv_b_rows(28, 8, 128, 4, 0) is not None
    assert oracle.tp_qkv_b_rows(30, 8, 128, 8, 0) is None      # 30 q heads over 8 ranks
    assert oracle.tp_qkv_b_rows(32, 6, 128, 4, 0) is None      # neither 4 | 6 nor 6 | 4
    assert oracle.tp_qkv_b_rows(32, 8, 128, 4, 4) is None      # rank out of range


@pytest.mark.parametrize("nh,nkv,hd,tp", CASES)
def test_library_matches_oracle(nh, nkv, hd, tp):
    for r in range(tp):
        assert mlr.lora_tp_qkv_b_rows(nh, nkv, hd, tp, r) == oracle.tp_qkv_b_rows(nh, nkv, hd, tp, r)


def test_library_argument_checks():
    lib = mlr.library()
    out = (ctypes.c_int32 * 6)()
    n = ctypes.c_int32(0)
    f = lib.lora_tp_qkv_b_rows
    assert f(32, 8, 128, 8, 0, out, ctypes.byref(n)) == 0
    assert f(30, 8, 128, 8, 0, out, ctypes.byref(n)) == mlr.MLR_ERR_INVALID
    assert f(32, 6, 128, 4, 0, out, ctypes.byref(n)) == mlr.MLR_ERR_INVALID
    assert f(32, 8, 128, 4, 4, out, ctypes.byref(n)) == mlr.MLR_ERR_INVALID
    assert f(32, 8, 128, 4, -1, out, ctypes.byref(n)) == mlr.MLR_ERR_INVALID
    assert f(32, 8, 0, 4, 0, out, ctypes.byref(n)) == mlr.MLR_ERR_INVALID
    assert f(32, 8, 128, 4, 0, None, ctypes.byref(n)) == mlr.MLR_ERR_INVALID


@pytest.mark.parametrize("tp", [2, 4])
def test_rank_projection_is_a_column_block_of_the_full_one(tp):
    # 8 q heads, 2 KV heads of 16: tp 2 splits the KV heads, tp 4 replicates them
    nh, nkv, hd, D_in, T, L, R = 8, 2, 16, 40, 12, 2, 4
    D = (nh + 2 * nkv) * hd
    rng = np.random.default_rng(tp)
    x = rng.standard_normal((T, D_in))
    w = rng.standard_normal((D, D_in))
    a = rng.standard_normal((L, 1, R, D_in))
    b = rng.standard_normal((L, D, R))
    mapping = rng.integers(-1, L, T).astype(np.int32)
    ranks = np.array([4, 2], np.int32)
    scal = np.array([0.5, 2.0], np.float32)
    st, y = oracle.lora_linear(x, mapping, ranks, scal, w, a, b, [0, D])
    assert st == oracle.OK
    for r in range(tp):
        ranges, n = oracle.tp_qkv_b_rows(nh, nkv, hd, tp, r)
        rows = rows_of(ranges)
        st, yr = oracle.lora_linear(x, mapping, ranks, scal, w[rows], a, b[:, rows], [0, n])
        assert st == oracle.OK
        np.testing.assert_allclose(yr, y[:, rows], rtol=1e-12, atol=1e-12)


def test_take_rows_helper_matches_index_selection():
    import torch
    ranges, n = mlr.lora_tp_qkv_b_rows(8, 2, 16, 4, 3)
    b = torch.arange(3 * 192 * 4, dtype=torch.float32).reshape(3, 192, 4)
    rows = rows_of(ranges)
    assert torch.equal(mlr.tp_take_rows(b, ranges, dim=1), b[:, rows])
    assert mlr.tp_take_rows(b[0], ranges, dim=0).shape == (n, 4)
