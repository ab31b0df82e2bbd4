"""Pins for the oracle's (lora, expert) align (CPU only).

The page (sglang PR #14105, section 实现拆解) says only that the align kernel
sorts tokens by LoRA adapter and expert id and pads to block_size.  The oracle
is pinned by brute force -- Python's stable sorted() on the key
(expert, adapter + 1, pair index) plus the padding rule -- and by the
invariants every valid output must satisfy.
"""
import ctypes

import numpy as np
import pytest

import oracle


def brute_force(topk_ids, mapping, E, L, bs):
    T, K = topk_ids.shape
    P = T * K
    key = lambda p: (int(topk_ids[p // K, p % K]), int(mapping[p // K]) + 1, p)
    order = sorted(range(P), key=key)
    out, bexp, blora = [], [], []
    i = 0
    while i < P:
        e, c, _ = key(order[i])
        j = i
        while j < P and key(order[j])[:2] == (e, c):
            j += 1
        run = order[i:j]
        padded = -(-len(run) // bs) * bs
        out += run + [P] * (padded - len(run))
        bexp += [e] * (padded // bs)
        blora += [c - 1] * (padded // bs)
        i = j
    return out, bexp, blora, len(out)


def _case(seed, T, K, E, L, p_none=0.2):
    rng = np.random.default_rng(seed)
    topk = np.stack([rng.choice(E, size=K, replace=K > E) for _ in range(T)]).astype(np.int32) \
        if T > 0 else np.zeros((0, K), np.int32)
    mapping = rng.integers(0, L, size=T).astype(np.int32) if L > 0 else np.full(T, -1, np.int32)
    mapping[rng.random(T) < p_none] = -1
    return topk.reshape(T, K), mapping


@pytest.mark.parametrize("seed,T,K,E,L,bs", [
    (0, 1, 1, 1, 0, 1),
    (1, 7, 2, 4, 2, 4),
    (2, 33, 3, 5, 3, 16),
    (3, 64, 2, 8, 4, 16),
    (4, 50, 4, 3, 1, 1),
    (5, 20, 8, 16, 6, 8),
    (6, 0, 2, 4, 2, 16),
    (7, 40, 2, 2, 0, 5),
    (8, 25, 6, 3, 7, 64),
])
def test_matches_brute_force(seed, T, K, E, L, bs):
    topk, mapping = _case(seed, T, K, E, L)
    st, s, be, bl, n = oracle.align(topk, mapping, E, L, bs)
    assert st == oracle.OK
    ref_s, ref_be, ref_bl, ref_n = brute_force(topk, mapping, E, L, bs)
    assert n == ref_n
    assert s.tolist() == ref_s
    assert be.tolist() == ref_be
    assert bl.tolist() == ref_bl


def test_duplicate_experts_within_a_token():
    # topk_ids need not be distinct per token: ties fall back to ascending k.
    topk = np.array([[1, 1, 0], [0, 1, 1]], np.int32)
    mapping = np.array([0, 0], np.int32)
    st, s, be, bl, n = oracle.align(topk, mapping, 2, 1, 2)
    assert st == oracle.OK
    ref = brute_force(topk, mapping, 2, 1, 2)
    assert (s.tolist(), be.tolist(), bl.tolist(), n) == ref


def test_invariants_medium():
    T, K, E, L, bs = 3000, 8, 64, 8, 16
    topk, mapping = _case(11, T, K, E, L)
    st, s, be, bl, n = oracle.align(topk, mapping, E, L, bs)
    assert st == oracle.OK
    P = T * K
    assert n % bs == 0 and n <= oracle.align_capacity(T, K, E, L, bs)
    # multiset of real ids is exactly {0..P-1}
    real = s[s != P]
    assert np.array_equal(np.sort(real), np.arange(P))
    # every block holds a single (expert, lora) and only pairs with that key
    blocks = s.reshape(-1, bs)
    for b in range(blocks.shape[0]):
        ids = blocks[b][blocks[b] != P]
        assert ids.size > 0
        assert np.all(topk.reshape(-1)[ids] == be[b])
        assert np.all(mapping[ids // K] == bl[b])
        assert np.all(np.diff(ids) > 0)  # stable: ascending pair index
    # padding lies only at bucket tails and is < bs per bucket
    keys = be.astype(np.int64) * (L + 1) + bl + 1
    assert np.all(np.diff(keys) >= 0)
    for k in np.unique(keys):
        seg = blocks[keys == k].reshape(-1)
        npad = int(np.sum(seg == P))
        assert npad < bs and np.all(seg[seg.size - npad:] == P)


@pytest.mark.parametrize("bad_e,bad_l", [(8, 0), (-1, 0), (0, 4), (0, -2)])
def test_out_of_range_ids(bad_e, bad_l):
    topk = np.array([[0, 1], [bad_e, 2]], np.int32)
    mapping = np.array([0, bad_l], np.int32)
    st, *_ = oracle.align(topk, mapping, 8, 4, 4)
    assert st == oracle.INDEX


def test_capacity_too_small():
    topk, mapping = _case(3, 64, 2, 8, 4)
    st, s, *_ , n = oracle.align(topk, mapping, 8, 4, 16)
    assert st == oracle.OK
    lib = oracle._load()
    out = np.zeros(n, np.int32)
    blk = np.zeros(n // 16, np.int32)
    blk2 = np.zeros(n // 16, np.int32)
    npad = np.zeros(1, np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    st = lib.oracle_align(p(np.ascontiguousarray(topk)), p(mapping), 64, 2, 8, 4, 16,
                          p(out), p(blk), p(blk2), p(npad), n - 1)
    assert st == oracle.CAPACITY


def test_capacity_bound_formula():
    # P + min(P, buckets) * (bs - 1), rounded up to bs
    assert oracle.align_capacity(64, 2, 8, 4, 16) == -(-(128 + 40 * 15) // 16) * 16
    assert oracle.align_capacity(1, 1, 100, 100, 16) == 16
    assert oracle.align_capacity(0, 8, 4, 4, 16) == 0
