"""Pins for the oracle's batch-info expand (CPU only).

The worked example and the under-coverage case come from the sglang PR #24160
page (section 关键源码片段, test_moe_lora_info.py); random cases are checked
against torch.repeat_interleave and the page's scatter rule written with torch
ops, both independent of the oracle's C loops.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "batch_info_worked_example.json")


def _gold():
    with open(GOLD) as f:
        return json.load(f)


def _indptr(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def test_worked_example_matches_page():
    g = _gold()
    ip = _indptr(g["seg_lens"])
    st, mapping, enabled = oracle.batch_info(ip, g["weight_indices"], g["lora_ranks"],
                                             int(ip[-1]), max_len=max(g["seg_lens"]))
    assert st == oracle.OK
    assert mapping.tolist() == g["expected_token_lora_mapping"]
    assert enabled.tolist() == g["expected_adapter_enabled"]


def test_worked_example_matches_page_rules_via_torch():
    g = _gold()
    wi = torch.tensor(g["weight_indices"], dtype=torch.int32)
    lens = torch.tensor(g["seg_lens"], dtype=torch.int32)
    ranks = torch.tensor(g["lora_ranks"], dtype=torch.int32)
    exp_map = torch.repeat_interleave(wi, lens)
    exp_en = torch.zeros_like(ranks).scatter_(0, wi.long(), (ranks[wi.long()] > 0).int())
    assert exp_map.tolist() == g["expected_token_lora_mapping"]
    assert exp_en.tolist() == g["expected_adapter_enabled"]


def test_undercovered_launch_rejected():
    u = _gold()["undercovered"]
    st, _, _ = oracle.batch_info(u["seg_indptr"], u["weight_indices"], u["lora_ranks"],
                                 u["num_tokens"], max_len=u["max_len"])
    assert st == oracle.UNDERCOVERED


def test_segment_longer_than_hint_rejected():
    # bs * max_len covers the tokens, but one segment is longer than the hint.
    st, _, _ = oracle.batch_info([0, 1, 5], [0, 0], [8], 5, max_len=3)
    assert st == oracle.UNDERCOVERED
    st, _, _ = oracle.batch_info([0, 1, 5], [0, 0], [8], 5, max_len=4)
    assert st == oracle.OK


@pytest.mark.parametrize("seed", range(6))
def test_random_matches_repeat_interleave_and_scatter(seed):
    g = torch.Generator().manual_seed(seed)
    bs = int(torch.randint(1, 40, (1,), generator=g))
    L = int(torch.randint(1, 12, (1,), generator=g))
    lens = torch.randint(0, 30, (bs,), generator=g).int()
    wi = torch.randint(0, L, (bs,), generator=g).int()
    ranks = torch.randint(0, 3, (L,), generator=g).int() * 8
    ip = _indptr(lens.numpy())
    T = int(ip[-1])
    st, mapping, enabled = oracle.batch_info(ip, wi.numpy(), ranks.numpy(), T)
    assert st == oracle.OK
    assert mapping.tolist() == torch.repeat_interleave(wi, lens).tolist()
    exp_en = torch.zeros_like(ranks).scatter_(0, wi.long(), (ranks[wi.long()] > 0).int())
    assert enabled.tolist() == exp_en.tolist()


def test_minus_one_adapter_maps_to_minus_one_and_is_skipped():
    # Reading: -1 (no adapter) is copied into the mapping and leaves adapter_enabled alone.
    ip = _indptr([3, 2, 4])
    st, mapping, enabled = oracle.batch_info(ip, [-1, 1, -1], [16, 8, 4], 9)
    assert st == oracle.OK
    assert mapping.tolist() == [-1, -1, -1, 1, 1, -1, -1, -1, -1]
    assert enabled.tolist() == [0, 1, 0]


def test_empty_batch_and_zero_loras():
    st, mapping, enabled = oracle.batch_info([0], [], [], 0)
    assert st == oracle.OK and mapping.size == 0 and enabled.size == 0
    st, mapping, enabled = oracle.batch_info([0, 0, 0], [1, 0], [4, 0], 0)
    assert st == oracle.OK and mapping.size == 0 and enabled.tolist() == [1, 0]


@pytest.mark.parametrize("ip,wi,T", [
    ([1, 4], [0], 4),        # does not start at 0
    ([0, 4, 3], [0, 0], 3),  # decreasing
    ([0, 4], [0], 5),        # does not end at num_tokens
])
def test_bad_indptr_invalid(ip, wi, T):
    st, _, _ = oracle.batch_info(ip, wi, [8], T)
    assert st == oracle.INVALID


@pytest.mark.parametrize("bad", [1, 5, -2])
def test_out_of_range_adapter(bad):
    st, _, _ = oracle.batch_info([0, 2], [bad], [8], 2)
    assert st == oracle.INDEX
