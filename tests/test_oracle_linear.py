"""Pins of the oracle's dense projection with per-segment LoRA and split B.

The page (DeepSeek-V3 MLA fused projection, ReplicatedLinearWithLoRA) applies
LoRA to the fused q_a_proj + kv_a_proj_with_mqa projection with its B split
into two parts, each applied to its own part's shrink.  Each pin below fails
for a plausible mistake: a part reading the other part's z, a dropped or
doubled scaling, rank padding read, the adapter rule inverted.
"""
import numpy as np
import pytest

import oracle


def test_worked_example_by_hand():
    # x = [1, 2]; W rows [1,0], [0,1], [1,1] -> base [1, 2, 3]
    # part 0 (rows 0-1): A = [1, 1] -> z0 = 3;  part 1 (row 2): A = [1, -2] -> z1 = -3
    # B rows [2], [-1], [4]; scaling 0.5:
    #   y0 = 1 + 0.5*2*3 = 4,  y1 = 2 + 0.5*(-1)*3 = 0.5,  y2 = 3 + 0.5*4*(-3) = -3
    x = np.array([[1.0, 2.0]])
    w = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    a = np.array([[[[1.0, 1.0]], [[1.0, -2.0]]]])      # [L=1, S=2, R=1, D_in=2]
    b = np.array([[[2.0], [-1.0], [4.0]]])              # [L=1, D_out=3, R=1]
    st, y = oracle.lora_linear(x, [0], [1], [0.5], w, a, b, [0, 2, 3])
    assert st == 0
    assert y.tolist() == [[4.0, 0.5, -3.0]]
    st, y = oracle.lora_linear(x, [-1], [1], [0.5], w, a, b, [0, 2, 3])
    assert y.tolist() == [[1.0, 2.0, 3.0]]


def _case(seed, T=37, D_in=40, D_out=56, L=3, R=8, offs=(0, 32, 56)):
    g = np.random.default_rng(seed)
    S = len(offs) - 1
    x = g.standard_normal((T, D_in))
    w = g.standard_normal((D_out, D_in))
    a = g.standard_normal((L, S, R, D_in))
    b = g.standard_normal((L, D_out, R))
    ranks = np.array([R, 3, 0][:L], dtype=np.int32)
    scal = np.array([0.25, 1.5, 2.0][:L], dtype=np.float32)
    mapping = g.integers(-1, L, T).astype(np.int32)
    return x, w, a, b, ranks, scal, mapping, list(offs)


def test_no_adapter_reduces_to_the_base_matmul():
    x, w, a, b, ranks, scal, mapping, offs = _case(0)
    st, y = oracle.lora_linear(x, np.full(len(x), -1, np.int32), ranks, scal, w, a, b, offs)
    assert st == 0
    np.testing.assert_allclose(y, x @ w.T, rtol=1e-12, atol=1e-12)


def test_factored_form_equals_the_materialised_weight_per_part():
    x, w, a, b, ranks, scal, mapping, offs = _case(1)
    st, y = oracle.lora_linear(x, mapping, ranks, scal, w, a, b, offs)
    assert st == 0
    for t in range(len(x)):
        l = mapping[t]
        weff = w.copy()
        if l >= 0 and ranks[l] > 0:
            r = ranks[l]
            for s in range(len(offs) - 1):
                o0, o1 = offs[s], offs[s + 1]
                weff[o0:o1] += float(scal[l]) * (b[l, o0:o1, :r] @ a[l, s, :r])
        np.testing.assert_allclose(y[t], weff @ x[t], rtol=1e-10, atol=1e-10)


def test_each_part_reads_only_its_own_A():
    x, w, a, b, ranks, scal, mapping, offs = _case(2)
    mapping[:] = 0  # every token uses the full-rank adapter
    st, y0 = oracle.lora_linear(x, mapping, ranks, scal, w, a, b, offs)
    a2 = a.copy()
    a2[0, 0] += 1.0  # part 0's A only
    st, y1 = oracle.lora_linear(x, mapping, ranks, scal, w, a2, b, offs)
    assert np.abs(y1[:, :offs[1]] - y0[:, :offs[1]]).max() > 1e-3
    assert np.array_equal(y1[:, offs[1]:], y0[:, offs[1]:])


def test_rank_padding_is_not_read_and_rank_zero_is_the_base():
    x, w, a, b, ranks, scal, mapping, offs = _case(3)
    st, y0 = oracle.lora_linear(x, mapping, ranks, scal, w, a, b, offs)
    a2, b2 = a.copy(), b.copy()
    a2[1, :, 3:] = 1e6   # adapter 1 has rank 3: rows >= 3 are padding
    b2[1, :, 3:] = -1e6
    a2[2] = 7.0          # adapter 2 has rank 0
    b2[2] = 7.0
    st, y1 = oracle.lora_linear(x, mapping, ranks, scal, w, a2, b2, offs)
    assert np.array_equal(y0, y1)
    base = x @ w.T
    none = (mapping == -1) | (mapping == 2)
    np.testing.assert_allclose(y0[none], base[none], rtol=1e-12, atol=1e-12)
    assert np.abs(y0[~none] - base[~none]).max() > 1e-3


def test_one_part_is_the_plain_lora_linear_and_scaling_is_linear():
    x, w, a, b, ranks, scal, mapping, offs = _case(4, offs=(0, 56))
    st, y1 = oracle.lora_linear(x, mapping, ranks, scal, w, a, b, offs)
    st, y2 = oracle.lora_linear(x, mapping, ranks, 2 * scal, w, a, b, offs)
    base = x @ w.T
    np.testing.assert_allclose(y2 - base, 2 * (y1 - base), rtol=1e-9, atol=1e-9)


def test_sampled_tokens_and_argument_checks():
    x, w, a, b, ranks, scal, mapping, offs = _case(5)
    st, y = oracle.lora_linear(x, mapping, ranks, scal, w, a, b, offs)
    st, ys = oracle.lora_linear(x, mapping, ranks, scal, w, a, b, offs, tokens=[5, 0, 36])
    assert st == 0 and np.array_equal(ys, y[[5, 0, 36]])
    assert oracle.lora_linear(x, mapping, ranks, scal, w, a, b, [0, 40, 40])[0] == oracle.INVALID
    bad = mapping.copy(); bad[0] = 3
    assert oracle.lora_linear(x, bad, ranks, scal, w, a, b, offs)[0] == oracle.INDEX
