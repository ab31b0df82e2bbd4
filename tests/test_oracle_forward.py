"""Pins for the oracle's forward (CPU only).

What the sglang PR #14105 page (section 实现拆解) fixes is the layer formula
  y = (W_down + a/r B_d A_d)[SiLU((W_gate + a/r B_g A_g)x) (.) ((W_up + a/r B_u A_u)x)]
applied per selected expert and summed with the top-k weights.  The oracle's
C loops are pinned here against things other than themselves:
  * one expert, top-1, weight 1 is a dense SwiGLU MLP computed with torch
    (F.silu and matmul);
  * the factored LoRA form equals the dense-materialised W + s*B*A (numpy
    matmul) run with the adapter switched off, per adapter class, with garbage
    in the rank padding so that reading past r_l fails;
  * B = 0, adapter -1 and rank 0 all reduce exactly to the base MoE;
  * the top-k combine is linear in the weights, invariant to the order of the
    k slots and to a relabelling of the experts;
  * bf16 operands are widened exactly.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def make(seed, T=12, K=2, E=4, H=24, I=20, L=3, R=6, ranks=(3, 0, 6), scal=(1.5, 2.0, 0.75),
         garbage_pad=False, p_none=0.25):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    topk = np.stack([rng.choice(E, size=K, replace=K > E) for _ in range(T)]).astype(np.int32) \
        if T > 0 else np.zeros((0, K), np.int32)
    w = rng.random((T, K)).astype(np.float32) + 0.1
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    mapping = rng.integers(0, max(L, 1), T).astype(np.int32) if L > 0 else np.full(T, -1, np.int32)
    mapping[rng.random(T) < p_none] = -1
    Wgu = rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)
    Wd = rng.standard_normal((E, H, I)) / np.sqrt(I)
    Agu = rng.standard_normal((L, E, 2, R, H)) / np.sqrt(H)
    Bgu = rng.standard_normal((L, E, 2, I, R)) / np.sqrt(max(R, 1))
    Ad = rng.standard_normal((L, E, R, I)) / np.sqrt(I)
    Bd = rng.standard_normal((L, E, H, R)) / np.sqrt(max(R, 1))
    ranks = np.asarray(ranks[:L], np.int32)
    for l in range(L):
        r = ranks[l]
        fill = 1e6 if garbage_pad else 0.0
        Agu[l, :, :, r:, :] = fill
        Bgu[l, :, :, :, r:] = fill
        Ad[l, :, r:, :] = fill
        Bd[l, :, :, r:] = fill
    return dict(x=x, topk_ids=topk, topk_weights=w, token_lora_mapping=mapping,
                lora_ranks=ranks, scalings=np.asarray(scal[:L], np.float32),
                w_gate_up=Wgu, w_down=Wd, lora_a_gu=Agu, lora_b_gu=Bgu,
                lora_a_down=Ad, lora_b_down=Bd)


def run(d, **kw):
    st, y = oracle.forward(**{**d, **kw})
    assert st == oracle.OK
    return y


def swiglu_torch(x, Wgu, Wd):
    I = Wgu.shape[0] // 2
    x, Wgu, Wd = (torch.from_numpy(np.asarray(a, np.float64)) for a in (x, Wgu, Wd))
    return (F.silu(x @ Wgu[:I].T) * (x @ Wgu[I:].T) @ Wd.T).numpy()


def test_single_expert_is_dense_swiglu():
    d = make(0, T=9, K=1, E=1, L=0, R=4)
    d["topk_weights"] = np.ones((9, 1), np.float32)
    y = run(d)
    ref = swiglu_torch(d["x"], d["w_gate_up"][0], d["w_down"][0])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_one_hot_weight_selects_that_expert():
    d = make(1, T=10, K=3, E=5, L=0, R=2)
    for k in range(3):
        w = np.zeros((10, 3), np.float32)
        w[:, k] = 1.0
        y = run(d, topk_weights=w)
        for t in range(10):
            e = d["topk_ids"][t, k]
            ref = swiglu_torch(d["x"][t:t + 1], d["w_gate_up"][e], d["w_down"][e])[0]
            np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-12)


def test_combine_linear_in_weights():
    d = make(2)
    rng = np.random.default_rng(5)
    wa = rng.random(d["topk_weights"].shape).astype(np.float32)
    wb = rng.random(d["topk_weights"].shape).astype(np.float32)
    ya, yb, yab = run(d, topk_weights=wa), run(d, topk_weights=wb), run(d, topk_weights=wa + wb)
    # wa + wb is rounded to float32 once; the combine is linear up to that rounding
    np.testing.assert_allclose(ya + yb, yab, rtol=1e-6, atol=1e-6)
    y2 = run(d, topk_weights=2 * wa)
    np.testing.assert_allclose(2 * ya, y2, rtol=1e-12, atol=1e-12)


def test_combine_invariant_to_k_order_and_expert_labels():
    d = make(3, E=6, K=3)
    y = run(d)
    perm_k = np.array([2, 0, 1])
    y_k = run(d, topk_ids=d["topk_ids"][:, perm_k], topk_weights=d["topk_weights"][:, perm_k])
    np.testing.assert_allclose(y, y_k, rtol=1e-12, atol=1e-12)
    pe = np.random.default_rng(0).permutation(6)     # new label of old expert e is pe[e]
    inv = np.argsort(pe)
    relabel = dict(
        topk_ids=pe[d["topk_ids"]].astype(np.int32),
        w_gate_up=d["w_gate_up"][inv], w_down=d["w_down"][inv],
        lora_a_gu=d["lora_a_gu"][:, inv], lora_b_gu=d["lora_b_gu"][:, inv],
        lora_a_down=d["lora_a_down"][:, inv], lora_b_down=d["lora_b_down"][:, inv])
    np.testing.assert_allclose(y, run(d, **relabel), rtol=1e-12, atol=1e-12)


def test_factored_equals_dense_materialised():
    d = make(4, T=16, K=2, E=4, L=3, R=6, ranks=(3, 0, 6), scal=(1.5, 2.0, 0.75),
             garbage_pad=True, p_none=0.2)
    y = run(d)
    base_map = np.full_like(d["token_lora_mapping"], -1)
    for l in range(3):
        toks = np.nonzero(d["token_lora_mapping"] == l)[0]
        if toks.size == 0:
            continue
        r, s = int(d["lora_ranks"][l]), float(d["scalings"][l])
        Wgu = d["w_gate_up"].copy()
        Wd = d["w_down"].copy()
        I = Wgu.shape[1] // 2
        for e in range(Wgu.shape[0]):
            if r == 0:
                continue
            Wgu[e, :I] += s * d["lora_b_gu"][l, e, 0, :, :r] @ d["lora_a_gu"][l, e, 0, :r, :]
            Wgu[e, I:] += s * d["lora_b_gu"][l, e, 1, :, :r] @ d["lora_a_gu"][l, e, 1, :r, :]
            Wd[e] += s * d["lora_b_down"][l, e, :, :r] @ d["lora_a_down"][l, e, :r, :]
        yd = run(d, token_lora_mapping=base_map, w_gate_up=Wgu, w_down=Wd, tokens=toks)
        np.testing.assert_allclose(y[toks], yd, rtol=1e-10, atol=1e-10)
    assert (d["token_lora_mapping"] == 0).any() and (d["token_lora_mapping"] == 2).any()


def test_gate_and_up_adapters_are_distinct():
    # Swapping the gate and up LoRA factors must change the output (a packed
    # gate_up that mixes the two is the bug class the PR #14105 review found).
    d = make(5, ranks=(4, 4, 4), p_none=0.0)
    y = run(d)
    sw = dict(lora_a_gu=d["lora_a_gu"][:, :, ::-1].copy(), lora_b_gu=d["lora_b_gu"][:, :, ::-1].copy())
    assert np.abs(run(d, **sw) - y).max() > 1e-3


@pytest.mark.parametrize("how", ["zero_b", "minus_one", "rank_zero"])
def test_reduces_exactly_to_base(how):
    d = make(6, p_none=0.0, ranks=(3, 5, 6))
    base = run(d, token_lora_mapping=np.full_like(d["token_lora_mapping"], -1))
    if how == "zero_b":
        y = run(d, lora_b_gu=np.zeros_like(d["lora_b_gu"]), lora_b_down=np.zeros_like(d["lora_b_down"]))
    elif how == "minus_one":
        y = base
    else:
        y = run(d, lora_ranks=np.zeros(3, np.int32))
    assert np.array_equal(y, base)
    assert np.abs(run(d) - base).max() > 1e-3   # the adapters do change the output


def test_bf16_operands_widened_exactly():
    d = make(7, ranks=(3, 2, 6))
    tb = {k: torch.from_numpy(np.asarray(d[k])).to(torch.bfloat16)
          for k in ("x", "w_gate_up", "w_down", "lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")}
    as_bits = {k: v.view(torch.int16).numpy().view(np.uint16) for k, v in tb.items()}
    as_f64 = {k: v.double().numpy() for k, v in tb.items()}
    assert np.array_equal(run(d, **as_bits), run(d, **as_f64))


def test_token_subset_rows_match():
    d = make(8, T=20)
    y = run(d)
    toks = np.array([19, 0, 7, 7, 3])
    np.testing.assert_array_equal(run(d, tokens=toks), y[toks])


def test_input_errors():
    d = make(9)
    bad = d["token_lora_mapping"].copy(); bad[0] = 3
    assert oracle.forward(**{**d, "token_lora_mapping": bad})[0] == oracle.INDEX
    bad = d["topk_ids"].copy(); bad[1, 0] = 4
    assert oracle.forward(**{**d, "topk_ids": bad})[0] == oracle.INDEX
    assert oracle.forward(**{**d, "lora_ranks": np.array([7, 0, 1], np.int32)})[0] == oracle.INVALID


def test_empty_tokens():
    d = make(10, T=0)
    st, y = oracle.forward(**d)
    assert st == oracle.OK and y.shape == (0, 24)
