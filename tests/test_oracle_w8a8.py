"""Pins for the oracle's FP8 W8A8 forward (power-of-two block scales) -- CPU only.

The sglang PR #22323 page (功能与动机, 实现拆解 item 1) names the FP8 method
whose scales reach the LoRA MoE layer.  This format is a reading, the one the
FP8 tensor cores take: E4M3 weight codes whose 128 x 128 block scales are
powers of two (biased 8-bit exponents, scale 2^(e-127)), and activations
quantised per token and 128-channel group with a power-of-two scale 2^s, s
the smallest integer with max|group| x 2^-s <= 448, each element rounded to
the nearest E4M3 value (ties to even).  The intermediate a = SiLU(g) * u is
rounded to bf16 first; the LoRA shrinks read the unquantised x and a.  The
decision on a's codes depends on the LoRA delta, so this layer takes it at
the kernels' precision: the scaled LoRA intermediates s * (A x) and
s * (A_d a) are rounded to bf16 before B multiplies them.

Pinned against things other than the oracle's own loops:
  * the E4M3 rounding against torch's float8_e4m3fn cast, on every tie
    between neighbouring E4M3 values and on random values of every binade;
  * the group exponent against the closed form ceil(log2(amax / 448)) and
    the boundary cases 448, 224 and the clamps;
  * the whole layer against a torch float64 re-derivation that quantises with
    torch's float8 cast, takes the exponent from log2, rounds a to bf16 with
    torch (through a round-to-odd float32 step, so there is no double
    rounding) and broadcasts the block exponents with repeat; ragged shapes
    leave partial groups, partial blocks and a block shared by gate and up;
  * planted mistakes in that re-derivation (x or a not quantised, LoRA fed
    the quantised operands, the exponent one too large, a or z not rounded)
    must each change the layer.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from test_oracle_forward import make


def test_e4m3_round_matches_torch_on_ties_and_random_values():
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    grid = np.unique(np.abs(vals[np.isfinite(vals)]))
    mids = (grid[:-1] + grid[1:]) / 2  # every tie
    rng = np.random.default_rng(3)
    rand = (rng.uniform(-1, 1, 20000) * np.ldexp(1.0, rng.integers(-14, 9, 20000))).astype(np.float32)
    rand = rand[np.abs(rand) <= 448].astype(np.float64)
    for v in (grid, -grid, mids, -mids, rand):
        ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        ours = np.array([oracle.e4m3_round(float(a)) for a in v])
        assert (ours == ref).all()


def test_group_exponent_closed_form_and_boundaries():
    rng = np.random.default_rng(4)
    # bf16-representable magnitudes over a wide range (8 significant bits)
    m = rng.integers(128, 256, 5000)
    amax = np.ldexp(m.astype(np.float64), rng.integers(-60, 60, 5000))
    ref = np.clip(np.ceil(np.log2(amax / 448.0)), -127, 127).astype(int)
    ours = np.array([oracle.mx_group_exp(float(a)) for a in amax])
    assert (ours == ref).all()
    assert oracle.mx_group_exp(448.0) == 0 and oracle.mx_group_exp(449.0) == 1
    assert oracle.mx_group_exp(224.0) == -1 and oracle.mx_group_exp(1.0) == -8
    assert oracle.mx_group_exp(0.0) == 0
    assert oracle.mx_group_exp(2.0 ** -200) == -127 and oracle.mx_group_exp(2.0 ** 200) == 127


def _bf16_values(a):
    """float64 array -> the nearest bf16 values, ties to even (torch's cast from float32)."""
    return torch.tensor(np.asarray(a), dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def _to_bf16_direct(a):
    """Round float64 -> bf16 with one rounding: float32 by round-to-odd (exact
    when a fits, else truncated with the last bit set), then torch's cast to
    bf16 (ties to even).  Round-to-odd with more bits than the target keeps the
    final rounding correct."""
    a = np.asarray(a, np.float64)
    f = a.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(a)
    f = np.where(over, np.nextafter(f, np.float32(0)), f)
    inexact = f.astype(np.float64) != a
    bits = f.view(np.uint32) | inexact.astype(np.uint32)
    f = bits.view(np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).to(torch.float64)


def _quant_torch(v, mistake=None):
    """Quantise-dequantise v [n] per 128-element group with torch's E4M3 cast."""
    out = torch.empty_like(v)
    for g0 in range(0, v.shape[0], 128):
        grp = v[g0:g0 + 128]
        amax = float(grp.abs().max())
        s = 0 if amax == 0 else int(np.clip(np.ceil(np.log2(amax / 448.0)), -127, 127))
        if mistake == "exp_off":
            s += 1
        scaled = (grp * 2.0 ** -s).to(torch.float32)  # exact: bf16 values times a power of two
        out[g0:g0 + 128] = scaled.to(torch.float8_e4m3fn).to(torch.float64) * 2.0 ** s
    return out


def _dequant_blocks(codes, ex):
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    rows, cols = codes.shape[1], codes.shape[2]
    sc = torch.from_numpy(np.ldexp(1.0, ex.astype(np.int64) - 127))
    sc = sc.repeat_interleave(128, dim=1).repeat_interleave(128, dim=2)[:, :rows, :cols]
    return vals * sc


def _torch_layer(d, wq, we, dq, de, mistake=None):
    x = torch.from_numpy(np.asarray(d["x"], np.float64))
    T, H = x.shape
    Wgu, Wd = _dequant_blocks(wq, we), _dequant_blocks(dq, de)
    I = Wgu.shape[1] // 2
    Agu, Bgu, Ad, Bd = (torch.from_numpy(np.asarray(d[k], np.float64))
                        for k in ("lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down"))
    topk, w, mp = d["topk_ids"], d["topk_weights"], d["token_lora_mapping"]
    ranks, scal = d["lora_ranks"], d["scalings"]
    y = torch.zeros(T, H, dtype=torch.float64)
    for t in range(T):
        xv = x[t]
        xq = xv if mistake == "no_xq" else _quant_torch(xv, mistake)
        l = int(mp[t])
        r = int(ranks[l]) if l >= 0 else 0
        s = float(scal[l]) if r > 0 else 0.0
        for k in range(topk.shape[1]):
            e = int(topk[t, k])
            g, u = Wgu[e, :I] @ xq, Wgu[e, I:] @ xq
            zr = (lambda z: s * z) if mistake == "no_zround" else (lambda z: _to_bf16_direct((s * z).numpy()))
            if r > 0:
                xl = xq if mistake == "lora_q" else xv
                g = g + Bgu[l, e, 0, :, :r] @ zr(Agu[l, e, 0, :r] @ xl)
                u = u + Bgu[l, e, 1, :, :r] @ zr(Agu[l, e, 1, :r] @ xl)
            a = F.silu(g) * u
            if mistake != "no_bf16":
                a = _to_bf16_direct(a.numpy())
            aq = a if mistake == "no_hq" else _quant_torch(a, mistake)
            dd = Wd[e] @ aq
            if r > 0:
                al = aq if mistake == "lora_q" else a
                dd = dd + Bd[l, e, :, :r] @ zr(Ad[l, e, :r] @ al)
            y[t] += float(w[t, k]) * dd
    return y.numpy()


def _weights(rng, E, H, I):
    def codes(shape):
        c = rng.integers(0, 256, shape).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x30  # no NaN codes
        return c

    wq, dq = codes((E, 2 * I, H)), codes((E, H, I))
    we = rng.integers(113, 121, (E, (2 * I + 127) // 128, (H + 127) // 128)).astype(np.uint8)
    de = rng.integers(113, 121, (E, (H + 127) // 128, (I + 127) // 128)).astype(np.uint8)
    return wq, we, dq, de


def _keep(d):
    return {k: v for k, v in d.items() if k not in ("w_gate_up", "w_down")}


@pytest.mark.parametrize("H,I", [(200, 80), (136, 72), (256, 128)])
def test_layer_matches_torch_rederivation(H, I):
    d = make(31, T=10, K=2, E=3, H=H, I=I, L=3, R=6)
    d["x"] = _bf16_values(d["x"] * 3.0)  # the layer's input is bf16
    wq, we, dq, de = _weights(np.random.default_rng(6), 3, H, I)
    st, y = oracle.forward_fp8_w8a8(**_keep(d), w_gate_up_q=wq, w_gate_up_exp=we, w_down_q=dq, w_down_exp=de)
    assert st == oracle.OK
    ref = _torch_layer(d, wq, we, dq, de)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())
    for mistake in ("no_xq", "no_hq", "lora_q", "exp_off", "no_bf16", "no_zround"):
        bad = _torch_layer(d, wq, we, dq, de, mistake)
        assert np.abs(bad - y).max() > 1e-6 * np.abs(y).max(), mistake


def test_zero_and_tiny_groups():
    # an all-zero token (every group's exponent 0) and a token whose values
    # are far below E4M3's range before scaling
    d = make(32, T=3, K=1, E=2, H=256, I=128, L=0, R=0)
    x = _bf16_values(d["x"])
    x[0] = 0.0
    x[1] = _bf16_values(x[1] * 2.0 ** -40)
    d["x"] = x
    wq, we, dq, de = _weights(np.random.default_rng(7), 2, 256, 128)
    st, y = oracle.forward_fp8_w8a8(**_keep(d), w_gate_up_q=wq, w_gate_up_exp=we, w_down_q=dq, w_down_exp=de)
    assert st == oracle.OK
    assert (y[0] == 0).all()
    ref = _torch_layer(d, wq, we, dq, de)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-300)
    assert np.abs(y[1]).max() > 0
