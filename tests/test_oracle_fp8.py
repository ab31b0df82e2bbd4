"""Pins for the oracle's FP8-expert forward (CPU only).

The sglang PR #22323 page (功能与动机, 实现拆解 item 1) says that quantised MoE
experts hand their scales to the LoRA MoE layer; the format is a reading:
E4M3 codes with one float scale per 128 x 128 block of each expert matrix,
the weight being code value x scale, LoRA and activations in bf16.  Pinned
here against things other than the oracle's own loops:
  * the E4M3 decoder against the format's defining values and against
    torch's float8_e4m3fn conversion for all 256 codes;
  * with every scale 1 the layer is the (already pinned) bf16/fp64 forward
    run on the decoded weights, exactly;
  * with power-of-two scales per block (exact products) it is the fp64
    forward on weights dequantised with numpy's block broadcast, exactly; the
    shapes leave ragged edge blocks and a block shared by gate and up rows, so
    a swapped or mis-divided block index fails.
"""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_forward import make


def test_e4m3_defining_values():
    fixed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0, 0x80: -0.0}
    for code, v in fixed.items():
        assert oracle.e4m3_value(code) == v, hex(code)
    assert np.signbit(oracle.e4m3_value(0x80))
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()


def decoded_table():
    return np.array([oracle.e4m3_value(c) for c in range(256)])


def quantised(d, seed, scale_fn):
    """Random non-NaN E4M3 codes for both expert matrices and block scales."""
    rng = np.random.default_rng(seed)
    E, I2, H = d["w_gate_up"].shape
    I = I2 // 2
    ok = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    # codes of moderate magnitude (exponent field <= 8: |v| < 4) keep the layer well scaled
    ok = ok[((ok >> 3) & 15) <= 8]
    wq = rng.choice(ok, size=(E, 2 * I, H)).astype(np.uint8)
    dq = rng.choice(ok, size=(E, H, I)).astype(np.uint8)
    ws = scale_fn(rng, (E, (2 * I + 127) // 128, (H + 127) // 128))
    ds = scale_fn(rng, (E, (H + 127) // 128, (I + 127) // 128))
    return wq, ws, dq, ds


def dequant(q, s, table):
    rows, cols = q.shape[1], q.shape[2]
    full = np.repeat(np.repeat(s.astype(np.float64), 128, axis=1), 128, axis=2)[:, :rows, :cols]
    return table[q] * full


def fp8_args(d, wq, ws, dq, ds):
    keep = {k: v for k, v in d.items() if k not in ("w_gate_up", "w_down")}
    return dict(keep, w_gate_up_q=wq, w_gate_up_scale=ws, w_down_q=dq, w_down_scale=ds)


def test_unit_scales_equal_decoded_forward():
    d = make(11, T=10, K=2, E=3, H=40, I=24, L=3, R=6)
    wq, ws, dq, ds = quantised(d, 1, lambda rng, shp: np.ones(shp, np.float32))
    tab = decoded_table()
    st, y8 = oracle.forward_fp8(**fp8_args(d, wq, ws, dq, ds))
    assert st == oracle.OK
    st, y = oracle.forward(**{**d, "w_gate_up": tab[wq], "w_down": tab[dq]})
    assert st == oracle.OK
    assert (y8 == y).all()


@pytest.mark.parametrize("H,I", [(200, 80), (256, 128), (136, 72)])
def test_block_scales_match_numpy_dequant(H, I):
    # I = 80: gate rows 0..79 and up rows 0..47 share row block 0 of W_gate_up;
    # H = 200 / 136 leaves ragged column (gate_up) and row (down) blocks
    d = make(12, T=8, K=2, E=3, H=H, I=I, L=3, R=6)
    wq, ws, dq, ds = quantised(d, 2, lambda rng, shp: np.ldexp(1.0, rng.integers(-6, 5, shp)).astype(np.float32))
    tab = decoded_table()
    st, y8 = oracle.forward_fp8(**fp8_args(d, wq, ws, dq, ds))
    assert st == oracle.OK
    st, y = oracle.forward(**{**d, "w_gate_up": dequant(wq, ws, tab), "w_down": dequant(dq, ds, tab)})
    assert st == oracle.OK
    assert (y8 == y).all()
    # a transposed scale layout would give a different layer
    if ws.shape[1] == ws.shape[2]:
        st, yt = oracle.forward_fp8(**fp8_args(d, wq, np.ascontiguousarray(ws.transpose(0, 2, 1)), dq, ds))
        assert not np.allclose(yt, y8)


def test_scale_of_one_block_moves_only_its_rows():
    # doubling the scale of W_down's row block 1 of expert e doubles that block's
    # contribution: y changes only in output columns 128..255 of tokens routed to e
    d = make(13, T=8, K=1, E=2, H=256, I=64, L=0, R=0)
    d["topk_weights"] = np.ones((8, 1), np.float32)
    wq, ws, dq, ds = quantised(d, 3, lambda rng, shp: np.ones(shp, np.float32))
    st, y0 = oracle.forward_fp8(**fp8_args(d, wq, ws, dq, ds))
    ds2 = ds.copy()
    ds2[1, 1, 0] = 2.0
    st, y1 = oracle.forward_fp8(**fp8_args(d, wq, ws, dq, ds2))
    routed = d["topk_ids"][:, 0] == 1
    assert (y1[~routed] == y0[~routed]).all()
    assert (y1[routed][:, :128] == y0[routed][:, :128]).all()
    np.testing.assert_allclose(y1[routed][:, 128:], 2 * y0[routed][:, 128:], rtol=1e-15, atol=0)
