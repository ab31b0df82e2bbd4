"""Pins for the oracle's INT8 and W4A16 expert forwards (CPU only).

The sglang PR #22323 page (功能与动机, 实现拆解 item 1) names the quantisation
methods whose scales reach the LoRA MoE layer: FP8, INT8 (blockwise_int8) and
WNA16.  The formats are readings:
  * INT8: two's-complement int8 codes with one float scale per 128 x 128 block
    (the FP8 layer's layout), weight = code x scale;
  * W4A16: uint4 codes two per byte along a row (even column in the low
    nibble), one float scale and one zero point per row and group of 128
    input columns, weight = (code - zero) x scale.
Pinned against things other than the oracle's own loops: the int8 decode
against numpy's int8 view of the same bytes; the layers against the pinned
fp64 forward on weights dequantised by numpy (block and group broadcasts,
nibble unpacking with shifts), exactly, with power-of-two scales; and planted
mistakes in that dequantisation (nibbles swapped, zero point ignored, groups
along rows instead of columns) that must change the layer.
"""
import numpy as np
import pytest

import oracle
from test_oracle_forward import make


def _pow2(rng, shp):
    return np.ldexp(1.0, rng.integers(-6, 3, shp)).astype(np.float32)


def _keep(d):
    return {k: v for k, v in d.items() if k not in ("w_gate_up", "w_down")}


def _block_dequant(q_int, s):
    rows, cols = q_int.shape[1], q_int.shape[2]
    full = np.repeat(np.repeat(s.astype(np.float64), 128, axis=1), 128, axis=2)[:, :rows, :cols]
    return q_int.astype(np.float64) * full


@pytest.mark.parametrize("H,I", [(200, 80), (136, 72), (256, 128)])
def test_int8_matches_numpy_dequant(H, I):
    d = make(21, T=8, K=2, E=3, H=H, I=I, L=3, R=6)
    rng = np.random.default_rng(5)
    E = 3
    wq = rng.integers(-128, 128, (E, 2 * I, H)).astype(np.int8)
    dq = rng.integers(-128, 128, (E, H, I)).astype(np.int8)
    ws = _pow2(rng, (E, (2 * I + 127) // 128, (H + 127) // 128)) / 64
    ds = _pow2(rng, (E, (H + 127) // 128, (I + 127) // 128)) / 64
    st, y8 = oracle.forward_int8(**_keep(d), w_gate_up_q=wq, w_gate_up_scale=ws, w_down_q=dq, w_down_scale=ds)
    assert st == oracle.OK
    st, y = oracle.forward(**{**d, "w_gate_up": _block_dequant(wq, ws), "w_down": _block_dequant(dq, ds)})
    assert st == oracle.OK
    assert (y8 == y).all()
    # the same bytes read as unsigned would be another layer
    st, yu = oracle.forward(**{**d, "w_gate_up": _block_dequant(wq.view(np.uint8), ws),
                               "w_down": _block_dequant(dq.view(np.uint8), ds)})
    assert not np.allclose(yu, y8)


def test_int8_extreme_codes():
    # codes -128, -1, 0, 127 through a one-token, one-expert layer with unit
    # scales and an identity-like setup: compare with the decoded forward
    d = make(22, T=4, K=1, E=1, H=128, I=128, L=0, R=0)
    wq = np.zeros((1, 256, 128), np.int8)
    dq = np.zeros((1, 128, 128), np.int8)
    wq[0, :, :4] = np.array([-128, -1, 0, 127], np.int8)
    dq[0, :, :4] = np.array([127, 0, -1, -128], np.int8)
    ones = lambda shp: np.ones(shp, np.float32)  # noqa: E731
    st, y8 = oracle.forward_int8(**_keep(d), w_gate_up_q=wq, w_gate_up_scale=ones((1, 2, 1)), w_down_q=dq,
                                 w_down_scale=ones((1, 1, 1)))
    st, y = oracle.forward(**{**d, "w_gate_up": wq.astype(np.float64), "w_down": dq.astype(np.float64)})
    assert (y8 == y).all() and np.abs(y).max() > 1


def _pack_uint4(codes):
    """[.., cols] uint4 codes -> [.., cols/2] bytes, even column in the low nibble."""
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _group_dequant(codes, scale, zero, rows_groups=False):
    g = np.repeat(scale.astype(np.float64), 128, axis=2)[..., :codes.shape[2]]
    z = np.repeat(zero.astype(np.float64), 128, axis=2)[..., :codes.shape[2]]
    return (codes.astype(np.float64) - z) * g


def _w4(d, H, I, seed):
    rng = np.random.default_rng(seed)
    E = d["w_gate_up"].shape[0]
    wc = rng.integers(0, 16, (E, 2 * I, H)).astype(np.uint8)
    dc = rng.integers(0, 16, (E, H, I)).astype(np.uint8)
    ws = _pow2(rng, (E, 2 * I, (H + 127) // 128)) / 8
    ds = _pow2(rng, (E, H, (I + 127) // 128)) / 8
    wz = rng.integers(0, 16, ws.shape).astype(np.uint8)
    dz = rng.integers(0, 16, ds.shape).astype(np.uint8)
    return wc, ws, wz, dc, ds, dz


@pytest.mark.parametrize("H,I", [(200, 80), (256, 128), (136, 72)])
def test_w4a16_matches_numpy_dequant(H, I):
    d = make(23, T=8, K=2, E=3, H=H, I=I, L=3, R=6)
    wc, ws, wz, dc, ds, dz = _w4(d, H, I, 6)
    args = dict(_keep(d), w_gate_up_q=_pack_uint4(wc), w_gate_up_scale=ws, w_gate_up_zero=wz,
                w_down_q=_pack_uint4(dc), w_down_scale=ds, w_down_zero=dz)
    st, y4 = oracle.forward_w4a16(**args)
    assert st == oracle.OK
    st, y = oracle.forward(**{**d, "w_gate_up": _group_dequant(wc, ws, wz), "w_down": _group_dequant(dc, ds, dz)})
    assert st == oracle.OK
    assert (y4 == y).all()
    # planted mistakes in the reading change the layer
    swapped = dict(args, w_gate_up_q=_pack_uint4(wc[..., ::-1].copy())[..., ::-1].copy())
    st, ys = oracle.forward_w4a16(**swapped)
    assert not np.allclose(ys, y4)
    st, yz = oracle.forward(**{**d, "w_gate_up": _group_dequant(wc, ws, np.zeros_like(wz)),
                               "w_down": _group_dequant(dc, ds, np.zeros_like(dz))})
    assert not np.allclose(yz, y4)


def test_w4a16_one_group_scale_is_local():
    # doubling the scale of one (row, group) of W_down for expert 1 with zero
    # point 0 doubles that group's contribution to one output row only
    d = make(24, T=6, K=1, E=2, H=128, I=256, L=0, R=0)
    d["topk_weights"] = np.ones((6, 1), np.float32)
    wc, ws, wz, dc, ds, dz = _w4(d, 128, 256, 7)
    dz[:] = 0
    base = dict(_keep(d), w_gate_up_q=_pack_uint4(wc), w_gate_up_scale=ws, w_gate_up_zero=wz,
                w_down_q=_pack_uint4(dc), w_down_scale=ds, w_down_zero=dz)
    st, y0 = oracle.forward_w4a16(**base)
    ds2 = ds.copy()
    ds2[1, 5, 1] *= 2
    st, y1 = oracle.forward_w4a16(**dict(base, w_down_scale=ds2))
    routed = d["topk_ids"][:, 0] == 1
    cols = [c for c in range(128) if c != 5]
    assert (y1[~routed] == y0[~routed]).all()
    assert (y1[routed][:, cols] == y0[routed][:, cols]).all()
    if routed.any():
        assert not np.allclose(y1[routed][:, 5], y0[routed][:, 5])
