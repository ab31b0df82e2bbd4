"""Seeded synthetic inputs for the LoRA MoE expert layer.

This module only draws random inputs: it holds none of the layer's arithmetic
(no adapter mapping, no bucketing, no projections), so that both the CUDA path
and the CPU oracle can be fed from it without sharing any of the method.

Distributions (the same for every workload):
  * x ~ N(0, 1);  W_gate_up ~ N(0, 1/H);  W_down ~ N(0, 1/I)
  * LoRA A, B ~ N(0, 0.02^2) on the first r_l rank rows/columns of slot l and
    exactly zero in the rank padding up to R ([num_loras, num_experts, rank, dim]
    stacks as in the adapter memory pool).  With ``lora_std="fan_in"`` they are
    N(0, 1/fan_in) instead, which makes the LoRA delta O(1).
  * router logits ~ N(0, 1) (plus a fixed per-expert bias where stated),
    softmax, top-k (sorted), renormalised to sum 1.  topk_ids int32,
    topk_weights float32.
  * x, W, A, B are stored as bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    hidden: int            # H
    intermediate: int      # I (per expert)
    num_experts: int       # E
    topk: int              # K
    num_loras: int         # L
    max_rank: int          # R
    block_size: int        # align block size
    num_tokens: int        # T
    description: str


CONFIGS = {
    "tiny": LayerConfig(
        "tiny", 256, 512, 8, 2, 4, 16, 16, 64,
        "hidden 256, intermediate 512, 8 experts top-2, 4 slots ranks [0,8,16,8] alpha 16, "
        "64 tokens in segments [10,22,7,25] with adapters [1,-1,2,3]"),
    "qwen_moe_prefill": LayerConfig(
        "qwen_moe_prefill", 2048, 768, 128, 8, 8, 64, 16, 4096,
        "Qwen-MoE-like prefill: hidden 2048, intermediate 768, 128 experts top-8, 8 slots ranks "
        "{8,16,32,64} alpha=2r, 4096 tokens in 16 segments (lens U{64..512} rescaled), one adapter -1"),
    "decode": LayerConfig(
        "decode", 2048, 768, 128, 8, 32, 32, 16, 256,
        "decode: hidden 2048, intermediate 768, 128 experts top-8, 32 slots ranks {0,8,16,32} "
        "alpha=2r, 256 requests x 1 token, adapters uniform with 10% -1"),
    "deepseek_v3_prefill": LayerConfig(
        "deepseek_v3_prefill", 7168, 2048, 256, 8, 4, 64, 16, 8192,
        "DeepSeek-V3-like prefill: hidden 7168, intermediate 2048, 256 experts top-8, 4 slots ranks "
        "{16,32,64,64} alpha=2r, 8192 tokens in 8 segments of 1024, router bias N(0,0.5)"),
    # One eighth of the DeepSeek-V3-like prefill (32 experts, 1024 tokens; the
    # same shapes, ranks, routing bias and about 256 pairs per expert): a
    # 2.8 GB case for counter captures whose per-expert traffic scales to the
    # full batch.
    "deepseek_v3_slice": LayerConfig(
        "deepseek_v3_slice", 7168, 2048, 32, 8, 4, 64, 16, 1024,
        "one eighth of the DeepSeek-V3-like prefill: hidden 7168, intermediate 2048, 32 experts top-8, "
        "4 slots ranks {16,32,64,64} alpha=2r, 1024 tokens in 8 segments of 128, router bias N(0,0.5)"),
    "metadata_stress": LayerConfig(
        "metadata_stress", 0, 0, 256, 8, 64, 64, 64, 1048576,
        "metadata stress: 1,048,576 tokens in 4096 segments (geometric lens, mean 256), 64 slots "
        "ranks uniform {0,8,16,32,64}, top-8 of 256 experts, block size 64"),
}


@dataclasses.dataclass
class Batch:
    """Per-batch request structure and routing (inputs of batch_info and align)."""
    seg_lens: torch.Tensor        # int32 [bs]
    seg_indptr: torch.Tensor      # int32 [bs+1]
    weight_indices: torch.Tensor  # int32 [bs]
    lora_ranks: torch.Tensor      # int32 [L]
    scalings: torch.Tensor        # float32 [L]  alpha_l / r_l (0 for rank 0)
    topk_ids: torch.Tensor        # int32 [T, K]
    topk_weights: torch.Tensor    # float32 [T, K]


@dataclasses.dataclass
class LayerWeights:
    w_gate_up: torch.Tensor    # bf16 [E, 2I, H]  (gate rows, then up rows)
    w_down: torch.Tensor       # bf16 [E, H, I]
    lora_a_gu: torch.Tensor    # bf16 [L, E, 2, R, H]
    lora_b_gu: torch.Tensor    # bf16 [L, E, 2, I, R]
    lora_a_down: torch.Tensor  # bf16 [L, E, R, I]
    lora_b_down: torch.Tensor  # bf16 [L, E, H, R]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _rescale_lengths(raw: torch.Tensor, total: int) -> torch.Tensor:
    """Scale positive lengths to sum exactly `total`: floor, remainder to the largest."""
    raw = raw.double()
    scaled = torch.floor(raw * total / raw.sum()).long().clamp_min(1)
    diff = total - int(scaled.sum())
    scaled[int(torch.argmax(scaled))] += diff
    assert int(scaled.sum()) == total and int(scaled.min()) >= 1
    return scaled.int()


def _indptr(seg_lens: torch.Tensor) -> torch.Tensor:
    out = torch.zeros(seg_lens.numel() + 1, dtype=torch.int64)
    out[1:] = torch.cumsum(seg_lens.long(), 0)
    return out.int()


def route(num_tokens: int, num_experts: int, topk: int, g: torch.Generator, device,
          expert_bias_std: float = 0.0, chunk: int = 1 << 16):
    """Softmax top-k routing from N(0,1) logits (+ optional fixed per-expert bias)."""
    bias = None
    if expert_bias_std > 0:
        bias = torch.randn(num_experts, generator=g, device=device) * expert_bias_std
    ids = torch.empty(num_tokens, topk, dtype=torch.int32, device=device)
    wts = torch.empty(num_tokens, topk, dtype=torch.float32, device=device)
    for t0 in range(0, num_tokens, chunk):
        t1 = min(num_tokens, t0 + chunk)
        logits = torch.randn(t1 - t0, num_experts, generator=g, device=device)
        if bias is not None:
            logits += bias
        probs = torch.softmax(logits, dim=-1)
        w, i = torch.topk(probs, topk, dim=-1, sorted=True)
        w = w / w.sum(dim=-1, keepdim=True)
        ids[t0:t1] = i.int()
        wts[t0:t1] = w.float()
    return ids, wts


def _ranks_and_scalings(cfg: LayerConfig, g: torch.Generator):
    L = cfg.num_loras
    if cfg.name == "tiny":
        ranks = [0, 8, 16, 8]
        scal = [0.0 if r == 0 else 16.0 / r for r in ranks]
    elif cfg.name == "qwen_moe_prefill":
        ranks = [[8, 16, 32, 64][l % 4] for l in range(L)]
        scal = [2.0] * L
    elif cfg.name == "decode":
        ranks = [[0, 8, 16, 32][l % 4] for l in range(L)]
        scal = [0.0 if r == 0 else 2.0 for r in ranks]
    elif cfg.name in ("deepseek_v3_prefill", "deepseek_v3_slice"):
        ranks = [16, 32, 64, 64]
        scal = [2.0] * L
    elif cfg.name == "metadata_stress":
        choices = torch.tensor([0, 8, 16, 32, 64])
        ranks = choices[torch.randint(0, 5, (L,), generator=g)].tolist()
        scal = [0.0 if r == 0 else 2.0 for r in ranks]
    else:
        raise KeyError(cfg.name)
    return torch.tensor(ranks, dtype=torch.int32), torch.tensor(scal, dtype=torch.float32)


def _segments(cfg: LayerConfig, g: torch.Generator):
    """Request segment lengths and adapter ids (CPU generator, small)."""
    T, L = cfg.num_tokens, cfg.num_loras
    if cfg.name == "tiny":
        lens = torch.tensor([10, 22, 7, 25], dtype=torch.int32)
        adapters = torch.tensor([1, -1, 2, 3], dtype=torch.int32)
    elif cfg.name == "qwen_moe_prefill":
        raw = torch.randint(64, 513, (16,), generator=g)
        lens = _rescale_lengths(raw, T)
        adapters = torch.randint(0, L, (16,), generator=g).int()
        adapters[int(torch.randint(0, 16, (1,), generator=g))] = -1
    elif cfg.name == "decode":
        lens = torch.ones(256, dtype=torch.int32)
        adapters = torch.randint(0, L, (256,), generator=g).int()
        none = torch.rand(256, generator=g) < 0.1
        adapters[none] = -1
    elif cfg.name in ("deepseek_v3_prefill", "deepseek_v3_slice"):
        lens = torch.full((8,), T // 8, dtype=torch.int32)
        adapters = torch.randint(0, L, (8,), generator=g).int()
    elif cfg.name == "metadata_stress":
        u = torch.rand(4096, generator=g, dtype=torch.float64).clamp_min(1e-12)
        p = 1.0 / 256.0
        geo = torch.floor(torch.log(u) / math.log1p(-p)) + 1  # geometric on {1,2,...}, mean 256
        lens = _rescale_lengths(geo, T)
        adapters = torch.randint(0, L, (4096,), generator=g).int()
    else:
        raise KeyError(cfg.name)
    return lens, adapters


def make_batch(cfg: LayerConfig, device="cpu", seed: int = 0) -> Batch:
    """Request segments, adapter ids, ranks/scalings and routing for one batch."""
    gc = _gen("cpu", seed)
    lens, adapters = _segments(cfg, gc)
    ranks, scal = _ranks_and_scalings(cfg, gc)
    gd = _gen(device, seed + 1)
    bias = 0.5 if cfg.name in ("deepseek_v3_prefill", "deepseek_v3_slice") else 0.0
    ids, wts = route(cfg.num_tokens, cfg.num_experts, cfg.topk, gd, device, expert_bias_std=bias)
    return Batch(lens.to(device), _indptr(lens).to(device), adapters.to(device),
                 ranks.to(device), scal.to(device), ids, wts)


def make_weights(cfg: LayerConfig, ranks: torch.Tensor, device="cpu", seed: int = 0,
                 lora_std: Optional[str] = None) -> LayerWeights:
    """Expert weights and zero-padded LoRA stacks, bf16."""
    E, H, I, L, R = cfg.num_experts, cfg.hidden, cfg.intermediate, cfg.num_loras, cfg.max_rank
    g = _gen(device, seed + 2)
    bf = torch.bfloat16

    def randn(shape, std):
        return torch.randn(shape, generator=g, device=device, dtype=bf).mul_(std)

    w_gate_up = torch.empty(E, 2 * I, H, dtype=bf, device=device)
    w_down = torch.empty(E, H, I, dtype=bf, device=device)
    for e in range(E):  # per expert keeps temporaries small at large sizes
        w_gate_up[e] = randn((2 * I, H), 1.0 / math.sqrt(H))
        w_down[e] = randn((H, I), 1.0 / math.sqrt(I))
    a_gu = torch.zeros(L, E, 2, R, H, dtype=bf, device=device)
    b_gu = torch.zeros(L, E, 2, I, R, dtype=bf, device=device)
    a_d = torch.zeros(L, E, R, I, dtype=bf, device=device)
    b_d = torch.zeros(L, E, H, R, dtype=bf, device=device)
    ranks_l = [int(r) for r in ranks.tolist()]
    for l in range(L):
        r = ranks_l[l]
        if r == 0:
            continue
        if lora_std == "fan_in":
            sa_gu, sb_gu, sa_d, sb_d = 1 / math.sqrt(H), 1 / math.sqrt(r), 1 / math.sqrt(I), 1 / math.sqrt(r)
        else:
            sa_gu = sb_gu = sa_d = sb_d = 0.02
        a_gu[l, :, :, :r, :] = randn((E, 2, r, H), sa_gu)
        b_gu[l, :, :, :, :r] = randn((E, 2, I, r), sb_gu)
        a_d[l, :, :r, :] = randn((E, r, I), sa_d)
        b_d[l, :, :, :r] = randn((E, H, r), sb_d)
    return LayerWeights(w_gate_up, w_down, a_gu, b_gu, a_d, b_d)


@dataclasses.dataclass
class Fp8Experts:
    w_gate_up_q: torch.Tensor      # uint8 [E, 2I, H], FP8 E4M3 codes
    w_gate_up_scale: torch.Tensor  # float32 [E, ceil(2I/128), ceil(H/128)]
    w_down_q: torch.Tensor         # uint8 [E, H, I]
    w_down_scale: torch.Tensor     # float32 [E, ceil(H/128), ceil(I/128)]


def make_fp8_experts(cfg: LayerConfig, device="cpu", seed: int = 0) -> Fp8Experts:
    """FP8 E4M3 expert weights with one float32 scale per 128 x 128 block.

    Codes are N(0, 32^2) samples cast to E4M3 (torch's float8_e4m3fn); each
    block's scale is U(0.75, 1.25) / (32 sqrt(fan_in)), so code x scale has
    about the bf16 weights' N(0, 1/fan_in) spread and the scales are not
    powers of two.
    """
    E, H, I = cfg.num_experts, cfg.hidden, cfg.intermediate
    g = _gen(device, seed + 5)
    nb = lambda n: (n + 127) // 128  # noqa: E731

    def mat(rows, cols, fan_in):
        z = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).mul_(32.0)
        codes = z.to(torch.float8_e4m3fn).view(torch.uint8)
        u = torch.rand((nb(rows), nb(cols)), generator=g, device=device, dtype=torch.float32)
        return codes, (u * 0.5 + 0.75) / (32.0 * math.sqrt(fan_in))

    wq = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
    ws = torch.empty(E, nb(2 * I), nb(H), dtype=torch.float32, device=device)
    dq = torch.empty(E, H, I, dtype=torch.uint8, device=device)
    ds = torch.empty(E, nb(H), nb(I), dtype=torch.float32, device=device)
    for e in range(E):  # per expert keeps temporaries small at large sizes
        wq[e], ws[e] = mat(2 * I, H, H)
        dq[e], ds[e] = mat(H, I, I)
    return Fp8Experts(wq, ws, dq, ds)


@dataclasses.dataclass
class Fp8W8A8Experts:
    w_gate_up_q: torch.Tensor    # uint8 [E, 2I, H], FP8 E4M3 codes
    w_gate_up_exp: torch.Tensor  # uint8 [E, ceil(2I/128), ceil(H/128)], biased block exponents
    w_down_q: torch.Tensor       # uint8 [E, H, I]
    w_down_exp: torch.Tensor     # uint8 [E, ceil(H/128), ceil(I/128)]


def make_fp8_w8a8_experts(cfg: LayerConfig, device="cpu", seed: int = 0) -> Fp8W8A8Experts:
    """FP8 E4M3 expert weights with power-of-two block scales.

    Codes are N(0, 32^2) samples cast to E4M3 (torch's float8_e4m3fn); each
    128 x 128 block's exponent is e0 or e0 + 1 at random, with 2^(e0 - 127)
    the largest power of two at or below 1 / (32 sqrt(fan_in)), so code x
    2^(e - 127) has about the bf16 weights' N(0, 1/fan_in) spread within a
    factor of two.
    """
    E, H, I = cfg.num_experts, cfg.hidden, cfg.intermediate
    g = _gen(device, seed + 8)
    nb = lambda n: (n + 127) // 128  # noqa: E731

    def mat(rows, cols, fan_in):
        z = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).mul_(32.0)
        codes = z.to(torch.float8_e4m3fn).view(torch.uint8)
        e0 = 127 + math.floor(math.log2(1.0 / (32.0 * math.sqrt(fan_in))))
        ex = torch.randint(0, 2, (nb(rows), nb(cols)), generator=g, device=device, dtype=torch.int32) + e0
        return codes, ex.to(torch.uint8)

    wq = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
    we = torch.empty(E, nb(2 * I), nb(H), dtype=torch.uint8, device=device)
    dq = torch.empty(E, H, I, dtype=torch.uint8, device=device)
    de = torch.empty(E, nb(H), nb(I), dtype=torch.uint8, device=device)
    for e in range(E):
        wq[e], we[e] = mat(2 * I, H, H)
        dq[e], de[e] = mat(H, I, I)
    return Fp8W8A8Experts(wq, we, dq, de)


@dataclasses.dataclass
class Int8Experts:
    w_gate_up_q: torch.Tensor      # int8 [E, 2I, H]
    w_gate_up_scale: torch.Tensor  # float32 [E, ceil(2I/128), ceil(H/128)]
    w_down_q: torch.Tensor         # int8 [E, H, I]
    w_down_scale: torch.Tensor     # float32 [E, ceil(H/128), ceil(I/128)]


def make_int8_experts(cfg: LayerConfig, device="cpu", seed: int = 0) -> Int8Experts:
    """Block-wise INT8 expert weights: codes round(N(0, 40^2)) clipped to
    [-127, 127], one float32 scale per 128 x 128 block of U(0.75, 1.25) /
    (40 sqrt(fan_in)), so code x scale has about the bf16 weights' spread."""
    E, H, I = cfg.num_experts, cfg.hidden, cfg.intermediate
    g = _gen(device, seed + 6)
    nb = lambda n: (n + 127) // 128  # noqa: E731

    def mat(rows, cols, fan_in):
        z = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).mul_(40.0)
        codes = z.round_().clamp_(-127, 127).to(torch.int8)
        u = torch.rand((nb(rows), nb(cols)), generator=g, device=device, dtype=torch.float32)
        return codes, (u * 0.5 + 0.75) / (40.0 * math.sqrt(fan_in))

    wq = torch.empty(E, 2 * I, H, dtype=torch.int8, device=device)
    ws = torch.empty(E, nb(2 * I), nb(H), dtype=torch.float32, device=device)
    dq = torch.empty(E, H, I, dtype=torch.int8, device=device)
    ds = torch.empty(E, nb(H), nb(I), dtype=torch.float32, device=device)
    for e in range(E):
        wq[e], ws[e] = mat(2 * I, H, H)
        dq[e], ds[e] = mat(H, I, I)
    return Int8Experts(wq, ws, dq, ds)


@dataclasses.dataclass
class W4A16Experts:
    w_gate_up_q: torch.Tensor      # uint8 [E, 2I, H/2], two uint4 codes per byte (even column low)
    w_gate_up_scale: torch.Tensor  # float32 [E, 2I, ceil(H/128)]
    w_gate_up_zero: torch.Tensor   # uint8 [E, 2I, ceil(H/128)], 0..15
    w_down_q: torch.Tensor         # uint8 [E, H, I/2]
    w_down_scale: torch.Tensor     # float32 [E, H, ceil(I/128)]
    w_down_zero: torch.Tensor      # uint8 [E, H, ceil(I/128)]


def make_w4a16_experts(cfg: LayerConfig, device="cpu", seed: int = 0) -> W4A16Experts:
    """4-bit expert weights: uniform codes 0..15, zero points uniform in 6..9,
    one float32 scale per row and 128-column group of U(0.75, 1.25) /
    sqrt(22.5 fan_in): code - zero has mean 0 and mean square 21.25 + 1.25 =
    22.5, so (code - zero) x scale has about the bf16 weights' N(0, 1/fan_in)
    spread."""
    E, H, I = cfg.num_experts, cfg.hidden, cfg.intermediate
    g = _gen(device, seed + 7)
    nb = lambda n: (n + 127) // 128  # noqa: E731

    def mat(rows, cols, fan_in):
        codes = torch.randint(0, 16, (rows, cols), generator=g, device=device, dtype=torch.int32)
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
        u = torch.rand((rows, nb(cols)), generator=g, device=device, dtype=torch.float32)
        zero = torch.randint(6, 10, (rows, nb(cols)), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
        return packed, (u * 0.5 + 0.75) / math.sqrt(22.5 * fan_in), zero

    wq = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
    ws = torch.empty(E, 2 * I, nb(H), dtype=torch.float32, device=device)
    wz = torch.empty(E, 2 * I, nb(H), dtype=torch.uint8, device=device)
    dq = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
    ds = torch.empty(E, H, nb(I), dtype=torch.float32, device=device)
    dz = torch.empty(E, H, nb(I), dtype=torch.uint8, device=device)
    for e in range(E):
        wq[e], ws[e], wz[e] = mat(2 * I, H, H)
        dq[e], ds[e], dz[e] = mat(H, I, I)
    return W4A16Experts(wq, ws, wz, dq, ds, dz)


def make_x(cfg: LayerConfig, device="cpu", seed: int = 0) -> torch.Tensor:
    g = _gen(device, seed + 3)
    return torch.randn(cfg.num_tokens, cfg.hidden, generator=g, device=device,
                       dtype=torch.bfloat16)


def custom_config(name: str = "custom", **kw) -> LayerConfig:
    """A LayerConfig with explicit sizes (tests of ragged and edge shapes)."""
    base = dict(hidden=256, intermediate=512, num_experts=8, topk=2, num_loras=4, max_rank=16,
                block_size=16, num_tokens=64, description="custom")
    base.update(kw)
    return LayerConfig(name=name, **base)
