"""CPU oracle for the multi-adapter LoRA MoE expert layer (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs are the only callers.
The CUDA library never imports, links or loads anything here, and this module
imports nothing from the CUDA package.

The arithmetic lives in ``moe_lora_oracle.c`` (plain C, fp64 accumulation);
this module only compiles it with gcc on first use and marshals numpy arrays.
bf16 tensors are passed as their uint16 bit patterns (widened exactly in C);
float64 arrays are accepted for the same operands so that tests can feed values
that bf16 cannot hold (the dense-materialised W + s*B*A check).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_lora_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libmoe_lora_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
INVALID = -1
UNDERCOVERED = -2
INDEX = -3
CAPACITY = -4
NOMEM = -7


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP) into oracle/_build; return the path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-std=c11", "-Wall", "-shared", "-fPIC",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            vp = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_batch_info.restype = ctypes.c_int
            lib.oracle_batch_info.argtypes = [i32p, i32p, i32p, i32, i32, i32, i32, i32p, i32p]
            lib.oracle_align_capacity.restype = i64
            lib.oracle_align_capacity.argtypes = [i32, i32, i32, i32, i32]
            lib.oracle_align.restype = ctypes.c_int
            lib.oracle_align.argtypes = [i32p, i32p, i32, i32, i32, i32, i32,
                                         i32p, i32p, i32p, i32p, i64]
            lib.oracle_forward.restype = ctypes.c_int
            lib.oracle_forward.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp,
                                           vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                           i64, i64, i64, i64, i64, i64, i64,
                                           vp, i64, vp, ctypes.c_int]
            lib.oracle_forward_fp8.restype = ctypes.c_int
            lib.oracle_forward_fp8.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp,
                                               vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                               i64, i64, i64, i64, i64, i64, i64,
                                               vp, i64, vp, ctypes.c_int]
            lib.oracle_forward_int8.restype = ctypes.c_int
            lib.oracle_forward_int8.argtypes = lib.oracle_forward_fp8.argtypes
            lib.oracle_forward_w4a16.restype = ctypes.c_int
            lib.oracle_forward_w4a16.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp,
                                                 vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                                 i64, i64, i64, i64, i64, i64, i64,
                                                 vp, i64, vp, ctypes.c_int]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint32]
            lib.oracle_forward_fp8_w8a8.restype = ctypes.c_int
            lib.oracle_forward_fp8_w8a8.argtypes = lib.oracle_forward_fp8.argtypes
            lib.oracle_e4m3_round.restype = ctypes.c_double
            lib.oracle_e4m3_round.argtypes = [ctypes.c_double]
            lib.oracle_mx_group_exp.restype = ctypes.c_int
            lib.oracle_mx_group_exp.argtypes = [ctypes.c_double]
            lib.oracle_lora_linear.restype = ctypes.c_int
            lib.oracle_lora_linear.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                               i64, i64, i64, i64, i64, i64, vp, vp, i64, vp, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def batch_info(seg_indptr, weight_indices, lora_ranks, num_tokens: int, max_len: int = 0):
    """Returns (status, token_lora_mapping[num_tokens], adapter_enabled[num_loras])."""
    seg_indptr, weight_indices, lora_ranks = _i32(seg_indptr), _i32(weight_indices), _i32(lora_ranks)
    bs = weight_indices.shape[0]
    if seg_indptr.shape[0] != bs + 1:
        return INVALID, None, None
    mapping = np.zeros(max(num_tokens, 0), dtype=np.int32)
    enabled = np.zeros(lora_ranks.shape[0], dtype=np.int32)
    st = _load().oracle_batch_info(_p32(seg_indptr), _p32(weight_indices), _p32(lora_ranks),
                                   bs, lora_ranks.shape[0], num_tokens, max_len,
                                   _p32(mapping), _p32(enabled))
    return int(st), mapping, enabled


def align_capacity(num_tokens: int, topk: int, num_experts: int, num_loras: int,
                   block_size: int) -> int:
    return int(_load().oracle_align_capacity(num_tokens, topk, num_experts, num_loras, block_size))


def align(topk_ids, token_lora_mapping, num_experts: int, num_loras: int, block_size: int):
    """Returns (status, sorted_token_ids[npad], block_expert_ids[npad/bs],
    block_lora_ids[npad/bs], npad); arrays are trimmed to the valid prefix."""
    topk_ids = _i32(topk_ids)
    if topk_ids.ndim != 2:
        return INVALID, None, None, None, 0
    T, K = topk_ids.shape
    mapping = _i32(token_lora_mapping)
    cap = align_capacity(T, K, num_experts, num_loras, block_size)
    if cap < 0:
        return INVALID, None, None, None, 0
    sorted_ids = np.zeros(max(cap, 1), dtype=np.int32)
    nblk = max(cap // block_size, 1)
    bexp = np.zeros(nblk, dtype=np.int32)
    blora = np.zeros(nblk, dtype=np.int32)
    npad = np.zeros(1, dtype=np.int32)
    st = _load().oracle_align(_p32(topk_ids), _p32(mapping), T, K, num_experts, num_loras,
                              block_size, _p32(sorted_ids), _p32(bexp), _p32(blora),
                              _p32(npad), cap)
    n = int(npad[0])
    if st != OK:
        return int(st), None, None, None, 0
    return int(st), sorted_ids[:n].copy(), bexp[: n // block_size].copy(), \
        blora[: n // block_size].copy(), n


def _operand(a):
    """(pointer, dtype code, keep-alive array) for a bf16-bits or float64 operand."""
    a = np.asarray(a)
    if a.dtype == np.uint16 or a.dtype == np.int16:
        a = np.ascontiguousarray(a.view(np.uint16))
        return a.ctypes.data, 0, a
    if a.dtype == np.float64:
        a = np.ascontiguousarray(a)
        return a.ctypes.data, 1, a
    raise TypeError(f"oracle operands are bf16 bit patterns (uint16) or float64, got {a.dtype}")


def forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
            w_gate_up, w_down, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down,
            tokens=None, threads: int = 0):
    """Returns (status, y) with y float64 [len(tokens) or T, H].

    Shapes: x [T,H]; topk_ids/topk_weights [T,K]; mapping [T]; ranks/scalings [L];
    w_gate_up [E,2I,H]; w_down [E,H,I]; lora_a_gu [L,E,2,R,H]; lora_b_gu [L,E,2,I,R];
    lora_a_down [L,E,R,I]; lora_b_down [L,E,H,R].  Weight operands must all share
    one dtype (bf16 bits or float64).
    """
    x_np = np.asarray(x)
    T, H = x_np.shape
    topk_ids = _i32(topk_ids)
    K = topk_ids.shape[1]
    topk_weights = np.ascontiguousarray(np.asarray(topk_weights, dtype=np.float32))
    mapping = _i32(token_lora_mapping)
    lora_ranks = _i32(lora_ranks)
    scalings = np.ascontiguousarray(np.asarray(scalings, dtype=np.float32))
    E, I2, H2 = np.asarray(w_gate_up).shape
    I = I2 // 2
    L, _, _, R, _ = np.asarray(lora_a_gu).shape
    assert H2 == H and np.asarray(w_down).shape == (E, H, I)
    assert np.asarray(lora_b_gu).shape == (L, E, 2, I, R)
    assert np.asarray(lora_a_down).shape == (L, E, R, I)
    assert np.asarray(lora_b_down).shape == (L, E, H, R)
    xp, xdt, xk = _operand(x_np)
    ops = [_operand(a) for a in (w_gate_up, w_down, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down)]
    wdt = ops[0][1]
    if any(o[1] != wdt for o in ops):
        raise TypeError("weight operands must share one dtype")
    if tokens is None:
        tok = None
        n_out = T
        tok_ptr = None
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        n_out = tok.shape[0]
        tok_ptr = tok.ctypes.data
    y = np.zeros((n_out, H), dtype=np.float64)
    st = _load().oracle_forward(
        xp, xdt, topk_ids.ctypes.data, topk_weights.ctypes.data, mapping.ctypes.data,
        lora_ranks.ctypes.data, scalings.ctypes.data,
        ops[0][0], ops[1][0], ops[2][0], ops[3][0], ops[4][0], ops[5][0], wdt,
        T, K, E, H, I, L, R, tok_ptr, n_out, y.ctypes.data, int(threads))
    del xk, tok
    return int(st), y


def e4m3_value(code: int) -> float:
    """The value of an FP8 E4M3 code (0..255)."""
    return float(_load().oracle_e4m3_value(int(code)))


def forward_fp8(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                w_gate_up_q, w_gate_up_scale, w_down_q, w_down_scale,
                lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens=None, threads: int = 0):
    """The layer with FP8 E4M3 base experts.  Returns (status, y) with y float64.

    w_gate_up_q [E,2I,H] and w_down_q [E,H,I] are uint8 E4M3 codes;
    w_gate_up_scale [E,ceil(2I/128),ceil(H/128)] and w_down_scale
    [E,ceil(H/128),ceil(I/128)] float32 scales of their 128 x 128 blocks.  The
    other operands are as in forward() (LoRA operands share one dtype).
    """
    x_np = np.asarray(x)
    T, H = x_np.shape
    topk_ids = _i32(topk_ids)
    K = topk_ids.shape[1]
    topk_weights = np.ascontiguousarray(np.asarray(topk_weights, dtype=np.float32))
    mapping = _i32(token_lora_mapping)
    lora_ranks = _i32(lora_ranks)
    scalings = np.ascontiguousarray(np.asarray(scalings, dtype=np.float32))
    wq = np.ascontiguousarray(np.asarray(w_gate_up_q, dtype=np.uint8))
    dq = np.ascontiguousarray(np.asarray(w_down_q, dtype=np.uint8))
    E, I2, H2 = wq.shape
    I = I2 // 2
    L, _, _, R, _ = np.asarray(lora_a_gu).shape
    assert H2 == H and dq.shape == (E, H, I)
    ws = np.ascontiguousarray(np.asarray(w_gate_up_scale, dtype=np.float32))
    ds = np.ascontiguousarray(np.asarray(w_down_scale, dtype=np.float32))
    assert ws.shape == (E, (2 * I + 127) // 128, (H + 127) // 128)
    assert ds.shape == (E, (H + 127) // 128, (I + 127) // 128)
    assert np.asarray(lora_b_gu).shape == (L, E, 2, I, R)
    assert np.asarray(lora_a_down).shape == (L, E, R, I)
    assert np.asarray(lora_b_down).shape == (L, E, H, R)
    xp, xdt, xk = _operand(x_np)
    ops = [_operand(a) for a in (lora_a_gu, lora_b_gu, lora_a_down, lora_b_down)]
    ldt = ops[0][1]
    if any(o[1] != ldt for o in ops):
        raise TypeError("LoRA operands must share one dtype")
    if tokens is None:
        tok, n_out, tok_ptr = None, T, None
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        n_out, tok_ptr = tok.shape[0], tok.ctypes.data
    y = np.zeros((n_out, H), dtype=np.float64)
    st = _load().oracle_forward_fp8(
        xp, xdt, topk_ids.ctypes.data, topk_weights.ctypes.data, mapping.ctypes.data,
        lora_ranks.ctypes.data, scalings.ctypes.data, wq.ctypes.data, ws.ctypes.data,
        dq.ctypes.data, ds.ctypes.data, ops[0][0], ops[1][0], ops[2][0], ops[3][0], ldt,
        T, K, E, H, I, L, R, tok_ptr, n_out, y.ctypes.data, int(threads))
    del xk, tok
    return int(st), y


def _quant_common(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                  lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens):
    x_np = np.asarray(x)
    T, H = x_np.shape
    topk_ids = _i32(topk_ids)
    c = dict(T=T, H=H, K=topk_ids.shape[1], topk_ids=topk_ids,
             topk_weights=np.ascontiguousarray(np.asarray(topk_weights, dtype=np.float32)),
             mapping=_i32(token_lora_mapping), lora_ranks=_i32(lora_ranks),
             scalings=np.ascontiguousarray(np.asarray(scalings, dtype=np.float32)))
    L, E, _, R, _ = np.asarray(lora_a_gu).shape
    c.update(L=L, E=E, R=R)
    c["x"] = _operand(x_np)
    ops = [_operand(a) for a in (lora_a_gu, lora_b_gu, lora_a_down, lora_b_down)]
    ldt = ops[0][1]
    if any(o[1] != ldt for o in ops):
        raise TypeError("LoRA operands must share one dtype")
    c.update(ops=ops, ldt=ldt)
    if tokens is None:
        c.update(tok=None, n_out=T, tok_ptr=None)
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        c.update(tok=tok, n_out=tok.shape[0], tok_ptr=tok.ctypes.data)
    return c


def forward_int8(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                 w_gate_up_q, w_gate_up_scale, w_down_q, w_down_scale,
                 lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens=None, threads: int = 0):
    """The layer with block-wise INT8 base experts.  Returns (status, y) float64.

    w_gate_up_q [E,2I,H] and w_down_q [E,H,I] hold int8 codes (int8 or uint8
    arrays of the two's-complement bytes); the scales are float32 per 128 x 128
    block, laid out as in forward_fp8; weight = code x scale.
    """
    c = _quant_common(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                      lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens)
    wq = np.ascontiguousarray(np.asarray(w_gate_up_q).view(np.uint8))
    dq = np.ascontiguousarray(np.asarray(w_down_q).view(np.uint8))
    T, H, K, E, L, R = c["T"], c["H"], c["K"], c["E"], c["L"], c["R"]
    I = wq.shape[1] // 2
    assert wq.shape == (E, 2 * I, H) and dq.shape == (E, H, I)
    ws = np.ascontiguousarray(np.asarray(w_gate_up_scale, dtype=np.float32))
    ds = np.ascontiguousarray(np.asarray(w_down_scale, dtype=np.float32))
    assert ws.shape == (E, (2 * I + 127) // 128, (H + 127) // 128)
    assert ds.shape == (E, (H + 127) // 128, (I + 127) // 128)
    y = np.zeros((c["n_out"], H), dtype=np.float64)
    ops = c["ops"]
    st = _load().oracle_forward_int8(
        c["x"][0], c["x"][1], c["topk_ids"].ctypes.data, c["topk_weights"].ctypes.data, c["mapping"].ctypes.data,
        c["lora_ranks"].ctypes.data, c["scalings"].ctypes.data, wq.ctypes.data, ws.ctypes.data,
        dq.ctypes.data, ds.ctypes.data, ops[0][0], ops[1][0], ops[2][0], ops[3][0], c["ldt"],
        T, K, E, H, I, L, R, c["tok_ptr"], c["n_out"], y.ctypes.data, int(threads))
    return int(st), y


def e4m3_round(v: float) -> float:
    """The nearest E4M3 value to v (ties to even); |v| <= 448."""
    return float(_load().oracle_e4m3_round(float(v)))


def mx_group_exp(amax: float) -> int:
    """The power-of-two scale exponent of a 128-element group with largest magnitude amax."""
    return int(_load().oracle_mx_group_exp(float(amax)))


def forward_fp8_w8a8(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                     w_gate_up_q, w_gate_up_exp, w_down_q, w_down_exp,
                     lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens=None, threads: int = 0):
    """The layer on FP8 tensor cores: W8A8 with power-of-two block scales.  Returns (status, y) float64.

    w_gate_up_q [E,2I,H] and w_down_q [E,H,I] hold E4M3 codes (uint8 bytes);
    w_gate_up_exp [E,ceil(2I/128),ceil(H/128)] and w_down_exp
    [E,ceil(H/128),ceil(I/128)] the biased exponent e of each 128 x 128 block
    (scale 2^(e-127)).  x and the intermediate are quantised per token and
    128-channel group before the base GEMMs; the LoRA paths read them unquantised.
    """
    c = _quant_common(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                      lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens)
    wq = np.ascontiguousarray(np.asarray(w_gate_up_q).view(np.uint8))
    dq = np.ascontiguousarray(np.asarray(w_down_q).view(np.uint8))
    T, H, K, E, L, R = c["T"], c["H"], c["K"], c["E"], c["L"], c["R"]
    I = wq.shape[1] // 2
    assert wq.shape == (E, 2 * I, H) and dq.shape == (E, H, I)
    we = np.ascontiguousarray(np.asarray(w_gate_up_exp, dtype=np.uint8))
    de = np.ascontiguousarray(np.asarray(w_down_exp, dtype=np.uint8))
    assert we.shape == (E, (2 * I + 127) // 128, (H + 127) // 128)
    assert de.shape == (E, (H + 127) // 128, (I + 127) // 128)
    y = np.zeros((c["n_out"], H), dtype=np.float64)
    ops = c["ops"]
    st = _load().oracle_forward_fp8_w8a8(
        c["x"][0], c["x"][1], c["topk_ids"].ctypes.data, c["topk_weights"].ctypes.data, c["mapping"].ctypes.data,
        c["lora_ranks"].ctypes.data, c["scalings"].ctypes.data, wq.ctypes.data, we.ctypes.data,
        dq.ctypes.data, de.ctypes.data, ops[0][0], ops[1][0], ops[2][0], ops[3][0], c["ldt"],
        T, K, E, H, I, L, R, c["tok_ptr"], c["n_out"], y.ctypes.data, int(threads))
    return int(st), y


def forward_w4a16(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                  w_gate_up_q, w_gate_up_scale, w_gate_up_zero, w_down_q, w_down_scale, w_down_zero,
                  lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens=None, threads: int = 0):
    """The layer with 4-bit base experts and 16-bit activations.  Returns (status, y).

    w_gate_up_q [E,2I,H/2] and w_down_q [E,H,I/2] are uint8 bytes each holding
    two uint4 codes (the even column in the low nibble); w_*_scale float32 and
    w_*_zero uint8 (0..15) are [E, rows, ceil(cols/128)]: one scale and zero
    point per row and group of 128 columns; weight = (code - zero) x scale.
    """
    c = _quant_common(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                      lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, tokens)
    T, H, K, E, L, R = c["T"], c["H"], c["K"], c["E"], c["L"], c["R"]
    wq = np.ascontiguousarray(np.asarray(w_gate_up_q, dtype=np.uint8))
    dq = np.ascontiguousarray(np.asarray(w_down_q, dtype=np.uint8))
    I = wq.shape[1] // 2
    assert wq.shape == (E, 2 * I, H // 2) and dq.shape == (E, H, I // 2)
    arrs = []
    for a, dt, shp in ((w_gate_up_scale, np.float32, (E, 2 * I, (H + 127) // 128)),
                       (w_gate_up_zero, np.uint8, (E, 2 * I, (H + 127) // 128)),
                       (w_down_scale, np.float32, (E, H, (I + 127) // 128)),
                       (w_down_zero, np.uint8, (E, H, (I + 127) // 128))):
        a = np.ascontiguousarray(np.asarray(a, dtype=dt))
        assert a.shape == shp
        arrs.append(a)
    y = np.zeros((c["n_out"], H), dtype=np.float64)
    ops = c["ops"]
    st = _load().oracle_forward_w4a16(
        c["x"][0], c["x"][1], c["topk_ids"].ctypes.data, c["topk_weights"].ctypes.data, c["mapping"].ctypes.data,
        c["lora_ranks"].ctypes.data, c["scalings"].ctypes.data, wq.ctypes.data, arrs[0].ctypes.data,
        arrs[1].ctypes.data, dq.ctypes.data, arrs[2].ctypes.data, arrs[3].ctypes.data,
        ops[0][0], ops[1][0], ops[2][0], ops[3][0], c["ldt"],
        T, K, E, H, I, L, R, c["tok_ptr"], c["n_out"], y.ctypes.data, int(threads))
    return int(st), y


def lora_linear(x, token_lora_mapping, lora_ranks, scalings, w, lora_a, lora_b, slice_offsets,
                tokens=None, threads: int = 0):
    """Dense projection with per-segment LoRA and split B.  Returns (status, y)
    with y float64 [len(tokens) or T, D_out].

    Shapes: x [T, D_in]; w [D_out, D_in]; lora_a [L, S, R, D_in] (part s has its
    own A); lora_b [L, D_out, R] (rows slice_offsets[s] .. slice_offsets[s+1]
    multiply part s's z); slice_offsets: S + 1 increasing ints from 0 to D_out.
    """
    x_np = np.asarray(x)
    T, D_in = x_np.shape
    mapping = _i32(token_lora_mapping)
    lora_ranks = _i32(lora_ranks)
    scalings = np.ascontiguousarray(np.asarray(scalings, dtype=np.float32))
    D_out, D_in2 = np.asarray(w).shape
    L, S, R, D_in3 = np.asarray(lora_a).shape
    assert D_in2 == D_in and D_in3 == D_in and np.asarray(lora_b).shape == (L, D_out, R)
    offs = np.ascontiguousarray(np.asarray(slice_offsets, dtype=np.int64))
    assert offs.shape == (S + 1,)
    xp, xdt, xk = _operand(x_np)
    ops = [_operand(a) for a in (w, lora_a, lora_b)]
    wdt = ops[0][1]
    if any(o[1] != wdt for o in ops):
        raise TypeError("weight operands must share one dtype")
    if tokens is None:
        tok, n_out, tok_ptr = None, T, None
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        n_out, tok_ptr = tok.shape[0], tok.ctypes.data
    y = np.zeros((n_out, D_out), dtype=np.float64)
    st = _load().oracle_lora_linear(
        xp, xdt, mapping.ctypes.data, lora_ranks.ctypes.data, scalings.ctypes.data,
        ops[0][0], ops[1][0], ops[2][0], wdt, T, D_in, D_out, L, R, S, offs.ctypes.data,
        tok_ptr, n_out, y.ctypes.data, int(threads))
    del xk, tok
    return int(st), y


def tp_qkv_b_rows(num_heads: int, num_kv_heads: int, head_dim: int, tp_size: int, tp_rank: int):
    """Rows of a fused q/k/v LoRA B held by one tensor-parallel rank, or None.

    [PR24420] page ("qkv_proj LoRA B sizing under KV-head replication"),
    关键源码片段, restated in two steps as the page gives them:
      1. the per-rank B output size (mem_pool.py): an even split of
         q + 2 kv rows, unless tp_size exceeds the KV heads; then 1/tp of q
         plus one whole head (head_dim rows) of k and of v;
      2. the rows taken (layers.py slice_lora_b_weights): q rows
         [q_shard * rank, +q_shard); k and v rows of KV shard rank // replicas
         (replicas = tp_size / num_kv_heads when the heads are replicated, else
         1), offset by the full q size and, for v, the full k size.
    Returns ([(q0, q1), (k0, k1), (v0, v1)], per_rank_rows).
    """
    if min(num_heads, num_kv_heads, head_dim, tp_size) < 1 or not 0 <= tp_rank < tp_size:
        return None
    if num_heads % tp_size:
        return None
    q_size = num_heads * head_dim
    k_size = num_kv_heads * head_dim  # the k block of B, as the checkpoint stores it
    replicated = tp_size > num_kv_heads
    if replicated and tp_size % num_kv_heads:
        return None
    if not replicated and num_kv_heads % tp_size:
        return None
    # step 1: the per-rank size
    if not replicated:
        per_rank = (q_size + 2 * k_size) // tp_size
    else:
        per_rank = q_size // tp_size + 2 * head_dim
    # step 2: the slices
    replicas = tp_size // num_kv_heads if replicated else 1
    q_shard = q_size // tp_size
    kv_shard = head_dim if replicated else k_size // tp_size
    kv_id = tp_rank // replicas
    q = (q_shard * tp_rank, q_shard * (tp_rank + 1))
    k = (q_size + kv_shard * kv_id, q_size + kv_shard * (kv_id + 1))
    v = (q_size + k_size + kv_shard * kv_id, q_size + k_size + kv_shard * (kv_id + 1))
    assert per_rank == sum(b - a for a, b in (q, k, v))
    return [q, k, v], per_rank
