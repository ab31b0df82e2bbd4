"""Python binding of the sm_103a LoRA MoE expert-layer library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_lib/libmoe_lora.so`` behind the C ABI in ``include/moe_lora.h``.
PyTorch supplies device memory (outputs, workspace) and the current stream.
The functions carry the C names:

  moe_lora_batch_info    -- per batch: token_lora_mapping, adapter_enabled
  moe_lora_align         -- per layer: (expert, adapter) buckets padded to block_size
  fused_moe_lora_forward -- the LoRA MoE expert layer

If the library has not been built (``__graft_entry__.build()`` or
``python -m lora_moe_expert_info_gb300._build``) every call raises: there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import functools
import inspect
import os
import threading
from typing import Optional, Tuple

import torch

from . import _build

__all__ = ["moe_lora_batch_info", "moe_lora_align", "moe_lora_align_capacity",
           "moe_lora_align_workspace_bytes", "fused_moe_lora_forward", "fused_moe_lora_forward_fp8",
           "fused_moe_lora_forward_int8", "fused_moe_lora_forward_w4a16", "fused_moe_lora_forward_fp8_w8a8",
           "fused_moe_lora_workspace_bytes", "fused_moe_lora_workspace_bytes_fp8_w8a8", "lora_linear_forward", "lora_tp_qkv_b_rows", "tp_take_rows",
           "set_wait_limit_ns", "wait_limit_ns", "set_deterministic", "deterministic", "library", "library_path", "MoeLoraError", "STATUS_BITS"]

MLR_OK = 0
MLR_ERR_INVALID = -1
MLR_ERR_UNDERCOVERED = -2
MLR_ERR_INDEX = -3
MLR_ERR_CAPACITY = -4
MLR_ERR_CUDA = -5
MLR_ERR_TIMEOUT = -6
MLR_ERR_UNSUPPORTED = -8

STATUS_BITS = {0x01: "bad seg_indptr", 0x02: "under-covers tokens", 0x04: "id out of range",
               0x08: "capacity exceeded", 0x10: "device wait timed out",
               0x20: "rank out of range"}

_lock = threading.Lock()
_lib = None


class MoeLoraError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(what)


def library_path() -> str:
    return _build.LIB


def library() -> ctypes.CDLL:
    """Load the in-tree CUDA library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    f"CUDA library {_build.LIB} is missing: run __graft_entry__.build() "
                    "(nvcc, sm_103a); there is no CPU fallback")
            lib = ctypes.CDLL(_build.LIB)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            lib.moe_lora_version.restype = ctypes.c_char_p
            lib.moe_lora_status_string.restype = ctypes.c_char_p
            lib.moe_lora_status_string.argtypes = [ctypes.c_int]
            lib.moe_lora_batch_info.restype = ctypes.c_int
            lib.moe_lora_batch_info.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
            lib.moe_lora_align_capacity.restype = i64
            lib.moe_lora_align_capacity.argtypes = [i32, i32, i32, i32, i32]
            lib.moe_lora_align_workspace_bytes.restype = sz
            lib.moe_lora_align_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            lib.moe_lora_align.restype = ctypes.c_int
            lib.moe_lora_align.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, i64,
                                           vp, sz, vp, vp]
            lib.moe_lora_profile_stages.restype = ctypes.c_int
            lib.moe_lora_profile_stages.argtypes = [ctypes.c_uint32]
            lib.moe_lora_profile_begin.restype = ctypes.c_int
            lib.moe_lora_profile_begin.argtypes = [i32]
            lib.moe_lora_profile_end.restype = ctypes.c_int
            lib.moe_lora_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), i32,
                                                 ctypes.POINTER(i32), ctypes.POINTER(i32)]
            lib.moe_lora_profile_stage_name.restype = ctypes.c_char_p
            lib.moe_lora_profile_stage_name.argtypes = [i32]
            lib.moe_lora_launch_count.restype = ctypes.c_uint64
            lib.moe_lora_launch_count.argtypes = []
            lib.moe_lora_set_wait_limit_ns.restype = ctypes.c_int
            lib.moe_lora_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.moe_lora_wait_limit_ns.restype = ctypes.c_uint64
            lib.moe_lora_wait_limit_ns.argtypes = []
            lib.moe_lora_set_deterministic.restype = ctypes.c_int
            lib.moe_lora_set_deterministic.argtypes = [i32]
            lib.moe_lora_deterministic.restype = i32
            lib.moe_lora_deterministic.argtypes = []
            if hasattr(lib, "fused_moe_lora_forward"):
                lib.fused_moe_lora_workspace_bytes.restype = sz
                lib.fused_moe_lora_workspace_bytes.argtypes = [i32] * 7
                lib.fused_moe_lora_forward.restype = ctypes.c_int
                lib.fused_moe_lora_forward.argtypes = [vp] * 12 + [i32] * 7 + [vp, vp, sz, vp, vp]
                lib.fused_moe_lora_forward_fp8.restype = ctypes.c_int
                lib.fused_moe_lora_forward_fp8.argtypes = [vp] * 14 + [i32] * 7 + [vp, vp, sz, vp, vp]
                lib.fused_moe_lora_forward_int8.restype = ctypes.c_int
                lib.fused_moe_lora_forward_int8.argtypes = [vp] * 14 + [i32] * 7 + [vp, vp, sz, vp, vp]
                lib.fused_moe_lora_forward_w4a16.restype = ctypes.c_int
                lib.fused_moe_lora_forward_w4a16.argtypes = [vp] * 16 + [i32] * 7 + [vp, vp, sz, vp, vp]
                lib.fused_moe_lora_workspace_bytes_fp8_w8a8.restype = sz
                lib.fused_moe_lora_workspace_bytes_fp8_w8a8.argtypes = [i32] * 7
                lib.fused_moe_lora_forward_fp8_w8a8.restype = ctypes.c_int
                lib.fused_moe_lora_forward_fp8_w8a8.argtypes = [vp] * 14 + [i32] * 7 + [vp, vp, sz, vp, vp]
            if hasattr(lib, "lora_linear_forward"):
                lib.lora_linear_workspace_bytes.restype = sz
                lib.lora_linear_workspace_bytes.argtypes = [i32] * 6
                lib.lora_linear_forward.restype = ctypes.c_int
                lib.lora_linear_forward.argtypes = [vp] * 8 + [i32] * 6 + [vp, vp, sz, vp, vp]
            if hasattr(lib, "lora_tp_qkv_b_rows"):
                lib.lora_tp_qkv_b_rows.restype = ctypes.c_int
                lib.lora_tp_qkv_b_rows.argtypes = [i32] * 5 + [ctypes.POINTER(i32), ctypes.POINTER(i32)]
            _lib = lib
    return _lib


def set_wait_limit_ns(ns: int) -> None:
    """Give-up limit of the GEMM kernels' pipeline waits for later launches
    (process-wide; default 2 s).  A wait that runs out sets the device status
    bit "device wait timed out" and the kernel returns early."""
    _check_host(library().moe_lora_set_wait_limit_ns(int(ns)), "moe_lora_set_wait_limit_ns")


def wait_limit_ns() -> int:
    return int(library().moe_lora_wait_limit_ns())


def set_deterministic(on: bool) -> None:
    """Top-k combine of the MoE forward for later calls (process-wide): False =
    fp32 atomic reductions (order-dependent last bits), True = per-pair rows
    summed in increasing k (bit-identical between runs)."""
    _check_host(library().moe_lora_set_deterministic(1 if on else 0), "moe_lora_set_deterministic")


def deterministic() -> bool:
    return bool(library().moe_lora_deterministic())


def _on_stream(fn):
    """Runs a wrapper with its `stream` argument as torch's current stream, so
    that the outputs, workspace and status word it allocates (and zeroes) are
    ordered on the stream the kernels are enqueued on, the caching allocator
    records them there, and the status read synchronises that stream."""
    sig = inspect.signature(fn)

    @functools.wraps(fn)
    def run(*args, **kw):
        bound = sig.bind(*args, **kw)
        s = bound.arguments.get("stream")
        if s is None:
            return fn(*args, **kw)
        with torch.cuda.stream(s):
            return fn(*args, **kw)
    return run


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_host(code: int, fn: str):
    if code == MLR_OK:
        return
    text = library().moe_lora_status_string(code).decode()
    if code == MLR_ERR_UNDERCOVERED:
        raise AssertionError(f"{fn}: launch under-covers tokens ({text})")
    if code == MLR_ERR_INVALID:
        raise ValueError(f"{fn}: {text}")
    raise MoeLoraError(code, f"{fn}: {text} (code {code})")


def _check_device(status: torch.Tensor, fn: str):
    bits = int(status.item())  # synchronises the stream
    if bits == 0:
        return
    names = ", ".join(v for k, v in STATUS_BITS.items() if bits & k)
    if bits & 0x02:
        raise AssertionError(f"{fn}: kernel under-covers tokens ({names})")
    if bits & 0x10:
        raise MoeLoraError(MLR_ERR_TIMEOUT, f"{fn}: {names}")
    raise MoeLoraError(MLR_ERR_INDEX if bits & 0x24 else MLR_ERR_CAPACITY, f"{fn}: {names}")


def _req(t: torch.Tensor, name: str, dtype, dev):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != dev:
        raise ValueError(f"{name} must be on {dev}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


@_on_stream
def moe_lora_batch_info(seg_indptr: torch.Tensor, weight_indices: torch.Tensor,
                        lora_ranks: torch.Tensor, num_tokens: int, max_len: int = 0,
                        adapter_enabled: Optional[torch.Tensor] = None,
                        token_lora_mapping: Optional[torch.Tensor] = None,
                        stream=None, check: bool = True) -> Tuple[torch.Tensor, torch.Tensor]:
    """Returns (adapter_enabled[num_loras], token_lora_mapping[num_tokens]).

    Preallocated buffers are written in place and the returned tensors alias
    them (the mapping view covers the first num_tokens entries).  With
    check=True the stream is synchronised and device-detected errors raise;
    an under-covering launch raises AssertionError("... under-covers tokens").
    """
    dev = seg_indptr.device
    for t, n in ((seg_indptr, "seg_indptr"), (weight_indices, "weight_indices"),
                 (lora_ranks, "lora_ranks")):
        _req(t, n, torch.int32, dev)
    bs, L = weight_indices.numel(), lora_ranks.numel()
    if seg_indptr.numel() != bs + 1:
        raise ValueError("seg_indptr must have bs + 1 entries")
    if adapter_enabled is None:
        adapter_enabled = torch.empty(L, dtype=torch.int32, device=dev)
    _req(adapter_enabled, "adapter_enabled", torch.int32, dev)
    if adapter_enabled.numel() != L:
        raise ValueError("adapter_enabled must have num_loras entries")
    if token_lora_mapping is None:
        token_lora_mapping = torch.empty(num_tokens, dtype=torch.int32, device=dev)
    _req(token_lora_mapping, "token_lora_mapping", torch.int32, dev)
    if token_lora_mapping.numel() < num_tokens:
        raise ValueError("token_lora_mapping holds fewer than num_tokens entries")
    status = torch.zeros(1, dtype=torch.int32, device=dev) if check else None
    code = library().moe_lora_batch_info(
        _ptr(seg_indptr), _ptr(weight_indices), _ptr(lora_ranks), bs, L, int(num_tokens),
        int(max_len), _ptr(token_lora_mapping), _ptr(adapter_enabled), _ptr(status), _stream(stream))
    _check_host(code, "moe_lora_batch_info")
    if check:
        _check_device(status, "moe_lora_batch_info")
    return adapter_enabled, token_lora_mapping[:num_tokens]


def moe_lora_align_capacity(num_tokens, topk, num_experts, num_loras, block_size) -> int:
    return int(library().moe_lora_align_capacity(num_tokens, topk, num_experts, num_loras, block_size))


def moe_lora_align_workspace_bytes(num_tokens, topk, num_experts, num_loras, block_size) -> int:
    return int(library().moe_lora_align_workspace_bytes(num_tokens, topk, num_experts, num_loras,
                                                        block_size))


@_on_stream
def moe_lora_align(topk_ids: torch.Tensor, token_lora_mapping: torch.Tensor, num_experts: int,
                   num_loras: int, block_size: int, out=None, workspace=None, stream=None,
                   check: bool = True):
    """Returns (sorted_token_ids, block_expert_ids, block_lora_ids, num_tokens_post_pad).

    The arrays have capacity length (moe_lora_align_capacity); the valid prefix
    is num_tokens_post_pad entries (a device int32[1]).  With check=True the
    stream is synchronised and device-detected errors raise.
    """
    dev = topk_ids.device
    _req(topk_ids, "topk_ids", torch.int32, dev)
    _req(token_lora_mapping, "token_lora_mapping", torch.int32, dev)
    if topk_ids.dim() != 2:
        raise ValueError("topk_ids must be [num_tokens, topk]")
    T, K = topk_ids.shape
    if token_lora_mapping.numel() < T:
        raise ValueError("token_lora_mapping holds fewer than num_tokens entries")
    lib = library()
    cap = int(lib.moe_lora_align_capacity(T, K, num_experts, num_loras, block_size))
    if cap < 0:
        raise ValueError("moe_lora_align: unsupported sizes")
    if out is None:
        out = (torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
               torch.empty(max(cap // block_size, 1), dtype=torch.int32, device=dev),
               torch.empty(max(cap // block_size, 1), dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev))
    sorted_ids, bexp, blora, npad = out
    wsb = int(lib.moe_lora_align_workspace_bytes(T, K, num_experts, num_loras, block_size))
    if workspace is None:
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev) if check else None
    code = lib.moe_lora_align(_ptr(topk_ids), _ptr(token_lora_mapping), T, K, num_experts, num_loras,
                              block_size, _ptr(sorted_ids), _ptr(bexp), _ptr(blora), _ptr(npad),
                              min(cap, sorted_ids.numel()), _ptr(workspace), workspace.numel(),
                              _ptr(status), _stream(stream))
    _check_host(code, "moe_lora_align")
    if check:
        _check_device(status, "moe_lora_align")
    return sorted_ids, bexp, blora, npad


def fused_moe_lora_workspace_bytes(T, K, E, H, I, L, R) -> int:
    return int(library().fused_moe_lora_workspace_bytes(T, K, E, H, I, L, R))


@_on_stream
def fused_moe_lora_forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                           w_gate_up, w_down, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down,
                           y: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None,
                           check: bool = True, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The LoRA MoE expert layer; returns y bf16 [T, H] (written in place if given).

    Shapes: x [T,H]; topk_ids, topk_weights [T,K]; token_lora_mapping [T];
    lora_ranks, scalings [L]; w_gate_up [E,2I,H]; w_down [E,H,I];
    lora_a_gu [L,E,2,R,H]; lora_b_gu [L,E,2,I,R]; lora_a_down [L,E,R,I];
    lora_b_down [L,E,H,R].
    """
    lib = library()
    if not hasattr(lib, "fused_moe_lora_forward"):
        raise RuntimeError("library built without fused_moe_lora_forward")
    dev = x.device
    bf = torch.bfloat16
    _req(x, "x", bf, dev)
    _req(topk_ids, "topk_ids", torch.int32, dev)
    _req(topk_weights, "topk_weights", torch.float32, dev)
    _req(token_lora_mapping, "token_lora_mapping", torch.int32, dev)
    _req(lora_ranks, "lora_ranks", torch.int32, dev)
    _req(scalings, "scalings", torch.float32, dev)
    for t, n in ((w_gate_up, "w_gate_up"), (w_down, "w_down"), (lora_a_gu, "lora_a_gu"),
                 (lora_b_gu, "lora_b_gu"), (lora_a_down, "lora_a_down"), (lora_b_down, "lora_b_down")):
        _req(t, n, bf, dev)
    T, H = x.shape
    K = topk_ids.shape[1]
    E, I2, H2 = w_gate_up.shape
    I = I2 // 2
    L, _, _, R, _ = lora_a_gu.shape
    if (H2 != H or tuple(w_down.shape) != (E, H, I) or tuple(lora_a_gu.shape) != (L, E, 2, R, H)
            or tuple(lora_b_gu.shape) != (L, E, 2, I, R) or tuple(lora_a_down.shape) != (L, E, R, I)
            or tuple(lora_b_down.shape) != (L, E, H, R) or tuple(topk_ids.shape) != (T, K)
            or tuple(topk_weights.shape) != (T, K) or token_lora_mapping.numel() < T
            or lora_ranks.numel() != L or scalings.numel() != L):
        raise ValueError("fused_moe_lora_forward: inconsistent shapes")
    if y is None:
        y = torch.empty(T, H, dtype=bf, device=dev)
    _req(y, "y", bf, dev)
    wsb = int(lib.fused_moe_lora_workspace_bytes(T, K, E, H, I, L, R))
    if wsb == 0 and T > 0:
        raise ValueError("fused_moe_lora_forward: unsupported sizes")
    if workspace is None:
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    if check and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = lib.fused_moe_lora_forward(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(token_lora_mapping), _ptr(lora_ranks),
        _ptr(scalings), _ptr(w_gate_up), _ptr(w_down), _ptr(lora_a_gu), _ptr(lora_b_gu),
        _ptr(lora_a_down), _ptr(lora_b_down), T, K, E, H, I, L, R, _ptr(y), _ptr(workspace),
        workspace.numel(), _ptr(status), _stream(stream))
    _check_host(code, "fused_moe_lora_forward")
    if check:
        _check_device(status, "fused_moe_lora_forward")
    return y


def _codes(t: torch.Tensor, name: str, dev) -> torch.Tensor:
    """FP8 E4M3 weights as their byte codes (uint8 or float8_e4m3fn tensors)."""
    if hasattr(torch, "float8_e4m3fn") and t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    _req(t, name, torch.uint8, dev)
    return t


@_on_stream
def fused_moe_lora_forward_fp8(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                               w_gate_up_q, w_gate_up_scale, w_down_q, w_down_scale,
                               lora_a_gu, lora_b_gu, lora_a_down, lora_b_down,
                               y: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, stream=None,
                               check: bool = True, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The layer with FP8 E4M3 base experts and 128 x 128 block scales.

    w_gate_up_q [E,2I,H] and w_down_q [E,H,I]: uint8 (or float8_e4m3fn) codes;
    w_gate_up_scale [E,ceil(2I/128),ceil(H/128)] and w_down_scale
    [E,ceil(H/128),ceil(I/128)]: float32, weight = code value x block scale.
    Everything else as in fused_moe_lora_forward.
    """
    lib = library()
    if not hasattr(lib, "fused_moe_lora_forward_fp8"):
        raise RuntimeError("library built without fused_moe_lora_forward_fp8")
    dev = x.device
    bf = torch.bfloat16
    _req(x, "x", bf, dev)
    _req(topk_ids, "topk_ids", torch.int32, dev)
    _req(topk_weights, "topk_weights", torch.float32, dev)
    _req(token_lora_mapping, "token_lora_mapping", torch.int32, dev)
    _req(lora_ranks, "lora_ranks", torch.int32, dev)
    _req(scalings, "scalings", torch.float32, dev)
    wq = _codes(w_gate_up_q, "w_gate_up_q", dev)
    dq = _codes(w_down_q, "w_down_q", dev)
    _req(w_gate_up_scale, "w_gate_up_scale", torch.float32, dev)
    _req(w_down_scale, "w_down_scale", torch.float32, dev)
    for t, n in ((lora_a_gu, "lora_a_gu"), (lora_b_gu, "lora_b_gu"), (lora_a_down, "lora_a_down"),
                 (lora_b_down, "lora_b_down")):
        _req(t, n, bf, dev)
    T, H = x.shape
    K = topk_ids.shape[1]
    E, I2, H2 = wq.shape
    I = I2 // 2
    L, _, _, R, _ = lora_a_gu.shape
    cb = lambda n: (n + 127) // 128  # noqa: E731
    if (H2 != H or tuple(dq.shape) != (E, H, I)
            or tuple(w_gate_up_scale.shape) != (E, cb(2 * I), cb(H))
            or tuple(w_down_scale.shape) != (E, cb(H), cb(I))
            or tuple(lora_a_gu.shape) != (L, E, 2, R, H)
            or tuple(lora_b_gu.shape) != (L, E, 2, I, R) or tuple(lora_a_down.shape) != (L, E, R, I)
            or tuple(lora_b_down.shape) != (L, E, H, R) or tuple(topk_ids.shape) != (T, K)
            or tuple(topk_weights.shape) != (T, K) or token_lora_mapping.numel() < T
            or lora_ranks.numel() != L or scalings.numel() != L):
        raise ValueError("fused_moe_lora_forward_fp8: inconsistent shapes")
    if y is None:
        y = torch.empty(T, H, dtype=bf, device=dev)
    _req(y, "y", bf, dev)
    wsb = int(lib.fused_moe_lora_workspace_bytes(T, K, E, H, I, L, R))
    if wsb == 0 and T > 0:
        raise ValueError("fused_moe_lora_forward_fp8: unsupported sizes")
    if workspace is None:
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    if check and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = lib.fused_moe_lora_forward_fp8(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(token_lora_mapping), _ptr(lora_ranks),
        _ptr(scalings), _ptr(wq), _ptr(w_gate_up_scale), _ptr(dq), _ptr(w_down_scale), _ptr(lora_a_gu),
        _ptr(lora_b_gu), _ptr(lora_a_down), _ptr(lora_b_down), T, K, E, H, I, L, R, _ptr(y),
        _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _check_host(code, "fused_moe_lora_forward_fp8")
    if check:
        _check_device(status, "fused_moe_lora_forward_fp8")
    return y


def _quant_forward(fn_name, x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings, quant,
                   lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, y, workspace, stream, check, status,
                   I_of, code_shapes, side_shapes, ws_fn="fused_moe_lora_workspace_bytes"):
    """Shared marshalling of the quantised-expert forwards: `quant` is the list of
    (tensor, name, dtype) of the code / scale / zero arrays in C argument order;
    code_shapes(E, I, H) and side_shapes(E, I, H) give their expected shapes."""
    lib = library()
    if not hasattr(lib, fn_name):
        raise RuntimeError(f"library built without {fn_name}")
    dev = x.device
    bf = torch.bfloat16
    _req(x, "x", bf, dev)
    _req(topk_ids, "topk_ids", torch.int32, dev)
    _req(topk_weights, "topk_weights", torch.float32, dev)
    _req(token_lora_mapping, "token_lora_mapping", torch.int32, dev)
    _req(lora_ranks, "lora_ranks", torch.int32, dev)
    _req(scalings, "scalings", torch.float32, dev)
    for t, n, dt in quant:
        _req(t, n, dt, dev)
    for t, n in ((lora_a_gu, "lora_a_gu"), (lora_b_gu, "lora_b_gu"), (lora_a_down, "lora_a_down"),
                 (lora_b_down, "lora_b_down")):
        _req(t, n, bf, dev)
    T, H = x.shape
    K = topk_ids.shape[1]
    E = quant[0][0].shape[0]
    I = I_of(quant[0][0])
    L, _, _, R, _ = lora_a_gu.shape
    expect = list(code_shapes(E, I, H)) + list(side_shapes(E, I, H))
    if (any(tuple(t.shape) != shp for (t, _, _), shp in zip(quant, expect))
            or tuple(lora_a_gu.shape) != (L, E, 2, R, H)
            or tuple(lora_b_gu.shape) != (L, E, 2, I, R) or tuple(lora_a_down.shape) != (L, E, R, I)
            or tuple(lora_b_down.shape) != (L, E, H, R) or tuple(topk_ids.shape) != (T, K)
            or tuple(topk_weights.shape) != (T, K) or token_lora_mapping.numel() < T
            or lora_ranks.numel() != L or scalings.numel() != L):
        raise ValueError(f"{fn_name}: inconsistent shapes")
    if y is None:
        y = torch.empty(T, H, dtype=bf, device=dev)
    _req(y, "y", bf, dev)
    wsb = int(getattr(lib, ws_fn)(T, K, E, H, I, L, R))
    if wsb == 0 and T > 0:
        raise ValueError(f"{fn_name}: unsupported sizes")
    if workspace is None:
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    if check and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = getattr(lib, fn_name)(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(token_lora_mapping), _ptr(lora_ranks),
        _ptr(scalings), *[_ptr(t) for t, _, _ in quant], _ptr(lora_a_gu), _ptr(lora_b_gu), _ptr(lora_a_down),
        _ptr(lora_b_down), T, K, E, H, I, L, R, _ptr(y), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream))
    _check_host(code, fn_name)
    if check:
        _check_device(status, fn_name)
    return y


@_on_stream
def fused_moe_lora_forward_int8(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                                w_gate_up_q, w_gate_up_scale, w_down_q, w_down_scale,
                                lora_a_gu, lora_b_gu, lora_a_down, lora_b_down,
                                y: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None, stream=None,
                                check: bool = True, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The layer with block-wise INT8 base experts: w_gate_up_q [E,2I,H] and
    w_down_q [E,H,I] int8 codes, scales laid out as for the FP8 layer
    (float32 per 128 x 128 block); weight = code x scale."""
    cb = lambda n: (n + 127) // 128  # noqa: E731
    quant = [(w_gate_up_q, "w_gate_up_q", torch.int8), (w_gate_up_scale, "w_gate_up_scale", torch.float32),
             (w_down_q, "w_down_q", torch.int8), (w_down_scale, "w_down_scale", torch.float32)]
    return _quant_forward("fused_moe_lora_forward_int8", x, topk_ids, topk_weights, token_lora_mapping,
                          lora_ranks, scalings, quant, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, y,
                          workspace, stream, check, status, lambda w: w.shape[1] // 2,
                          lambda E, I, H: [(E, 2 * I, H), (E, cb(2 * I), cb(H)), (E, H, I), (E, cb(H), cb(I))],
                          lambda E, I, H: [])


@_on_stream
def fused_moe_lora_forward_w4a16(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                                 w_gate_up_q, w_gate_up_scale, w_gate_up_zero, w_down_q, w_down_scale,
                                 w_down_zero, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down,
                                 y: Optional[torch.Tensor] = None,
                                 workspace: Optional[torch.Tensor] = None, stream=None,
                                 check: bool = True, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The layer with 4-bit base experts: w_gate_up_q [E,2I,H/2] and w_down_q
    [E,H,I/2] uint8 bytes of two uint4 codes (even column in the low nibble);
    scales (float32) and zero points (uint8) [E, rows, ceil(cols/128)], one per
    row and 128-column group; weight = (code - zero) x scale."""
    cb = lambda n: (n + 127) // 128  # noqa: E731
    quant = [(w_gate_up_q, "w_gate_up_q", torch.uint8), (w_gate_up_scale, "w_gate_up_scale", torch.float32),
             (w_gate_up_zero, "w_gate_up_zero", torch.uint8), (w_down_q, "w_down_q", torch.uint8),
             (w_down_scale, "w_down_scale", torch.float32), (w_down_zero, "w_down_zero", torch.uint8)]
    return _quant_forward("fused_moe_lora_forward_w4a16", x, topk_ids, topk_weights, token_lora_mapping,
                          lora_ranks, scalings, quant, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, y,
                          workspace, stream, check, status, lambda w: w.shape[1] // 2,
                          lambda E, I, H: [(E, 2 * I, H // 2), (E, 2 * I, cb(H)), (E, 2 * I, cb(H)),
                                           (E, H, I // 2), (E, H, cb(I)), (E, H, cb(I))],
                          lambda E, I, H: [])


def fused_moe_lora_workspace_bytes_fp8_w8a8(T, K, E, H, I, L, R) -> int:
    return int(library().fused_moe_lora_workspace_bytes_fp8_w8a8(T, K, E, H, I, L, R))


@_on_stream
def fused_moe_lora_forward_fp8_w8a8(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                                    w_gate_up_q, w_gate_up_exp, w_down_q, w_down_exp,
                                    lora_a_gu, lora_b_gu, lora_a_down, lora_b_down,
                                    y: Optional[torch.Tensor] = None,
                                    workspace: Optional[torch.Tensor] = None, stream=None,
                                    check: bool = True, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The layer on the FP8 tensor cores: w_gate_up_q [E,2I,H] and w_down_q
    [E,H,I] E4M3 codes (uint8), w_gate_up_exp [E,ceil(2I/128),ceil(H/128)] and
    w_down_exp [E,ceil(H/128),ceil(I/128)] uint8 biased block exponents (scale
    2^(e-127)); the activations of the base GEMMs are quantised per token and
    128-channel group on the way (see the C header)."""
    cb = lambda n: (n + 127) // 128  # noqa: E731
    quant = [(w_gate_up_q, "w_gate_up_q", torch.uint8), (w_gate_up_exp, "w_gate_up_exp", torch.uint8),
             (w_down_q, "w_down_q", torch.uint8), (w_down_exp, "w_down_exp", torch.uint8)]
    return _quant_forward("fused_moe_lora_forward_fp8_w8a8", x, topk_ids, topk_weights, token_lora_mapping,
                          lora_ranks, scalings, quant, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down, y,
                          workspace, stream, check, status, lambda w: w.shape[1] // 2,
                          lambda E, I, H: [(E, 2 * I, H), (E, cb(2 * I), cb(H)), (E, H, I), (E, cb(H), cb(I))],
                          lambda E, I, H: [], ws_fn="fused_moe_lora_workspace_bytes_fp8_w8a8")


@_on_stream
def lora_linear_forward(x, w, token_lora_mapping, lora_ranks, scalings, lora_a, lora_b, slice_offsets,
                        y: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None, check: bool = True,
                        status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Dense projection with per-segment LoRA and split B; returns y bf16 [T, D_out].

    Shapes: x [T, D_in]; w [D_out, D_in]; token_lora_mapping [T]; lora_ranks,
    scalings [L]; lora_a [L, S, R, D_in] (part s's A); lora_b [L, D_out, R];
    slice_offsets: S + 1 ints (host), 0 = offsets[0] < ... < offsets[S] = D_out.
    """
    lib = library()
    if not hasattr(lib, "lora_linear_forward"):
        raise RuntimeError("library built without lora_linear_forward")
    dev = x.device
    bf = torch.bfloat16
    _req(x, "x", bf, dev)
    _req(w, "w", bf, dev)
    _req(token_lora_mapping, "token_lora_mapping", torch.int32, dev)
    _req(lora_ranks, "lora_ranks", torch.int32, dev)
    _req(scalings, "scalings", torch.float32, dev)
    _req(lora_a, "lora_a", bf, dev)
    _req(lora_b, "lora_b", bf, dev)
    T, D_in = x.shape
    D_out = w.shape[0]
    L, S, R, _ = lora_a.shape
    offs = (ctypes.c_int32 * (S + 1))(*[int(v) for v in slice_offsets])
    if (len(slice_offsets) != S + 1 or tuple(w.shape) != (D_out, D_in) or tuple(lora_a.shape) != (L, S, R, D_in)
            or tuple(lora_b.shape) != (L, D_out, R) or token_lora_mapping.numel() < T
            or lora_ranks.numel() != L or scalings.numel() != L):
        raise ValueError("lora_linear_forward: inconsistent shapes")
    if y is None:
        y = torch.empty(T, D_out, dtype=bf, device=dev)
    _req(y, "y", bf, dev)
    wsb = int(lib.lora_linear_workspace_bytes(T, D_in, D_out, L, R, S))
    if wsb == 0 and T > 0:
        raise ValueError("lora_linear_forward: unsupported sizes")
    if workspace is None:
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    if check and status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = lib.lora_linear_forward(
        _ptr(x), _ptr(w), _ptr(token_lora_mapping), _ptr(lora_ranks), _ptr(scalings), _ptr(lora_a),
        _ptr(lora_b), ctypes.cast(offs, ctypes.c_void_p), T, D_in, D_out, L, R, S, _ptr(y), _ptr(workspace),
        workspace.numel(), _ptr(status), _stream(stream))
    _check_host(code, "lora_linear_forward")
    if check:
        _check_device(status, "lora_linear_forward")
    return y


def lora_tp_qkv_b_rows(num_heads: int, num_kv_heads: int, head_dim: int, tp_size: int, tp_rank: int):
    """Rows of a fused q/k/v projection's LoRA B (and base weight) that one
    tensor-parallel rank holds, with KV heads replicated when tp_size exceeds
    num_kv_heads.  Returns ([(q0, q1), (k0, k1), (v0, v1)], per_rank_rows)."""
    lib = library()
    r = (ctypes.c_int32 * 6)()
    n = ctypes.c_int32(0)
    code = lib.lora_tp_qkv_b_rows(num_heads, num_kv_heads, head_dim, tp_size, tp_rank, r, ctypes.byref(n))
    _check_host(code, "lora_tp_qkv_b_rows")
    return [(r[0], r[1]), (r[2], r[3]), (r[4], r[5])], int(n.value)


def tp_take_rows(t: torch.Tensor, ranges, dim: int = 0) -> torch.Tensor:
    """A rank's shard of an output-row-stacked tensor: the given row ranges of
    dimension `dim`, concatenated (load-time layout step, as for the rank's
    copy of W or LoRA B; the per-token path runs in lora_linear_forward)."""
    return torch.cat([t.narrow(dim, a, b - a) for a, b in ranges], dim=dim).contiguous()
