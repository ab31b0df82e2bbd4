"""Expert parallelism over ranks: dispatch, exchange, owner forward, combine.

The experts are split over n ranks in equal contiguous ranges (rank d owns
experts [d*E/n, (d+1)*E/n)) and each rank holds only its experts' weights and
LoRA stacks ([L, E/n, ...]).  One step on every rank:

  1. ep_dispatch (CUDA): this rank's (token, slot) pairs packed by owner rank,
     each rank's in increasing pair order, with pair_pos recording the place
     of every pair;
  2. an all-to-all of the packed rows (`Exchange`; torch.distributed on the
     caller's process group, NCCL between GPUs);
  3. fused_moe_lora_forward on the received rows with top-1 routing over the
     local experts: each output row is w * (expert output);
  4. the reverse all-to-all returns those rows in this rank's send order;
  5. ep_combine (CUDA): y_t = sum over k, in increasing k, of t's rows.

Only the exchange moves data between GPUs, and it is the process group's
collective; every arithmetic step runs in the library's kernels.
"""
from __future__ import annotations

import ctypes
from typing import List, Optional

import torch

from . import (_check_device, _check_host, _on_stream, _ptr, _req, _stream, fused_moe_lora_forward,
               library)

__all__ = ["ep_dispatch", "ep_combine", "ep_fused_moe_lora_forward", "Exchange", "TorchDistExchange",
           "local_expert_slice"]


def _lib():
    lib = library()
    if not hasattr(lib.moe_lora_ep_dispatch, "_mlr_typed"):
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        lib.moe_lora_ep_workspace_bytes.restype = ctypes.c_size_t
        lib.moe_lora_ep_workspace_bytes.argtypes = [i32, i32, i32]
        lib.moe_lora_ep_dispatch.restype = ctypes.c_int
        lib.moe_lora_ep_dispatch.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                             vp, ctypes.c_size_t, vp, vp]
        lib.moe_lora_ep_combine.restype = ctypes.c_int
        lib.moe_lora_ep_combine.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        lib.moe_lora_ep_dispatch._mlr_typed = True
    return lib


@_on_stream
def ep_dispatch(x, topk_ids, topk_weights, token_lora_mapping, num_experts: int, n_ranks: int,
                stream=None, check: bool = True):
    """Packs this rank's pairs by owner rank.  Returns a dict with send_x
    [T*K, H], send_expert, send_weight, send_lora [T*K] (the first
    sum(send_counts) rows are valid), send_counts int32 [n_ranks] (device) and
    pair_pos int32 [T*K] (-1 for a dropped pair)."""
    lib = _lib()
    dev = x.device
    _req(x, "x", torch.bfloat16, dev)
    _req(topk_ids, "topk_ids", torch.int32, dev)
    _req(topk_weights, "topk_weights", torch.float32, dev)
    _req(token_lora_mapping, "token_lora_mapping", torch.int32, dev)
    T, H = x.shape
    K = topk_ids.shape[1]
    if tuple(topk_ids.shape) != (T, K) or tuple(topk_weights.shape) != (T, K) or token_lora_mapping.numel() < T:
        raise ValueError("ep_dispatch: inconsistent shapes")
    P = T * K
    out = {"send_x": torch.empty(P, H, dtype=torch.bfloat16, device=dev),
           "send_expert": torch.empty(P, dtype=torch.int32, device=dev),
           "send_weight": torch.empty(P, dtype=torch.float32, device=dev),
           "send_lora": torch.empty(P, dtype=torch.int32, device=dev),
           "send_counts": torch.zeros(n_ranks, dtype=torch.int32, device=dev),
           "pair_pos": torch.empty(P, dtype=torch.int32, device=dev)}
    wsb = int(lib.moe_lora_ep_workspace_bytes(T, K, n_ranks))
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev) if check else None
    code = lib.moe_lora_ep_dispatch(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(token_lora_mapping), T, K, H,
                                    int(num_experts), int(n_ranks), _ptr(out["send_x"]), _ptr(out["send_expert"]),
                                    _ptr(out["send_weight"]), _ptr(out["send_lora"]), _ptr(out["send_counts"]),
                                    _ptr(out["pair_pos"]), _ptr(ws), ws.numel(), _ptr(status), _stream(stream))
    _check_host(code, "moe_lora_ep_dispatch")
    if check:
        _check_device(status, "moe_lora_ep_dispatch")
    return out


@_on_stream
def ep_combine(rows, pair_pos, num_tokens: int, topk: int, y: Optional[torch.Tensor] = None, stream=None):
    """y[t] = sum over k (increasing) of rows[pair_pos[t*K + k]], skipping -1."""
    lib = _lib()
    dev = pair_pos.device
    _req(pair_pos, "pair_pos", torch.int32, dev)
    _req(rows, "rows", torch.bfloat16, dev)
    H = rows.shape[1]
    if y is None:
        y = torch.empty(num_tokens, H, dtype=torch.bfloat16, device=dev)
    _req(y, "y", torch.bfloat16, dev)
    code = lib.moe_lora_ep_combine(_ptr(rows) if rows.numel() else None, _ptr(pair_pos), int(num_tokens),
                                   int(topk), H, _ptr(y), _stream(stream))
    _check_host(code, "moe_lora_ep_combine")
    return y


def local_expert_slice(t: torch.Tensor, rank: int, n_ranks: int, dim: int) -> torch.Tensor:
    """A rank's experts of a stacked tensor (load time): the contiguous range
    [rank*E/n, (rank+1)*E/n) of dimension `dim`."""
    E = t.shape[dim]
    if E % n_ranks:
        raise ValueError("the experts must split evenly over the ranks")
    per = E // n_ranks
    return t.narrow(dim, rank * per, per).contiguous()


class Exchange:
    """All-to-all of row tensors between the ranks of one step."""

    def counts(self, send_counts: torch.Tensor) -> List[int]:
        raise NotImplementedError

    def rows(self, t: torch.Tensor, send: List[int], recv: List[int]) -> torch.Tensor:
        raise NotImplementedError


class TorchDistExchange(Exchange):
    """torch.distributed all_to_all_single on a process group (NCCL between
    GPUs; gloo on CPU tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group

    def counts(self, send_counts: torch.Tensor) -> List[int]:
        recv = torch.empty_like(send_counts)
        self.dist.all_to_all_single(recv, send_counts.contiguous(), group=self.group)
        return [int(v) for v in recv.cpu().tolist()]

    def rows(self, t: torch.Tensor, send: List[int], recv: List[int]) -> torch.Tensor:
        out = torch.empty((sum(recv),) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        self.dist.all_to_all_single(out, t[:sum(send)].contiguous(), output_split_sizes=recv,
                                    input_split_sizes=send, group=self.group)
        return out


def ep_fused_moe_lora_forward(x, topk_ids, topk_weights, token_lora_mapping, lora_ranks, scalings,
                              w_gate_up, w_down, lora_a_gu, lora_b_gu, lora_a_down, lora_b_down,
                              num_experts: int, exchange: Exchange, n_ranks: int):
    """One expert-parallel step of the layer on this rank.  The weights are this
    rank's experts only (w_gate_up [E/n, 2I, H], lora_a_gu [L, E/n, 2, R, H],
    ...); x, topk_ids (global expert ids), topk_weights and the mapping are this
    rank's own tokens.  Returns y bf16 [T, H]."""
    T, H = x.shape
    K = topk_ids.shape[1]
    d = ep_dispatch(x, topk_ids, topk_weights, token_lora_mapping, num_experts, n_ranks)
    send = [int(v) for v in d["send_counts"].cpu().tolist()]
    recv = exchange.counts(d["send_counts"])
    rx = exchange.rows(d["send_x"], send, recv)
    re = exchange.rows(d["send_expert"], send, recv)
    rw = exchange.rows(d["send_weight"], send, recv)
    rl = exchange.rows(d["send_lora"], send, recv)
    n = rx.shape[0]
    y_rows = fused_moe_lora_forward(rx, re.view(n, 1), rw.view(n, 1), rl, lora_ranks, scalings, w_gate_up, w_down,
                                    lora_a_gu, lora_b_gu, lora_a_down, lora_b_down)
    back = exchange.rows(y_rows, recv, send)
    return ep_combine(back, d["pair_pos"], T, K)
