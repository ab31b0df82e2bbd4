"""Expert parallelism across two processes on CPU (gloo, world size 2).

Each rank holds its own batch and only half of the experts.  The pairs are
ordered by owner with the oracle's dispatch, exchanged with the library's
TorchDistExchange (torch.distributed all_to_all_single, here over gloo on CPU
tensors), each owner runs the oracle layer on the rows it received (top-1
routing over its local experts), the weighted rows travel back through the
same exchange and are combined.  Every rank's result must equal the oracle
layer on its own batch over all experts.  No GPU is involved: this checks the
exchange plumbing (split sizes, order of the returned rows) and the protocol.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

KEYS = ("w_gate_up", "w_down", "lora_a_gu", "lora_b_gu", "lora_a_down", "lora_b_down")
DIMS = (0, 0, 1, 1, 1, 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits(a):
    return a.contiguous().view(torch.int16).numpy().view(np.uint16)


def _worker(rank, world, port, out):
    import oracle
    from oracle import ep as oep
    from lora_moe_expert_info_gb300 import workloads
    from lora_moe_expert_info_gb300.ep import TorchDistExchange, local_expert_slice
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        E, K, H, I, L, R, T = 8, 2, 64, 32, 3, 16, 24 + 7 * rank
        cfg = workloads.custom_config(hidden=H, intermediate=I, num_experts=E, topk=K, num_loras=L, max_rank=R,
                                      num_tokens=T)
        ranks = np.array([8, 0, 16], dtype=np.int32)
        scal = np.array([0.5, 0.0, 0.5], dtype=np.float32)
        w = workloads.make_weights(cfg, torch.from_numpy(ranks), seed=11, lora_std="fan_in")  # same on every rank
        local = [_bits(local_expert_slice(getattr(w, k), rank, world, d)) for k, d in zip(KEYS, DIMS)]
        g = torch.Generator().manual_seed(100 + rank)                                       # own batch
        x = torch.randn(T, H, generator=g).to(torch.bfloat16)
        ids, wts = workloads.route(T, E, K, g, "cpu")
        mapping = torch.randint(-1, L, (T,), generator=g).int()
        st, order, counts, pos = oep.ep_dispatch(ids.numpy(), E, world)
        assert st == oep.OK
        ex = TorchDistExchange()
        send = counts.tolist()
        recv = ex.counts(torch.from_numpy(counts))
        per = E // world
        flat_ids = ids.reshape(-1)[torch.from_numpy(order).long()]
        send_x = x[torch.from_numpy(order // K).long()]
        send_e = (flat_ids % per).int()
        send_w = wts.reshape(-1)[torch.from_numpy(order).long()]
        send_l = mapping[torch.from_numpy(order // K).long()]
        rx, re = ex.rows(send_x, send, recv), ex.rows(send_e, send, recv)
        rw, rl = ex.rows(send_w, send, recv), ex.rows(send_l, send, recv)
        n = rx.shape[0]
        st, rows = oracle.forward(_bits(rx), re.numpy().reshape(n, 1), rw.numpy().reshape(n, 1), rl.numpy(),
                                  ranks, scal, *local)
        assert st == 0
        back = ex.rows(torch.from_numpy(rows), recv, send)
        y = oep.ep_combine(back.numpy(), pos, T, K)
        st, y_ref = oracle.forward(_bits(x), ids.numpy(), wts.numpy(), mapping.numpy(), ranks, scal,
                                   *[_bits(getattr(w, k)) for k in KEYS])
        assert st == 0
        out[rank] = (float(np.abs(y - y_ref).max()), float(np.abs(y_ref).max()), send, recv)
    finally:
        dist.destroy_process_group()


def test_two_ranks_match_the_single_process_layer():
    import oracle
    oracle.build()
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    for rank in range(world):
        err, scale, send, recv = got[rank]
        assert scale > 0.1
        assert err <= 1e-12 * scale
    # what rank 0 sent to rank 1 is what rank 1 received from rank 0, and back
    assert got[0][2][1] == got[1][3][0] and got[1][2][0] == got[0][3][1]
    assert sum(got[0][2]) == 2 * (24 + 0) and sum(got[1][2]) == 2 * (24 + 7)
