"""moe_lora_align_noalloc: the align for callers that cannot allocate device memory.

Some callers of this library may not allocate GPU memory at all (engines that
own every byte through their own pools, latency-critical paths where
cudaMalloc/cudaFree could synchronise the device, layers given no allocator).
The no-allocation entry point keeps its scratch in a fixed array inside the
library.  These tests call it through the C ABI and check that its results
equal, bit for bit, both the workspace-taking moe_lora_align and the CPU oracle
on calls in a row (each later call reuses the shared scratch the one before it
left behind, on the single-block path and on the chunked path with differently
shaped count matrices), and that sizes beyond the fixed scratch are
refused.  The file is named to be collected last and needs no state from other
tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import lora_moe_expert_info_gb300 as mlr
import oracle

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    lib = mlr.library()
    fn = lib.moe_lora_align_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, ctypes.c_int64, vp, vp]
    return fn


def _inputs(seed, T, K, E, L, dev):
    rng = np.random.default_rng(seed)
    topk = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)
    mapping = rng.integers(-1, L, T).astype(np.int32)
    return torch.from_numpy(topk).to(dev), torch.from_numpy(mapping).to(dev)


def _call_noalloc(topk, mapping, E, L, bs):
    dev = topk.device
    T, K = topk.shape
    cap = mlr.moe_lora_align_capacity(T, K, E, L, bs)
    fill = -7
    out = (torch.full((cap + 8,), fill, dtype=torch.int32, device=dev),
           torch.full((cap // bs + 8,), fill, dtype=torch.int32, device=dev),
           torch.full((cap // bs + 8,), fill, dtype=torch.int32, device=dev),
           torch.full((1,), fill, dtype=torch.int32, device=dev))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = _noalloc_fn()(p(topk), p(mapping), T, K, E, L, bs, p(out[0]), p(out[1]), p(out[2]),
                       p(out[3]), cap, p(status),
                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out, status


def _check_same_as_workspace_call(topk, mapping, E, L, bs):
    rc, (s, be, bl, n), status = _call_noalloc(topk, mapping, E, L, bs)
    assert rc == mlr.MLR_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rs, rbe, rbl, rn = mlr.moe_lora_align(topk, mapping, E, L, bs)   # takes a workspace
    npad = int(rn.item())
    assert int(n.item()) == npad
    assert torch.equal(s[:npad], rs[:npad])
    assert torch.equal(be[:npad // bs], rbe[:npad // bs])
    assert torch.equal(bl[:npad // bs], rbl[:npad // bs])
    assert torch.all(s[mlr.moe_lora_align_capacity(*topk.shape, E, L, bs):] == -7)  # never past capacity
    # and the CPU oracle's canonical order
    st, os_, obe, obl, on = oracle.align(topk.cpu().numpy(), mapping.cpu().numpy(), E, L, bs)
    assert st == 0 and on == npad
    assert np.array_equal(s[:npad].cpu().numpy(), os_)
    assert np.array_equal(be[:npad // bs].cpu().numpy(), obe)
    assert np.array_equal(bl[:npad // bs].cpu().numpy(), obl)


def test_two_calls_in_a_row_match_workspace_align(cuda_device):
    # Qwen-MoE-like routing shape, then a different decode-like shape: the second
    # call reuses the scratch the first call filled.
    t1, m1 = _inputs(1, 4096, 8, 128, 8, cuda_device)
    _check_same_as_workspace_call(t1, m1, 128, 8, 16)
    t2, m2 = _inputs(2, 256, 8, 128, 32, cuda_device)
    _check_same_as_workspace_call(t2, m2, 128, 32, 16)


def test_chunked_calls_in_a_row_with_other_shapes(cuda_device):
    # Both calls take the chunked path (more than 16384 pairs); the second has
    # fewer chunks and another bucket count, so its count matrix overlaps the
    # stale one of the first call with a different layout.
    t1, m1 = _inputs(3, 5000, 8, 128, 8, cuda_device)     # 40000 pairs, 128 x 9 buckets
    assert 5000 * 8 > 16384
    _check_same_as_workspace_call(t1, m1, 128, 8, 16)
    t2, m2 = _inputs(4, 6000, 6, 64, 4, cuda_device)      # 36000 pairs, 64 x 5 buckets
    assert 6000 * 6 > 16384
    _check_same_as_workspace_call(t2, m2, 64, 4, 32)


def test_sizes_beyond_the_fixed_scratch_are_refused(cuda_device):
    # 1,048,576 tokens x top-8 over 256 experts and 65 adapter classes needs ~17 MB
    # of align scratch: refused before anything is enqueued.
    T, K, E, L, bs = 1048576, 8, 256, 64, 64
    assert mlr.moe_lora_align_workspace_bytes(T, K, E, L, bs) > (4 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device=cuda_device)
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = _noalloc_fn()(p, p, T, K, E, L, bs, p, p, p, p, 16, None,
                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == mlr.MLR_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.all(dummy == 0)
