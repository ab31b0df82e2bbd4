"""The C-ABI library builds, loads and exports every function include/*.h declares.

CPU only: nothing here launches a kernel.  The host-side argument checks that
return before any CUDA call are exercised with never-dereferenced pointers.
"""
import ctypes
import glob
import os
import re

import pytest

import __graft_entry__
import lora_moe_expert_info_gb300 as mlr
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return mlr.library()


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("moe_lora_batch_info", "moe_lora_align", "fused_moe_lora_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_library_is_the_in_tree_build(lib):
    assert os.path.realpath(lib._name).startswith(os.path.realpath(ROOT))
    assert lib.moe_lora_version().decode().startswith("moe_lora")


@pytest.mark.parametrize("T,K,E,L,bs", [(64, 2, 8, 4, 16), (4096, 8, 128, 8, 16), (0, 8, 4, 4, 16),
                                        (1, 1, 100, 100, 16), (1048576, 8, 256, 64, 64)])
def test_align_capacity_matches_oracle_bound(lib, T, K, E, L, bs):
    assert mlr.moe_lora_align_capacity(T, K, E, L, bs) == oracle.align_capacity(T, K, E, L, bs)
    assert mlr.moe_lora_align_workspace_bytes(T, K, E, L, bs) > 0


def test_align_rejects_bad_sizes(lib):
    assert mlr.moe_lora_align_capacity(-1, 2, 8, 4, 16) == -1
    assert mlr.moe_lora_align_capacity(4, 0, 8, 4, 16) == -1
    assert mlr.moe_lora_align_workspace_bytes(4, 2, 0, 4, 16) == 0
    assert mlr.moe_lora_align_capacity(4, 2, 1024, 64, 16) == -1   # E*(L+1) above the limit


def test_batch_info_host_checks(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the call returns before any launch
    f = lib.moe_lora_batch_info
    assert f(fake, fake, fake, -1, 4, 8, 0, fake, fake, None, None) == mlr.MLR_ERR_INVALID
    assert f(None, fake, fake, 1, 4, 8, 0, fake, fake, None, None) == mlr.MLR_ERR_INVALID
    # the page's under-covered launch: bs=1, max_len=1, 300 tokens
    assert f(fake, fake, fake, 1, 1, 300, 1, fake, fake, None, None) == mlr.MLR_ERR_UNDERCOVERED
    assert f(fake, fake, fake, 1, 70000, 8, 0, fake, fake, None, None) == mlr.MLR_ERR_UNSUPPORTED


def test_align_host_checks(lib):
    fake = ctypes.c_void_p(0x1000)
    f = lib.moe_lora_align
    ws = mlr.moe_lora_align_workspace_bytes(64, 2, 8, 4, 16)
    cap = mlr.moe_lora_align_capacity(64, 2, 8, 4, 16)
    assert f(fake, fake, 64, 2, 8, 4, 0, fake, fake, fake, fake, cap, fake, ws, None, None) \
        == mlr.MLR_ERR_INVALID
    assert f(fake, fake, 64, 2, 8, 4, 16, fake, fake, fake, fake, cap, fake, ws - 1, None, None) \
        == mlr.MLR_ERR_CAPACITY
    assert f(fake, fake, 64, 2, 8, 4, 16, fake, fake, fake, None, cap, fake, ws, None, None) \
        == mlr.MLR_ERR_INVALID


def test_forward_host_checks(lib):
    ws = lib.fused_moe_lora_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws(4096, 8, 128, 2048, 768, 8, 64) > 0
    assert ws(64, 2, 8, 256, 512, 4, 24) == 0          # R not a multiple of 16
    assert ws(64, 2, 8, 120, 512, 4, 16) == 0          # H below 128
    assert ws(64, 2, 256, 256, 512, 63, 16) > 0        # E*(L+1) = 16384: the limit
    assert ws(64, 2, 256, 256, 512, 64, 16) == 0       # E*(L+1) = 16640: above it
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the call returns before any launch
    f = lib.fused_moe_lora_forward
    args = [fake] * 12 + [64, 2, 256, 256, 512, 64, 16, fake, fake, ctypes.c_size_t(1 << 30), None, None]
    assert f(*args) == mlr.MLR_ERR_UNSUPPORTED


def test_linear_host_checks(lib):
    ws = lib.lora_linear_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws(8192, 7168, 2112, 4, 64, 2) > 0           # the MLA fused projection
    assert ws(64, 120, 256, 2, 16, 1) == 0              # D_in below 128
    assert ws(64, 256, 256, 2, 24, 1) == 0              # R not a multiple of 16
    assert ws(64, 256, 256, 2, 16, 3) == 0              # more than two parts
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the calls return before any launch
    f = lib.lora_linear_forward
    f.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int32] * 6 + [ctypes.c_void_p, ctypes.c_void_p,
                                                               ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]

    def call(offsets, D_out=512, S=2):
        offs = (ctypes.c_int32 * len(offsets))(*offsets)
        return f(fake, fake, fake, fake, fake, fake, fake, ctypes.cast(offs, ctypes.c_void_p), 64, 256, D_out, 2, 16,
                 S, fake, fake, ctypes.c_size_t(1 << 30), None, None)

    assert call([0, 200, 512]) == mlr.MLR_ERR_INVALID   # second part not on a 256-row block
    assert call([0, 256, 500]) == mlr.MLR_ERR_INVALID   # last offset is not D_out
    assert call([0, 512, 512]) == mlr.MLR_ERR_INVALID   # empty second part
    assert call([0, 512], S=1, D_out=510) == mlr.MLR_ERR_INVALID


def test_status_strings(lib):
    assert b"under-covers" in lib.moe_lora_status_string(mlr.MLR_ERR_UNDERCOVERED)
    assert lib.moe_lora_status_string(0) == b"ok"


def test_profile_stage_selection_checks(lib):
    # host-side only: selecting stages records nothing until a forward runs
    assert lib.moe_lora_profile_stages(0) == mlr.MLR_ERR_INVALID
    assert lib.moe_lora_profile_stages(1 << 7) == mlr.MLR_ERR_INVALID
    n = 0
    while lib.moe_lora_profile_stage_name(n) is not None:
        n += 1
    assert n == 7
    assert lib.moe_lora_profile_stages(1 << 3) == 0
    assert lib.moe_lora_profile_stages((1 << n) - 1) == 0  # back to every stage


def test_fp8_forward_host_checks(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the calls return before any launch
    f = lib.fused_moe_lora_forward_fp8
    big = ctypes.c_size_t(1 << 30)
    # hidden 136: a multiple of 8 (fine for bf16) but not of 16 (FP8 rows are bytes)
    assert f(*([fake] * 14 + [64, 2, 8, 136, 512, 4, 16, fake, fake, big, None, None])) == mlr.MLR_ERR_UNSUPPORTED
    assert f(*([fake] * 14 + [64, 2, 8, 256, 520, 4, 16, fake, fake, big, None, None])) == mlr.MLR_ERR_UNSUPPORTED
    # a missing scale array
    args = [fake] * 7 + [None] + [fake] * 6 + [64, 2, 8, 256, 512, 4, 16, fake, fake, big, None, None]
    assert f(*args) == mlr.MLR_ERR_INVALID
    args = [fake] * 9 + [None] + [fake] * 4 + [64, 2, 8, 256, 512, 4, 16, fake, fake, big, None, None]
    assert f(*args) == mlr.MLR_ERR_INVALID


def test_fp8_binding_rejects_bad_inputs_before_any_call():
    # CPU tensors: every case must fail in the binding's checks, never reach the library
    import pytest
    import torch
    T, K, E, H, I, L, R = 8, 2, 3, 128, 64, 2, 16
    bf = torch.bfloat16
    x = torch.zeros(T, H, dtype=bf)
    ids = torch.zeros(T, K, dtype=torch.int32)
    wts = torch.zeros(T, K, dtype=torch.float32)
    mp = torch.zeros(T, dtype=torch.int32)
    ranks = torch.zeros(L, dtype=torch.int32)
    scal = torch.zeros(L, dtype=torch.float32)
    wq = torch.zeros(E, 2 * I, H, dtype=torch.uint8)
    ws = torch.zeros(E, 1, 1, dtype=torch.float32)
    dq = torch.zeros(E, H, I, dtype=torch.uint8)
    ds = torch.zeros(E, 1, 1, dtype=torch.float32)
    lo = dict(lora_a_gu=torch.zeros(L, E, 2, R, H, dtype=bf), lora_b_gu=torch.zeros(L, E, 2, I, R, dtype=bf),
              lora_a_down=torch.zeros(L, E, R, I, dtype=bf), lora_b_down=torch.zeros(L, E, H, R, dtype=bf))
    f = mlr.fused_moe_lora_forward_fp8
    with pytest.raises(ValueError):   # scale of W_gate_up has the wrong number of row blocks
        f(x, ids, wts, mp, ranks, scal, wq, torch.zeros(E, 2, 1), dq, ds, **lo)
    with pytest.raises(ValueError):   # W_down codes of the wrong shape
        f(x, ids, wts, mp, ranks, scal, wq, ws, torch.zeros(E, I, H, dtype=torch.uint8), ds, **lo)
    with pytest.raises(TypeError):    # codes must be bytes
        f(x, ids, wts, mp, ranks, scal, wq.to(bf), ws, dq, ds, **lo)
    with pytest.raises(TypeError):    # scales must be float32
        f(x, ids, wts, mp, ranks, scal, wq, ws.double(), dq, ds, **lo)
