"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (for example code inside a host application that owns all device memory
through its own pool, or a serving path where cudaMalloc is not allowed).

The entry point uses one fixed scratch array that the library keeps in device
memory instead of a caller-provided workspace. Each test calls it through the
C ABI twice in a row (the second call sees the first call's leftovers in the
shared array) and checks both results against fa_bwd with a freshly allocated
workspace, using the same tolerances as the other parity tests. This file is
named to be collected last.
"""
import ctypes
import math

import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv
from parity_utils import TOL_BF16_GRAD, TOL_F32_ABS, max_abs, rel_max

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, do, lse, scale, dtype_code):
    """One fa_bwd_noalloc call through the C ABI; returns (dQ, dK, dV) and the
    change in the device's free memory across the call itself (the outputs
    are allocated before the first reading)."""
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    rc = lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                            ctypes.c_float(scale), dtype_code,
                            torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK, fa.fa_status_string(rc)
    assert fa.fa_check_device_status() == fa.FA_OK
    free1 = torch.cuda.mem_get_info()[0]
    return (dq, dk, dv), free0 - free1


@pytest.mark.parametrize("B,H,N,d", [(1, 4, 1000, 128), (2, 3, 333, 64)])
def test_bf16_noalloc_matches_fa_bwd_twice(B, H, N, d):
    lib = fa.load_library()
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.bfloat16, seed=N + d))
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale)
    ref = fa.fa_bwd(q, k, v, o, do, lse, scale)
    for call in range(2):
        got, used = _noalloc(lib, q, k, v, o, do, lse, scale, fa.FA_BF16)
        if call == 1:
            assert used == 0  # the second call (module loaded, scratch address cached) allocates nothing
        for g, r in zip(got, ref):
            assert rel_max(g, r) <= TOL_BF16_GRAD


def test_f32_noalloc_matches_fa_bwd_twice():
    lib = fa.load_library()
    q, k, v, do = (t.cuda() for t in random_qkv(1, 2, 77, 40, torch.float32, seed=5))
    scale = 1 / math.sqrt(40)
    o, lse = fa.fa_fwd(q, k, v, scale)
    ref = fa.fa_bwd(q, k, v, o, do, lse, scale)
    for call in range(2):
        got, used = _noalloc(lib, q, k, v, o, do, lse, scale, fa.FA_F32)
        if call == 1:
            assert used == 0
        for g, r in zip(got, ref):
            assert max_abs(g, r) <= TOL_F32_ABS


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = fa.load_library()
    B, H, N, d = 1, 16, 4096, 128  # needs ~34 MB of workspace > 32 MiB
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) > 32 << 20
    fake = 0x10000  # never dereferenced: the size check comes first
    rc = lib.fa_bwd_noalloc(*([fake] * 9), B, H, N, d, ctypes.c_float(0.088), fa.FA_BF16, None)
    assert rc == fa.FA_ERR_UNSUPPORTED
