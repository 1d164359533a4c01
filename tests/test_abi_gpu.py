"""The plain fa_fwd / fa_bwd entry points, called through ctypes exactly as a C
caller would (raw device pointers, sizes, a stream handle), against the fp64
oracle.

The Python binding routes through the extended entry points (fa_fwd_ws,
fa_bwd_ex); these tests make sure the two calls that define the boundary launch
the kernels themselves and give the oracle's result. Bars as in the other parity
tests: bf16 O within 2e-2 and dQ/dK/dV within 5e-2 of max|ref|, LSE within
1e-3; fp32 within 1e-5 absolute."""
import ctypes
import math

import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv
from oracle import attention_bwd_batched, attention_fwd_batched
from parity_utils import (TOL_BF16_GRAD, TOL_BF16_LSE, TOL_BF16_O, TOL_F32_ABS, max_abs,
                          rel_max, to64)

pytestmark = pytest.mark.gpu


def _raw_fwd_bwd(q, k, v, do, scale):
    lib = fa.load_library()
    B, H, N, d = q.shape
    code = fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_F32
    stream = torch.cuda.current_stream().cuda_stream
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    rc = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    B, H, N, d, ctypes.c_float(scale), code, stream)
    assert rc == fa.FA_OK, fa.fa_status_string(rc)
    ws_bytes = lib.fa_bwd_workspace_bytes(B, H, N, d, code)
    assert ws_bytes > 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                    ctypes.c_size_t(ws_bytes), B, H, N, d, ctypes.c_float(scale), code, stream)
    assert rc == fa.FA_OK, fa.fa_status_string(rc)
    assert lib.fa_check_device_status(ctypes.c_void_p(stream)) == fa.FA_OK
    return o, lse, (dq, dk, dv)


@pytest.mark.parametrize("B,H,N,d", [(1, 2, 300, 128), (2, 2, 257, 64)])
def test_raw_fa_fwd_fa_bwd_bf16_against_oracle(B, H, N, d):
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.bfloat16, seed=900 + N + d))
    scale = 1 / math.sqrt(d)
    o, lse, grads = _raw_fwd_bwd(q, k, v, do, scale)
    O, LSE = attention_fwd_batched(to64(q), to64(k), to64(v), scale)
    ref = attention_bwd_batched(to64(q), to64(k), to64(v), to64(do), scale)
    assert rel_max(o, O) <= TOL_BF16_O
    assert max_abs(lse, LSE) <= TOL_BF16_LSE
    for g, r in zip(grads, ref):
        assert rel_max(g, r) <= TOL_BF16_GRAD


def test_raw_fa_fwd_fa_bwd_f32_against_oracle():
    B, H, N, d = 1, 2, 45, 24
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.float32, seed=77))
    scale = 1 / math.sqrt(d)
    o, lse, grads = _raw_fwd_bwd(q, k, v, do, scale)
    O, LSE = attention_fwd_batched(to64(q), to64(k), to64(v), scale)
    ref = attention_bwd_batched(to64(q), to64(k), to64(v), to64(do), scale)
    assert max_abs(o, O) <= TOL_F32_ABS and max_abs(lse, LSE) <= TOL_F32_ABS
    for g, r in zip(grads, ref):
        assert max_abs(g, r) <= TOL_F32_ABS * max(1.0, float(abs(to64(r)).max()))
