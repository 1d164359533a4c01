"""Canary checks for the paths added on top of the plain forward/backward
(compute-sanitizer is not available): outputs live inside larger NaN-filled
buffers; after the call every output element must be finite (written) and the
guard regions before and after it untouched. Determinism: a second call gives
bitwise the same forward outputs."""
import math

import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv, random_varlen

pytestmark = pytest.mark.gpu

GUARD = 4096


def _guarded(shape, dtype):
    n = math.prod(shape)
    buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(*shape)


def _check(buf, view):
    assert torch.isfinite(view.float()).all(), "an output element was not written"
    assert torch.isnan(buf[:GUARD].float()).all() and torch.isnan(buf[-GUARD:].float()).all(), \
        "a write landed outside the output"


@pytest.mark.parametrize("d", [64, 128])
def test_causal_fwd_bwd_canaries(d):
    B, H, N = 2, 3, 700
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.bfloat16, seed=d))
    ob, o = _guarded((B, H, N, d), torch.bfloat16)
    lb, lse = _guarded((B, H, N), torch.float32)
    fa.fa_fwd(q, k, v, out=o, lse=lse, causal=True)
    _check(ob, o)
    _check(lb, lse)
    gb = [_guarded((B, H, N, d), torch.bfloat16) for _ in range(3)]
    fa.fa_bwd(q, k, v, o, do, lse, dq=gb[0][1], dk=gb[1][1], dv=gb[2][1], causal=True)
    assert fa.fa_check_device_status() == fa.FA_OK
    for buf, view in gb:
        _check(buf, view)
    o2, l2 = fa.fa_fwd(q, k, v, causal=True)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_canaries(causal):
    lens = [1, 300, 0, 129, 1000]
    H, d = 2, 128
    q, k, v, do, cu = random_varlen(lens, H, d, torch.bfloat16, seed=7)
    q, k, v, do, cu = (t.cuda() for t in (q, k, v, do, cu))
    total = q.shape[0]
    ob, o = _guarded((total, H, d), torch.bfloat16)
    lb, lse = _guarded((H, total), torch.float32)
    fa.fa_fwd_varlen(q, k, v, cu, max(lens), causal=causal, out=o, lse=lse)
    _check(ob, o)
    _check(lb, lse)
    dq, dk, dv = fa.fa_bwd_varlen(q, k, v, o, do, lse, cu, max(lens), causal=causal)
    assert fa.fa_check_device_status() == fa.FA_OK
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()
    o2, l2 = fa.fa_fwd_varlen(q, k, v, cu, max(lens), causal=causal)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("nq", [1, 8])
def test_decode_canaries(nq):
    B, H, nk, d = 2, 3, 5000, 128
    q, k, v, _ = random_qkv(B, H, nq, d, torch.bfloat16, seed=nq, with_do=False, n_k=nk)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ob, o = _guarded((B, H, nq, d), torch.bfloat16)
    lb, lse = _guarded((B, H, nq), torch.float32)
    fa.fa_decode(q, k, v, out=o, lse=lse)
    assert fa.fa_check_device_status() == fa.FA_OK
    _check(ob, o)
    _check(lb, lse)


@pytest.mark.parametrize("cols", [100, 4096, 20000])
def test_softmax_rows_canaries(cols):
    rows = 37
    x = torch.randn(rows, cols, device="cuda")
    yb, y = _guarded((rows, cols), torch.float32)
    fa.fa_softmax_rows(x, out=y)
    _check(yb, y)
