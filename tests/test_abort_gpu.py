"""The attention kernels' own abort path, driven without a fault.

fa_debug_fwd_skip_load / fa_debug_bwd_skip_load make the producer of every CTA
skip one tile load (neither the copy nor its expected-bytes arrival is issued,
so nothing is left in flight). The consumers' bounded waits on that tile then
run out after a short limit: each CTA records FA_ERR_TIMEOUT in the device
status word, drains the copies and products it issued, frees its tensor memory
and exits. The tests check that the status is reported (and cleared by the
read), and that ordinary calls on the same context afterwards still match the
fp64 oracle.
"""
import ctypes
import math

import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv
from oracle import attention_bwd, attention_fwd
from parity_utils import TOL_BF16_GRAD, TOL_BF16_LSE, TOL_BF16_O, max_abs, rel_max, to64

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000  # 2 ms per bounded wait


def _ptrs(*ts):
    return [t.data_ptr() for t in ts]


def _check_fwd(q, k, v, o, lse, scale):
    q64, k64, v64 = to64(q), to64(k), to64(v)
    for h in sorted({0, q.shape[1] // 2, q.shape[1] - 1}):
        O, LSE = attention_fwd(q64[0, h], k64[0, h], v64[0, h], scale)
        assert rel_max(o[0, h], O) <= TOL_BF16_O
        assert max_abs(lse[0, h], LSE) <= TOL_BF16_LSE


@pytest.mark.parametrize("d,H", [(128, 4), (64, 4), (64, 128)])
def test_forward_skipped_key_tile_times_out_then_recovers(d, H):
    """H = 4: the two-tile kernels (8 CTAs at d = 64); H = 128 at d = 64: the
    four-query-tile kernel (256 CTAs, at least 3/4 of the SMs)."""
    lib = fa.load_library()
    B, N = 1, 1024  # nothing split
    q, k, v, _ = (t.cuda() if t is not None else None
                  for t in random_qkv(B, H, N, d, torch.bfloat16, seed=41 + d, with_do=False))
    scale = 1 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    assert fa.fa_check_device_status() == fa.FA_OK
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    rc = lib.fa_debug_fwd_skip_load(*_ptrs(q, k, v, o, lse), B, H, N, d, ctypes.c_float(scale), 3,
                                    LIMIT_NS, stream)
    assert rc == fa.FA_OK
    assert fa.fa_check_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK  # the read cleared it
    o2, lse2 = fa.fa_fwd(q, k, v, scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    _check_fwd(q, k, v, o2, lse2, scale)


@pytest.mark.parametrize("d,H,N", [(128, 2, 768), (64, 2, 768), (128, 10, 2000)])
def test_backward_skipped_query_tile_times_out_then_recovers(d, H, N):
    """H = 2, N = 768: 6 query tiles per unit, 12 units, one per CTA. H = 10,
    N = 2000: 160 units, the last 8 split into query ranges, so 32 CTAs walk a
    whole unit and then a range (each CTA skips the third tile of its walk)."""
    lib = fa.load_library()
    B = 1
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.bfloat16, seed=51 + d))
    scale = 1 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    o, lse = fa.fa_fwd(q, k, v, scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = lib.fa_debug_bwd_skip_load(*_ptrs(q, k, v, o, do, lse, dq, dk, dv, ws), ws_bytes, B, H, N,
                                    d, ctypes.c_float(scale), 2, LIMIT_NS, stream)
    assert rc == fa.FA_OK
    assert fa.fa_check_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK
    grads = fa.fa_bwd(q, k, v, o, do, lse, scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    for h in sorted({0, H - 1}):
        ref = attention_bwd(q64[0, h], k64[0, h], v64[0, h], do64[0, h], scale)
        for g, r in zip(grads, ref):
            assert rel_max(g[0, h], r) <= TOL_BF16_GRAD


def test_skip_hooks_reject_tiles_outside_the_problem():
    lib = fa.load_library()
    fake = 0x10000  # never dereferenced: validation comes first
    for bad in (0, 8, -1):
        assert lib.fa_debug_fwd_skip_load(*([fake] * 5), 1, 1, 1024, 128, ctypes.c_float(0.1), bad,
                                          LIMIT_NS, None) == fa.FA_ERR_INVALID_ARG
        assert lib.fa_debug_bwd_skip_load(*([fake] * 10), 1 << 30, 1, 1, 1024, 128,
                                          ctypes.c_float(0.1), bad, LIMIT_NS,
                                          None) == fa.FA_ERR_INVALID_ARG
        assert lib.fa_debug_bwd_skip_load_ex(*([fake] * 10), 1 << 30, 1, 1, 1024, 128,
                                             ctypes.c_float(0.1), fa.FA_CAUSAL, bad, LIMIT_NS,
                                             None) == fa.FA_ERR_INVALID_ARG
    # flags other than FA_CAUSAL
    assert lib.fa_debug_bwd_skip_load_ex(*([fake] * 10), 1 << 30, 1, 1, 1024, 128, ctypes.c_float(0.1),
                                         2, 1, LIMIT_NS, None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [64, 128])
def test_causal_backward_skipped_query_tile_times_out_then_recovers(d):
    """The causal backward: persistent CTAs taking units from the device
    counter and passing them on through the item ring. Every CTA skips the
    third tile of its walk; the bounded waits (tile and ring) run out, the
    timeout is reported, and a normal causal call afterwards matches the
    oracle."""
    lib = fa.load_library()
    B, H, N = 1, 24, 768
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.bfloat16, seed=61 + d))
    scale = 1 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    o, lse = fa.fa_fwd(q, k, v, scale, causal=True)
    assert fa.fa_check_device_status() == fa.FA_OK
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, N, d)  # covers the causal layout (no split partials)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = lib.fa_debug_bwd_skip_load_ex(*_ptrs(q, k, v, o, do, lse, dq, dk, dv, ws), ws_bytes, B, H, N,
                                       d, ctypes.c_float(scale), fa.FA_CAUSAL, 2, LIMIT_NS, stream)
    assert rc == fa.FA_OK
    assert fa.fa_check_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK
    grads = fa.fa_bwd(q, k, v, o, do, lse, scale, causal=True)
    assert fa.fa_check_device_status() == fa.FA_OK
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    for h in (0, H - 1):
        ref = attention_bwd(q64[0, h], k64[0, h], v64[0, h], do64[0, h], scale, causal=True)
        for g, r in zip(grads, ref):
            assert rel_max(g[0, h], r) <= TOL_BF16_GRAD
