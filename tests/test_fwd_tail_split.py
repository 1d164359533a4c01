"""GPU parity of the bf16 forward when the last wave of its schedule is split
into key ranges (fa_fwd_ws; the Python fa_fwd passes the scratch).

A split unit's rows come out of a merge (a second kernel) of 2-4 partial
softmaxes, each over a range of key tiles, combined through their maxima and
sums. Checks, through the C ABI:
  * rows of split units and of whole units against the fp64 oracle, with the
    bf16 bars of the other forward tests;
  * the split schedule against the plain one (fa_fwd_ex, no scratch) on the
    whole output;
  * a second call on the same scratch gives the same bits (the scratch
    carries nothing from one call to the next), whatever the scratch held
    before, and every row is written;
  * a scratch that is too small is refused before launch.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv
from oracle import attention_fwd_rows
from parity_utils import TOL_BF16_LSE, TOL_BF16_O, max_abs, rel_max, to64

pytestmark = pytest.mark.gpu


def _plain(q, k, v, scale):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lib = fa.load_library()
    rc = lib.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                       scale, 0, fa.FA_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    return o, lse


def _split(q, k, v, scale, ws):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lib = fa.load_library()
    rc = lib.fa_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       ws.data_ptr(), ws.numel(), B, H, N, d, scale, 0, fa.FA_BF16,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    return o, lse


def _unit_heads(B, H, N, n_full):
    """(b, h) of the first whole unit's head and of every head holding a split unit."""
    qblocks = -(-N // 256)
    split_heads = sorted({u // qblocks for u in range(n_full, B * H * qblocks)})
    return [divmod(0, H)] + [divmod(bh, H) for bh in split_heads]


@pytest.mark.parametrize("B,H,N,d", [(1, 10, 4096, 128), (1, 12, 4096, 128), (1, 10, 4000, 64), (1, 13, 3001, 128),
                                     (2, 16, 4096, 128), (1, 2, 20000, 64)])
def test_split_tail_matches_oracle_and_plain_schedule(B, H, N, d):
    n_full, n_tail, splits = fa.fa_fwd_plan(B, H, N, d)
    if splits == 1:
        pytest.skip("this GPU's schedule splits nothing for this shape")
    assert n_tail > 0
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=N + H + d, with_do=False)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    scale = 1 / math.sqrt(d)
    ws_bytes = fa.fa_fwd_workspace_bytes(B, H, N, d)
    assert ws_bytes > 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o, lse = _split(qc, kc, vc, scale, ws)
    o_ref, lse_ref = _plain(qc, kc, vc, scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    # same attention as the plain schedule (fp32 rounding order differs)
    assert rel_max(to64(o), to64(o_ref)) <= TOL_BF16_O
    assert max_abs(to64(lse), to64(lse_ref)) <= TOL_BF16_LSE
    # oracle rows: every 256-row block of the split units' heads, and a whole unit
    q64, k64, v64 = to64(q), to64(k), to64(v)
    o64, l64 = to64(o), to64(lse)
    rng = np.random.default_rng(N)
    for b, h in _unit_heads(B, H, N, n_full):
        rows = np.unique(np.concatenate([np.arange(0, N, 256), [N - 1], rng.choice(N, 24, replace=False)]))
        O, LSE = attention_fwd_rows(q64[b, h], k64[b, h], v64[b, h], scale, rows)
        assert rel_max(o64[b, h][rows], O) <= TOL_BF16_O, (b, h)
        assert max_abs(l64[b, h][rows], LSE) <= TOL_BF16_LSE, (b, h)


def test_split_tail_repeats_bit_for_bit_on_the_same_scratch():
    B, H, N, d = 1, 10, 4096, 128
    if fa.fa_fwd_plan(B, H, N, d)[2] == 1:
        pytest.skip("this GPU's schedule splits nothing for this shape")
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=5, with_do=False)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    ws = torch.full((fa.fa_fwd_workspace_bytes(B, H, N, d),), 0x7F, dtype=torch.uint8, device="cuda")
    o1, l1 = _split(qc, kc, vc, 0.1, ws)
    o2, l2 = _split(qc, kc, vc, 0.1, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # the Python entry point takes the same schedule
    o3, l3 = fa.fa_fwd(qc, kc, vc, 0.1)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


@pytest.mark.parametrize("B,H,N,d", [(1, 10, 4096, 128), (1, 2, 20000, 64)])
def test_split_tail_is_deterministic_for_any_scratch(B, H, N, d):
    """Twenty calls on scratch filled with 0x00, 0xFF, 0x7F bytes and then on
    the previous call's leftovers: O starts as NaN each time and comes out
    with the same bits as the first call."""
    if fa.fa_fwd_plan(B, H, N, d)[2] == 1:
        pytest.skip("this GPU's schedule splits nothing for this shape")
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=11 + d, with_do=False)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    scale = 1 / math.sqrt(d)
    nbytes = fa.fa_fwd_workspace_bytes(B, H, N, d)
    ref = None
    for i in range(20):
        ws = torch.full((nbytes,), (0x00, 0xFF, 0x7F)[i % 3], dtype=torch.uint8, device="cuda") if i < 3 else ws
        o = torch.full_like(qc, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        lib = fa.load_library()
        rc = lib.fa_fwd_ws(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           ws.data_ptr(), ws.numel(), B, H, N, d, scale, 0, fa.FA_BF16,
                           torch.cuda.current_stream().cuda_stream)
        assert rc == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_check_device_status() == fa.FA_OK
        assert not torch.isnan(o).any() and not torch.isnan(lse).any(), i
        if ref is None:
            ref = (o, lse)
        else:
            assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1]), i


def test_split_tail_refuses_a_small_scratch():
    B, H, N, d = 1, 10, 4096, 128
    need = fa.fa_fwd_workspace_bytes(B, H, N, d)
    if need == 0:
        pytest.skip("this GPU's schedule splits nothing for this shape")
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    lib = fa.load_library()
    rc = lib.fa_fwd_ws(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       ws.data_ptr(), need - 1, B, H, N, d, 0.1, 0, fa.FA_BF16,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_ERR_INVALID_ARG
    rc = lib.fa_fwd_ws(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       ws.data_ptr() + 16, need, B, H, N, d, 0.1, 0, fa.FA_BF16,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_ERR_INVALID_ARG
