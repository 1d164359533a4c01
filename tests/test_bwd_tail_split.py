"""GPU parity of the bf16 backward when the last wave of its schedule is split
into ranges of query tiles (fa_bwd_plan; the split units' partial dK and dV
are added up by the dQ-convert stage).

Checks, against the fp64 oracle with the bf16 gradient bar (5e-2 of max|ref|):
  * every head that holds a split unit, and a head of whole units, in full;
  * a second run gives the same bits for dK and dV (the partial sums are added
    in a fixed order) and dQ within fp32 rounding;
  * running the three stages one by one (fa_bwd_stage) gives the same result.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv
from oracle import attention_bwd
from parity_utils import grad_within, rel_max, to64

pytestmark = pytest.mark.gpu


def _split_heads(B, H, N, n_full):
    """(b, h) of the first head and of every head that holds a split unit."""
    kblocks = -(-N // 128)
    heads = sorted({u // kblocks for u in range(n_full, B * H * kblocks)})
    return sorted({divmod(0, H)} | {divmod(bh, H) for bh in heads})


@pytest.mark.parametrize("B,H,N,d", [(4, 16, 1024, 64), (1, 10, 2000, 128), (1, 16, 4096, 128), (2, 7, 2048, 64)])
def test_split_backward_matches_oracle(B, H, N, d):
    n_full, n_tail, splits = fa.fa_bwd_plan(B, H, N, d)
    if splits == 1:
        pytest.skip("this GPU's schedule splits nothing for this shape")
    assert n_tail > 0
    q, k, v, do = random_qkv(B, H, N, d, torch.bfloat16, seed=N + H + d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(qc, kc, vc, scale)
    grads = fa.fa_bwd(qc, kc, vc, o, doc, lse, scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    g64 = [to64(g) for g in grads]
    for b, h in _split_heads(B, H, N, n_full):
        ref = attention_bwd(q64[b, h], k64[b, h], v64[b, h], do64[b, h], scale)
        cancel = float(np.abs(do64[b, h]).max() * np.abs(v64[b, h]).max() * d)
        for name, got, r in zip(("dQ", "dK", "dV"), g64, ref):
            assert grad_within(got[b, h], r, cancel), (name, b, h, rel_max(got[b, h], r))


def test_split_backward_is_repeatable_and_stagewise_equal():
    B, H, N, d = 4, 16, 1024, 64
    if fa.fa_bwd_plan(B, H, N, d)[2] == 1:
        pytest.skip("this GPU's schedule splits nothing for this shape")
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.bfloat16, seed=3))
    o, lse = fa.fa_fwd(q, k, v)
    ws = torch.full((fa.fa_bwd_workspace_bytes(B, H, N, d),), 0x7F, dtype=torch.uint8, device="cuda")
    g1 = fa.fa_bwd(q, k, v, o, do, lse, workspace=ws)
    g2 = fa.fa_bwd(q, k, v, o, do, lse, workspace=ws)
    outs = [torch.empty_like(q) for _ in range(3)]
    for stage in (fa.FA_BWD_PREPROCESS, fa.FA_BWD_MAIN, fa.FA_BWD_DQ_CONVERT):
        fa.fa_bwd_stage(stage, q, k, v, o, do, lse, workspace=ws, dq=outs[0], dk=outs[1], dv=outs[2])
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    for a_, b_, c_ in zip(g1[1:], g2[1:], outs[1:]):
        assert torch.equal(a_, b_) and torch.equal(a_, c_)
    # dQ is added by the TMA engine in whatever order the CTAs arrive
    for x in (g2[0], outs[0]):
        assert (x.float() - g1[0].float()).abs().max() <= 1e-2 * g1[0].float().abs().max()


@pytest.mark.parametrize("B,H,N,d", [(8, 50, 1024, 64), (3, 60, 1536, 128)])
def test_split_backward_many_heads(B, H, N, d):
    """Many heads of short sequences (a 2-D grid's worth of units in the split
    schedule's 1-D grid); sampled heads against the oracle, split ones included."""
    n_full, n_tail, splits = fa.fa_bwd_plan(B, H, N, d)
    q, k, v, do = random_qkv(B, H, N, d, torch.bfloat16, seed=B * H + N)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(qc, kc, vc, scale)
    grads = fa.fa_bwd(qc, kc, vc, o, doc, lse, scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    kblocks = -(-N // 128)
    heads = {0, B * H - 1, (n_full // kblocks) if splits > 1 else B * H // 2}
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    for bh in sorted(heads):
        b, h = divmod(bh, H)
        ref = attention_bwd(q64[b, h], k64[b, h], v64[b, h], do64[b, h], scale)
        for name, got, r in zip(("dQ", "dK", "dV"), grads, ref):
            assert rel_max(to64(got[b, h]), r) <= 5e-2, (name, b, h)
