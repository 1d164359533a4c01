"""GPU parity of causal attention and packed variable-length batches.

Causal: query row r sees keys c <= r (the oracle masks the scores to -inf
there). Variable length: a packed [total, H, d] batch with offsets
cu_seqlens, every sequence attended to on its own. Both are checked, forward
and backward, against the fp64 oracle on the same seeded inputs, with the
bars of the other parity tests: bf16 O <= 2e-2 and dQ/dK/dV <= 5e-2 (max error
relative to max |ref|), LSE <= 1e-3 absolute; fp32 1e-5 absolute.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv, random_varlen
from oracle import attention_bwd, attention_fwd, attention_fwd_rows, varlen_attention_bwd, varlen_attention_fwd
from parity_utils import (TOL_BF16_GRAD, TOL_BF16_LSE, TOL_BF16_O, TOL_F32_ABS, grad_within, max_abs,
                          rel_max, to64)

pytestmark = pytest.mark.gpu


def _fwd_bwd_fixed(B, H, N, d, dtype, seed, causal=True):
    q, k, v, do = random_qkv(B, H, N, d, dtype, seed=seed)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(qc, kc, vc, scale, causal=causal)
    dq, dk, dv = fa.fa_bwd(qc, kc, vc, o, doc, lse, scale, causal=causal)
    assert fa.fa_check_device_status() == fa.FA_OK
    return (q, k, v, do), (o, lse, dq, dk, dv), scale


@pytest.mark.parametrize("N", [1, 100, 128, 129, 256, 257, 383, 640, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_causal_bf16_fwd_bwd(N, d):
    (q, k, v, do), (o, lse, dq, dk, dv), scale = _fwd_bwd_fixed(1, 2, N, d, torch.bfloat16, N + d)
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    for h in range(2):
        O, LSE = attention_fwd(q64[0, h], k64[0, h], v64[0, h], scale, causal=True)
        assert rel_max(o[0, h], O) <= TOL_BF16_O, h
        assert max_abs(lse[0, h], LSE) <= TOL_BF16_LSE, h
        grads = attention_bwd(q64[0, h], k64[0, h], v64[0, h], do64[0, h], scale, causal=True)
        cancel = float(np.abs(do64[0, h]).max() * np.abs(v64[0, h]).max() * d)
        for g, r in zip((dq, dk, dv), grads):
            assert grad_within(g[0, h], r, cancel), h


@pytest.mark.parametrize("N,d", [(1, 8), (33, 40), (100, 128), (257, 64)])
def test_causal_f32_fwd_bwd(N, d):
    (q, k, v, do), (o, lse, dq, dk, dv), scale = _fwd_bwd_fixed(2, 1, N, d, torch.float32, N * 3 + d)
    for b in range(2):
        O, LSE = attention_fwd(to64(q[b, 0]), to64(k[b, 0]), to64(v[b, 0]), scale, causal=True)
        assert max_abs(o[b, 0], O) <= TOL_F32_ABS
        assert max_abs(lse[b, 0], LSE) <= TOL_F32_ABS
        grads = attention_bwd(to64(q[b, 0]), to64(k[b, 0]), to64(v[b, 0]), to64(do[b, 0]), scale,
                              causal=True)
        for g, r in zip((dq, dk, dv), grads):
            assert max_abs(g[b, 0], r) <= TOL_F32_ABS * max(1.0, float(np.abs(r).max()))


def test_causal_bf16_long_sequence_sampled():
    """1x4x4096x128, the bench's causal shape per head: two whole heads
    (forward and backward) and sampled rows of the other two."""
    B, H, N, d = 1, 4, 4096, 128
    (q, k, v, do), (o, lse, dq, dk, dv), scale = _fwd_bwd_fixed(B, H, N, d, torch.bfloat16, 4)
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    for h in (0, 3):
        O, LSE = attention_fwd(q64[0, h], k64[0, h], v64[0, h], scale, causal=True)
        assert rel_max(o[0, h], O) <= TOL_BF16_O
        assert max_abs(lse[0, h], LSE) <= TOL_BF16_LSE
        grads = attention_bwd(q64[0, h], k64[0, h], v64[0, h], do64[0, h], scale, causal=True)
        for g, r in zip((dq, dk, dv), grads):
            assert rel_max(g[0, h], r) <= TOL_BF16_GRAD
    rows = np.random.default_rng(0).choice(N, 64, replace=False)
    rows[:3] = [0, 127, N - 1]
    o64, l64 = to64(o), to64(lse)
    for h in (1, 2):
        O, LSE = attention_fwd_rows(q64[0, h], k64[0, h], v64[0, h], scale, rows, causal=True)
        assert rel_max(o64[0, h][rows], O) <= TOL_BF16_O
        assert max_abs(l64[0, h][rows], LSE) <= TOL_BF16_LSE


def test_causal_differs_from_full_and_flags_are_independent():
    """The same inputs through the causal and the full path: the last rows agree
    (they see every key), the first rows do not; a later full call is unaffected."""
    q, k, v, _ = random_qkv(1, 1, 300, 64, torch.bfloat16, seed=8, with_do=False)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o_full, l_full = fa.fa_fwd(q, k, v)
    o_c, l_c = fa.fa_fwd(q, k, v, causal=True)
    o_full2, _ = fa.fa_fwd(q, k, v)
    assert torch.equal(o_full, o_full2)
    assert (l_c[0, 0, -1] - l_full[0, 0, -1]).abs().item() < 1e-3
    assert (l_c[0, 0, :10] - l_full[0, 0, :10]).abs().max().item() > 0.1


LENS = [
    [1000],
    [1, 127, 128, 129, 300, 1000, 7],
    [0, 256, 0, 513, 64],
    [40] * 9,
]


@pytest.mark.parametrize("lens", LENS, ids=lambda l: "x".join(map(str, l[:4])))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_varlen_bf16_fwd_bwd(lens, causal, d):
    H = 3
    q, k, v, do, cu = random_varlen(lens, H, d, torch.bfloat16, seed=sum(lens) + d)
    scale = 1 / math.sqrt(d)
    args = [t.cuda() for t in (q, k, v)]
    cuc = cu.cuda()
    o, lse = fa.fa_fwd_varlen(*args, cuc, max(lens), scale, causal=causal)
    dq, dk, dv = fa.fa_bwd_varlen(*args, o, do.cuda(), lse, cuc, max(lens), scale, causal=causal)
    assert fa.fa_check_device_status() == fa.FA_OK
    O, LSE = varlen_attention_fwd(to64(q), to64(k), to64(v), cu.tolist(), scale, causal)
    assert rel_max(o, O) <= TOL_BF16_O
    assert max_abs(lse, LSE) <= TOL_BF16_LSE
    grads = varlen_attention_bwd(to64(q), to64(k), to64(v), to64(do), cu.tolist(), scale, causal)
    for g, r in zip((dq, dk, dv), grads):
        assert rel_max(g, r) <= TOL_BF16_GRAD


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_f32_fwd_bwd(causal):
    lens = [3, 40, 0, 77, 1]
    q, k, v, do, cu = random_varlen(lens, 2, 24, torch.float32, seed=13)
    args = [t.cuda() for t in (q, k, v)]
    cuc = cu.cuda()
    o, lse = fa.fa_fwd_varlen(*args, cuc, max(lens), 0.3, causal=causal)
    dq, dk, dv = fa.fa_bwd_varlen(*args, o, do.cuda(), lse, cuc, max(lens), 0.3, causal=causal)
    assert fa.fa_check_device_status() == fa.FA_OK
    O, LSE = varlen_attention_fwd(to64(q), to64(k), to64(v), cu.tolist(), 0.3, causal)
    assert max_abs(o, O) <= TOL_F32_ABS and max_abs(lse, LSE) <= TOL_F32_ABS
    grads = varlen_attention_bwd(to64(q), to64(k), to64(v), to64(do), cu.tolist(), 0.3, causal)
    for g, r in zip((dq, dk, dv), grads):
        assert max_abs(g, r) <= TOL_F32_ABS * max(1.0, float(np.abs(r).max()))


def test_varlen_single_sequence_matches_fixed_layout():
    """One packed sequence [N, H, d] equals the fixed layout [1, H, N, d]."""
    N, H, d = 700, 4, 128
    q, k, v, do, cu = random_varlen([N], H, d, torch.bfloat16, seed=1)
    qc, kc, vc, doc, cuc = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu.cuda()
    for causal in (False, True):
        o, lse = fa.fa_fwd_varlen(qc, kc, vc, cuc, N, causal=causal)
        grads = fa.fa_bwd_varlen(qc, kc, vc, o, doc, lse, cuc, N, causal=causal)
        t = lambda x: x.transpose(0, 1).unsqueeze(0).contiguous()  # [N,H,d] -> [1,H,N,d]
        o2, lse2 = fa.fa_fwd(t(qc), t(kc), t(vc), causal=causal)
        grads2 = fa.fa_bwd(t(qc), t(kc), t(vc), o2, t(doc), lse2, causal=causal)
        assert torch.equal(t(o), o2) and torch.equal(lse, lse2[0])
        for g, g2 in zip(grads, grads2):
            assert rel_max(t(g), to64(g2)) <= 1e-2  # dQ sums in a different order


def test_varlen_inconsistent_offsets_are_reported_and_skipped():
    """Offsets that decrease or pass `total` are caught in the kernels: the bad
    sequences are skipped (their rows keep the sentinel) and the status word
    reports FA_ERR_INVALID_ARG; valid sequences are still computed."""
    H, d = 2, 64
    q, k, v, _, _ = random_varlen([100, 50, 80], H, d, torch.bfloat16, seed=2, with_do=False)
    cu = torch.tensor([0, 100, 60, 230], dtype=torch.int32).cuda()  # seq 1 decreasing, seq 2 longer than max_seqlen
    out = torch.full_like(q, 7.0).cuda()
    lse = torch.full((H, 230), 7.0, dtype=torch.float32).cuda()
    fa.fa_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu, 100, out=out, lse=lse)
    assert fa.fa_check_device_status() == fa.FA_ERR_INVALID_ARG
    assert bool((out[100:] == 7.0).all()) and bool((lse[:, 100:] == 7.0).all())
    O, LSE = varlen_attention_fwd(to64(q[:100]), to64(k[:100]), to64(v[:100]), [0, 100], 1 / 8)
    assert rel_max(out[:100], O) <= TOL_BF16_O
    assert fa.fa_check_device_status() == fa.FA_OK  # cleared by the read
