"""Edge cases of the attention kernels on the GPU: the largest grids the C ABI
accepts, a long sequence, degenerate inputs with closed forms, and extreme
score ranges for the online softmax. Same bars as the other parity tests."""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv
from oracle import attention_bwd, attention_fwd, attention_fwd_rows
from parity_utils import TOL_BF16_GRAD, TOL_BF16_LSE, TOL_BF16_O, grad_within, max_abs, rel_max, to64

pytestmark = pytest.mark.gpu


def test_largest_head_count():
    """B*H = 65535 (a grid dimension): forward and backward on every head, a few checked."""
    B, H, N, d = 65535, 1, 5, 64
    q, k, v, do = random_qkv(B, H, N, d, torch.bfloat16, seed=1)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.fa_fwd(qc, kc, vc)
    grads = fa.fa_bwd(qc, kc, vc, o, doc, lse)
    assert fa.fa_check_device_status() == fa.FA_OK
    scale = 1 / math.sqrt(d)
    for b in (0, 1, 32767, 65534):
        Q, K, V, dO = (to64(t[b, 0]) for t in (q, k, v, do))
        O, LSE = attention_fwd(Q, K, V, scale)
        assert rel_max(o[b, 0], O) <= TOL_BF16_O and max_abs(lse[b, 0], LSE) <= TOL_BF16_LSE
        ref = attention_bwd(Q, K, V, dO, scale)
        cancel = float(np.abs(dO).max() * np.abs(V).max() * d)
        for g, r in zip(grads, ref):
            assert grad_within(g[b, 0], r, cancel)


def test_long_sequence_sampled_rows():
    """One head of 131072 rows (1024 key tiles per query tile), forward, causal and not."""
    B, H, N, d = 1, 1, 131072, 128
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=2, with_do=False)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    rows = np.array([0, 1, 127, 128, 70000, N - 129, N - 1])
    for causal in (False, True):
        o, lse = fa.fa_fwd(qc, kc, vc, causal=causal)
        assert fa.fa_check_device_status() == fa.FA_OK
        O, LSE = attention_fwd_rows(to64(q[0, 0]), to64(k[0, 0]), to64(v[0, 0]), 1 / math.sqrt(d), rows,
                                    causal=causal)
        assert rel_max(to64(o[0, 0])[rows], O) <= TOL_BF16_O
        assert max_abs(to64(lse[0, 0])[rows], LSE) <= TOL_BF16_LSE


@pytest.mark.parametrize("d", [64, 128])
def test_zero_queries_give_the_mean_of_the_values(d):
    """Q = 0: every score is 0, so P is uniform, O is the mean of V and
    LSE = ln N; dV = P^T dO gives every key the column sums of dO over N, and
    dK = dS^T Q is exactly 0."""
    B, H, N = 1, 2, 777
    _, k, v, do = random_qkv(B, H, N, d, torch.bfloat16, seed=3)
    q = torch.zeros_like(k)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.fa_fwd(qc, kc, vc)
    dq, dk, dv = fa.fa_bwd(qc, kc, vc, o, doc, lse)
    V64 = to64(v)
    mean = V64.mean(axis=2, keepdims=True)
    assert rel_max(o, np.broadcast_to(mean, V64.shape)) <= TOL_BF16_O
    assert max_abs(lse, np.full((B, H, N), math.log(N))) <= TOL_BF16_LSE
    dv_ref = np.broadcast_to(to64(do).sum(axis=2, keepdims=True) / N, V64.shape)
    assert rel_max(dv, dv_ref) <= TOL_BF16_GRAD
    assert float(dk.float().abs().max()) == 0.0


@pytest.mark.parametrize("causal", [False, True])
def test_extreme_score_ranges(causal):
    """Scores spanning thousands (Q, K scaled up, every 64th key larger still):
    the running max moves by far more than the rescale threshold many times."""
    B, H, N, d = 1, 2, 1000, 128
    q, k, v, do = random_qkv(B, H, N, d, torch.bfloat16, seed=4, big_key_every=64)
    q = (q.float() * 8).to(torch.bfloat16)
    k = (k.float() * 8).to(torch.bfloat16)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(qc, kc, vc, scale, causal=causal)
    grads = fa.fa_bwd(qc, kc, vc, o, doc, lse, scale, causal=causal)
    assert fa.fa_check_device_status() == fa.FA_OK
    for h in range(H):
        Q, K, V, dO = (to64(t[0, h]) for t in (q, k, v, do))
        O, LSE = attention_fwd(Q, K, V, scale, causal=causal)
        assert np.isfinite(to64(o[0, h])).all()
        assert rel_max(o[0, h], O) <= TOL_BF16_O
        assert max_abs(lse[0, h], LSE) <= TOL_BF16_LSE
        ref = attention_bwd(Q, K, V, dO, scale, causal=causal)
        cancel = float(np.abs(dO).max() * np.abs(V).max() * d)
        for g, r in zip(grads, ref):
            assert grad_within(g[0, h], r, cancel)
