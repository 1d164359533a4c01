"""Seeded sweep of bf16 forward + backward shapes against the fp64 oracle.

Shapes are drawn (seeded) so that, between them, they reach every schedule
the library picks: one unit per CTA and several per CTA (the backward's
persistent grid), split last rounds (forward key ranges, backward query
ranges), causal item lists whose last head group is padded, more than 32
key tiles, the four-tile d = 64 forward, and ragged last tiles. Each
case checks O, LSE, dQ, dK and dV of three heads (first, last, one drawn)
with the bars of the other bf16 tests.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv
from oracle import attention_bwd, attention_fwd
from parity_utils import TOL_BF16_LSE, TOL_BF16_O, grad_within, max_abs, rel_max, to64

pytestmark = pytest.mark.gpu


def _cases():
    rng = np.random.default_rng(20261202)
    out = []
    for i in range(24):
        d = (64, 128)[i % 2]
        causal = (i // 2) % 2 == 1
        N = int(rng.integers(1, 3000))
        if i % 8 == 7:
            N = int(rng.integers(4097, 5200))  # more than 32 key tiles
        BH = int(rng.integers(1, 64)) if N > 1000 else int(rng.integers(1, 300))
        H = int(rng.integers(1, 9))
        B = max(1, BH // H)
        out.append((B, H, N, d, causal))
    return out


@pytest.mark.parametrize("B,H,N,d,causal", _cases())
def test_sweep_forward_backward(B, H, N, d, causal):
    q, k, v, do = random_qkv(B, H, N, d, torch.bfloat16, seed=B * 7919 + H * 104729 + N * 31 + d + int(causal))
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(qc, kc, vc, scale, causal=causal)
    grads = fa.fa_bwd(qc, kc, vc, o, doc, lse, scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    o64, l64 = to64(o), to64(lse)
    g64 = [to64(g) for g in grads]
    rng = np.random.default_rng(N + B + H)
    heads = sorted({0, B * H - 1, int(rng.integers(0, B * H))})
    for bh in heads:
        b, h = divmod(bh, H)
        O, LSE = attention_fwd(q64[b, h], k64[b, h], v64[b, h], scale, causal=causal)
        assert rel_max(o64[b, h], O) <= TOL_BF16_O, ("O", b, h)
        assert max_abs(l64[b, h], LSE) <= TOL_BF16_LSE, ("LSE", b, h)
        ref = attention_bwd(q64[b, h], k64[b, h], v64[b, h], do64[b, h], scale, causal=causal)
        cancel = float(np.abs(do64[b, h]).max() * np.abs(v64[b, h]).max() * d)
        for name, got, r in zip(("dQ", "dK", "dV"), g64, ref):
            assert grad_within(got[b, h], r, cancel), (name, b, h, rel_max(got[b, h], r))
