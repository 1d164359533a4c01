"""GPU parity of the bf16 backward's persistent grid: fixed-length problems
run as one CTA per SM taking (batch*head, key tile) items in list order from
a device counter, so a CTA carries its rings, barriers and tensor memory from
one item to the next.

Checks, against the fp64 oracle with the bf16 gradient bar, EVERY head of
problems where each CTA takes several items: ragged key and query tiles,
whole items followed by the query ranges of a split tail, short items of one
query tile, and causal items of decreasing length. A second run gives the
same dK and dV bits (each item's dK and dV come from one CTA whatever the
order the items are taken in).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import random_qkv, random_varlen
from oracle import attention_bwd, varlen_attention_bwd
from parity_utils import TOL_BF16_GRAD, grad_within, rel_max, to64

pytestmark = pytest.mark.gpu


def _items(B, H, N, d):
    n_full, n_tail, splits = fa.fa_bwd_plan(B, H, N, d)
    return n_full + n_tail * splits


@pytest.mark.parametrize("B,H,N,d,causal", [
    (3, 67, 300, 64, False),    # 603 items of 3 query tiles, ragged last key and query tiles
    (1, 40, 1000, 128, False),  # 320 units: 304 whole, then 16 split into query ranges
    (2, 90, 128, 128, False),   # 180 items of a single query tile
    (4, 40, 520, 64, False),    # 800 items of 5 tiles, 8 rows in the last
    (3, 67, 300, 64, True),     # causal: 603 items of 3, 2 and 1 query tiles, longest first
    (1, 40, 1000, 128, True),   # causal: 320 items of 8 down to 1 query tile
    (2, 30, 2048, 64, True),    # causal: head groups, items of 16 down to 1 tile
])
def test_persistent_backward_every_head(B, H, N, d, causal):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * H * -(-N // 128) > sms  # some CTA walks more than one item
    if not causal:
        assert _items(B, H, N, d) > sms
    q, k, v, do = random_qkv(B, H, N, d, torch.bfloat16, seed=B * H + N + d + int(causal))
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(qc, kc, vc, scale, causal=causal)
    grads = fa.fa_bwd(qc, kc, vc, o, doc, lse, scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    g64 = [to64(g) for g in grads]
    for b in range(B):
        for h in range(H):
            ref = attention_bwd(q64[b, h], k64[b, h], v64[b, h], do64[b, h], scale, causal=causal)
            cancel = float(np.abs(do64[b, h]).max() * np.abs(v64[b, h]).max() * d)
            for name, got, r in zip(("dQ", "dK", "dV"), g64, ref):
                assert grad_within(got[b, h], r, cancel), (name, b, h, rel_max(got[b, h], r))


def test_persistent_backward_repeats_dk_dv_bit_for_bit():
    B, H, N, d = 1, 40, 1000, 128
    q, k, v, do = (t.cuda() for t in random_qkv(B, H, N, d, torch.bfloat16, seed=77))
    o, lse = fa.fa_fwd(q, k, v)
    g1 = fa.fa_bwd(q, k, v, o, do, lse)
    g2 = fa.fa_bwd(q, k, v, o, do, lse)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    # dQ is added by the TMA engine in whatever order the items arrive
    assert (g1[0].float() - g2[0].float()).abs().max() <= 1e-2 * g1[0].float().abs().max()


def _varlen_case(lens, H, d, causal, seed):
    q, k, v, do, cu = random_varlen(lens, H, d, torch.bfloat16, seed=seed)
    scale = 1 / math.sqrt(d)
    args = [t.cuda() for t in (q, k, v)]
    cuc = cu.cuda()
    o, lse = fa.fa_fwd_varlen(*args, cuc, max(lens), scale, causal=causal)
    grads = fa.fa_bwd_varlen(*args, o, do.cuda(), lse, cuc, max(lens), scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    ref = varlen_attention_bwd(to64(q), to64(k), to64(v), to64(do), cu.tolist(), scale, causal)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        assert rel_max(g, r) <= TOL_BF16_GRAD, (name, rel_max(g, r))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_persistent_backward_packed_batch_many_sequences(d, causal):
    """A packed batch of 40 sequences (empty ones among them) whose units
    outnumber the SMs: the preprocess ranks the sequences by length and the
    CTAs take the units, longest sequence first, from the device counter."""
    rng = np.random.default_rng(40 + d)
    lens = [int(x) for x in rng.integers(0, 700, size=40)]
    lens[3] = lens[17] = 0
    _varlen_case(lens, 4, d, causal, seed=d + int(causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_persistent_backward_packed_batch_past_1024_sequences(d, causal):
    """More than 1024 sequences: the schedule keeps their index order."""
    rng = np.random.default_rng(1100)
    lens = [int(x) for x in rng.integers(1, 48, size=1100)]
    _varlen_case(lens, 1, d, causal, seed=7 + d + int(causal))


@pytest.mark.parametrize("causal", [False, True])
def test_persistent_backward_packed_batch_long_sequences(causal):
    """Six sequences of 1500-4100 keys (12 to 33 key tiles), 12 heads: long
    units, the longest sequences' units first."""
    lens = [1500, 4100, 2049, 3333, 1999, 2600]
    _varlen_case(lens, 12, 128, causal, seed=99 + int(causal))
