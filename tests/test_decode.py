"""GPU parity of KV-cache decode (fa_decode) against the fp64 oracle.

Decode is attention of Nq <= 16 new queries per head against Nk cached keys
(one query on CUDA cores, more on the tensor cores);
the oracle is the plain definition (``attention_fwd`` on the rectangular
problem). The library splits the keys into ranges and merges the partial
results; the tests cover one range and many, a ragged last range, fewer keys
than one 64-key tile, every query-count bucket, both head sizes and the
full-size decode workload (sampled heads). Bar as for the bf16 forward:
max|O - O_ref| / max|O_ref| <= 2e-2, max|LSE - LSE_ref| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import DECODE_WORKLOADS, decode_inputs, random_qkv
from oracle import attention_fwd
from parity_utils import TOL_BF16_LSE, TOL_BF16_O, max_abs, rel_max, to64

pytestmark = pytest.mark.gpu


def _check(q, k, v, o, lse, scale, heads):
    q64, o64, l64 = to64(q), to64(o), to64(lse)
    for b, h in heads:
        O, LSE = attention_fwd(q64[b, h], to64(k[b, h]), to64(v[b, h]), scale)
        assert rel_max(o64[b, h], O) <= TOL_BF16_O, (b, h)
        assert max_abs(l64[b, h], LSE) <= TOL_BF16_LSE, (b, h)


def _run(B, H, nq, nk, d, seed, big_key_every=0):
    q, k, v, _ = random_qkv(B, H, nq, d, torch.bfloat16, seed=seed, with_do=False, n_k=nk,
                            big_key_every=big_key_every)
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    return q, k, v, o, lse, scale


@pytest.mark.parametrize("nk", [1, 17, 63, 64, 65, 1000, 4097])
@pytest.mark.parametrize("nq", [1, 3, 8, 16])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_cache_lengths(nk, nq, d):
    q, k, v, o, lse, scale = _run(1, 3, nq, nk, d, seed=nk * 10 + nq + d)
    _check(q, k, v, o, lse, scale, [(0, 0), (0, 1), (0, 2)])


@pytest.mark.parametrize("nq", [1, 2, 4, 5, 8, 11, 16])
def test_every_query_bucket_with_many_splits(nq):
    B, H, nk, d = 2, 2, 3000, 128
    splits, kps = fa.fa_decode_plan(B, H, nq, nk, d)
    assert splits > 1 and nk % kps != 0  # several ranges, the last one ragged
    q, k, v, o, lse, scale = _run(B, H, nq, nk, d, seed=nq)
    _check(q, k, v, o, lse, scale, [(b, h) for b in range(B) for h in range(H)])


def test_single_range():
    # enough heads that the planner keeps one range per head
    B, H, nq, nk, d = 16, 64, 1, 256, 64
    assert fa.fa_decode_plan(B, H, nq, nk, d)[0] == 1
    q, k, v, o, lse, scale = _run(B, H, nq, nk, d, seed=11)
    _check(q, k, v, o, lse, scale, [(0, 0), (7, 33), (15, 63)])


def test_moving_max_across_ranges():
    # every 64th key scaled by 4: the per-range maxima differ widely
    q, k, v, o, lse, scale = _run(1, 2, 4, 20000, 128, seed=5, big_key_every=64)
    _check(q, k, v, o, lse, scale, [(0, 0), (0, 1)])


def test_growing_keys_force_rescale_within_a_range():
    B, H, nq, nk, d = 1, 2, 2, 2048, 64
    q, k, v, _ = random_qkv(B, H, nq, d, torch.bfloat16, seed=9, with_do=False, n_k=nk)
    ramp = torch.linspace(0.1, 6.0, nk).view(1, 1, nk, 1)
    k = (k.float().abs() * ramp).to(torch.bfloat16)
    q = (q.float().abs() + 0.5).to(torch.bfloat16)
    o, lse = fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), 0.125)
    _check(q, k, v, o, lse, 0.125, [(0, 0), (0, 1)])


def test_decode_matches_forward_on_square_problems():
    """With Nq = Nk the decode path and the tensor-core forward compute the same thing."""
    q, k, v, _ = random_qkv(1, 4, 8, 128, torch.bfloat16, seed=2, with_do=False)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.fa_decode(q, k, v)
    o2, l2 = fa.fa_fwd(q, k, v)
    assert rel_max(o1, to64(o2)) <= TOL_BF16_O
    assert max_abs(l1, to64(l2)) <= TOL_BF16_LSE


def test_reused_workspace_and_outputs():
    B, H, nq, nk, d = 2, 4, 4, 5000, 128
    q, k, v, _ = random_qkv(B, H, nq, d, torch.bfloat16, seed=21, with_do=False, n_k=nk)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ws = torch.full((fa.fa_decode_workspace_bytes(B, H, nq, nk, d),), 255, dtype=torch.uint8,
                    device="cuda")  # garbage (NaN bit patterns) on entry
    o1, l1 = fa.fa_decode(q, k, v, workspace=ws)
    o2, l2 = fa.fa_decode(q, k, v, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)  # deterministic
    _check(q.cpu(), k.cpu(), v.cpu(), o1, l1, 1 / math.sqrt(d), [(0, 0), (1, 3)])


@pytest.mark.parametrize("name", sorted(DECODE_WORKLOADS))
def test_full_size_decode_workload_sampled_heads(name):
    w = DECODE_WORKLOADS[name]
    q, k, v = decode_inputs(w, seed=0)
    o, lse = fa.fa_decode(q.cuda(), k.cuda(), v.cuda(), w.scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    rng = np.random.default_rng(1)
    heads = [(int(b), int(h)) for b, h in zip(rng.integers(0, w.B, 6), rng.integers(0, w.H, 6))]
    heads += [(0, 0), (w.B - 1, w.H - 1)]
    _check(q, k, v, o, lse, w.scale, heads)
