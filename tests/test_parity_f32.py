"""GPU parity of the float32 CUDA-core path against the fp64 oracle.

Bar: max |gpu - oracle| <= 1e-5 (absolute) for O and LSE of the mini-lab
workload; backward outputs within 1e-5 * max(1, max|ref|)."""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import WORKLOADS, random_qkv, workload_inputs
from oracle import attention_bwd_batched, attention_fwd_batched
from parity_utils import TOL_F32_ABS, max_abs, to64

pytestmark = pytest.mark.gpu


def test_minilab_workload_forward():
    w = WORKLOADS["minilab_f32_1x1x16x8"]
    q, k, v, _ = workload_inputs(w)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), w.scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    O, LSE = attention_fwd_batched(to64(q), to64(k), to64(v), w.scale)
    assert max_abs(o, O) <= TOL_F32_ABS
    assert max_abs(lse, LSE) <= TOL_F32_ABS


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 8), (1, 2, 5, 1), (2, 1, 33, 33), (1, 3, 100, 64),
                                     (1, 1, 257, 128), (2, 2, 70, 100), (1, 1, 31, 31)])
def test_forward_shapes(B, H, N, d):
    q, k, v, _ = random_qkv(B, H, N, d, torch.float32, seed=N * 7 + d, with_do=False)
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), scale)
    O, LSE = attention_fwd_batched(to64(q), to64(k), to64(v), scale)
    assert max_abs(o, O) <= TOL_F32_ABS
    assert max_abs(lse, LSE) <= TOL_F32_ABS


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 16, 8), (1, 1, 1, 4), (2, 2, 37, 33), (1, 2, 100, 64),
                                     (1, 1, 129, 128)])
def test_backward_shapes(B, H, N, d):
    q, k, v, do = random_qkv(B, H, N, d, torch.float32, seed=1000 + N + d)
    scale = 1 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.fa_fwd(qc, kc, vc, scale)
    dq, dk, dv = fa.fa_bwd(qc, kc, vc, o, doc, lse, scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    dQ, dK, dV = attention_bwd_batched(to64(q), to64(k), to64(v), to64(do), scale)
    for got, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        assert max_abs(got, ref) <= TOL_F32_ABS * max(1.0, np.abs(ref).max())


def test_forward_is_deterministic():
    q, k, v, _ = random_qkv(1, 2, 200, 64, torch.float32, seed=5, with_do=False)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.fa_fwd(q, k, v)
    o2, l2 = fa.fa_fwd(q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
