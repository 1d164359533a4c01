"""GPU parity of the bf16 tcgen05 forward kernel against the fp64 oracle.

Bar: max|O_gpu - O_ref| / max|O_ref| <= 2e-2 and max|LSE_gpu - LSE_ref| <= 1e-3.
Inputs are the exact bf16 values the kernel sees, upcast to fp64. Full-size
workloads are checked on whole heads plus sampled rows of every head."""
import math

import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300.inputs import WORKLOADS, random_qkv, workload_inputs
from oracle import attention_fwd, attention_fwd_rows
from parity_utils import TOL_BF16_LSE, TOL_BF16_O, max_abs, rel_max, to64

pytestmark = pytest.mark.gpu


def _check_heads(q, k, v, o, lse, scale, heads, rows_per_head=0, seed=0):
    q64, k64, v64 = to64(q), to64(k), to64(v)
    o64, l64 = to64(o), to64(lse)
    B, H, N, _ = q64.shape
    for b, h in heads:
        O, LSE = attention_fwd(q64[b, h], k64[b, h], v64[b, h], scale)
        assert rel_max(o64[b, h], O) <= TOL_BF16_O, (b, h)
        assert max_abs(l64[b, h], LSE) <= TOL_BF16_LSE, (b, h)
    if rows_per_head:
        rng = np.random.default_rng(seed)
        for b in range(B):
            for h in range(H):
                rows = rng.choice(N, size=min(rows_per_head, N), replace=False)
                rows[0] = N - 1  # always include the ragged tail row
                O, LSE = attention_fwd_rows(q64[b, h], k64[b, h], v64[b, h], scale, rows)
                assert rel_max(o64[b, h][rows], O) <= TOL_BF16_O, (b, h)
                assert max_abs(l64[b, h][rows], LSE) <= TOL_BF16_LSE, (b, h)


@pytest.mark.parametrize("N", [1, 17, 128, 129, 255, 256, 257, 383, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_lengths(N, d):
    q, k, v, _ = random_qkv(1, 2, N, d, torch.bfloat16, seed=N + d, with_do=False)
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    _check_heads(q, k, v, o, lse, scale, [(0, 0), (0, 1)])


def test_growing_max_forces_rescale():
    # keys grow along the sequence so the running max rises on every tile
    B, H, N, d = 1, 2, 1024, 64
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=3, with_do=False)
    ramp = torch.linspace(0.1, 6.0, N).view(1, 1, N, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    q = (q.float().abs() + 0.5).to(torch.bfloat16)
    k = k.abs()
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), 0.125)
    _check_heads(q, k, v, o, lse, 0.125, [(0, 0), (0, 1)])


def test_large_scores_do_not_overflow():
    B, H, N, d = 1, 1, 640, 128
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=11, with_do=False)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), 1.0)  # scores ~ N(0, 128)
    _check_heads(q, k, v, o, lse, 1.0, [(0, 0)])


def test_workload_fwd_4x16x1024x64():
    w = WORKLOADS["fwd_bf16_4x16x1024x64"]
    q, k, v, _ = workload_inputs(w)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), w.scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    _check_heads(q, k, v, o, lse, w.scale, heads)


def test_workload_fwd_2x16x4096x128():
    w = WORKLOADS["fwd_bf16_2x16x4096x128"]
    q, k, v, _ = workload_inputs(w)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), w.scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]  # every head, whole
    _check_heads(q, k, v, o, lse, w.scale, heads)


def test_workload_fwd_1x32x16384x128_with_big_keys():
    w = WORKLOADS["fwdbwd_bf16_1x32x16384x128"]
    q, k, v, _ = workload_inputs(w)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), w.scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    _check_heads(q, k, v, o, lse, w.scale, [(0, 0), (0, 31)], rows_per_head=16, seed=2)


def test_forward_is_deterministic_bf16():
    q, k, v, _ = random_qkv(2, 4, 777, 128, torch.bfloat16, seed=9, with_do=False)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.fa_fwd(q, k, v)
    o2, l2 = fa.fa_fwd(q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_outputs_written_everywhere_and_nowhere_else():
    # NaN-filled outputs inside larger NaN canaries: every element of O/LSE must
    # be written and the guard regions left untouched.
    B, H, N, d = 1, 3, 300, 64
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=21, with_do=False)
    n = B * H * N * d
    guard = 4096
    obuf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * N + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    o = obuf[guard:guard + n].view(B, H, N, d)
    lse = lbuf[guard:guard + B * H * N].view(B, H, N)
    fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), 0.125, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert torch.isnan(obuf[:guard]).all() and torch.isnan(obuf[guard + n:]).all()
    assert torch.isnan(lbuf[:guard]).all() and torch.isnan(lbuf[guard + B * H * N:]).all()


def _runs_on_four_tile_kernel(B, H, N, d):
    """The routing rule fa.h states for fa_fwd_plan: bf16, d = 64, causal or not,
    B*H*ceil(N/512) >= 3/4 of the SMs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return d == 64 and 4 * B * H * -(-N // 512) >= 3 * sms


@pytest.mark.parametrize("N,H", [(1, 160), (63, 160), (64, 160), (65, 160), (300, 160), (511, 160),
                                 (512, 160), (513, 80), (1000, 80), (1536, 60), (2049, 40)])
def test_four_tile_d64_forward_ragged_lengths(N, H):
    """Ragged lengths on the four-query-tile d = 64 kernel: key tiles of 64
    with a masked last tile, query tiles past N inside a 512-row block, and
    rows past N not written."""
    B, d = 1, 64
    assert _runs_on_four_tile_kernel(B, H, N, d)
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=7000 + N, with_do=False)
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), scale)
    assert fa.fa_check_device_status() == fa.FA_OK
    _check_heads(q, k, v, o, lse, scale, [(0, 0), (0, H // 2), (0, H - 1)])


def test_four_tile_d64_forward_rescale_and_large_scores():
    # keys growing along the sequence (the reference max moves on every key
    # tile, so O is rescaled in TMEM) and scale 1 (scores ~ N(0, 64))
    B, H, N, d = 1, 128, 1024, 64
    assert _runs_on_four_tile_kernel(B, H, N, d)
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=71, with_do=False)
    ramp = torch.linspace(0.1, 6.0, N).view(1, 1, N, 1)
    kr = (k.float().abs() * ramp).to(torch.bfloat16)
    qr = (q.float().abs() + 0.5).to(torch.bfloat16)
    o, lse = fa.fa_fwd(qr.cuda(), kr.cuda(), v.cuda(), 0.125)
    _check_heads(qr, kr, v, o, lse, 0.125, [(0, 0), (0, 127)])
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), 1.0)
    assert fa.fa_check_device_status() == fa.FA_OK
    _check_heads(q, k, v, o, lse, 1.0, [(0, 3), (0, 100)])


def test_four_tile_d64_outputs_written_everywhere_and_nowhere_else():
    B, H, N, d = 1, 120, 700, 64
    assert _runs_on_four_tile_kernel(B, H, N, d)
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=23, with_do=False)
    n = B * H * N * d
    guard = 4096
    obuf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * N + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    o = obuf[guard:guard + n].view(B, H, N, d)
    lse = lbuf[guard:guard + B * H * N].view(B, H, N)
    fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), 0.125, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert torch.isnan(obuf[:guard]).all() and torch.isnan(obuf[guard + n:]).all()
    assert torch.isnan(lbuf[:guard]).all() and torch.isnan(lbuf[guard + B * H * N:]).all()
    # deterministic
    o2, l2 = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), 0.125)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("N,H", [(1, 160), (100, 160), (512, 160), (513, 80), (1000, 80), (2048, 40)])
def test_four_tile_d64_causal_forward(N, H):
    """Causal attention on the four-query-tile d = 64 kernel: each query tile
    stops at its diagonal, the last two 64-key tiles masked per row, blocks
    scheduled longest first."""
    B, d = 1, 64
    assert _runs_on_four_tile_kernel(B, H, N, d)
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=9000 + N, with_do=False)
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), scale, causal=True)
    assert fa.fa_check_device_status() == fa.FA_OK
    q64, k64, v64 = to64(q), to64(k), to64(v)
    o64, l64 = to64(o), to64(lse)
    for h in (0, H // 2, H - 1):
        O, LSE = attention_fwd(q64[0, h], k64[0, h], v64[0, h], scale, causal=True)
        assert rel_max(o64[0, h], O) <= TOL_BF16_O, h
        assert max_abs(l64[0, h], LSE) <= TOL_BF16_LSE, h


@pytest.mark.parametrize("B,H,N,causal", [(1, 16, 16384, False), (1, 16, 16384, True), (1, 32, 12289, False),
                                          (1, 8, 32768, True)])
def test_four_tile_d64_long_sequences(B, H, N, causal):
    """Long sequences on the four-query-tile d = 64 kernel: sampled rows of
    every head (the first and last rows of every 512-row block among them, and
    the ragged tail) against the oracle, causal or not."""
    d = 64
    assert _runs_on_four_tile_kernel(B, H, N, d)
    q, k, v, _ = random_qkv(B, H, N, d, torch.bfloat16, seed=N + H + int(causal), with_do=False)
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    q64, k64, v64 = to64(q), to64(k), to64(v)
    o64, l64 = to64(o), to64(lse)
    rng = np.random.default_rng(N)
    edges = np.concatenate([np.arange(0, N, 512), np.arange(511, N, 512), [N - 1]])
    for h in range(H):
        rows = np.unique(np.concatenate([edges[h % 2::2], rng.choice(N, 16, replace=False)]))
        O, LSE = attention_fwd_rows(q64[0, h], k64[0, h], v64[0, h], scale, rows, causal=causal)
        assert rel_max(o64[0, h][rows], O) <= TOL_BF16_O, h
        assert max_abs(l64[0, h][rows], LSE) <= TOL_BF16_LSE, h
