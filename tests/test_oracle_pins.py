"""Pins of the fp64 oracle to facts fixed outside the oracle itself.

Each test compares the oracle with a value the pages print, a closed form, an
invariant, a library routine (PyTorch/scipy in float64 on the CPU), or central
finite differences. Chosen so that a dropped term, a wrong sign or index or a
transposed operand in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import (attention_bwd, attention_bwd_batched, attention_fwd, attention_fwd_batched,
                    attention_fwd_rows, merge_partials, online_softmax_stats, row_softmax, scores,
                    split_kv_attention_fwd, tiled_attention_fwd, varlen_attention_bwd,
                    varlen_attention_fwd)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    out = {}
    blocks = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "block":
                blocks.append([float(v) for v in vals])
            else:
                out[key] = [float(v) for v in vals]
    out["blocks"] = blocks
    return out


def _rand(shape, seed):
    return np.random.default_rng(seed).normal(size=shape)


# --- worked example ("FlashAttention and Triton" §19.5) ---------------------------------

def test_worked_example_online_equals_one_shot():
    fx = _read_fixture("worked_example.txt")
    blocks = fx["blocks"]
    assert blocks == [[1.0, 2.0], [3.0, 4.0]]
    stats = online_softmax_stats(blocks)
    e = math.exp
    l1 = 1 + e(-1)
    l2 = 1 + e(-1) + e(-2) + e(-3)
    assert stats[0][0] == 2.0 and abs(stats[0][1] - l1) <= 1e-15
    assert stats[1][0] == 4.0 and abs(stats[1][1] - l2) <= 1e-15
    # one-shot softmax of the whole row, through the oracle's softmax
    P, m, l = row_softmax(np.array([[1.0, 2.0, 3.0, 4.0]]))
    assert m[0] == 4.0 and abs(l[0] - l2) <= 1e-15
    p_expected = np.array([e(-3), e(-2), e(-1), 1.0]) / l2
    assert np.abs(P[0] - p_expected).max() <= 1e-15
    # the same row as an attention problem: q = [1], keys 1..4, scale 1
    q = np.array([[1.0]])
    K = np.array([[1.0], [2.0], [3.0], [4.0]])
    V = _rand((4, 3), 7)
    O, LSE = attention_fwd(q, K, V, 1.0)
    assert abs(LSE[0] - (4.0 + math.log(l2))) <= 1e-14
    assert np.abs(O[0] - p_expected @ V).max() <= 1e-14
    Ot, LSEt = tiled_attention_fwd(q, K, V, 1.0, q_tile=1, k_tile=2)
    assert np.abs(Ot - O).max() <= 1e-15 and abs(LSEt[0] - LSE[0]) <= 1e-15


# --- mini lab ("FlashAttention and Triton" §19.12) ---------------------------------------

def _minilab():
    rng = np.random.default_rng(0)
    return rng.normal(size=(16, 8)), rng.normal(size=(16, 8)), rng.normal(size=(16, 8))


def test_minilab_tiled_equals_naive():
    fx = _read_fixture("minilab.txt")
    Q, K, V = _minilab()
    assert Q.shape == tuple(int(x) for x in fx["shape"])
    scale = 1 / math.sqrt(8)
    ref, lse = attention_fwd(Q, K, V, scale)
    qt, kt = int(fx["q_tile"][0]), int(fx["k_tile"][0])
    sim, lse_t = tiled_attention_fwd(Q, K, V, scale, q_tile=qt, k_tile=kt)
    assert np.abs(ref - sim).max() < fx["max_abs_diff"][0]
    assert np.allclose(ref, sim, atol=fx["atol"][0])
    assert np.abs(lse - lse_t).max() < 1e-12


@pytest.mark.parametrize("qt,kt", [(1, 1), (3, 5), (16, 16), (5, 16), (16, 3), (7, 1)])
def test_minilab_ragged_tiles(qt, kt):
    Q, K, V = _minilab()
    scale = 1 / math.sqrt(8)
    ref, lse = attention_fwd(Q, K, V, scale)
    sim, lse_t = tiled_attention_fwd(Q, K, V, scale, q_tile=qt, k_tile=kt)
    assert np.abs(ref - sim).max() < 1e-12
    assert np.abs(lse - lse_t).max() < 1e-12


# --- softmax invariants ------------------------------------------------------------------

def test_rows_of_P_are_stochastic():
    S = scores(_rand((33, 16), 1), _rand((45, 16), 2), 0.25) * 7.0
    P, m, l = row_softmax(S)
    assert (P >= 0).all()
    assert np.abs(P.sum(axis=1) - 1).max() <= 1e-14 * 45
    assert np.allclose(m, S.max(axis=1))
    assert np.argmax(P, axis=1).tolist() == np.argmax(S, axis=1).tolist()


def test_lse_matches_scipy_logsumexp():
    from scipy.special import logsumexp
    Q, K, V = _rand((20, 8), 3), _rand((30, 8), 4), _rand((30, 5), 5)
    _, LSE = attention_fwd(Q, K, V, 0.3)
    assert np.abs(LSE - logsumexp(0.3 * (Q @ K.T), axis=1)).max() <= 1e-13


# --- closed forms ------------------------------------------------------------------------

def test_single_key_gives_that_value_row():
    Q, K, V = _rand((6, 4), 10), _rand((1, 4), 11), _rand((1, 3), 12)
    O, LSE = attention_fwd(Q, K, V, 0.7)
    assert np.abs(O - V[0]).max() <= 1e-15
    assert np.abs(LSE - 0.7 * (Q @ K[0])).max() <= 1e-14


def test_zero_queries_average_the_values_and_have_closed_form_grads():
    N, d, scale = 9, 5, 0.4
    Q = np.zeros((N, d))
    K, V, dO = _rand((N, d), 20), _rand((N, d), 21), _rand((N, d), 22)
    O, LSE = attention_fwd(Q, K, V, scale)
    assert np.abs(O - V.mean(axis=0)).max() <= 1e-15
    assert np.abs(LSE - math.log(N)).max() <= 1e-15
    dQ, dK, dV = attention_bwd(Q, K, V, dO, scale)
    # P = 1/N everywhere
    assert np.abs(dV - dO.sum(axis=0) / N).max() <= 1e-14
    assert np.abs(dK).max() == 0.0
    Vc = V - V.mean(axis=0)
    dQ_expected = (scale / N) * (dO @ Vc.T) @ K
    assert np.abs(dQ - dQ_expected).max() <= 1e-14


def test_dominant_key_selects_its_value():
    Q = _rand((4, 6), 30)
    K = _rand((12, 6), 31) * 0.01
    K[5] = 0.0
    V = _rand((12, 3), 32)
    S_other = Q @ K.T
    # an extra dimension that only key 5 and the queries use lifts key 5's
    # score more than 50 above every other key for every query
    Qx = np.concatenate([Q, np.ones((4, 1))], axis=1)
    Kx = np.concatenate([K, np.zeros((12, 1))], axis=1)
    Kx[5, -1] = 50.0 + np.abs(S_other).max() + 1.0
    O, _ = attention_fwd(Qx, Kx, V, 1.0)
    assert np.abs(O - V[5]).max() <= 1e-18 + 12 * math.exp(-50) * np.abs(V).max()


def test_equal_value_rows_give_that_row():
    Q, K = _rand((7, 4), 40), _rand((11, 4), 41)
    v = _rand((1, 6), 42)
    O, _ = attention_fwd(Q, K, np.repeat(v, 11, axis=0), 2.0)
    assert np.abs(O - v).max() <= 1e-14


def test_identity_values_return_P():
    Q, K = _rand((5, 3), 50), _rand((8, 3), 51)
    O, _ = attention_fwd(Q, K, np.eye(8), 1.3)
    P, _, _ = row_softmax(1.3 * Q @ K.T)
    assert np.abs(O - P).max() <= 1e-15
    assert np.abs(O.sum(axis=1) - 1).max() <= 1e-14


def test_joint_permutation_of_keys_and_values():
    Q, K, V, dO = _rand((10, 4), 60), _rand((13, 4), 61), _rand((13, 5), 62), _rand((10, 5), 63)
    perm = np.random.default_rng(64).permutation(13)
    O, LSE = attention_fwd(Q, K, V, 0.5)
    Op, LSEp = attention_fwd(Q, K[perm], V[perm], 0.5)
    assert np.abs(O - Op).max() <= 1e-14 and np.abs(LSE - LSEp).max() <= 1e-14
    dQ, dK, dV = attention_bwd(Q, K, V, dO, 0.5)
    dQp, dKp, dVp = attention_bwd(Q, K[perm], V[perm], dO, 0.5)
    assert np.abs(dQ - dQp).max() <= 1e-13
    assert np.abs(dK[perm] - dKp).max() <= 1e-13
    assert np.abs(dV[perm] - dVp).max() <= 1e-13


def test_key_shift_leaves_P_unchanged():
    Q, K, V = _rand((6, 4), 70), _rand((9, 4), 71), _rand((9, 2), 72)
    c = _rand((4,), 73)
    O, LSE = attention_fwd(Q, K, V, 0.8)
    Os, LSEs = attention_fwd(Q, K + c, V, 0.8)
    assert np.abs(O - Os).max() <= 1e-13
    assert np.abs(LSEs - LSE - 0.8 * (Q @ c)).max() <= 1e-13


def test_rows_subset_matches_full():
    Q, K, V = _rand((40, 8), 80), _rand((50, 8), 81), _rand((50, 8), 82)
    O, LSE = attention_fwd(Q, K, V, 0.35)
    rows = [0, 7, 39, 13]
    Or, LSEr = attention_fwd_rows(Q, K, V, 0.35, rows)
    assert np.array_equal(Or, O[rows]) or np.abs(Or - O[rows]).max() <= 1e-15
    assert np.abs(LSEr - LSE[rows]).max() <= 1e-15


# --- library routine: PyTorch float64 on the CPU -----------------------------------------

@pytest.mark.parametrize("nq,nk,scale", [(37, 37, None), (37, 29, 0.173), (5, 64, 1.0)])
def test_against_torch_sdpa_and_autograd_float64(nq, nk, scale):
    B, H, d = 2, 3, 16
    g = torch.Generator().manual_seed(nq * 100 + nk)
    q = torch.randn(B, H, nq, d, dtype=torch.float64, generator=g, requires_grad=True)
    k = torch.randn(B, H, nk, d, dtype=torch.float64, generator=g, requires_grad=True)
    v = torch.randn(B, H, nk, d + 3, dtype=torch.float64, generator=g, requires_grad=True)
    do = torch.randn(B, H, nq, d + 3, dtype=torch.float64, generator=g)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    o.backward(do)
    s = 1 / math.sqrt(d) if scale is None else scale
    for b in range(B):
        for h in range(H):
            Q, K, V, dO = (t[b, h].detach().numpy() for t in (q, k, v, do))
            O, _ = attention_fwd(Q, K, V, s)
            assert np.abs(O - o[b, h].detach().numpy()).max() <= 1e-12
            dQ, dK, dV = attention_bwd(Q, K, V, dO, s)
            assert np.abs(dQ - q.grad[b, h].numpy()).max() <= 1e-12
            assert np.abs(dK - k.grad[b, h].numpy()).max() <= 1e-12
            assert np.abs(dV - v.grad[b, h].numpy()).max() <= 1e-12


# --- central finite differences ----------------------------------------------------------

@pytest.mark.parametrize("N,d", [(3, 2), (5, 4), (3, 4), (5, 2)])
def test_backward_against_central_differences(N, d):
    rng = np.random.default_rng(N * 10 + d)
    Q, K, V, G = (rng.normal(size=(N, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    h = 1e-6

    def loss(Q_, K_, V_):
        return float((attention_fwd(Q_, K_, V_, scale)[0] * G).sum())

    dQ, dK, dV = attention_bwd(Q, K, V, G, scale)
    for X, dX, which in ((Q, dQ, 0), (K, dK, 1), (V, dV, 2)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args_p = [Q.copy(), K.copy(), V.copy()]
            args_m = [Q.copy(), K.copy(), V.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - dX).max() / max(np.abs(dX).max(), 1e-300)
        assert err <= 1e-7, (which, err)


def test_D_identity_rowsum_dP_P_equals_rowsum_dO_O():
    Q, K, V, dO = _rand((12, 6), 90), _rand((15, 6), 91), _rand((15, 6), 92), _rand((12, 6), 93)
    scale = 0.45
    P, _, _ = row_softmax(scale * Q @ K.T)
    O, _ = attention_fwd(Q, K, V, scale)
    dP = dO @ V.T
    assert np.abs((dP * P).sum(axis=1) - (dO * O).sum(axis=1)).max() <= 1e-12


# ---------------------------------------------------------------- split-KV merge
@pytest.mark.parametrize("nq,nk,kps", [(1, 1, 1), (1, 200, 64), (3, 7, 3), (8, 130, 64), (2, 50, 50)])
def test_split_kv_merge_equals_one_shot(nq, nk, kps):
    """Merging per-range results reproduces attention over all keys (the pages'
    claim that the online (m, l) update is exact), to rounding."""
    rng = np.random.default_rng(nq * 1000 + nk)
    Q, K, V = rng.normal(size=(nq, 16)), rng.normal(size=(nk, 16)), rng.normal(size=(nk, 16))
    O1, L1 = attention_fwd(Q, K, V, 0.25)
    O2, L2 = split_kv_attention_fwd(Q, K, V, 0.25, kps)
    assert np.abs(O1 - O2).max() < 1e-12
    assert np.abs(L1 - L2).max() < 1e-12


def test_split_merge_on_the_worked_example():
    """The worked example's score row [1, 2, 3, 4] as two key ranges of two:
    one query q = [1], keys k_j = [j], scale 1. The merged log-sum-exp is the
    closed form 4 + ln(1 + e^-1 + e^-2 + e^-3), and with values v_j = [j] the
    merged output is sum_j j e^(j-4) / l."""
    Q = np.array([[1.0]])
    K = np.array([[1.0], [2.0], [3.0], [4.0]])
    V = K.copy()
    O, L = split_kv_attention_fwd(Q, K, V, 1.0, 2)
    l = 1 + math.exp(-1) + math.exp(-2) + math.exp(-3)
    assert abs(L[0] - (4 + math.log(l))) < 1e-14
    expect = sum(j * math.exp(j - 4) for j in range(1, 5)) / l
    assert abs(O[0, 0] - expect) < 1e-14


def test_merge_of_a_dominant_range_returns_it():
    """A range whose log-sum-exp exceeds the others by far carries all weight."""
    O_a, O_b = np.full((1, 2), 3.0), np.full((1, 2), -5.0)
    O, L = merge_partials([O_a, O_b], [np.array([800.0]), np.array([0.0])])
    assert np.allclose(O, 3.0, rtol=0, atol=1e-300) and abs(L[0] - 800.0) < 1e-12


# ---------------------------------------------------------------- causal and variable length
def test_causal_against_brute_force_loops():
    """Pure-Python loops over visible keys only (c <= r), math.exp / math.log."""
    rng = np.random.default_rng(77)
    n, d, scale = 6, 3, 0.7
    Q, K, V = rng.normal(size=(n, d)), rng.normal(size=(n, d)), rng.normal(size=(n, d))
    O, LSE = attention_fwd(Q, K, V, scale, causal=True)
    for r in range(n):
        s = [scale * sum(Q[r, i] * K[c, i] for i in range(d)) for c in range(r + 1)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        l = sum(w)
        for j in range(d):
            assert abs(O[r, j] - sum(w[c] * V[c, j] for c in range(r + 1)) / l) < 1e-14
        assert abs(LSE[r] - (m + math.log(l))) < 1e-14


def test_causal_closed_forms():
    """Row 0 sees only key 0 (O_0 = V_0, LSE_0 = scale q_0.k_0); the last row
    sees every key (equal to the non-causal last row)."""
    rng = np.random.default_rng(78)
    Q, K, V = rng.normal(size=(9, 5)), rng.normal(size=(9, 5)), rng.normal(size=(9, 4))
    O, LSE = attention_fwd(Q, K, V, 0.4, causal=True)
    assert np.abs(O[0] - V[0]).max() < 1e-15 and abs(LSE[0] - 0.4 * Q[0] @ K[0]) < 1e-14
    O2, LSE2 = attention_fwd(Q, K, V, 0.4)
    assert np.abs(O[-1] - O2[-1]).max() < 1e-14 and abs(LSE[-1] - LSE2[-1]) < 1e-14
    rows = np.array([8, 0, 4])
    Or, Lr = attention_fwd_rows(Q, K, V, 0.4, rows, causal=True)
    assert np.abs(Or - O[rows]).max() < 1e-15 and np.abs(Lr - LSE[rows]).max() < 1e-15


@pytest.mark.parametrize("n", [1, 7, 33])
def test_causal_against_torch_sdpa_and_autograd_float64(n):
    B, H, d = 1, 2, 8
    g = torch.Generator().manual_seed(n)
    q, k, v = (torch.randn(B, H, n, d, dtype=torch.float64, generator=g, requires_grad=True)
               for _ in range(3))
    do = torch.randn(B, H, n, d, dtype=torch.float64, generator=g)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    o.backward(do)
    s = 1 / math.sqrt(d)
    for h in range(H):
        Q, K, V, dO = (t[0, h].detach().numpy() for t in (q, k, v, do))
        O, _ = attention_fwd(Q, K, V, s, causal=True)
        assert np.abs(O - o[0, h].detach().numpy()).max() <= 1e-12
        dQ, dK, dV = attention_bwd(Q, K, V, dO, s, causal=True)
        for mine, ref in ((dQ, q.grad), (dK, k.grad), (dV, v.grad)):
            assert np.abs(mine - ref[0, h].numpy()).max() <= 1e-12


def test_causal_backward_against_central_differences():
    rng = np.random.default_rng(5)
    N, d, h = 4, 3, 1e-6
    Q, K, V, G = (rng.normal(size=(N, d)) for _ in range(4))

    def loss(Q_, K_, V_):
        return float((attention_fwd(Q_, K_, V_, 0.6, causal=True)[0] * G).sum())

    grads = attention_bwd(Q, K, V, G, 0.6, causal=True)
    for which, dX in enumerate(grads):
        X = (Q, K, V)[which]
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args_p, args_m = [Q.copy(), K.copy(), V.copy()], [Q.copy(), K.copy(), V.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.abs(num - dX).max() / max(np.abs(dX).max(), 1e-300) <= 1e-7


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_against_torch_sdpa_per_sequence(causal):
    """A packed batch equals independent attention per sequence (torch float64)."""
    lens = [5, 1, 12, 0, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    total, H, d = int(cu[-1]), 3, 4
    g = torch.Generator().manual_seed(3)
    q, k, v, do = (torch.randn(total, H, d, dtype=torch.float64, generator=g) for _ in range(4))
    O, LSE = varlen_attention_fwd(q.numpy(), k.numpy(), v.numpy(), cu, 0.5, causal)
    dQ, dK, dV = varlen_attention_bwd(q.numpy(), k.numpy(), v.numpy(), do.numpy(), cu, 0.5, causal)
    for b in range(len(lens)):
        s, e = int(cu[b]), int(cu[b + 1])
        if s == e:
            continue
        qs, ks, vs = (t[s:e].transpose(0, 1).clone().requires_grad_(True) for t in (q, k, v))
        o = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=0.5, is_causal=causal)
        o.backward(do[s:e].transpose(0, 1))
        assert np.abs(O[s:e] - o.detach().transpose(0, 1).numpy()).max() <= 1e-12
        for mine, ref in ((dQ, qs.grad), (dK, ks.grad), (dV, vs.grad)):
            assert np.abs(mine[s:e] - ref.transpose(0, 1).numpy()).max() <= 1e-12
        # LSE from its definition: log of the sum of exp over the visible scores
        for h in range(H):
            S = 0.5 * q[s:e, h].numpy() @ k[s:e, h].numpy().T
            if causal:
                S = np.where(np.tril(np.ones_like(S, dtype=bool)), S, -np.inf)
            ref_lse = np.log(np.exp(S - S.max(1, keepdims=True)).sum(1)) + S.max(1)
            assert np.abs(LSE[h, s:e] - ref_lse).max() <= 1e-12


# --- the [B, H, N, d] batch wrappers against the library's batched routine -----------

def _torch_batch(B, H, N, d, dv, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, d, dtype=torch.float64, generator=g, requires_grad=True)
    k = torch.randn(B, H, N, d, dtype=torch.float64, generator=g, requires_grad=True)
    v = torch.randn(B, H, N, dv, dtype=torch.float64, generator=g, requires_grad=True)
    do = torch.randn(B, H, N, dv, dtype=torch.float64, generator=g)
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
def test_batched_wrappers_against_torch_batched_sdpa_float64(causal):
    """Every (b, h) of the wrappers' output against torch's batched SDPA + autograd.

    The heads differ (distinct seeded draws), so a swapped b/h index, a head
    computed from another head's K or V, or dQ/dK/dV returned in the wrong
    slot fails here. LSE is checked against its definition computed by torch.
    """
    B, H, N, d, dv, scale = 2, 3, 19, 8, 5, 0.3
    q, k, v, do = _torch_batch(B, H, N, d, dv, 11 + causal)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale, is_causal=causal)
    o.backward(do)
    Q, K, V, dO = (t.detach().numpy() for t in (q, k, v, do))
    O, LSE = attention_fwd_batched(Q, K, V, scale, causal=causal)
    dQ, dK, dV = attention_bwd_batched(Q, K, V, dO, scale, causal=causal)
    assert O.shape == (B, H, N, dv) and LSE.shape == (B, H, N)
    assert np.abs(O - o.detach().numpy()).max() <= 1e-12
    s = scale * torch.einsum("bhnd,bhmd->bhnm", q.detach(), k.detach())
    if causal:
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), -math.inf)
    assert np.abs(LSE - torch.logsumexp(s, dim=-1).numpy()).max() <= 1e-12
    for mine, ref in ((dQ, q.grad), (dK, k.grad), (dV, v.grad)):
        assert mine.shape == tuple(ref.shape)
        assert np.abs(mine - ref.numpy()).max() <= 1e-12


def test_batched_wrappers_head_subset_leaves_the_rest_nan():
    B, H, N, d = 2, 3, 9, 4
    q, k, v, do = _torch_batch(B, H, N, d, d, 5)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=0.7)
    o.backward(do)
    Q, K, V, dO = (t.detach().numpy() for t in (q, k, v, do))
    heads = [(1, 2), (0, 1)]
    O, LSE = attention_fwd_batched(Q, K, V, 0.7, heads=heads)
    grads = attention_bwd_batched(Q, K, V, dO, 0.7, heads=heads)
    for b in range(B):
        for h in range(H):
            if (b, h) in heads:
                assert np.abs(O[b, h] - o[b, h].detach().numpy()).max() <= 1e-12
                assert np.isfinite(LSE[b, h]).all()
                for mine, ref in zip(grads, (q.grad, k.grad, v.grad)):
                    assert np.abs(mine[b, h] - ref[b, h].numpy()).max() <= 1e-12
            else:
                assert np.isnan(O[b, h]).all() and np.isnan(LSE[b, h]).all()
                for mine in grads:
                    assert np.isnan(mine[b, h]).all()
