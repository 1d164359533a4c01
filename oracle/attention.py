"""Exact-attention oracle: plain, slow, fp64, CPU.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product path (``exact_attention_30_gb300``) never imports it and
shares no code with it: no kernels, helpers, constants or pre/post-processing.

What it computes (all arithmetic in float64, numpy; a BLAS matmul is the only
library primitive used as a step):

* ``attention_fwd`` -- the plain definition O = softmax(scale * Q K^T) V with
  S and P materialised, as written in "Lesson 1: FlashAttention core idea" §1
  and in the naive three-step decomposition of "Interview Q15: FlashAttention"
  (Step 1-3) and "FlashAttention and Triton" §19.2. The softmax is the
  max-subtracted one of "FlashAttention and Triton" §19.12
  (``standard_attention``) and §19.11. It also returns the per-row
  log-sum-exp LSE = m + ln(l) of the scaled scores: the per-row statistics
  that "Lesson 1" §5 says are the only thing kept for the backward pass.
* ``attention_bwd`` -- dQ, dK, dV from the chain rule through the same
  definition, in the notation of "Lesson 1" §5 (backward by recomputation):
  dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(dP o P)) * scale,
  dQ = dS K, dK = dS^T Q. The row sum is taken over the whole row of P.
* ``tiled_attention_fwd`` -- the tiled online-softmax algorithm, step by step
  as "Lesson 1" §4 and "FlashAttention and Triton" §19.12 (``tiled_attention``)
  describe it: query tiles outer, key/value tiles inner, running max m,
  running denominator l and unnormalised accumulator rescaled by exp(m - m_new).
  Used only to check the oracle against itself (the pages claim the two agree
  to < 1e-12), never as the reference for the GPU path.
* ``online_softmax_stats`` -- the (m, l) recurrence of "Lesson 1" §3 over a
  list of score blocks, for the worked example of "FlashAttention and Triton"
  §19.5 (scores [1, 2] then [3, 4]).
* ``merge_partials`` / ``split_kv_attention_fwd`` -- the same (m, l) rule
  applied to whole results: attention over disjoint key ranges computed
  separately, then merged. This is how decoding against a KV cache (the
  inference remark of "Interview Q15") is parallelised over the keys. The
  reference for decode parity is still ``attention_fwd`` on the rectangular
  problem (N_q new queries, N_k cached keys); the split form is checked
  against it.

* ``causal=True`` (every function above that takes it) -- not on the pages:
  the plainest adjacent variant of the definition for self-attention. Score
  S_rc of query row r and key c is kept only for c <= r; the others are set
  to -inf before the softmax, so P_rc = 0 there and the backward formulas
  above need no change (dS = 0 where P = 0).
* ``varlen_attention_fwd`` / ``varlen_attention_bwd`` -- a packed batch of
  sequences of different lengths ([total, H, d], offsets cu_seqlens): each
  sequence and head is attended to on its own, by the functions above.

Readings where the pages are silent (each also listed in the design notes):
* ``scale`` is a free argument; the pages fix 1/sqrt(d). dS carries exactly one
  factor of ``scale`` (the pages' "/ sqrt(d)" in the dS line).
* LSE is the natural-log log-sum-exp of the *scaled* scores.
* Inputs are taken exactly as given (bf16 or fp32 values upcast exactly to
  fp64); outputs are fp64.

Pins (tests/test_oracle_pins.py): the worked example, the mini-lab agreement
of naive and tiled paths, row-stochastic P, closed forms (N = 1, Q = 0, a
dominant key, permutation and key-shift invariance), PyTorch's float64 CPU
scaled_dot_product_attention + autograd (per head, and batched over [B, H] for
the ``*_batched`` wrappers, with a head subset left NaN), and central finite
differences for the backward pass. No function here is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "scores",
    "row_softmax",
    "attention_fwd",
    "attention_bwd",
    "attention_fwd_rows",
    "tiled_attention_fwd",
    "online_softmax_stats",
    "attention_fwd_batched",
    "attention_bwd_batched",
    "merge_partials",
    "split_kv_attention_fwd",
    "causal_mask",
    "varlen_attention_fwd",
    "varlen_attention_bwd",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def causal_mask(n_q: int, n_k: int, rows=None) -> np.ndarray:
    """Boolean [n_q, n_k]: True where key c is visible to query row r (c <= r).

    ``rows``: the global row indices of the n_q query rows (default 0..n_q-1).
    """
    r = np.arange(n_q) if rows is None else np.asarray(rows, dtype=np.int64)
    return np.arange(n_k)[None, :] <= r[:, None]


def scores(Q, K, scale: float, causal: bool = False, rows=None) -> np.ndarray:
    """S = scale * Q K^T, materialised (N_q x N_k); -inf where a causal mask hides a key.

    "Lesson 1: FlashAttention core idea" §1 (the formula and the explicit
    intermediate matrices); "Interview Q15" Step 1.
    """
    S = float(scale) * (_f64(Q) @ _f64(K).T)
    if causal:
        S = np.where(causal_mask(S.shape[0], S.shape[1], rows), S, -np.inf)
    return S


def row_softmax(S):
    """Numerically stable row softmax: returns (P, m, l).

    m_r = max_c S_rc, E = exp(S - m_r), l_r = sum_c E_rc, P = E / l_r.
    "FlashAttention and Triton" §19.12 (``standard_attention``) and §19.11
    (subtract the row max, exponentiate, sum, divide).
    """
    S = _f64(S)
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    P = E / l[:, None]
    return P, m, l


def attention_fwd(Q, K, V, scale: float, causal: bool = False, rows=None):
    """Exact attention forward for one head: (O, LSE).

    O = softmax(scale * Q K^T) V ("Lesson 1" §1; "Interview Q15" Steps 1-3;
    "FlashAttention and Triton" §19.2). LSE_r = m_r + ln(l_r): the per-row
    statistics that "Lesson 1" §5 keeps for the backward pass, folded into one
    number.
    Q: [N_q, d], K: [N_k, d], V: [N_k, d_v]. ``causal``/``rows``: see ``scores``.
    """
    S = scores(Q, K, scale, causal, rows)
    P, m, l = row_softmax(S)
    O = P @ _f64(V)
    LSE = m + np.log(l)
    return O, LSE


def attention_fwd_rows(Q, K, V, scale: float, rows, causal: bool = False):
    """The definition of ``attention_fwd`` evaluated for the query rows ``rows`` only.

    Softmax is row-local ("FlashAttention and Triton" §19.11: one program per
    row), so row r of O and LSE depends only on query row r and all of K, V.
    """
    rows = np.asarray(rows, dtype=np.int64)
    return attention_fwd(_f64(Q)[rows], K, V, scale, causal, rows)


def attention_bwd(Q, K, V, dO, scale: float, causal: bool = False):
    """Exact attention backward for one head: (dQ, dK, dV).

    "Lesson 1: FlashAttention core idea" §5, written for whole matrices:
      S  = scale * Q K^T,  P = softmax(S)   (rows)
      dV = P^T dO
      dP = dO V^T
      dS = P o (dP - rowsum(dP o P)) * scale
      dQ = dS K
      dK = dS^T Q
    The row sum runs over the full row (the page shows it inside a per-tile
    loop; only the full-row sum is the gradient of softmax).
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    S = scores(Q, K, scale, causal)
    P, _, _ = row_softmax(S)
    dV = P.T @ dO
    dP = dO @ V.T
    D = (dP * P).sum(axis=1)
    dS = P * (dP - D[:, None]) * float(scale)
    dQ = dS @ K
    dK = dS.T @ Q
    return dQ, dK, dV


def tiled_attention_fwd(Q, K, V, scale: float, q_tile: int = 4, k_tile: int = 4):
    """Tiled forward with online softmax (self-check of the oracle only).

    The algorithm of "Lesson 1" §4 (query tiles outer, key/value tiles inner)
    as run by the CPU simulator of "FlashAttention and Triton" §19.12: per
    query tile keep a running max m (start -inf), a running denominator l
    (start 0) and an unnormalised accumulator acc (start 0); for each key tile
    form the local scores s, m_new = max(m, rowmax(s)), alpha = exp(m - m_new),
    p = exp(s - m_new), l = l * alpha + rowsum(p), acc = acc * alpha + p V_j,
    m = m_new; after the last key tile divide acc by l. Ragged last tiles are
    whatever remains (the pages' ceil(N / B)).
    Returns (O, LSE) with LSE = m + ln(l).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    n_q, n_k, d_v = Q.shape[0], K.shape[0], V.shape[1]
    O = np.zeros((n_q, d_v))
    LSE = np.zeros(n_q)
    for q0 in range(0, n_q, q_tile):
        q = Q[q0:q0 + q_tile]
        m = np.full(q.shape[0], -np.inf)
        l = np.zeros(q.shape[0])
        acc = np.zeros((q.shape[0], d_v))
        for k0 in range(0, n_k, k_tile):
            s = float(scale) * (q @ K[k0:k0 + k_tile].T)
            m_new = np.maximum(m, s.max(axis=1))
            alpha = np.exp(m - m_new)  # exp(-inf) = 0 on the first tile
            p = np.exp(s - m_new[:, None])
            l = l * alpha + p.sum(axis=1)
            acc = acc * alpha[:, None] + p @ V[k0:k0 + k_tile]
            m = m_new
        O[q0:q0 + q_tile] = acc / l[:, None]
        LSE[q0:q0 + q_tile] = m + np.log(l)
    return O, LSE


def online_softmax_stats(blocks):
    """Running (m, l) after each block of one score row.

    "Lesson 1" §3: m_new = max(m, m_tile);
    l_new = l * exp(m - m_new) + l_tile * exp(m_tile - m_new), where
    l_tile = sum(exp(block - m_tile)). Starts from m = -inf, l = 0.
    Returns a list of (m, l) pairs, one per block.
    """
    m, l = -np.inf, 0.0
    out = []
    for blk in blocks:
        blk = _f64(blk)
        m_tile = blk.max()
        l_tile = np.exp(blk - m_tile).sum()
        m_new = max(m, m_tile)
        l = l * np.exp(m - m_new) + l_tile * np.exp(m_tile - m_new)
        m = m_new
        out.append((float(m), float(l)))
    return out


def attention_fwd_batched(Q, K, V, scale: float, heads=None, causal: bool = False):
    """``attention_fwd`` applied to every (b, h) of [B, H, N, d] arrays.

    ``heads``: optional list of (b, h) pairs to compute; others stay NaN.
    Returns O [B, H, N, d_v] and LSE [B, H, N] (float64).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N = Q.shape[:3]
    O = np.full((B, H, N, V.shape[-1]), np.nan)
    LSE = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        O[b, h], LSE[b, h] = attention_fwd(Q[b, h], K[b, h], V[b, h], scale, causal)
    return O, LSE


def attention_bwd_batched(Q, K, V, dO, scale: float, heads=None, causal: bool = False):
    """``attention_bwd`` applied to every (b, h) of [B, H, N, d] arrays.

    ``heads``: optional list of (b, h) pairs to compute; others stay NaN.
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H = Q.shape[:2]
    dQ = np.full(Q.shape, np.nan)
    dK = np.full(K.shape, np.nan)
    dV = np.full(V.shape, np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        dQ[b, h], dK[b, h], dV[b, h] = attention_bwd(Q[b, h], K[b, h], V[b, h], dO[b, h], scale,
                                                     causal)
    return dQ, dK, dV


def merge_partials(O_parts, LSE_parts):
    """Merge attention results over disjoint key ranges: (O, LSE).

    Each part s covers some of the keys and gives its normalised output O_s
    [N_q, d_v] and log-sum-exp LSE_s = m_s + ln(l_s) [N_q]. The rule of
    "Lesson 1" §3 (m = max of the maxima, each l rescaled by exp(m_s - m)),
    with l_s exp(m_s - m) = exp(LSE_s - m):
      m = max_s LSE_s,  w_s = exp(LSE_s - m),  l = sum_s w_s,
      O = sum_s w_s O_s / l,  LSE = m + ln(l).
    """
    L = np.stack([_f64(x) for x in LSE_parts])          # [S, N_q]
    Os = np.stack([_f64(x) for x in O_parts])           # [S, N_q, d_v]
    m = L.max(axis=0)
    w = np.exp(L - m[None, :])
    l = w.sum(axis=0)
    O = (w[:, :, None] * Os).sum(axis=0) / l[:, None]
    return O, m + np.log(l)


def split_kv_attention_fwd(Q, K, V, scale: float, keys_per_split: int):
    """``attention_fwd`` over key ranges of ``keys_per_split`` keys, then ``merge_partials``.

    Ranges are [0, k), [k, 2k), ...; the last one holds what remains.
    """
    K, V = _f64(K), _f64(V)
    k = int(keys_per_split)
    parts = [attention_fwd(Q, K[s:s + k], V[s:s + k], scale) for s in range(0, K.shape[0], k)]
    return merge_partials([p[0] for p in parts], [p[1] for p in parts])


def varlen_attention_fwd(Q, K, V, cu_seqlens, scale: float, causal: bool = False):
    """Packed variable-length batch: Q, K, V [total, H, d]; sequence b is rows
    cu_seqlens[b]..cu_seqlens[b+1]-1. Returns O [total, H, d_v], LSE [H, total]."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    cu = [int(x) for x in cu_seqlens]
    total, H = Q.shape[:2]
    O = np.full((total, H, V.shape[-1]), np.nan)
    LSE = np.full((H, total), np.nan)
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        if e == s:
            continue
        for h in range(H):
            O[s:e, h], LSE[h, s:e] = attention_fwd(Q[s:e, h], K[s:e, h], V[s:e, h], scale, causal)
    return O, LSE


def varlen_attention_bwd(Q, K, V, dO, cu_seqlens, scale: float, causal: bool = False):
    """Backward of ``varlen_attention_fwd``: dQ, dK, dV [total, H, d]."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    cu = [int(x) for x in cu_seqlens]
    dQ, dK, dV = np.zeros(Q.shape), np.zeros(K.shape), np.zeros(V.shape)
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        if e == s:
            continue
        for h in range(Q.shape[1]):
            dQ[s:e, h], dK[s:e, h], dV[s:e, h] = attention_bwd(Q[s:e, h], K[s:e, h], V[s:e, h],
                                                              dO[s:e, h], scale, causal)
    return dQ, dK, dV
