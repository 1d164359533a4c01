"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws random numbers,
rounds them to the storage dtype and lays them out as contiguous [B, H, N, d]
CPU tensors. Both the CUDA path and the fp64 oracle consume exactly these bits.

Workloads (every one non-causal, Q/K/V/dO i.i.d. N(0, 1)):

* ``minilab_f32_1x1x16x8`` -- the CPU mini-lab of "FlashAttention and Triton"
  §19.12: numpy ``default_rng(0)``, Q, K, V drawn in that order, each
  ``normal(size=(16, 8))``, stored as float32; scale 1/sqrt(8); forward only.
* ``fwd_bf16_4x16x1024x64`` -- forward, bf16, B=4 H=16 N=1024 d=64.
* ``fwd_bf16_2x16x4096x128`` -- forward, bf16, B=2 H=16 N=4096 d=128.
* ``bwd_bf16_2x16x4096x128`` -- backward, bf16, same shape; O and LSE come
  from the forward pass.
* ``fwdbwd_bf16_1x32x16384x128`` -- forward + backward, bf16, B=1 H=32
  N=16384 d=128, every key row with n % 64 == 0 multiplied by 4 after the
  bf16 cast (exact: a power of two) so that the running max keeps moving.

KV-cache decode workloads (``DECODE_WORKLOADS``; the pages describe decoding
with a KV cache but print no decode configuration, so these stand in for a
serving step: one new query per sequence, or a group of queries that share a
K/V head):

* ``decode_bf16_8x32x1x32768x128`` -- B=8, H=32, Nq=1, Nk=32768, d=128.
* ``decode_bf16_8x8x8x32768x128`` -- B=8, H=8 K/V heads, Nq=8 queries per
  K/V head, Nk=32768, d=128.

Decode inputs are drawn like the others (Q [B,H,Nq,d], then K and V
[B,H,Nk,d], every 64th key row times 4).

bf16 workloads: ``torch.Generator().manual_seed(seed)``, ``torch.randn`` in
float32 of shape [B, H, N, d] in the order Q, K, V, dO, then round-to-nearest
to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "f32" or "bf16"
    fwd: bool
    bwd: bool
    big_key_every: int = 0  # scale key rows n % big_key_every == 0 by 4

    @property
    def scale(self) -> float:
        # the pages' 1/sqrt(d), rounded to float32 (the value both sides see)
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def fwd_flops(self) -> float:
        """4 * B * H * N^2 * d (two N x N x d contractions per head)."""
        return 4.0 * self.B * self.H * self.N * self.N * self.d

    def bwd_flops(self) -> float:
        """2.5x the forward count (five N x N x d contractions per head)."""
        return 2.5 * self.fwd_flops()


WORKLOADS = {
    w.name: w
    for w in [
        Workload("minilab_f32_1x1x16x8", 1, 1, 16, 8, "f32", True, False),
        Workload("fwd_bf16_4x16x1024x64", 4, 16, 1024, 64, "bf16", True, False),
        Workload("fwd_bf16_2x16x4096x128", 2, 16, 4096, 128, "bf16", True, False),
        Workload("bwd_bf16_2x16x4096x128", 2, 16, 4096, 128, "bf16", False, True),
        Workload("fwdbwd_bf16_1x32x16384x128", 1, 32, 16384, 128, "bf16", True, True, 64),
    ]
}


def minilab_inputs():
    """Q, K, V of the mini-lab: default_rng(0), three normal((16, 8)) draws."""
    rng = np.random.default_rng(0)
    Q = rng.normal(size=(16, 8))
    K = rng.normal(size=(16, 8))
    V = rng.normal(size=(16, 8))
    return Q, K, V


def random_qkv(B, H, N, d, dtype=torch.bfloat16, seed=0, with_do=True, big_key_every=0,
               n_k=None):
    """Seeded i.i.d. N(0,1) tensors [B,H,N,d] (K/V may have n_k rows), rounded to ``dtype``.

    Drawn in float32 in the order Q, K, V, dO from one CPU generator.
    """
    g = torch.Generator().manual_seed(seed)
    n_k = N if n_k is None else n_k
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(dtype)
    k = torch.randn((B, H, n_k, d), generator=g, dtype=torch.float32).to(dtype)
    v = torch.randn((B, H, n_k, d), generator=g, dtype=torch.float32).to(dtype)
    do = torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(dtype) if with_do else None
    if big_key_every:
        k[:, :, ::big_key_every, :] *= 4
    return q, k, v, do


def workload_inputs(w: Workload, seed: int = 0):
    """(q, k, v, do) CPU tensors for a named workload; do is None if forward only."""
    if w.name.startswith("minilab"):
        Q, K, V = minilab_inputs()
        t = lambda a: torch.from_numpy(a.astype(np.float32)).reshape(1, 1, 16, 8).contiguous()
        return t(Q), t(K), t(V), None
    return random_qkv(w.B, w.H, w.N, w.d, w.torch_dtype, seed=seed, with_do=w.bwd,
                      big_key_every=w.big_key_every)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d)))

    def flops(self) -> float:
        """4 * B * H * Nq * Nk * d (scores and P V)."""
        return 4.0 * self.B * self.H * self.Nq * self.Nk * self.d

    def hbm_bytes(self) -> float:
        """Bytes a decode call must move: K and V once, Q and O once (bf16), LSE (fp32)."""
        kv = 2 * self.B * self.H * self.Nk * self.d * 2
        qo = 2 * self.B * self.H * self.Nq * self.d * 2
        return float(kv + qo + self.B * self.H * self.Nq * 4)


DECODE_WORKLOADS = {
    w.name: w
    for w in [
        DecodeWorkload("decode_bf16_8x32x1x32768x128", 8, 32, 1, 32768, 128),
        DecodeWorkload("decode_bf16_8x8x8x32768x128", 8, 8, 8, 32768, 128),
    ]
}


def decode_inputs(w: DecodeWorkload, seed: int = 0):
    """(q, k, v) CPU bf16 tensors of a decode workload."""
    q, k, v, _ = random_qkv(w.B, w.H, w.Nq, w.d, torch.bfloat16, seed=seed, with_do=False,
                            big_key_every=64, n_k=w.Nk)
    return q, k, v


def random_varlen(lens, H, d, dtype=torch.bfloat16, seed=0, with_do=True):
    """Packed variable-length batch: (q, k, v, do, cu_seqlens) with tensors
    [total, H, d] drawn like ``random_qkv`` (order Q, K, V, dO) and
    cu_seqlens int32 [len(lens) + 1] (prefix sums of ``lens``), all on the CPU."""
    g = torch.Generator().manual_seed(seed)
    total = int(sum(lens))
    draw = lambda: torch.randn((total, H, d), generator=g, dtype=torch.float32).to(dtype)
    q, k, v = draw(), draw(), draw()
    do = draw() if with_do else None
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return q, k, v, do, cu
