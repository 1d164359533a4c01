"""Fused row softmax ("FlashAttention and Triton" §19.11) against the fp64 oracle.

Bar: fp32 max |gpu - ref| <= 2e-6 (outputs lie in [0, 1]); bf16 max |gpu - ref| /
max |ref| <= 1e-2 (one bf16 rounding of the output, 2^-9 relative)."""
import numpy as np
import pytest
import torch

import exact_attention_30_gb300 as fa
from oracle import row_softmax
from parity_utils import max_abs, rel_max, to64

pytestmark = pytest.mark.gpu


def _ref(x, scale):
    P, _, _ = row_softmax(scale * to64(x).reshape(-1, x.shape[-1]))
    return P.reshape(x.shape)


@pytest.mark.parametrize("cols", [1, 7, 31, 32, 100, 128, 129, 1000, 2048, 2049, 5000, 32768])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_shapes(cols, dtype):
    g = torch.Generator().manual_seed(cols)
    rows = 3 if cols > 4096 else 300
    x = (torch.randn(rows, cols, generator=g) * 3).to(dtype)
    y = fa.fa_softmax_rows(x.cuda(), scale=0.7)
    ref = _ref(x, 0.7)
    if dtype == torch.float32:
        assert max_abs(y, ref) <= 2e-6
    else:
        assert rel_max(y, ref) <= 1e-2
    assert np.abs(to64(y).sum(axis=-1) - 1).max() <= (1e-5 if dtype == torch.float32 else 2e-2)


def test_in_place_and_unaligned_rows():
    g = torch.Generator().manual_seed(3)
    base = torch.randn(1 + 37 * 250, generator=g).cuda()
    x = base[1:].view(37, 250)  # rows start 4 bytes off a 16-byte boundary
    ref = _ref(x.cpu(), 1.0)
    fa.fa_softmax_rows(x, out=x)
    torch.cuda.synchronize()
    assert max_abs(x, ref) <= 2e-6


def test_large_and_negative_scores_are_stable():
    x = torch.tensor([[1000.0, 999.0, -1000.0, 0.0], [-5e4, -5e4 + 1, -5e4 + 2, -5e4 + 3]]).cuda()
    y = fa.fa_softmax_rows(x)
    ref = _ref(x.cpu(), 1.0)
    assert torch.isfinite(y).all() and max_abs(y, ref) <= 2e-6


def test_many_rows_tail_block():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(1001, 64, generator=g).to(torch.bfloat16).cuda()  # rows not a multiple of 8
    assert rel_max(fa.fa_softmax_rows(x), _ref(x.cpu(), 1.0)) <= 1e-2
