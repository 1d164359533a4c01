"""The bounded-wait machinery on the GPU: a kernel that waits on a barrier
nothing arrives at gives up after its limit, records FA_ERR_TIMEOUT in the
status word, and leaves the context usable. No fault, trap or hang."""
import pytest
import torch

import exact_attention_30_gb300 as fa

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_cleared():
    assert fa.fa_check_device_status() == fa.FA_OK
    assert fa.fa_debug_timeout_probe(2_000_000) == fa.FA_OK  # 2 ms limit
    assert fa.fa_check_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK  # cleared by the read
    # the context still works
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0
