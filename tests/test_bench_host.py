"""Host-side rules of bench.py, on the CPU: which bf16 peak a tensor-bound
kernel's roofline fraction is taken against, the DRAM-traffic record's guard
against a changed kernel source, and the forward-kernel label's routing rule."""
import os

import pytest

import bench

PEAKS = {"bf16_tflops": 1898.0, "bf16_tflops_sustained": 1718.7, "hbm_gbs": 6795.5}


def test_burst_peak_unless_long_and_power_capped():
    capped = {"reasons": ["sw_power_cap"]}
    assert bench.bf16_peak(PEAKS, "measured", None, 10.0)[0] == 1898.0
    assert bench.bf16_peak(PEAKS, "measured", {"reasons": []}, 10.0)[0] == 1898.0
    assert bench.bf16_peak(PEAKS, "measured", capped, 0.85)[0] == 1898.0  # a burst under the cap
    assert bench.bf16_peak(PEAKS, "measured", capped, bench.SUSTAINED_MIN_SECONDS)[0] == 1718.7
    label = bench.bf16_peak(PEAKS, "measured", capped, 0.85)[1]
    assert "burst" in label and "0.85" in label


def test_traffic_record_matches_the_current_backward_source():
    """The committed record carries the hash of the kernel source it was
    captured from; the bench reports its bytes only while they agree."""
    got = bench.read_traffic()
    assert got is not None, "profiles/bwd_main_traffic.txt is stale for attn_bwd_bf16.cu"
    assert 1e8 < got < 1e9


def test_traffic_record_is_dropped_for_another_source(tmp_path, monkeypatch):
    with open(bench.TRAFFIC_FILE) as f:
        text = f.read()
    bad = tmp_path / "traffic.txt"
    bad.write_text(text.replace("source_sha256 ", "source_sha256 0"))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(bad))
    assert bench.read_traffic() is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", os.path.join(str(tmp_path), "missing.txt"))
    assert bench.read_traffic() is None


@pytest.mark.parametrize("shape,name", [((4, 16, 1024, 64), "fwd_bf16_q4_kernel"),
                                        ((2, 16, 4096, 64), "fwd_bf16_q4_kernel"),
                                        ((1, 2, 20000, 64), "fwd_bf16_kernel<64>"),
                                        ((1, 4, 1024, 64), "fwd_bf16_kernel<64>"),
                                        ((2, 16, 4096, 128), "fwd_bf16_kernel<128>")])
def test_forward_kernel_label_follows_the_routing_rule(shape, name):
    assert bench.fwd_kernel_name(*shape, 152) == name
