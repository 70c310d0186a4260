"""Host-side rules of bench.py: when the captured DRAM-traffic ratio of a
kernel may be reported, and that each stored ratio is keyed to the kernel
source hash its committed Nsight Compute summary names."""
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILE = {"gdpa_fwd": "tc_fwd_kernel_training_256seq.md",
           "gdpa_bwd": "tc_bwd_kernel_training_256seq.md"}


@pytest.fixture
def same_sources(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: bench.TRAFFIC_RATIO[k][0])


@pytest.mark.parametrize("kernel", ["gdpa_fwd", "gdpa_bwd"])
def test_traffic_scales_the_algorithmic_bytes(same_sources, kernel):
    ratio = bench.TRAFFIC_RATIO[kernel][1]
    got = bench.dram_traffic(kernel, 1.0e9, bench.TRAFFIC_WORKLOAD, False, False, False)
    assert got == pytest.approx(ratio * 1.0e9)
    assert 0.9 < ratio < 1.2   # a ratio far from 1 would mean re-reads or a wrong capture


@pytest.mark.parametrize("kernel", ["gdpa_fwd", "gdpa_bwd"])
@pytest.mark.parametrize("case", ["workload", "key_split", "softmax", "qk_norm"])
def test_traffic_only_where_the_capture_applies(same_sources, kernel, case):
    kw = dict(workload=bench.TRAFFIC_WORKLOAD, key_split=False, softmax=False, qk_norm=False)
    kw[case] = "pma_pooling" if case == "workload" else True
    assert bench.dram_traffic(kernel, 1.0e9, **kw) is None


@pytest.mark.parametrize("kernel", ["gdpa_fwd", "gdpa_bwd"])
def test_traffic_null_for_changed_sources(monkeypatch, kernel):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
    assert bench.dram_traffic(kernel, 1.0e9, bench.TRAFFIC_WORKLOAD, False, False, False) is None


@pytest.mark.parametrize("kernel", ["gdpa_fwd", "gdpa_bwd"])
def test_stored_ratio_names_the_profiled_source(kernel):
    with open(os.path.join(ROOT, "profiles", PROFILE[kernel])) as fh:
        text = fh.read()
    assert "Kernel source hash %s" % bench.TRAFFIC_RATIO[kernel][0] in text.replace("\n", " ")
