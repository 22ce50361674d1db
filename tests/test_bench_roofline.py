"""bench.py's roofline accounting, on the host: the algorithmic bytes and FLOPs
of the scope table for the pages' benchmark shape, and which bound (HBM or the
dense FP4 tensor peak) a workload is reported against."""
import importlib.util
import os

import pytest

from nvfp4_token_routed_gb300 import workloads as W


@pytest.fixture(scope="module")
def bench():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_layer_bytes_of_the_default_workload(bench):
    # H7168 / I3072 / E384 top-6 SwiGLU at T=4096, every expert touched: 15.2 GB,
    # of which the weights (codes and E4M3 scales, 9/16 byte each) are 14.3 GB
    wl = W.PAGES_E384.with_T(4096)
    R, U = 4096 * 6, 384
    B = bench.algorithmic_bytes(wl, R, U)
    weights = 384 * (2 * 3072 * 7168 + 7168 * 3072) * 9 / 16
    assert weights == pytest.approx(14.27e9, rel=1e-3)
    assert B["layer"] == pytest.approx(15.209e9, rel=1e-3)
    assert B["fc1"] == pytest.approx(384 * 2 * 3072 * 7168 * 9 / 16 + 4096 * 7168 * 9 / 16
                                     + R * 3072 * 9 / 16)
    # workspace-only traffic is reported apart, never in the algorithmic bytes
    assert B["workspace"] > 0 and B["layer"] + B["workspace"] > B["layer"]


def test_flops_and_bound(bench):
    hbm = 6791.4e9
    tpeak = 1682.9e12 * bench.FP4_OVER_BF16
    for wl, R, U, tensor in [(W.PAGES_E384.with_T(4096), 4096 * 6, 384, False),
                             (W.COMPUTE_PROBE.with_T(65536), 65536 * 2, 8, True)]:
        F = bench.algorithmic_flops(wl, R)
        N1 = 2 * wl.I
        assert F["fc1"] == 2.0 * R * wl.H * N1 and F["fc2"] == 2.0 * R * wl.I * wl.H
        B = bench.algorithmic_bytes(wl, R, U)
        assert (F["fc1"] / tpeak > B["fc1"] / hbm) == tensor


def test_fp4_peak_is_six_times_the_sustained_bf16_rate(bench):
    peak, src = bench.fp4_peak()
    assert bench.FP4_OVER_BF16 == 6.0
    assert "x 6" in src and peak > 0
