"""The benchmark's accounting of the method's own work (CPU only): per token at
the headline shape (b4 L8192 H64 P64 N128 G1 Q256, bf16) the forward+backward
reads and writes about 43 KB and does about 10.6 MFLOP counting the causal half
of the chunk products; the tensor-core kernels' shares add up to that."""
from __future__ import annotations

import pytest

import bench
from mamba2_ssd_selective_gb300.inputs import WORKLOADS


def test_method_work_at_the_headline_shape():
    shape, dtype, _ = WORKLOADS["mamba2-1b-fwdbwd"]
    m = bench.method_work(shape, dtype)
    assert m["fwd_bytes"] + m["bwd_bytes"] == pytest.approx(43e3, rel=0.01)
    assert m["fwd_flop"] == pytest.approx(3.18e6, rel=0.01)
    assert m["bwd_flop"] == pytest.approx(7.44e6, rel=0.01)
    k = m["per_kernel_flop_per_token"]
    # the chunk-state kernel runs in the forward and again in the backward's recompute
    fwd = k["tc_chunk_out"] + k["tc_chunk_state"]
    bwd = k["tc_chunk_state"] + k["tc_chunk_z"] + k["tc_bwd_row"] + k["tc_bwd_col"]
    assert fwd == m["fwd_flop"] and bwd == m["bwd_flop"]


def test_method_roofline_floor():
    shape, dtype, _ = WORKLOADS["mamba2-1b-fwdbwd"]
    peaks = {"hbm_gbs": 6686.8, "bf16_tflops": 1953.3, "bf16_tflops_sustained": 1742.8}
    kt = [("tc_bwd_col", 2, 1.4), ("conv_fwd", 4, 0.4)]
    r = bench.method_roofline(kt, shape, dtype, 2.919, peaks, backward=True)
    assert r["bytes_per_step"] == pytest.approx(1.41e9, rel=0.01)
    assert r["floor_ms"] == pytest.approx(0.21, rel=0.03)
    assert r["frac"] == pytest.approx(0.21 / 2.919, rel=0.03)
    d = r["dominant_contraction"]
    assert d["kernel"] == "tc_bwd_col" and d["method_flop_per_launch"] == pytest.approx(1.04e11, rel=0.01)
    assert d["frac_compute"] == pytest.approx(1.04e11 / 0.7e-3 / 1742.8e12, rel=0.01)
