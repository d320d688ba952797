"""The tensor-core rate probe runs and measures plausible rates: kind::f16
(bf16) near the GB300's dense bf16 rate, and the block-scaled E2M1 x E4M3
kind at a multiple of it (the rate the MXFP4 expert GEMMs are judged by)."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_probe_rates_are_plausible():
    import quantile_balanced_routing_gb300 as Q
    bf16 = Q.mma_peak_tflops("bf16", runs=2, iters=4000)
    mx = Q.mma_peak_tflops("mxf8f6f4", runs=2, iters=4000)
    # 152 SMs x 8192 bf16 flop/clk at 0.8-2.1 GHz
    assert 900 < bf16 < 2700, bf16
    assert 1.5 * bf16 < mx < 4.5 * bf16, (bf16, mx)


def test_probe_rejects_bad_arguments():
    import ctypes
    import quantile_balanced_routing_gb300 as Q
    lib = Q.load_library()
    ms, fl = ctypes.c_float(), ctypes.c_double()
    assert lib.qbmoe_mma_probe(7, 10, ctypes.byref(ms), ctypes.byref(fl)) == Q.QBMOE_EINVAL
    assert lib.qbmoe_mma_probe(0, 0, ctypes.byref(ms), ctypes.byref(fl)) == Q.QBMOE_EINVAL
