"""convrot_measure_engine_peak: the throughput ceilings of the engines that
compute the exact int8 product (tcgen05 kind::f16, mma.sync f16, dp4a,
mma.sync s8), which the benchmark reports next to its kernels' rates."""
import pytest

import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu

pytestmark = pytest.mark.gpu

ENGINES = {
    "tcgen05_f16": cr.CONVROT_PEAK_TCGEN05_F16,
    "mma_f16": cr.CONVROT_PEAK_MMA_F16,
    "dp4a": cr.CONVROT_PEAK_DP4A,
    "mma_s8": cr.CONVROT_PEAK_MMA_S8,
}


def _rate(engine, reps=2000):
    best = 0.0
    for _ in range(2):
        ops, ms = cr.convrot_measure_engine_peak(engine, reps)
        assert ops > 0 and ms > 0
        best = max(best, ops / (ms * 1e-3) / 1e12)
    return best


def test_engine_ceilings_order():
    # Plausible on any sm_103 part: the tensor-memory MMA is the fastest, the
    # fp16 warp MMA outruns the int8 warp MMA and dp4a; every rate is far
    # below the tcgen05 one and above zero.
    gu.require_gpu()
    r = {k: _rate(v) for k, v in ENGINES.items()}
    gu.check_no_device_error()
    print("engine ceilings (TOPS / TFLOP/s):", {k: round(v, 1) for k, v in r.items()})
    assert r["tcgen05_f16"] > r["mma_f16"] > r["mma_s8"] > 0
    assert r["mma_f16"] > r["dp4a"] > 0


def test_unknown_engine_rejected():
    gu.require_gpu()
    with pytest.raises(cr.ConvRotError):
        cr.convrot_measure_engine_peak(4, 10)
