"""The block-scaled tensor-rate loop that supplies the roofline denominator
(fp4attn_debug_mma_peak): it runs to completion, reports no timed-out wait,
and gives rates in the range a GB300 can reach (dense FP4 products at least
several PFLOP/s; the E4M3 product about half the E2M1 rate)."""
import pytest

pytestmark = pytest.mark.gpu


def test_mma_peak_rates():
    import blackwell_nvfp4_quantize_gb300 as fa

    r = {k: fa.debug_mma_peak(k, iters=1 << 16, launches=2) for k in ("nvf4", "mxf4", "mxf8")}
    assert fa.device_status() == fa.FP4ATTN_OK
    print("block-scaled MMA loop, TFLOP/s:", r)
    assert 3000.0 < r["nvf4"] < 20000.0
    assert 3000.0 < r["mxf4"] < 20000.0
    assert 0.35 < r["mxf8"] / r["mxf4"] < 0.65
