"""Failure detection without a GPU fault: a bounded device-side wait that
nothing completes gives up after its limit, the host reads the timeout from
the status word (once: the read clears it), and the context stays usable --
a forward afterwards still matches the oracle."""
import time

import numpy as np
import pytest
import torch

from blackwell_nvfp4_quantize_gb300 import workloads as wl
from _gpu_common import run_and_check

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import blackwell_nvfp4_quantize_gb300 as fa

    assert fa.device_status() == fa.FP4ATTN_OK
    t0 = time.perf_counter()
    fa.debug_wait_timeout(20000)  # 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert dt >= 0.015, dt  # the wait really waited
    assert fa.device_status() == fa.FP4ATTN_ERR_TIMEOUT
    assert fa.device_status() == fa.FP4ATTN_OK  # cleared by the read
    w = wl.WORKLOADS[1]
    q, k, v = wl.make_inputs(w)
    run_and_check(q, k, v, w.softmax_scale, [(0, 0, 0, 64)], np.arange(256, dtype=np.int64),
                  "after a timed-out wait")


def test_wait_timeout_argument_checks():
    import blackwell_nvfp4_quantize_gb300 as fa

    with pytest.raises(fa.Fp4AttnError):
        fa.debug_wait_timeout(0)
    with pytest.raises(fa.Fp4AttnError):
        fa.debug_wait_timeout(2000001)
