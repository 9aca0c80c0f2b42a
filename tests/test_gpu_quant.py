"""Bit-exact parity of the CUDA quantizers with the oracle: NVFP4 payloads,
E4M3 scale atoms and the fp32 tensor scale for Q and K; MXFP4 V^T payloads and
E8M0 scale atoms -- on full tensors of all five workloads and on edge cases."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl
from _gpu_common import mx_to_np, nv_to_np

pytestmark = pytest.mark.gpu


def _check_nvfp4(x):
    import blackwell_nvfp4_quantize_gb300 as fa

    t = fa.quant_qk_nvfp4(x.cuda())
    p, sf, g = nv_to_np(t)
    rp, rsf, rg = oracle.quant_nvfp4(wl.bf16_bits(x))
    assert g == rg, (g, rg)
    assert np.array_equal(sf, rsf), "scale atoms differ at %s" % np.argwhere(sf != rsf)[:5].tolist()
    assert np.array_equal(p, rp), "payload differs at %s" % np.argwhere(p != rp)[:5].tolist()


def _check_mxfp4(v):
    import blackwell_nvfp4_quantize_gb300 as fa

    t = fa.quant_v_mxfp4(v.cuda())
    p, sf = mx_to_np(t)
    rp, rsf = oracle.quant_mxfp4_v(wl.bf16_bits(v))
    assert np.array_equal(sf, rsf), "scale atoms differ at %s" % np.argwhere(sf != rsf)[:5].tolist()
    assert np.array_equal(p, rp), "payload differs at %s" % np.argwhere(p != rp)[:5].tolist()


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_quantizers_bit_exact_on_workloads(idx):
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    _check_nvfp4(q)
    _check_nvfp4(k)
    _check_mxfp4(v)
    del q, k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N", [1, 31, 77, 128, 129, 300])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", ["normal", "wide", "zeros"])
def test_quantizers_bit_exact_edge_cases(N, D, kind):
    q, k, v = wl.make_custom(2, 3, N, D, seed=100 + N + D, kind=kind, scale=3.0)
    _check_nvfp4(q)
    _check_nvfp4(k)
    _check_mxfp4(v)


def test_quantizer_hand_worked_block(golden_dir):
    import json
    import os

    import blackwell_nvfp4_quantize_gb300 as fa

    gold = json.load(open(os.path.join(golden_dir, "nvfp4_block.json")))
    x = torch.tensor(gold["values"], dtype=torch.float32).reshape(1, 1, 1, 128).to(torch.bfloat16)
    t = fa.quant_qk_nvfp4(x.cuda())
    p = t.payload.cpu().numpy().reshape(-1)
    codes = [(p[i // 2] >> (4 * (i % 2))) & 0xF for i in range(128)]
    assert codes == gold["codes"]
    sf = t.sf.cpu().numpy()
    assert [int(sf[kb % 4 + 512 * (kb // 4)]) for kb in range(8)] == gold["sf_by_block"]
    assert t.g.item() == gold["g"]


def test_quantizers_bit_exact_wrapping_grid_with_partial_chunk():
    # 7 heads of 100003 rows at D = 64: the amax pass has more 8 KB warp
    # chunks than warps (they wrap round the grid) and a partial last chunk
    # (424 vectors); the NVFP4 pass wraps its 128-block warp groups and ends
    # in a partial one (84 blocks); the V pass ends in a partial key tile
    q, k, v = wl.make_custom(1, 7, 100003, 64, seed=313, kind="normal", scale=2.0)
    import blackwell_nvfp4_quantize_gb300 as fa

    _check_nvfp4(q)
    _check_mxfp4(v)
    x = torch.zeros((1, 7, 100003, 64), dtype=torch.bfloat16)
    x.view(-1)[-1] = 1000.0  # the tensor maximum sits in the amax pass's last partial chunk
    t = fa.quant_qk_nvfp4(x.cuda())
    assert np.float32(t.g.item()) == np.float32(1000.0) / np.float32(2688.0)
    del q, k, v, x
    torch.cuda.empty_cache()
