"""Host-side checks of the Python binding: the C ABI takes plain pointers, so
the binding refuses operands and outputs whose shapes, byte counts, dtypes or
devices do not match before any call reaches a kernel.  CPU tensors stand in
for device buffers; every case must raise ValueError (no GPU is touched)."""
import pytest
import torch


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__

    __graft_entry__.build()
    import blackwell_nvfp4_quantize_gb300 as fa

    fa.lib()
    return fa


SHAPE = (1, 2, 200, 64)


def _nv(fa, shape=SHAPE, payload_n=None, sf_n=None):
    B, H, N, D = shape
    pb, sb = fa.nvfp4_bytes(B, H, N, D)
    return fa.NVFP4Tensor(torch.zeros(payload_n or pb, dtype=torch.uint8), torch.zeros(sf_n or sb, dtype=torch.uint8),
                          torch.zeros(1), tuple(shape))


def _mx(fa, shape=SHAPE, payload_n=None):
    B, H, N, D = shape
    pb, sb = fa.mxfp4_v_bytes(B, H, N, D)
    return fa.MXFP4Tensor(torch.zeros(payload_n or pb, dtype=torch.uint8), torch.zeros(sb, dtype=torch.uint8),
                          tuple(shape))


def test_well_formed_cpu_operands_stop_at_the_device_check(fa):
    with pytest.raises(ValueError, match="CUDA"):
        fa.fwd_directp(_nv(fa), _nv(fa), _mx(fa))


def test_mismatched_key_length(fa):
    k = _nv(fa, shape=(1, 2, 328, 64))
    with pytest.raises(ValueError, match="shape"):
        fa.fwd_directp(_nv(fa), k, _mx(fa))


def test_short_payload_and_scale_buffers(fa):
    with pytest.raises(ValueError, match="q.payload"):
        fa.fwd_directp(_nv(fa, payload_n=100), _nv(fa), _mx(fa))
    with pytest.raises(ValueError, match="k.sf"):
        fa.fwd_directp(_nv(fa), _nv(fa, sf_n=512), _mx(fa))
    with pytest.raises(ValueError, match="v.payload_t"):
        fa.fwd_directp(_nv(fa), _nv(fa), _mx(fa, payload_n=64))


def test_wrong_value_format(fa):
    B, H, N, D = SHAPE
    pb, sb = fa.mxfp8_v_bytes(B, H, N, D)
    v8 = fa.MXFP8Tensor(torch.zeros(pb, dtype=torch.uint8), torch.zeros(sb, dtype=torch.uint8), SHAPE)
    with pytest.raises(ValueError, match="MXFP4Tensor"):
        fa.fwd_directp(_nv(fa), _nv(fa), v8)
    with pytest.raises(ValueError, match="MXFP8Tensor"):
        fa.fwd_directp_fp8pv(_nv(fa), _nv(fa), _mx(fa))


def test_preallocated_outputs(fa):
    B, H, N, D = SHAPE
    q, k, v = _nv(fa), _nv(fa), _mx(fa)
    with pytest.raises(ValueError, match="o must be"):
        fa.fwd_directp(q, k, v, o=torch.zeros((B, H, N - 1, D), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="o must be"):
        fa.fwd_directp(q, k, v, o=torch.zeros((B, H, N, D), dtype=torch.float32))
    with pytest.raises(ValueError, match="lse must be"):
        fa.fwd_directp(q, k, v, o=torch.zeros((B, H, N, D), dtype=torch.bfloat16), lse=torch.zeros((B, H)))


def test_quantizer_inputs_and_outputs(fa):
    x = torch.zeros(SHAPE, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA bf16"):
        fa.quant_qk_nvfp4(x)
    with pytest.raises(ValueError, match="CUDA bf16"):
        fa.quant_v_mxfp4(x.float())


def test_noalloc_needs_caller_outputs(fa):
    B, H, N, D = SHAPE
    with pytest.raises(ValueError, match="caller-provided"):
        fa.fwd_directp_noalloc(_nv(fa), _nv(fa), _mx(fa), None, torch.zeros((B, H, N)))
    with pytest.raises(ValueError, match="caller-provided"):
        fa.fwd_directp_noalloc(_nv(fa), _nv(fa), _mx(fa), torch.zeros((B, H, N, D), dtype=torch.bfloat16), None)


def _fp8(fa, layout, fmt, shape=SHAPE, payload_n=None):
    B, H, N, D = shape
    pb, sb = (fa.mxfp8_rows_bytes if layout == "rows" else fa.mxfp8_v_bytes)(B, H, N, D)
    return fa.FP8Tensor(torch.zeros(payload_n or pb, dtype=torch.uint8), torch.zeros(sb, dtype=torch.uint8),
                        tuple(shape), layout, fmt)


def _bwd_args(fa, **over):
    B, H, N, D = SHAPE
    npad = (N + 127) // 128 * 128
    args = dict(q_saved=_nv(fa), k_saved=_nv(fa), v_rows=_fp8(fa, "rows", fa.FP8_E4M3),
                do_rows=_fp8(fa, "rows", fa.FP8_E5M2), do_t=_fp8(fa, "t", fa.FP8_E5M2),
                q_t=_fp8(fa, "t", fa.FP8_E4M3), k_t=_fp8(fa, "t", fa.FP8_E4M3),
                nl2=torch.zeros(B * H * npad), delta=torch.zeros(B * H * npad))
    args.update(over)
    return args


def test_backward_operands_checked(fa):
    # well-formed CPU operands stop at the device check
    with pytest.raises(ValueError, match="CUDA"):
        fa.bwd_directp_causal(**_bwd_args(fa))
    # a format or layout swapped, a short payload, a short workspace
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa, do_rows=_fp8(fa, "rows", fa.FP8_E4M3)))
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa, q_t=_fp8(fa, "rows", fa.FP8_E4M3)))
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa, k_t=_fp8(fa, "t", fa.FP8_E4M3, payload_n=10)))
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa, nl2=torch.zeros(5)))
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa, delta=torch.zeros(SHAPE[0] * SHAPE[1] * 256, dtype=torch.float64)))
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa, k_saved=_nv(fa, shape=(1, 2, 256, 64))))
    # preallocated gradients of the wrong size or dtype
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa), dq=torch.zeros(3))
    with pytest.raises(ValueError):
        fa.bwd_directp_causal(**_bwd_args(fa), dv=torch.zeros(SHAPE, dtype=torch.bfloat16))


def test_backward_quantizer_and_prep_inputs(fa):
    x = torch.zeros(SHAPE, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.quant_mxfp8_rows(x, fa.FP8_E5M2)  # CPU input
    with pytest.raises(ValueError):
        fa.quant_mxfp8_t(x.float(), fa.FP8_E4M3)  # not bf16
    with pytest.raises(ValueError):
        fa.empty_fp8(SHAPE, "cols", fa.FP8_E4M3, "cpu")
    with pytest.raises(ValueError):
        fa.bwd_prep(x, x, torch.zeros(SHAPE[:3]))  # CPU inputs


def test_host_batch_buffers_checked(fa):
    B, H, N, D = SHAPE
    x = [torch.zeros(SHAPE, dtype=torch.bfloat16)]
    o = [torch.zeros(SHAPE, dtype=torch.bfloat16)]
    lse = [torch.zeros((B, H, N), dtype=torch.float32)]
    ws = torch.zeros((fa.host_batch_workspace_bytes(B, H, N, D),), dtype=torch.uint8)
    with pytest.raises(ValueError):
        fa.fwd_host_batch(x, x, x, o, lse, workspace=ws)  # workspace not on a GPU
    with pytest.raises(ValueError):
        fa.fwd_host_batch(x, x, x, o, lse)  # no workspace
    with pytest.raises(ValueError):
        fa.fwd_host_batch(x, x, x + x, o, lse, workspace=ws)  # step counts differ
    with pytest.raises(ValueError):
        fa.fwd_host_batch([], [], [], [], [], workspace=ws)
    with pytest.raises(ValueError):
        fa.fwd_host_batch(x, x, [x[0].float()], o, lse, workspace=ws)  # not bf16
    with pytest.raises(ValueError):
        fa.fwd_host_batch(x, x, x, [o[0][:, :, :100]], lse, workspace=ws)  # short O
    with pytest.raises(ValueError):
        fa.fwd_host_batch(x, x, x, o, [lse[0].double()], workspace=ws)  # LSE not fp32
    with pytest.raises(ValueError):
        fa.fwd_host_batch(x, x, x, o, lse, workspace=ws[:-1])  # workspace too small (checked first as CPU)
