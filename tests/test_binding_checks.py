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
