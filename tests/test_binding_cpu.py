"""The Python binding's own argument checks, which run before any CUDA call
and so need no GPU: device-tensor entry points refuse host tensors, the
host-tensor entry point refuses malformed inputs and result buffers, and
unsupported dtypes are refused by name."""

import pytest

torch = pytest.importorskip("torch")

from exact_attention_16_gb300 import api  # noqa: E402


def _qkv(B=1, Sq=8, Sk=16, Hq=4, Hkv=2, D=64, dtype=torch.bfloat16):
    return (torch.zeros(B, Sq, Hq, D, dtype=dtype), torch.zeros(B, Sk, Hkv, D, dtype=dtype),
            torch.zeros(B, Sk, Hkv, D, dtype=dtype))


def test_device_entry_points_refuse_host_tensors():
    q, k, v = _qkv()
    with pytest.raises(TypeError, match="CUDA"):
        api.fa_fwd(q, k, v)
    with pytest.raises(ValueError, match="CUDA"):
        api.fa_fwd_decode(q, k, v)
    with pytest.raises(ValueError, match="CUDA"):
        api.fa_fwd_decode_noalloc(q, k, v)
    with pytest.raises(ValueError, match="CUDA"):
        api.fa_merge(torch.zeros(2, 1, 8, 4, 64, dtype=torch.bfloat16), torch.zeros(2, 1, 4, 8))


def test_merge_refuses_wrong_ranks_and_shapes():
    with pytest.raises(ValueError, match="o_parts"):
        api.fa_merge(torch.zeros(1, 8, 4, 64, dtype=torch.bfloat16), torch.zeros(2, 1, 4, 8))
    with pytest.raises(ValueError, match="lse_parts"):
        api.fa_merge(torch.zeros(2, 1, 8, 4, 64, dtype=torch.bfloat16), torch.zeros(2, 1, 8, 4))
    with pytest.raises(ValueError, match="lse_parts"):
        api.fa_merge(torch.zeros(2, 1, 8, 4, 64, dtype=torch.bfloat16),
                     torch.zeros(2, 1, 4, 8, dtype=torch.float64))


def test_host_entry_refuses_malformed_inputs():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="contiguous"):
        api.fa_fwd_host(q.transpose(1, 2), k, v)
    with pytest.raises(ValueError, match="4-D"):
        api.fa_fwd_host(q[0], k, v)
    with pytest.raises(TypeError, match="one dtype"):
        api.fa_fwd_host(q, k.to(torch.float16), v)
    with pytest.raises(ValueError, match="matching q"):
        api.fa_fwd_host(q, k, v[:, :15].contiguous())
    with pytest.raises(ValueError, match="matching q"):
        api.fa_fwd_host(q, k[..., :32].contiguous(), v[..., :32].contiguous())
    with pytest.raises(TypeError, match="unsupported dtype"):
        api.fa_fwd_host(*_qkv(dtype=torch.float32))


def test_host_entry_refuses_result_buffers_that_do_not_fit():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="out"):
        api.fa_fwd_host(q, k, v, out=torch.empty(1, 8, 2, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out"):
        api.fa_fwd_host(q, k, v, out=torch.empty(1, 8, 4, 64, dtype=torch.float16))
    with pytest.raises(ValueError, match="lse"):
        api.fa_fwd_host(q, k, v, out=torch.empty_like(q), lse=torch.empty(1, 8, 4))
    with pytest.raises(ValueError, match="lse"):
        api.fa_fwd_host(q, k, v, out=torch.empty_like(q), lse=torch.empty(1, 4, 8, dtype=torch.float64))


def test_strided_entry_is_the_same_call():
    # fa_fwd passes every tensor's strides, so it serves fa_fwd_strided too
    assert api.fa_fwd_strided is api.fa_fwd
