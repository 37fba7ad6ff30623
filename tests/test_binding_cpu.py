"""The Python binding's argument checks (no GPU): every malformed call is rejected with
ValueError before any CUDA call or kernel launch, in particular the buffers whose size
the library would otherwise trust (a caller's host result buffers, the backward's LSE)."""

import pytest
import torch

import online_softmax_07_gb300 as osf
from online_softmax_07_gb300 import abi
from online_softmax_07_gb300.build import build_library


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_library()
    return abi.load()


def _qkv(B=1, H=2, N=64, d=64, dtype=torch.bfloat16):
    return tuple(torch.zeros(B, H, N, d, dtype=dtype) for _ in range(3))


def test_forward_rejects_mixed_devices():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="one device"):
        osf.attention_forward(q, k.to("meta"), v)


def test_forward_rejects_mixed_dtypes_and_shapes():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="bf16"):
        osf.attention_forward(q, k.half(), v)
    with pytest.raises(ValueError, match="one shape"):
        osf.attention_forward(q, k[:, :, :32], v)
    with pytest.raises(ValueError, match="splits"):
        osf.attention_forward(q, k, v, splits=0)


@pytest.mark.parametrize("out_shape, out_dtype", [
    ((1, 2, 63, 64), torch.bfloat16),   # one row short: the copy out would overrun it
    ((1, 2, 64, 64), torch.float16),    # wrong element type
    ((2, 64, 64), torch.bfloat16),      # same size, wrong shape
])
def test_forward_host_rejects_wrong_out(out_shape, out_dtype):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="out must be"):
        osf.attention_forward(q, k, v, out=torch.empty(out_shape, dtype=out_dtype))


def test_forward_host_rejects_wrong_lse_out():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="lse_out must be"):
        osf.attention_forward(q, k, v, lse_out=torch.empty(1, 2, 32))
    with pytest.raises(ValueError, match="lse_out must be"):
        osf.attention_forward(q, k, v, lse_out=torch.empty(1, 2, 64, dtype=torch.float64))
    strided = torch.empty(1, 2, 128)[:, :, ::2]
    with pytest.raises(ValueError, match="lse_out must be"):
        osf.attention_forward(q, k, v, lse_out=strided)


def test_backward_rejects_wrong_lse():
    q, k, v = _qkv()
    o, do = torch.zeros_like(q), torch.zeros_like(q)
    with pytest.raises(ValueError, match="lse must be"):
        osf.attention_backward(q, k, v, o, torch.zeros(1, 2, 32), do)
    with pytest.raises(ValueError, match="lse must be"):
        osf.attention_backward(q, k, v, o, torch.zeros(1, 2, 64, dtype=torch.bfloat16), do)


def test_backward_rejects_host_tensors_and_fp32():
    q, k, v = _qkv()
    o, do = torch.zeros_like(q), torch.zeros_like(q)
    with pytest.raises(ValueError, match="CUDA"):
        osf.attention_backward(q, k, v, o, torch.zeros(1, 2, 64), do)
    qf, kf, vf = _qkv(dtype=torch.float32)
    with pytest.raises(ValueError, match="bf16 or all fp16"):
        osf.attention_backward(qf, kf, vf, torch.zeros_like(qf), torch.zeros(1, 2, 64),
                               torch.zeros_like(qf))


def test_row_kernels_reject_bad_input():
    with pytest.raises(ValueError, match="fp32"):
        osf.row_state(torch.zeros(4, 8, dtype=torch.float64))
    with pytest.raises(ValueError, match="fp32"):
        osf.row_state(torch.zeros(4, 8, 2))
    with pytest.raises(ValueError, match="CUDA"):
        osf.softmax(torch.zeros(4, 8))
