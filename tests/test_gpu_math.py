"""The polynomial exp2 that the tensor-core softmax runs on the FMA pipe,
checked against CUDA's exp2f (torch.exp2 on the GPU) over the range the
kernels feed it."""
import ctypes

import pytest
import torch

from online_softmax_attention_gb300 import _abi

pytestmark = pytest.mark.gpu


def test_fma_exp2_matches_cuda_exp2():
    x = torch.cat([torch.linspace(-120.0, 10.0, 1_000_001, device="cuda"),
                   torch.tensor([0.0, -0.5, 0.5, -1.0, 1.0, -0.25, 7.999], device="cuda")])
    y = torch.empty_like(x)
    lib = _abi.load()
    rc = lib.attn_selftest_exp2(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.numel(),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _abi.ATTN_OK
    ref = torch.exp2(x.double())
    rel = ((y.double() - ref).abs() / ref).max().item()
    assert rel <= 3.5e-6, rel
    assert float(y[x.numel() - 7]) == 1.0  # 2^0 exactly


def test_fma_exp2_saturates_outside_its_range():
    """Arguments above 127 give a finite value near 2^127 (not a wrapped
    exponent), below -126 about 2^-126: a stale or mismatched lse in the
    backward then shows up as huge gradients, never as silent garbage."""
    x = torch.tensor([127.0, 128.0, 200.0, 1e6, -126.0, -127.0, -1e6], device="cuda")
    y = torch.empty_like(x)
    lib = _abi.load()
    rc = lib.attn_selftest_exp2(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.numel(),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _abi.ATTN_OK
    y = y.double().cpu()
    top = 2.0 ** 127
    for i in range(4):
        assert abs(y[i].item() / top - 1.0) <= 3.5e-6
    for i in range(4, 7):
        assert abs(y[i].item() / 2.0 ** -126 - 1.0) <= 3.5e-6
