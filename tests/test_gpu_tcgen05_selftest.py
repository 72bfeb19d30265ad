"""GPU check of the tcgen05 (5th-generation tensor core) building blocks through the C ABI
self-test: a 128 x N x 64 bf16 GEMM with K-major and MN-major B and A read from shared or
tensor memory, accumulated in tensor memory, against a float64 product of the same bf16
inputs."""

import ctypes

import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv

pytestmark = pytest.mark.gpu


def _gemm(A, B, N, b_mn_major, a_tmem=False):
    lib = skv.load_library()
    f = lib.splitkv_selftest_umma_gemm
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
    f.restype = ctypes.c_int32
    C = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    st = f(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()), ctypes.c_void_p(C.data_ptr()), N,
           (1 if b_mn_major else 0) | (2 if a_tmem else 0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == skv.SKV_OK, skv.last_error()
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    return C


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("b_mn_major", [False, True])
@pytest.mark.parametrize("a_tmem", [False, True])
def test_umma_gemm(N, b_mn_major, a_tmem):
    g = torch.Generator(device="cuda").manual_seed(11 + N + int(b_mn_major))
    A = torch.randn((128, 64), generator=g, device="cuda").to(torch.bfloat16)
    if b_mn_major:
        B = torch.randn((64, N), generator=g, device="cuda").to(torch.bfloat16)
        ref = A.double() @ B.double()
    else:
        B = torch.randn((N, 64), generator=g, device="cuda").to(torch.bfloat16)
        ref = A.double() @ B.double().T
    C = _gemm(A, B, N, b_mn_major, a_tmem)
    err = (C.double() - ref).abs().max().item()
    assert err < 1e-3, err
