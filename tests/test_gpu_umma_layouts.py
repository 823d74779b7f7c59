"""The two tcgen05 operand layouts of the decode kernel, checked on known matrices.

Scores: K-major A and B with 128-byte swizzle, K advanced inside the swizzle atom.
Values: MN-major A (two 64-column chunks) and MN-major B written with the P^T row swizzle.
Scores with A in tensor memory: the rows written by the threads into TMEM lanes, two
16-bit values per 32-bit column (the FP8 path's dequantised keys).
A failure here localises a decode mismatch to one operand layout.
"""
import ctypes
import os

import pytest
import torch

pytestmark = pytest.mark.gpu
LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "native", "libumma_probe.so")


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(LIB):
        pytest.skip("probe not built")
    L = ctypes.CDLL(LIB)
    L.umma_probe.restype = ctypes.c_int
    L.umma_probe.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
    return L


def run(probe, mode, n, a, b):
    d = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert probe.umma_probe(mode, n, a.data_ptr(), b.data_ptr(), d.data_ptr(), err.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return d


@pytest.mark.parametrize("n", [16, 32, 64])
def test_scores_layout(probe, n):
    g = torch.Generator().manual_seed(n)
    a = torch.randn(128, 64, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(n, 64, generator=g).to(torch.bfloat16).cuda()
    d = run(probe, 0, n, a, b)
    ref = a.double() @ b.double().T
    assert torch.allclose(d.double(), ref, atol=1e-3, rtol=1e-4), (d - ref).abs().max()


@pytest.mark.parametrize("n", [16, 32, 64])
def test_values_layout(probe, n):
    g = torch.Generator().manual_seed(100 + n)
    v = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    p = torch.rand(128, n, generator=g).to(torch.bfloat16).cuda()
    d = run(probe, 1, n, v, p)
    ref = v.double().T @ p.double()
    assert torch.allclose(d.double(), ref, atol=1e-3, rtol=1e-4), (d - ref).abs().max()


@pytest.mark.parametrize("n", [16, 32, 64])
def test_scores_layout_a_in_tensor_memory(probe, n):
    g = torch.Generator().manual_seed(200 + n)
    a = torch.randn(128, 64, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(n, 64, generator=g).to(torch.bfloat16).cuda()
    d = run(probe, 2, n, a, b)
    ref = a.double() @ b.double().T
    assert torch.allclose(d.double(), ref, atol=1e-3, rtol=1e-4), (d - ref).abs().max()
