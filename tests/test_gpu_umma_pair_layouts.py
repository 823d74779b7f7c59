"""The CTA-pair (cta_group::2, M = 256) tcgen05 layouts of the 128-row decode kernel,
checked on known matrices with a cluster of two CTAs.

Scores: each CTA holds 128 of the 256 A rows (keys) and 64 of the 128 B rows (query rows),
K-major with 128-byte swizzle; each CTA's tensor memory receives its 128 A rows x all 128
B rows. Values: MN-major A (each CTA two 64-column chunks of V, i.e. 128 of the 256 output
rows) and MN-major B (each CTA 64 of the 128 P columns). The third case is the scores
layout with every TMA load completing on the even CTA's barrier, as the decode kernel's
loads do. A failure here localises a 128-row decode mismatch to one of these steps.
"""
import ctypes
import os

import pytest
import torch

pytestmark = pytest.mark.gpu
LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "native", "libumma_pair_probe.so")


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(LIB):
        pytest.skip("probe not built")
    L = ctypes.CDLL(LIB)
    L.umma_pair_probe.restype = ctypes.c_int
    L.umma_pair_probe.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 5
    return L


def run(probe, mode, a, b):
    d = torch.full((256, 128), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert probe.umma_pair_probe(mode, a.data_ptr(), b.data_ptr(), d.data_ptr(), err.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return d


@pytest.mark.parametrize("mode", [0, 2])
def test_pair_scores_layout(probe, mode):
    g = torch.Generator().manual_seed(300 + mode)
    a = torch.randn(256, 64, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(128, 64, generator=g).to(torch.bfloat16).cuda()
    d = run(probe, mode, a, b)
    ref = a.double() @ b.double().T
    assert torch.allclose(d.double(), ref, atol=1e-3, rtol=1e-4), (d - ref).abs().max()


def test_pair_values_layout(probe):
    g = torch.Generator().manual_seed(310)
    v = torch.randn(64, 256, generator=g).to(torch.bfloat16).cuda()
    p = torch.rand(64, 128, generator=g).to(torch.bfloat16).cuda()
    d = run(probe, 1, v, p)
    ref = v.double().T @ p.double()
    assert torch.allclose(d.double(), ref, atol=1e-3, rtol=1e-4), (d - ref).abs().max()
