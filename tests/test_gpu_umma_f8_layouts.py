"""The two 8-bit tcgen05 operand layouts (kind::f8f6f4, E4M3 x E4M3) of the FP8-cache
decode, checked on known matrices.

Scores: K-major A (TMA, 64-byte swizzle, the cache's key boxes) and K-major B written by
threads in the same layout; K advanced 32 bytes inside the swizzle atom.
Values: MN-major A straight from the cache's row layout (64-byte swizzle, two 64-column
chunks) and MN-major B (one 64-byte swizzled key row per thread), or MN-major B without
swizzle (each key row's N bytes as N / 16 core matrices of 16 bytes, for 16 to 64 query
rows).
The products of two E4M3 values are exact in float32, so on integer-valued operands the
sums are exact too and the comparison is strict; random codes use a relative bound.
"""
import ctypes
import os

import pytest
import torch

pytestmark = pytest.mark.gpu
LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "native", "libumma_f8_probe.so")


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(LIB):
        pytest.skip("probe not built")
    L = ctypes.CDLL(LIB)
    L.umma_f8_probe.restype = ctypes.c_int
    L.umma_f8_probe.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
    return L


def e4m3_codes(shape, gen, small_ints=False):
    """Random E4M3 bytes (no NaN codes). small_ints: values in {-8..8}, so that sums of
    products are small integers, exact in float32."""
    if small_ints:
        vals = torch.randint(-8, 9, shape, generator=gen).to(torch.float32)
        return vals.to(torch.float8_e4m3fn).view(torch.uint8)
    codes = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32)
    codes = torch.where((codes & 0x7F) == 0x7F, codes - 1, codes)
    return codes.to(torch.uint8)


def as_f64(codes):
    return codes.view(torch.float8_e4m3fn).to(torch.float64)


def run(probe, mode, n, a, b):
    d = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert probe.umma_f8_probe(mode, n, a.data_ptr(), b.data_ptr(), d.data_ptr(), err.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return d.double().cpu()


@pytest.mark.parametrize("n", [16, 32, 64])
@pytest.mark.parametrize("small_ints", [True, False])
def test_scores_layout_e4m3(probe, n, small_ints):
    g = torch.Generator().manual_seed(300 + n + 7 * small_ints)
    a = e4m3_codes((128, 128), g, small_ints)
    b = e4m3_codes((n, 128), g, small_ints)
    d = run(probe, 0, n, a.cuda(), b.cuda())
    ref = as_f64(a) @ as_f64(b).T
    if small_ints:
        assert torch.equal(d, ref), (d - ref).abs().max()
    else:
        bound = (as_f64(a).abs() @ as_f64(b).abs().T) * 2.0 ** -20
        assert ((d - ref).abs() <= bound).all(), ((d - ref).abs() / bound.clamp_min(1e-30)).max()


@pytest.mark.parametrize("small_ints", [True, False])
def test_values_layout_e4m3(probe, small_ints):
    g = torch.Generator().manual_seed(400 + small_ints)
    v = e4m3_codes((64, 128), g, small_ints)
    p = e4m3_codes((64, 64), g, small_ints)
    d = run(probe, 1, 64, v.cuda(), p.cuda())
    ref = as_f64(v).T @ as_f64(p)
    if small_ints:
        assert torch.equal(d, ref), (d - ref).abs().max()
    else:
        bound = (as_f64(v).abs().T @ as_f64(p).abs()) * 2.0 ** -20
        assert ((d - ref).abs() <= bound).all(), ((d - ref).abs() / bound.clamp_min(1e-30)).max()


@pytest.mark.parametrize("n", [16, 32, 64])
@pytest.mark.parametrize("small_ints", [True, False])
def test_values_layout_e4m3_unswizzled_p(probe, n, small_ints):
    g = torch.Generator().manual_seed(500 + n + small_ints)
    v = e4m3_codes((64, 128), g, small_ints)
    p = e4m3_codes((64, n), g, small_ints)
    d = run(probe, 2, n, v.cuda(), p.cuda())
    ref = as_f64(v).T @ as_f64(p)
    if small_ints:
        assert torch.equal(d, ref), (d - ref).abs().max()
    else:
        bound = (as_f64(v).abs().T @ as_f64(p).abs()) * 2.0 ** -20
        assert ((d - ref).abs() <= bound).all(), ((d - ref).abs() / bound.clamp_min(1e-30)).max()
