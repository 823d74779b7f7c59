"""Pins for the oracle's E4M3 codec (oracle/fp8_e4m3.py) against torch and brute force."""
import math
import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np
import pytest
import torch

from conftest import ROOT, read_golden
from oracle import fp8_e4m3


def test_decode_matches_torch_for_all_256_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8_e4m3.decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    # the sign of zero survives decoding
    assert math.copysign(1.0, got[0x80]) == -1.0


def test_decode_anchor_values_from_the_ocp_table():
    for code_s, val_s in read_golden("e4m3_anchor_values.txt"):
        code = int(code_s, 16)
        v = fp8_e4m3.decode(np.array([code], dtype=np.uint8))[0]
        if val_s == "nan":
            assert math.isnan(v), code_s
        else:
            assert v == float(val_s) and math.copysign(1, v) == math.copysign(1, float(val_s)), code_s


def test_encode_special_values():
    x = np.array([0.0, -0.0, 448.0, 449.0, 464.0, 1e30, np.inf, -np.inf, np.nan,
                  2.0 ** -9, 2.0 ** -10, 2.0 ** -10 * 1.0001, 1.5 * 2.0 ** -9, 1.0625, 1.1875],
                 dtype=np.float32)
    got = fp8_e4m3.encode_rne_satfinite(x).tolist()
    # 2^-10 is the tie between 0 and the smallest subnormal: even code 0 wins;
    # 1.5*2^-9 ties between codes 1 and 2: even code 2 wins; 1.0625 ties between
    # 1.0 (0x38) and 1.125 (0x39): 0x38; 1.1875 ties between 0x39 and 0x3A: 0x3A.
    assert got == [0x00, 0x80, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F,
                   0x01, 0x00, 0x01, 0x02, 0x38, 0x3A]


def test_encode_decode_roundtrip_of_every_finite_code():
    vals = fp8_e4m3.DECODE_TABLE.astype(np.float32)
    finite = ~np.isnan(vals)
    codes = np.arange(256, dtype=np.uint8)[finite]
    assert np.array_equal(fp8_e4m3.encode_rne_satfinite(vals[finite]), codes)


def _pool():
    os.environ["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests")] +
                                               os.environ.get("PYTHONPATH", "").split(os.pathsep))
    return ProcessPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)),
                               mp_context=mp.get_context("spawn"))


def _run(ranges):
    from e4m3_sweep import sweep_chunk
    total, bad = 0, []
    with _pool() as ex:
        for n, b in ex.map(sweep_chunk, [r[0] for r in ranges], [r[1] for r in ranges]):
            total += n
            bad += b
    return total, bad


def test_encode_exhaustive_over_the_rounding_range():
    """Every float32 with |x| in [2^-17, 2^9) (exponent fields 110..135, both signs,
    all 2^23 mantissas): the whole range where rounding can pick a non-zero,
    non-saturated code, checked against torch and the brute-force nearest search."""
    ranges = [((s << 31) | (e << 23), 1 << 23) for s in (0, 1) for e in range(110, 136)]
    total, bad = _run(ranges)
    assert total == 52 * (1 << 23)
    assert not bad, bad[:10]


def test_encode_outside_the_rounding_range_sampled():
    """The flush-to-zero and saturation ranges (all other exponent fields, including
    infinities and NaNs), with the first/last 4096 mantissas and a stride-97 sample."""
    from e4m3_sweep import sweep_chunk
    for s in (0, 1):
        for e in list(range(0, 110)) + list(range(136, 256)):
            base = (s << 31) | (e << 23)
            for start, cnt in ((base, 4096), (base + (1 << 23) - 4096, 4096)):
                n, bad = sweep_chunk(start, cnt)
                assert not bad, bad
    # strided sample through each field
    bits = np.concatenate([np.arange((s << 31) | (e << 23), ((s << 31) | (e << 23)) + (1 << 23), 97,
                                     dtype=np.uint64)
                           for s in (0, 1) for e in (0, 1, 50, 109, 136, 200, 254, 255)]).astype(np.uint32)
    from e4m3_sweep import brute_force_encode
    x = bits.view(np.float32)
    assert np.array_equal(fp8_e4m3.encode_rne_satfinite(x), brute_force_encode(x))


@pytest.mark.skipif(os.environ.get("MLA_EXHAUSTIVE") != "1",
                    reason="all 2^32 float32 patterns: set MLA_EXHAUSTIVE=1 (several CPU-minutes)")
def test_encode_exhaustive_all_float32():
    ranges = [(i << 24, 1 << 24) for i in range(256)]
    total, bad = _run(ranges)
    assert total == 1 << 32
    assert not bad, bad[:10]
