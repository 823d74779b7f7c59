"""Exhaustive float32 -> E4M3 check of the oracle encoder (worker for test_oracle_fp8).

For a contiguous range of float32 bit patterns this compares the oracle's
``encode_rne_satfinite`` with two references that share none of its arithmetic:

1. torch's ``float32 -> float8_e4m3fn`` conversion, wherever |x| <= 448 (torch rounds
   to nearest-even there but does not saturate above it);
2. a brute-force search for the nearest finite E4M3 value among the 127 non-negative
   codes (ties to the even code), with saturation to 448 above the range and 0x7F
   for NaN — the definition of round-to-nearest-even with satfinite, written out.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import fp8_e4m3

_POS_VALUES = fp8_e4m3.DECODE_TABLE[:127]          # codes 0x00..0x7E, ascending


def brute_force_encode(x: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        a = np.abs(x.astype(np.float64))
    sign = ((x.view(np.uint32) >> 31) & 1).astype(np.uint8) << 7
    out = np.empty(x.shape, dtype=np.uint8)
    nan = np.isnan(a)
    sat = (~nan) & (a > 448.0)
    mid = (~nan) & (~sat)
    am = a[mid]
    hi = np.searchsorted(_POS_VALUES, am, side="left")          # values[hi] >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = am - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - am
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    out[mid] = code
    out[sat] = 0x7E
    out = out | sign
    out[nan] = 0x7F
    return out


def sweep_chunk(start: int, count: int):
    """Check bit patterns [start, start+count); return (checked, first mismatches)."""
    bits = np.arange(start, start + count, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    got = fp8_e4m3.encode_rne_satfinite(x)
    bad = []
    ref = brute_force_encode(x)
    m = np.nonzero(got != ref)[0]
    bad += [("brute", int(bits[i]), int(got[i]), int(ref[i])) for i in m[:5]]
    a = np.abs(x)
    inr = (~np.isnan(a)) & (a <= 448.0)
    t = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    m2 = np.nonzero(got[inr] != t)[0]
    sel = bits[inr]
    bad += [("torch", int(sel[i]), int(got[inr][i]), int(t[i])) for i in m2[:5]]
    return count, bad
