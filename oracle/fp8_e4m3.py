"""OCP FP8 E4M3 ("fn") codec — oracle, test infrastructure only (see ``oracle/__init__``).

The FP8 KV cache of "[Attention] Blackwell FP8 MLA support with CUTLASS_MLA backend"
(Purpose: "Enable FP8 KV cache support"; the kernel-test log in the comment by
elvischenv names the element type ``torch.float8_e4m3fn``) stores each latent value
as one E4M3 byte. The pages do not define the format; its definition is the OCP
"OFP8 Formats for Deep Learning" specification (v1.0), E4M3 column:

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
* exponent field 0 encodes subnormals ``(-1)^s * m * 2**-9``;
* exponent field 1..15 encodes ``(-1)^s * (1 + m/8) * 2**(e - 7)``, except
  ``S.1111.111`` which is NaN. There are no infinities; the largest finite
  magnitude is ``S.1111.110`` = 448.

Encoding (the cache write) is round-to-nearest, ties-to-even on the exact float32
input, with saturation of every finite or infinite magnitude above 448 to ±448
("satfinite"). The sign of zero is kept. NaN encodes to 0x7F.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def _decode_one(code: int) -> float:
    """Value of one E4M3 byte, straight from the OCP field definition."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:
        return sign * mant * 2.0 ** -9
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


#: float64 value of every byte 0..255 (NaN for 0x7F and 0xFF).
DECODE_TABLE = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)


def decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 bytes (uint8 array, any shape) -> float64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    return DECODE_TABLE[codes]


def encode_rne_satfinite(x: np.ndarray) -> np.ndarray:
    """float32 array -> E4M3 bytes, round-to-nearest-even with saturation.

    The input is taken as exact float32 values (float64 holds every float32 exactly,
    so every step below is exact until the one rounding ``np.rint``, which rounds
    half to even). For a finite magnitude ``a <= 448`` with ``2**k <= a < 2**(k+1)``:

    * the spacing of E4M3 values around ``a`` is ``2**(k-3)`` for ``k >= -6`` and
      ``2**-9`` below (the subnormal range), i.e. ``2**(max(k, -6) - 3)``;
    * ``q = rint(a / spacing)`` lies in 8..16 for normals (0..8 for subnormals);
    * the code is ``8 * (max(k, -6) + 7) + (q - 8)``: exponent field times 8 plus the
      mantissa. ``q == 16`` (or 8 from a subnormal) carries into the next exponent
      field on its own, and for subnormals the formula reduces to ``q``.

    Magnitudes above 448 (and infinities) saturate to code 0x7E; NaN gives 0x7F; the
    sign bit is copied from the input, so -0.0 encodes to 0x80.
    """
    x = np.asarray(x, dtype=np.float32)
    sign = (((x.view(np.uint32) >> 31) & 1).astype(np.uint8) << 7)
    with np.errstate(invalid="ignore"):
        a = np.abs(x.astype(np.float64))
    nan = np.isnan(a)
    big = (~nan) & (a > E4M3_MAX)
    a_in = np.where(nan | big, 0.0, a)
    _, e2 = np.frexp(a_in)                       # a = f * 2**e2, f in [0.5, 1)
    k = np.where(a_in < 2.0 ** -6, -6, e2.astype(np.int64) - 1)
    q = np.rint(np.ldexp(a_in, 3 - k)).astype(np.int64)
    code = 8 * (k + 7) + (q - 8)
    code = np.where(big, 0x7E, code).astype(np.uint8) | sign
    code[nan] = E4M3_NAN_CODE
    return code
