"""FP8 E4M3 (the "fn" variant: no infinities, two NaN codes) from its definition.

Test infrastructure only (see oracle/__init__.py).

Format, as used by the FP8 K/V caches ("KvQuantSparseFlashAttention" README,
参数说明 table, key/value dtype FLOAT8_E4M3; "[Triton] FP8 with FA v3 API",
Technical Details): bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0
mantissa.  Exponent field 0 encodes subnormals m/8 * 2^-6; exponent field
15 with mantissa 7 (codes 0x7F / 0xFF) is NaN; the largest finite value is
1.75 * 2^8 = 448.
"""
import numpy as np

E4M3_MAX = 448.0


def _decode_one(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


#: value of every byte, float64 (exact: every E4M3 value is a dyadic rational)
DECODE_TABLE = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)


def decode(codes: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values (exact)."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode_rne_satfinite(x: np.ndarray) -> np.ndarray:
    """float32 values -> uint8 E4M3 codes, round to nearest even, saturating.

    |x| >= 448 maps to +-448 (saturation to the largest finite value instead
    of NaN); NaN maps to 0x7F; the sign of zero is kept.  The quantum at
    magnitude v is 2^(floor(log2 v) - 3) for normals and 2^-9 below 2^-6;
    dividing by a power of two is exact in float64, so ``rint`` applies the
    ties-to-even rule to the exact quotient.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    sat = a >= E4M3_MAX
    a = np.where(sat, 0.0, a)

    # exponent of the quantum: normals use floor(log2 a) - 3, subnormals -9
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.exp2(e - 3.0)
    n = np.rint(a / quantum)          # integer count of quanta, ties to even
    v = n * quantum                   # rounded magnitude (exact)

    code = np.zeros(x.shape, dtype=np.int64)
    sub = v < 2.0 ** -6
    code = np.where(sub, (v / 2.0 ** -9).astype(np.int64), code)
    with np.errstate(divide="ignore"):
        ev = np.floor(np.log2(np.where(sub | (v == 0), 1.0, v)))
    mant = np.where(sub, 0.0, v / np.exp2(ev) * 8.0 - 8.0)
    normal_code = ((ev.astype(np.int64) + 7) << 3) | mant.astype(np.int64)
    code = np.where(sub, code, normal_code)
    code = np.where(sat, 0x7E, code)
    code = code | np.where(sign, 0x80, 0)
    code = np.where(nan, 0x7F, code)
    out[...] = code.astype(np.uint8)
    return out
