"""E4M3 codec and BF16 rounding written from the format definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

E4M3 ("E4M3FN" in the OCP 8-bit floating point specification, the FP8
activation and weight format of FlashInfer PR #4287's W8A8 path):

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
* exponent field 0 is subnormal: value = m/8 * 2**-6;
* otherwise value = (1 + m/8) * 2**(e - 7);
* S.1111.111 is NaN; there are no infinities; the largest finite value is
  S.1111.110 = 448.

Encoding rule used throughout (the reading fixed for the whole build):
round to nearest, ties to the even mantissa; finite values beyond 448 and
infinities saturate to +-448 ("satfinite"); NaN encodes to 0x7F; the sign of
zero is kept.

BF16: 1 sign, 8 exponent, 7 mantissa bits (the FP32 exponent range);
conversion from FP32 rounds to nearest, ties to even, overflow goes to
infinity as IEEE 754 prescribes.
"""

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Decode E4M3 codes (uint8 array) to float64 values, NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int32)
    e = (c >> 3) & 0xF
    m = c & 0x7
    # subnormal: m * 2^-9; normal: (8 + m) * 2^(e - 10)
    mag = np.ldexp(np.where(e == 0, m, 8 + m).astype(np.float64), np.where(e == 0, -9, e - 10))
    val = np.where((c >> 7) == 1, -mag, mag)
    return np.where((e == 15) & (m == 7), np.nan, val)


def e4m3_encode(x):
    """Encode real values to E4M3 codes (uint8).

    ``x`` may be float32 or float64; the rounding is done on the exact value
    (float32 inputs are exact in float64).  Within the binade
    [2**E, 2**(E+1)) the spacing of E4M3 values is 2**(E-3); below 2**-6 the
    subnormal spacing 2**-9 applies, which is the same formula with E clamped
    to -6.  So r = |x| / 2**(E-3) is exact, and ``np.round`` (halves to the
    even integer) rounds it to the nearest representable multiple; an even r
    is an even mantissa, so this is round-to-nearest-even on the E4M3 grid.
    r lies in [8, 16] for normal binades (16 carries into the next binade)
    and in [0, 8] below 2**-6.
    """
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    neg = np.signbit(x)
    a = np.where(nan, 0.0, np.abs(x))
    a = np.minimum(a, E4M3_MAX)             # satfinite: beyond 448 (and inf) -> 448
    _, ex = np.frexp(a)                     # a = f * 2**ex, f in [0.5, 1)
    E = np.maximum(ex - 1, -6)              # binade exponent, subnormals share -6
    r = np.round(np.ldexp(a, 3 - E)).astype(np.int32)
    carry = r == 16
    E = E + carry
    r = np.where(carry, 8, r)
    normal = r >= 8
    e_field = np.where(normal, E + 7, 0)
    m_field = np.where(normal, r - 8, r)
    code = (neg.astype(np.int32) << 7) | (e_field << 3) | m_field
    return np.where(nan, 0x7F, code).astype(np.uint8)


def bf16_round(x):
    """Round float32 values to the nearest BF16 value (ties to even).

    Returns float32 values that are exactly representable in BF16.  The
    spacing of BF16 values in the binade [2**E, 2**(E+1)) is 2**(E-7), with E
    clamped to -126 for subnormals (BF16 shares FP32's exponent range).
    Values that round beyond the largest finite BF16 become infinity.
    """
    x = np.asarray(x, dtype=np.float32)
    out = x.astype(np.float64)
    fin = np.isfinite(out)
    a = np.where(fin, np.abs(out), 0.0)
    _, ex = np.frexp(a)
    E = np.maximum(ex - 1, -126)
    spacing = np.exp2((E - 7).astype(np.float64))
    r = np.round(a / spacing) * spacing
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(r > bf16_max, np.inf, r)
    r = np.where(np.signbit(out), -r, r)
    res = np.where(fin, r, out)
    return res.astype(np.float32)


def bf16_to_bits(x):
    """BF16-representable float32 values -> their uint16 bit patterns."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f32(bits):
    """BF16 bit patterns (uint16) -> float32 values."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32(x):
    """Round to float32 (round to nearest even), the FP32 step of the method."""
    return np.asarray(x, dtype=np.float32)
