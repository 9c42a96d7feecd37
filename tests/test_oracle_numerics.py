"""Pins for the oracle's E4M3 codec and BF16 rounding (CPU only).

The codec is pinned exhaustively: every one of the 256 codes, and every FP32
value in the binades where E4M3 rounding is non-trivial, is checked against a
brute-force nearest-value search written independently of the encoder.
"""

import os

import numpy as np
import pytest
import torch

from oracle.numerics import (
    bf16_round,
    bf16_to_bits,
    bits_to_f32,
    e4m3_decode,
    e4m3_encode,
)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _finite_table():
    """Sorted positive finite E4M3 values and their codes, by enumeration."""
    codes = np.arange(0x00, 0x7F, dtype=np.uint8)       # 0x00 .. 0x7E, positive
    vals = e4m3_decode(codes)
    order = np.argsort(vals, kind="stable")
    return vals[order], codes[order]


def _brute_force_encode_pos(a):
    """Nearest positive finite E4M3 value, ties to the even code, saturating."""
    vals, codes = _finite_table()
    a = np.minimum(a, vals[-1])
    hi = np.searchsorted(vals, a, side="left")          # vals[hi] >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - vals[lo]
    d_hi = vals[hi] - a
    pick_hi = d_hi < d_lo
    tie = d_hi == d_lo
    even_hi = (codes[hi] & 1) == 0
    pick_hi = np.where(tie, even_hi, pick_hi)
    return np.where(pick_hi, codes[hi], codes[lo])


def test_e4m3_spot_values_from_format_definition():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e4m3_spot_values.txt"))
            if l.strip() and not l.startswith("#")]
    for code_hex, val in rows:
        code = int(code_hex, 16)
        got = e4m3_decode(np.array([code], dtype=np.uint8))[0]
        if val == "nan":
            assert np.isnan(got), code_hex
        else:
            want = float(val)
            assert got == want and np.signbit(got) == np.signbit(want), (code_hex, got, want)


def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_all_codes_round_trip():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3_decode(codes)
    back = e4m3_encode(vals)
    nan = np.isnan(vals)
    assert nan.sum() == 2                     # 0x7F and 0xFF
    assert (back[~nan] == codes[~nan]).all()
    assert (back[nan] == 0x7F).all()
    finite = np.sort(np.abs(vals[~nan]))
    assert finite[-1] == 448.0 and np.unique(finite).size == 127


@pytest.mark.parametrize("biased_exp", list(range(116, 137)))
def test_e4m3_encode_exhaustive_binade(biased_exp):
    """Every positive FP32 value of one binade 2^-11 .. 2^9, against brute force.

    Below 2^-11 every value is closer to 0 than to 2^-9 and above 2^9 every
    value saturates; both tails are checked separately below.
    """
    bits = (np.uint32(biased_exp) << np.uint32(23)) | np.arange(1 << 23, dtype=np.uint32)
    x = bits.view(np.float32)
    got = e4m3_encode(x)
    want = _brute_force_encode_pos(x.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], want[bad[:5]])
    # sign symmetry on the same binade
    neg = e4m3_encode(-x[:: 97])
    assert (neg == (want[:: 97] | 0x80)).all()


def test_e4m3_encode_tails_and_specials():
    tiny = np.array([0.0, 2.0 ** -149, 2.0 ** -20, 2.0 ** -11, 2.0 ** -10, np.nextafter(np.float32(2.0 ** -10), np.float32(1))],
                    dtype=np.float32)
    assert list(e4m3_encode(tiny)) == [0, 0, 0, 0, 0, 1]     # 2^-10 is a tie -> even code 0
    assert list(e4m3_encode(-tiny)) == [0x80, 0x80, 0x80, 0x80, 0x80, 0x81]
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, 3.0e38, np.inf], dtype=np.float32)
    assert (e4m3_encode(big) == 0x7E).all()
    assert (e4m3_encode(-big) == 0xFE).all()
    assert e4m3_encode(np.array([np.nan], dtype=np.float32))[0] == 0x7F
    # the largest value below 2^-11 .. and the smallest above 2^9 region
    rng = np.random.default_rng(1)
    low = (rng.random(100000) * 2.0 ** -11).astype(np.float32)
    assert (e4m3_encode(low) == 0).all()
    high = (512.0 + rng.random(100000) * 1e30).astype(np.float32)
    assert (e4m3_encode(high) == 0x7E).all()


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(200000) * 50,
        rng.standard_normal(100000) * 0.01,
        (rng.random(50000) - 0.5) * 896,
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (e4m3_encode(x) == ref).all()


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, size=500000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # exact halfway cases: low 16 bits == 0x8000
    halves = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    halves = halves[np.isfinite(halves)]
    specials = np.array([0.0, -0.0, 1.0, 3.3895314e38, -3.3895314e38, 3.4028235e38,
                         1e-40, -1e-40, 1.17549435e-38, 2.0 ** -133, 2.0 ** -134], dtype=np.float32)
    for arr in (x, halves, specials):
        ours = bf16_round(arr)
        ref = torch.from_numpy(arr).to(torch.bfloat16).to(torch.float32).numpy()
        same = (ours.view(np.uint32) == ref.view(np.uint32))
        assert same.all(), (arr[~same][:5], ours[~same][:5], ref[~same][:5])


def test_bf16_bits_round_trip():
    rng = np.random.default_rng(4)
    b = rng.integers(0, 2 ** 16, size=100000, dtype=np.uint64).astype(np.uint16)
    f = bits_to_f32(b)
    ok = np.isfinite(f)
    assert (bf16_to_bits(f[ok]) == b[ok]).all()
    assert (bf16_round(f[ok]).view(np.uint32) == f[ok].view(np.uint32)).all()
