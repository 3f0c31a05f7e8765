"""Pins for the oracle's format codecs (CPU only).

Decoders are checked on every code against library conversions (torch's bf16/fp16/float8 dtypes).
Encoders (double -> 16-bit, round to nearest even, one rounding) are checked against numpy's direct
double -> binary16 conversion and, for bf16, against torch on inputs that are exactly binary32
values (where torch's float -> bf16 step is a single rounding), plus hand-derived codes for
doubles with more than 24 significant bits, where a double -> float -> bf16 path would round twice.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _same(a, b):
    """Equal values, NaN matching NaN, and the sign of zero respected."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nan = np.isnan(a) | np.isnan(b)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    assert np.array_equal(a[~nan], b[~nan])
    assert np.array_equal(np.signbit(a[~nan]), np.signbit(b[~nan]))


def test_dec_bf16_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    _same(oracle.dec_bf16(codes), ref.numpy())


def test_dec_f16_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.float16).to(torch.float64)
    _same(oracle.dec_f16(codes), ref.numpy())


def test_dec_e4m3_all_codes():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.dec_e4m3(codes)
    _same(got, ref)
    # the format's landmarks: largest finite 448, smallest subnormal 2^-9, NaN only at S.1111.111
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    assert [c for c in range(256) if math.isnan(got[c])] == [0x7F, 0xFF]


def test_dec_e5m2_all_codes():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
    got = oracle.dec_e5m2(codes)
    _same(got, ref)
    # landmarks: largest finite 57344, smallest subnormal 2^-16, 1.0 = 0x3C, inf at exponent 31
    # with a zero fraction, NaN with a non-zero one
    assert got[0x7B] == 57344.0 and got[0x01] == 2.0 ** -16 and got[0x3C] == 1.0
    assert got[0x7C] == math.inf and got[0xFC] == -math.inf
    assert [c for c in range(256) if math.isnan(got[c])] == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]


def test_dec_e8m0_all_codes():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = oracle.dec_e8m0(codes)
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        _same(got, ref)
    # closed form 2^(e-127), exact in double for every finite code; 0xFF is NaN
    assert all(got[e] == math.ldexp(1.0, e - 127) for e in range(255))
    assert math.isnan(got[255])


def test_enc_16bit_round_trips_every_code():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dec, enc in ((oracle.dec_bf16, oracle.enc_bf16), (oracle.dec_f16, oracle.enc_f16)):
        vals = dec(codes)
        finite = ~np.isnan(vals)
        assert np.array_equal(enc(vals[finite]), codes[finite])


def _f16_grid():
    """fp16 values, the midpoints between neighbours (exact ties) and points just off them."""
    codes = np.arange(0, 0x7C00, dtype=np.uint16)  # +0 .. largest finite
    v = oracle.dec_f16(codes)
    mids = (v[:-1] + v[1:]) / 2
    eps = np.abs(mids) * 2.0 ** -30
    pts = np.concatenate([v, mids, mids + eps, mids - eps, [65504.0, 65519.99, 65520.0, 1e6]])
    return np.concatenate([pts, -pts])


def test_enc_f16_matches_numpy_direct_rounding():
    pts = _f16_grid()
    with np.errstate(over="ignore"):
        ref = pts.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.enc_f16(pts), ref)


def test_enc_f16_random_doubles_match_numpy():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-30, 18, 20000))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.enc_f16(x), ref)


def test_enc_bf16_on_binary32_inputs_matches_torch():
    # every bf16 midpoint has 9 significant bits, so it is a binary32 value: torch's float -> bf16
    # conversion is then a single RNE rounding and a valid reference.
    codes = np.arange(0, 0x7F80, dtype=np.uint16)
    v = oracle.dec_bf16(codes)
    mids = (v[:-1] + v[1:]) / 2
    rng = np.random.default_rng(3)
    rnd = (rng.standard_normal(20000) * np.exp2(rng.integers(-100, 100, 20000))).astype(np.float32)
    pts = np.concatenate([v, mids, rnd.astype(np.float64)])
    pts = np.concatenate([pts, -pts])
    assert np.array_equal(pts.astype(np.float32).astype(np.float64), pts)
    ref = torch.from_numpy(pts.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(oracle.enc_bf16(pts), ref.view(np.uint16))


@pytest.mark.parametrize(
    "x,code",
    [
        # hand-derived: bf16 has 8 significant bits, spacing 2^-7 on [1,2)
        (1 + 2.0 ** -8, 0x3F80),  # exact tie -> even (1.0)
        (1 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),  # just above the tie: one rounding goes up
        (1 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),
        (1 + 3 * 2.0 ** -8, 0x3F82),  # tie between 0x3F81 and 0x3F82 -> even
        (257.0, 0x4380),  # tie 256|258 -> 256
        (259.0, 0x4382),  # tie 258|260 -> 260
        (-259.0, 0xC382),
        (2.0 ** 128, 0x7F80),  # overflow -> +inf
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),  # tie above the largest finite -> inf
        ((2 - 2.0 ** -8 - 2.0 ** -30) * 2.0 ** 127, 0x7F7F),  # below it -> largest finite
        (2.0 ** -133, 0x0001),  # smallest subnormal
        (2.0 ** -134, 0x0000),  # tie 0|2^-133 -> 0 (even)
        (1.5 * 2.0 ** -134, 0x0001),
        (-0.0, 0x8000),
        (float("inf"), 0x7F80),
        (float("-inf"), 0xFF80),
    ],
)
def test_enc_bf16_hand_derived(x, code):
    assert int(oracle.enc_bf16([x])[0]) == code


@pytest.mark.parametrize(
    "x,code",
    [
        (2049.0, 0x6800),  # tie 2048|2050 -> 2048
        (2051.0, 0x6802),  # tie 2050|2052 -> 2052 (mantissa 2: spacing is 2 at 2048)
        (1 + 2.0 ** -11 + 2.0 ** -40, 0x3C01),
        (65504.0, 0x7BFF),
        (65519.0, 0x7BFF),
        (65520.0, 0x7C00),  # tie between the largest finite and 2^16 -> even -> overflow
        (-70000.0, 0xFC00),
        (2.0 ** -24, 0x0001),
        (2.0 ** -25, 0x0000),  # tie -> 0
        (3 * 2.0 ** -26, 0x0001),
        (2.0 ** -14 - 2.0 ** -24, 0x03FF),  # largest subnormal
    ],
)
def test_enc_f16_hand_derived(x, code):
    assert int(oracle.enc_f16([x])[0]) == code
