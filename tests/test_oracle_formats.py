"""Pins of the oracle's other block-scaled formats (CPU only).

05 Blackwell TCGEN05 GEMM tutorial, "Advanced (not implemented here)", names "MXFP8 and other
block-scaled formats" without defining them; the oracle reads them as the OCP MX family (fp6
E2M3 / E3M2 and fp4 E2M1 elements with E8M0 scales per 32 or 128 K-elements) and NVFP4 (E2M1
elements with a UE4M3 scale per 16). Each part is pinned to something other than the oracle's own
formula: the OCP E2M1 table typed by hand, torch's fp8 decoders for the fp6 value sets and UE4M3,
hand-derived products in tests/golden/, a packer written here with numpy's bit routines, and
torch float64 matmul on the decoded operands.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def _torch_dec(codes, dtype):
    return torch.tensor(np.asarray(codes, dtype=np.uint8)).view(dtype).to(torch.float64).numpy()


# --- element decoders ---------------------------------------------------------------------------

def test_e2m1_matches_the_ocp_table():
    g = read_golden("ocp_mx_e2m1_values.txt")
    codes = [int(c, 16) for c in g["codes"][0]]
    want = np.array([float(v) for v in g["values"][0]])
    got = oracle.dec_e2m1(codes)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))  # -0 for code 0x8


@pytest.mark.parametrize("fmt,fp8,bits_scale,largest", [("e2m3", torch.float8_e4m3fn, 8, 7.5),
                                                        ("e3m2", torch.float8_e5m2, 16, 28.0)])
def test_fp6_value_sets_from_fp8(fmt, fp8, bits_scale, largest):
    # E2M3 has e4m3's 3 mantissa bits: its values are exactly the e4m3 values in [0, 7.5] that are
    # multiples of 1/8. E3M2 has e5m2's 2 mantissa bits: the e5m2 values in [0, 28] that are
    # multiples of 1/16. Codes 0..31 list them in increasing order; bit 5 is the sign.
    dec = getattr(oracle, "dec_" + fmt)
    pos = dec(range(32))
    ref = _torch_dec(range(256), fp8)
    ref = ref[np.isfinite(ref)]
    want = np.unique(ref[(ref >= 0) & (ref <= largest) & (ref * bits_scale == np.round(ref * bits_scale))])
    assert np.array_equal(pos, want)
    assert np.all(np.diff(pos) > 0) and pos[-1] == largest
    neg = dec(range(32, 64))
    assert np.array_equal(neg, -pos) and np.all(np.signbit(neg))


def test_e2m1_is_e2m3_with_a_shorter_mantissa():
    # both have 2 exponent bits with bias 1: fp4 code (s, e, m) is fp6 code (s, e, m << 2)
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        assert oracle.dec_e2m1([c])[0] == oracle.dec_e2m3([(s << 5) | (e << 3) | (m << 2)])[0]


def test_ue4m3_is_e4m3_without_sign():
    codes = np.arange(256)
    got = oracle.dec_ue4m3(codes)
    want = _torch_dec(codes[:128], torch.float8_e4m3fn)
    assert np.array_equal(got[:128], want, equal_nan=True)
    assert np.isnan(got[128:]).all()  # a set sign bit is not a UE4M3 scale


# --- packing (written independently with numpy's bit routines) ------------------------------------

BITS = {"e4m3": 8, "e5m2": 8, "e2m3": 6, "e3m2": 6, "e2m1": 4}


def pack_rows(codes, fmt):
    """[R, K] element codes -> [R, row_bytes] packed: element k in bits [b*k, b*k + b) of the row
    as a little-endian bit stream."""
    b = BITS[fmt]
    codes = np.asarray(codes, dtype=np.uint8)
    if b == 8:
        return codes.copy()
    R, K = codes.shape
    # each code's b bits, least significant first, laid end to end
    bits = ((codes[:, :, None] >> np.arange(b, dtype=np.uint8)) & 1).reshape(R, K * b)
    pad = (-bits.shape[1]) % 8
    bits = np.pad(bits, ((0, 0), (0, pad)))
    return np.packbits(bits, axis=1, bitorder="little")


def random_codes(rng, fmt, shape):
    return rng.integers(0, 1 << BITS[fmt], size=shape).astype(np.uint8)


def decode(codes, fmt):
    if fmt in ("e4m3", "e5m2"):
        return _torch_dec(codes.ravel(), torch.float8_e4m3fn if fmt == "e4m3" else
                          torch.float8_e5m2).reshape(codes.shape)
    return getattr(oracle, "dec_" + fmt)(codes.ravel()).reshape(codes.shape)


def _finite_fp8(rng, fmt, shape):
    c = random_codes(rng, fmt, shape)
    nan = np.isnan(decode(c, fmt)) | np.isinf(decode(c, fmt))
    c[nan] = 0
    return c


@pytest.mark.parametrize("a_fmt,b_fmt,scale,block,K", [
    ("e2m1", "e2m1", "e8m0", 32, 256),
    ("e2m3", "e3m2", "e8m0", 32, 128),
    ("e3m2", "e2m1", "e8m0", 128, 384),
    ("e2m1", "e4m3", "e8m0", 32, 160),   # a partial last block
    ("e5m2", "e2m3", "e8m0", 128, 256),
    ("e2m1", "e2m1", "ue4m3", 16, 192),  # NVFP4
    ("e2m1", "e2m1", "ue4m3", 16, 40),   # a partial last block
])
def test_packed_products_equal_torch_float64(a_fmt, b_fmt, scale, block, K):
    rng = np.random.default_rng(K + block)
    M, N = 5, 7
    ca = _finite_fp8(rng, a_fmt, (M, K))
    cb = _finite_fp8(rng, b_fmt, (N, K))
    kb = (K + block - 1) // block
    if scale == "e8m0":
        sfA = rng.integers(120, 135, (M, kb)).astype(np.uint8)
        sfB = rng.integers(120, 135, (N, kb)).astype(np.uint8)
        sa, sb = np.ldexp(1.0, sfA.astype(int) - 127), np.ldexp(1.0, sfB.astype(int) - 127)
    else:
        sfA = rng.integers(0x20, 0x50, (M, kb)).astype(np.uint8)  # positive finite e4m3 codes
        sfB = rng.integers(0x20, 0x50, (N, kb)).astype(np.uint8)
        sa, sb = _torch_dec(sfA, torch.float8_e4m3fn), _torch_dec(sfB, torch.float8_e4m3fn)
    av = decode(ca, a_fmt) * np.repeat(sa, block, axis=1)[:, :K]
    bv = decode(cb, b_fmt) * np.repeat(sb, block, axis=1)[:, :K]
    want = (torch.from_numpy(av) @ torch.from_numpy(bv).T).numpy()
    C, S = oracle.gemm_bs(pack_rows(ca, a_fmt), pack_rows(cb, b_fmt), sfA, sfB, M, N, K,
                          a_fmt=a_fmt, b_fmt=b_fmt, scale=scale, block=block, sums=True)
    assert np.allclose(S, want, rtol=1e-12, atol=1e-12)
    Cs, Ss = oracle.gemm_bs_sampled(pack_rows(ca, a_fmt), pack_rows(cb, b_fmt), sfA, sfB, M, N, K,
                                    np.repeat(np.arange(M), N), np.tile(np.arange(N), M),
                                    a_fmt=a_fmt, b_fmt=b_fmt, scale=scale, block=block)
    assert np.array_equal(Cs, C.ravel()) and np.array_equal(Ss, S.ravel())


def _golden_bs(name):
    g = read_golden(name)
    M, N, K = int(g["M"][0][0]), int(g["N"][0][0]), int(g["K"][0][0])
    a_fmt, b_fmt = g["A_fmt"][0][0], g["B_fmt"][0][0]
    block, scale = int(g["block"][0][0]), g["scale"][0][0]
    ca = np.zeros((M, K), np.uint8)
    cb = np.zeros((N, K), np.uint8)
    for r, k, c in g["A_nz"]:
        ca[int(r), int(k)] = int(c, 16)
    for r, k, c in g["B_nz"]:
        cb[int(r), int(k)] = int(c, 16)
    sfA = np.array([[int(x, 0) for x in row] for row in g["sfA"]], np.uint8)
    sfB = np.array([[int(x, 0) for x in row] for row in g["sfB"]], np.uint8)
    want = np.array([[float(x) for x in row] for row in g["C"]])
    return (pack_rows(ca, a_fmt), pack_rows(cb, b_fmt), sfA, sfB, M, N, K,
            dict(a_fmt=a_fmt, b_fmt=b_fmt, scale=scale, block=block), want)


@pytest.mark.parametrize("name", ["bs_1x2_k128_e2m1_e3m2_block32.txt",
                                  "nvfp4_1x1_k64_ue4m3_block16.txt"])
def test_golden_sub_byte_products(name):
    A, B, sfA, sfB, M, N, K, kw, want = _golden_bs(name)
    C, S = oracle.gemm_bs(A, B, sfA, sfB, M, N, K, sums=True, **kw)
    assert np.array_equal(S, want)
    dec = torch.from_numpy(C.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(dec, want)  # the sums are bf16 values: rounding keeps them


def test_block32_with_repeated_scales_equals_block128_for_fp4():
    rng = np.random.default_rng(3)
    M, N, K = 4, 6, 256
    ca, cb = random_codes(rng, "e2m1", (M, K)), random_codes(rng, "e2m1", (N, K))
    sa = rng.integers(122, 132, (M, 2)).astype(np.uint8)
    sb = rng.integers(122, 132, (N, 2)).astype(np.uint8)
    kw = dict(a_fmt="e2m1", b_fmt="e2m1")
    c128 = oracle.gemm_bs(pack_rows(ca, "e2m1"), pack_rows(cb, "e2m1"), sa, sb, M, N, K,
                          block=128, **kw)
    c32 = oracle.gemm_bs(pack_rows(ca, "e2m1"), pack_rows(cb, "e2m1"), np.repeat(sa, 4, 1),
                         np.repeat(sb, 4, 1), M, N, K, block=32, **kw)
    assert np.array_equal(c128, c32)


def test_fp8_members_agree_with_the_mx_entry():
    rng = np.random.default_rng(4)
    M, N, K = 6, 5, 192
    ca, cb = _finite_fp8(rng, "e4m3", (M, K)), _finite_fp8(rng, "e5m2", (N, K))
    sa = rng.integers(124, 131, (M, 2)).astype(np.uint8)
    sb = rng.integers(124, 131, (N, 2)).astype(np.uint8)
    a = oracle.gemm_bs(ca, cb, sa, sb, M, N, K, a_fmt="e4m3", b_fmt="e5m2", block=128)
    b = oracle.gemm_mx(ca, cb, sa, sb, M, N, K, a_fmt="e4m3", b_fmt="e5m2", block=128)
    assert np.array_equal(a, b)


def test_bad_format_arguments_are_refused():
    A = np.zeros((1, 64), np.uint8)
    s = np.zeros((1, 4), np.uint8)
    with pytest.raises(KeyError):
        oracle.gemm_bs(A, A, s, s, 1, 1, 64, a_fmt="e1m2", block=16)
    with pytest.raises(ValueError):  # a block size outside 16, 32, 128
        oracle.gemm_bs(np.zeros((1, 32), np.uint8), np.zeros((1, 32), np.uint8), np.zeros((1, 1), np.uint8),
                       np.zeros((1, 1), np.uint8), 1, 1, 64, a_fmt="e2m1", b_fmt="e2m1", block=64)
