"""Seeded synthetic workloads for the dense GEMM: shapes, seeds and host-side input bytes.

This module holds no GEMM arithmetic. It only draws random numbers and stores them in the
operand formats, so the same bytes can be handed to the CUDA library and to the CPU oracle.

Recipe (the pages measure on random matrices, not on a dataset: TileLang SM100 Support (Preview),
"Compilation and Usage", draws ``torch.randn(M, K)`` and ``torch.randn(N, K)``):

* 16-bit operands: ``torch.Generator().manual_seed(seed)``, then ``torch.randn`` in fp32 for A
  (shape [M,K]) and then B ([N,K] for "NT", [K,N] for "NN"), each rounded to bf16 or fp16 by
  torch's round-to-nearest-even conversion. Returned as uint16 code arrays.
* FP6 / FP4 block-scaled operands (the OCP MX element formats e2m3, e3m2, e2m1): the MXFP8
  recipe below with the element rounded to the nearest fp6 / fp4 value (ties to the even code,
  saturating at the largest magnitude); rows packed as a little-endian bit stream, element k at
  bit b*k.
* 2:4 structured-sparse A: the generator draws the stored values ~ N(0,1) [M, K/2] (rounded to
  bf16 / fp16), then B as for the dense product, then for every group of 4 K-elements two
  distinct positions (a uniformly random pair, in random order); metadata nibble = first | second
  << 2, two groups per byte, the even group in the low nibble.
* MXFP8 operands: the same generator draws x_A ~ N(0,1) [M,K], x_B ~ N(0,1) [N,K], then integer
  exponents u_A [M, ceil(K/128)] and u_B [N, ceil(K/128)] uniform in {-3..3}. Each element is
  stored as e4m3(x / 2^u) (torch's RNE conversion to float8_e4m3fn) and each scale as the E8M0
  code 127 + u, so that e4m3 * 2^(sf-127) is close to x. |x / 2^u| stays far below e4m3's
  largest finite value 448, so no element saturates.
"""
from dataclasses import dataclass

import numpy as np
import torch

SF_BLOCK = 128  # K-elements per E8M0 scale (granularity 128 along K for both operands)
BITS = {"e4m3": 8, "e5m2": 8, "e2m3": 6, "e3m2": 6, "e2m1": 4}  # bits per element


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "bf16", "f16", "mxfp8" (block-scaled, E8M0 scales), "nvfp4" (e2m1, UE4M3 scales
    #            per 16) or "bf16_sp24" / "f16_sp24" (2:4 sparse A)
    layout: str  # "NT" (B is [N,K]), "NN" (B is [K,N]); a leading "T" stores A as [K,M]
    M: int
    N: int
    K: int
    seed: int
    a_fmt: str = "e4m3"  # block-scaled product: element formats of A and B (fp8, fp6 or fp4)
    b_fmt: str = "e4m3"
    block: int = SF_BLOCK  # block-scaled product: K-elements per scale

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """Compulsory HBM traffic: read A and B (and the scales) once, write C once."""
        if self.kind == "mxfp8":
            kb = (self.K + self.block - 1) // self.block
            return (self.M * self.K * BITS[self.a_fmt] // 8 + self.N * self.K * BITS[self.b_fmt] // 8
                    + (self.M + self.N) * kb + 2 * self.M * self.N)
        if self.kind == "nvfp4":  # packed e2m1 rows, one scale byte per 16 elements, bf16 C
            return (self.M + self.N) * (self.K // 2 + self.K // 16) + 2 * self.M * self.N
        if self.kind.endswith("_sp24"):  # stored values, metadata, B, C
            return self.M * self.K + self.M * self.K // 8 + 2 * (self.N * self.K + self.M * self.N)
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


# The pages' example shapes (TileLang SM100 Support (Preview): NT 4096x4096x8192 with a
# 128x256x128 tile; tilelang (velog) 1.1-1.3: fp16 NN 1024^3) plus the large 2-CTA square, the
# memory-bound skinny product and the block-scaled variant; then the same 4096x4096x8192 product
# with A stored transposed (trans_A of T.gemm), to measure the MN-major A path, and block-scaled
# with the OCP MX 32-element scale blocks, in e4m3, e5m2, fp4 (e2m1) and fp6 (e2m3 x e3m2).
WORKLOADS = {
    w.name: w
    for w in [
        Workload("bf16_nt_256x256x512", "bf16", "NT", 256, 256, 512, 0),
        Workload("f16_nn_1024x1024x1024", "f16", "NN", 1024, 1024, 1024, 1),
        Workload("bf16_nt_4096x4096x8192", "bf16", "NT", 4096, 4096, 8192, 2),
        Workload("bf16_nt_8192x8192x8192", "bf16", "NT", 8192, 8192, 8192, 3),
        Workload("bf16_nt_128x8192x8192", "bf16", "NT", 128, 8192, 8192, 3),
        Workload("mxfp8_nt_4096x4096x8192", "mxfp8", "NT", 4096, 4096, 8192, 4),
        Workload("bf16_tn_4096x4096x8192", "bf16", "TN", 4096, 4096, 8192, 5),
        Workload("bf16_tt_4096x4096x8192", "bf16", "TT", 4096, 4096, 8192, 6),
        Workload("mxfp8_b32_nt_4096x4096x8192", "mxfp8", "NT", 4096, 4096, 8192, 7,
                 block=32),
        Workload("mx_e5m2_b32_nt_4096x4096x8192", "mxfp8", "NT", 4096, 4096, 8192, 8,
                 a_fmt="e5m2", b_fmt="e5m2", block=32),
        Workload("mxfp4_b32_nt_4096x4096x8192", "mxfp8", "NT", 4096, 4096, 8192, 9,
                 a_fmt="e2m1", b_fmt="e2m1", block=32),
        Workload("mxfp6_e2m3_e3m2_b32_nt_4096x4096x8192", "mxfp8", "NT", 4096, 4096, 8192, 10,
                 a_fmt="e2m3", b_fmt="e3m2", block=32),
        Workload("bf16_sp24_nt_4096x4096x8192", "bf16_sp24", "NT", 4096, 4096, 8192, 11),
        Workload("nvfp4_nt_4096x4096x8192", "nvfp4", "NT", 4096, 4096, 8192, 12,
                 a_fmt="e2m1", b_fmt="e2m1", block=16),
    ]
}

HEADLINE = "bf16_nt_4096x4096x8192"

_TORCH_16 = {"bf16": torch.bfloat16, "f16": torch.float16}


def randn16(kind: str, shape, gen: torch.Generator) -> np.ndarray:
    """N(0,1) fp32 draws rounded to bf16/fp16; returned as uint16 codes."""
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32).to(_TORCH_16[kind])
    return x.view(torch.int16).numpy().view(np.uint16)


def make16(kind: str, layout: str, M: int, N: int, K: int, seed: int):
    """(A, B) as uint16 codes: A [M,K] ([K,M] for layouts TN, TT), B [N,K] (NT, TT) or [K,N]
    (NN, TN)."""
    g = torch.Generator().manual_seed(seed)
    A = randn16(kind, (K, M) if layout[0] == "T" else (M, K), g)
    B = randn16(kind, (N, K) if layout[1] == "T" else (K, N), g)
    return A, B


_TORCH_8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def make_mx(M: int, N: int, K: int, seed: int, a_fmt: str = "e4m3", b_fmt: str = "e4m3",
            block: int = SF_BLOCK):
    """(A [M,K], B [N,K], sfA [M,kb], sfB [N,kb]) as uint8 codes: fp8 elements (e4m3 or e5m2) and
    E8M0 scales, one per row per `block` K-elements (kb = ceil(K/block)). Element = fp8(x / 2^u)
    with x ~ N(0,1) and u uniform in {-3..3} per (row, block); scale = 127 + u."""
    g = torch.Generator().manual_seed(seed)
    kb = (K + block - 1) // block
    xa = torch.randn((M, K), generator=g, dtype=torch.float32)
    xb = torch.randn((N, K), generator=g, dtype=torch.float32)
    ua = torch.randint(-3, 4, (M, kb), generator=g, dtype=torch.int32)
    ub = torch.randint(-3, 4, (N, kb), generator=g, dtype=torch.int32)

    def quantise(x, u, fmt):
        # per-element exponent of its (row, K-block); dividing by a power of two is exact in fp32
        ue = u.repeat_interleave(block, dim=1)[:, : x.shape[1]]
        q = torch.ldexp(x, -ue.to(torch.float32)).to(_TORCH_8[fmt])
        return q.view(torch.uint8).numpy()

    A = quantise(xa, ua, a_fmt)
    B = quantise(xb, ub, b_fmt)
    sfA = (ua + 127).to(torch.uint8).numpy()
    sfB = (ub + 127).to(torch.uint8).numpy()
    return A, B, sfA, sfB


def pack_rows(codes: np.ndarray, bits: int) -> np.ndarray:
    """[R, K] element codes of `bits` bits -> [R, ceil(K*bits/8)] bytes, element k at bit bits*k
    of the row read as a little-endian bit stream (one byte per element for 8 bits)."""
    codes = np.asarray(codes, dtype=np.uint8)
    if bits == 8:
        return codes.copy()
    R, K = codes.shape
    stream = ((codes[:, :, None] >> np.arange(bits, dtype=np.uint8)) & 1).reshape(R, K * bits)
    stream = np.pad(stream, ((0, 0), (0, (-stream.shape[1]) % 8)))
    return np.packbits(stream, axis=1, bitorder="little")


# Bit fields of the OCP MX sub-byte element formats: (exponent bits, mantissa bits, bias).
_SUB_BYTE_FIELDS = {"e2m3": (2, 3, 1), "e3m2": (3, 2, 3), "e2m1": (2, 1, 1)}


def _positive_values(fmt: str) -> np.ndarray:
    """Values of the non-negative codes 0 .. 2^(bits-1) - 1 of an fp6 / fp4 format, in code
    order (which is increasing): subnormals m * 2^(1-bias-mbits), normals (1 + m/2^mbits) *
    2^(e-bias)."""
    ebits, mbits, bias = _SUB_BYTE_FIELDS[fmt]
    vals = []
    for e in range(1 << ebits):
        for m in range(1 << mbits):
            if e == 0:
                vals.append(m * 2.0 ** (1 - bias - mbits))
            else:
                vals.append((1 + m / 2.0 ** mbits) * 2.0 ** (e - bias))
    return np.array(vals)


def quantise_sub_byte(x: np.ndarray, fmt: str) -> np.ndarray:
    """Codes of the nearest fp6 / fp4 values to x (ties to the even code), saturating at the
    largest magnitude (the OCP MX conversion saturates: these formats have no infinity)."""
    vals = _positive_values(fmt)
    sign_bit = 1 << (sum(_SUB_BYTE_FIELDS[fmt][:2]))
    a = np.minimum(np.abs(x), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 1, len(vals) - 1)
    lo = hi - 1
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    return (code | np.where(x < 0, sign_bit, 0)).astype(np.uint8)


def make_sub_byte(M: int, N: int, K: int, seed: int, a_fmt: str, b_fmt: str, block: int = 32):
    """(A [M, K*ba/8], B [N, K*bb/8] packed rows, sfA [M,kb], sfB [N,kb] E8M0 codes) for block-
    scaled products with fp6 / fp4 operands (an fp8 partner stays one byte per element): the
    MXFP8 recipe, element = fmt(x / 2^u) with x ~ N(0,1) and u uniform in {-3..3} per (row,
    block), scale = 127 + u; sub-byte elements round to nearest (ties to even) and saturate."""
    g = torch.Generator().manual_seed(seed)
    kb = (K + block - 1) // block
    xa = torch.randn((M, K), generator=g, dtype=torch.float32)
    xb = torch.randn((N, K), generator=g, dtype=torch.float32)
    ua = torch.randint(-3, 4, (M, kb), generator=g, dtype=torch.int32)
    ub = torch.randint(-3, 4, (N, kb), generator=g, dtype=torch.int32)

    def quantise(x, u, fmt):
        ue = u.repeat_interleave(block, dim=1)[:, : x.shape[1]]
        y = torch.ldexp(x, -ue.to(torch.float32))  # exact: a power-of-two scaling
        if fmt in _TORCH_8:
            return y.to(_TORCH_8[fmt]).view(torch.uint8).numpy()
        return quantise_sub_byte(y.numpy().astype(np.float64), fmt)

    A = pack_rows(quantise(xa, ua, a_fmt), BITS[a_fmt])
    B = pack_rows(quantise(xb, ub, b_fmt), BITS[b_fmt])
    return A, B, (ua + 127).to(torch.uint8).numpy(), (ub + 127).to(torch.uint8).numpy()


def make_nvfp4(M: int, N: int, K: int, seed: int):
    """(A [M, K/2], B [N, K/2] packed e2m1 rows, sfA [M, K/16], sfB [N, K/16] UE4M3 codes) of an
    NVFP4 product, K % 16 == 0. Elements: e2m1(2x) with x ~ N(0,1) (round to nearest, ties to the
    even code, saturating at 6), so the codes spread over the whole e2m1 range; scales: UE4M3
    codes with exponent field uniform in {4..10} and mantissa uniform in {0..7} (values 2^-3 ..
    1.875 * 2^3), independent per (row, 16-element block)."""
    g = torch.Generator().manual_seed(seed)
    kb = K // 16

    def operand(rows):
        x = 2.0 * torch.randn((rows, K), generator=g, dtype=torch.float32).numpy().astype(np.float64)
        e = torch.randint(4, 11, (rows, kb), generator=g, dtype=torch.int32)
        m = torch.randint(0, 8, (rows, kb), generator=g, dtype=torch.int32)
        return (pack_rows(quantise_sub_byte(x, "e2m1"), 4), ((e << 3) | m).to(torch.uint8).numpy())

    A, sfA = operand(M)
    B, sfB = operand(N)
    return A, B, sfA, sfB


def make_mxfp8(M: int, N: int, K: int, seed: int):
    """(A [M,K] e4m3, B [N,K] e4m3, sfA [M,kb] E8M0, sfB [N,kb] E8M0) as uint8 codes, kb =
    ceil(K/128)."""
    return make_mx(M, N, K, seed)


def make_sp24(kind: str, layout: str, M: int, N: int, K: int, seed: int):
    """(vals [M, K/2] uint16 codes, meta [M, ceil(K/8)] uint8, B) of a 2:4 structured-sparse
    product: B [N,K] for "NT", [K,N] for "NN". K % 4 == 0."""
    g = torch.Generator().manual_seed(seed)
    vals = randn16(kind, (M, K // 2), g)
    B = randn16(kind, (N, K) if layout[1] == "T" else (K, N), g)
    G = K // 4
    # a random pair of distinct positions per group: the first uniform in 0..3, the second one
    # of the other three
    first = torch.randint(0, 4, (M, G), generator=g)
    second = (first + torch.randint(1, 4, (M, G), generator=g)) % 4
    nib = (first | (second << 2)).numpy().astype(np.uint8)
    if G % 2:
        nib = np.concatenate([nib, np.zeros((M, 1), np.uint8)], axis=1)
    meta = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return vals, meta, B


def make(w: Workload):
    if w.kind == "nvfp4":
        return make_nvfp4(w.M, w.N, w.K, w.seed)
    if w.kind.endswith("_sp24"):
        return make_sp24(w.kind[:-5], w.layout, w.M, w.N, w.K, w.seed)
    if w.kind == "mxfp8" and (BITS[w.a_fmt] < 8 or BITS[w.b_fmt] < 8):
        return make_sub_byte(w.M, w.N, w.K, w.seed, w.a_fmt, w.b_fmt, w.block)
    if w.kind == "mxfp8":
        return make_mx(w.M, w.N, w.K, w.seed, w.a_fmt, w.b_fmt, w.block)
    return make16(w.kind, w.layout, w.M, w.N, w.K, w.seed)
