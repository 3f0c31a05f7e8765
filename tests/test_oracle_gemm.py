"""Pins for the oracle's GEMMs (CPU only): hand-derived fixtures, exact special cases, invariants
and an independent library routine (torch float64 matmul on torch-decoded operands).

The method's definition: C = A . B^T with B stored [N,K] ("NT": TileLang SM100 Support (Preview),
"Code Example" / "Compilation and Usage") or C = A . B with B stored [K,N] ("NN": tilelang
(velog), 1.1 Front-End DSL); a leading "T" stores A as [K,M] (trans_A of T.gemm, TileLang SM100
Support (Preview), "Current Limitations"); MXFP8 per the 05 Blackwell TCGEN05 GEMM tutorial, "Advanced"
(gemm_blockscaled, K-granularity 128 for both operands).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from dense_tensor_core_gb300 import workloads

T16 = {"bf16": torch.bfloat16, "f16": torch.float16}


def codes_of(vals, kind):
    """Exact decimal values -> 16-bit codes (torch conversion; every value used is representable)."""
    t = torch.tensor(np.asarray(vals, dtype=np.float64)).to(T16[kind])
    assert np.array_equal(t.to(torch.float64).numpy(), np.asarray(vals, dtype=np.float64))
    return t.view(torch.int16).numpy().view(np.uint16)


def values_of(codes, kind):
    t = torch.from_numpy(np.ascontiguousarray(codes).view(np.int16).copy()).view(T16[kind])
    return t.to(torch.float64).numpy()


def matrix(rows):
    return np.array([[float(v) for v in r] for r in rows], dtype=np.float64)


# --- hand-derived fixtures ----------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["NT", "NN"])
def test_golden_2x2(kind, layout):
    g = read_golden("gemm16_2x2_integers.txt")
    A, B = matrix(g["A"]), matrix(g["B"])
    C = oracle.gemm16(kind, layout, codes_of(A, kind), codes_of(B, kind), 2, 2, 2)
    assert np.array_equal(values_of(C, kind), matrix(g[f"C_{layout}_{kind}"]))


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["TN", "TT"])
def test_golden_transposed_a(kind, layout):
    g = read_golden("gemm16_2x3_k3_transposed_a.txt")
    A, B = matrix(g["A"]), matrix(g[f"B_{layout}"])
    C, S = oracle.gemm16(kind, layout, codes_of(A, kind), codes_of(B, kind), 2, 3, 3, sums=True)
    assert np.array_equal(S, matrix(g["C"]))
    assert np.array_equal(values_of(C, kind), matrix(g["C"]))


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["NT", "NN"])
def test_golden_4x4_rounding(kind, layout):
    g = read_golden("gemm16_4x4_dyadic_rounding.txt")
    A, Bnk = matrix(g["A"]), matrix(g["B"])
    B = Bnk if layout == "NT" else np.ascontiguousarray(Bnk.T)  # NN stores B^T as [K,N]
    C, S = oracle.gemm16(kind, layout, codes_of(A, kind), codes_of(B, kind), 4, 4, 4, sums=True)
    assert np.array_equal(S, matrix(g["S"]))
    assert np.array_equal(values_of(C, kind), matrix(g[f"C_NT_{kind}"]))


@pytest.mark.parametrize("kind", ["bf16", "f16"])
def test_golden_f16_ties_and_overflow(kind):
    g = read_golden("gemm16_1x3_f16_ties_overflow.txt")
    A, B = matrix(g["A"]), matrix(g["B"])
    C, S = oracle.gemm16(kind, "NT", codes_of(A, kind), codes_of(B, kind), 1, 3, 2, sums=True)
    assert np.array_equal(S, matrix(g["S"]))
    assert np.array_equal(values_of(C, kind), matrix(g[f"C_NT_{kind}"]))


def test_golden_mxfp8_blockscaled():
    g = read_golden("mxfp8_2x2_k256_blockscaled.txt")
    M, N, K = 2, 2, 256
    A = np.zeros((M, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    for r, k, c in g["A_nz"]:
        A[int(r), int(k)] = int(c, 16)
    for r, k, c in g["B_nz"]:
        B[int(r), int(k)] = int(c, 16)
    sfA = np.array(g["sfA"], dtype=np.uint8)
    sfB = np.array(g["sfB"], dtype=np.uint8)
    C, S = oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K, sums=True)
    assert np.array_equal(S, matrix(g["C"]))
    assert np.array_equal(values_of(C, "bf16"), matrix(g["C"]))


# --- exact special cases -------------------------------------------------------------------------

def _rand16(kind, shape, seed):
    return workloads.randn16(kind, shape, torch.Generator().manual_seed(seed))


def store_a(Aop, layout):
    """Aop [M,K] in the layout's storage order for A."""
    return np.ascontiguousarray(Aop.T if layout[0] == "T" else Aop)


def store_b(Bop, layout):
    """Bop [K,N] in the layout's storage order for B ([N,K] when its second letter is T)."""
    return np.ascontiguousarray(Bop.T if layout[1] == "T" else Bop)


def op_b(B, layout):
    return B.T if layout[1] == "T" else B


LAYOUTS = ["NT", "NN", "TN", "TT"]


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_identity_gives_B(kind, layout):
    # A = I (M = K): C = Bop exactly (each sum has one nonzero term, already a 16-bit value)
    K, N = 24, 40
    A = codes_of(np.eye(K), kind)
    B = _rand16(kind, oracle.b_shape(layout, N, K), 11)
    C = oracle.gemm16(kind, layout, A, B, K, N, K)
    assert np.array_equal(C, op_b(B, layout))


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_permutations_permute_exactly(kind, layout):
    M, N, K = 16, 12, 20  # M != K: a transposed A read as untransposed would not even line up
    rng = np.random.default_rng(5)
    p = rng.permutation(K)[:M]
    P = np.zeros((M, K))
    P[np.arange(M), p] = 1.0  # (P X)[i] = X[p[i]]
    B = _rand16(kind, oracle.b_shape(layout, N, K), 12)
    C = oracle.gemm16(kind, layout, codes_of(store_a(P, layout), kind), B, M, N, K)
    assert np.array_equal(C, op_b(B, layout)[p, :])
    # permutation on the other side: Bop = Q with Q[k, n] = 1 iff k = q[n] -> C[:, n] = Aop[:, q[n]]
    q = rng.permutation(K)[:N]
    Q = np.zeros((K, N))
    Q[q, np.arange(N)] = 1.0
    A = _rand16(kind, oracle.a_shape(layout, M, K), 13)
    Aop = A.T if layout[0] == "T" else A
    C2 = oracle.gemm16(kind, layout, A, codes_of(store_b(Q, layout), kind), M, N, K)
    assert np.array_equal(C2, Aop[:, q])


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("K", [512, 1024, 8192])
def test_all_ones_gives_K(kind, K):
    M, N = 3, 5
    one = codes_of([1.0], kind)[0]
    A = np.full((M, K), one, np.uint16)
    B = np.full((N, K), one, np.uint16)
    C, S = oracle.gemm16(kind, "NT", A, B, M, N, K, sums=True)
    assert np.all(S == K)
    assert np.all(values_of(C, kind) == K)  # powers of two: exact in both formats


@pytest.mark.parametrize("kind", ["bf16", "f16"])
def test_linearity_in_A(kind):
    M, N, K = 20, 18, 96
    A = _rand16(kind, (M, K), 21)
    B = _rand16(kind, (N, K), 22)
    A2 = codes_of(2.0 * values_of(A, kind), kind)  # doubling is exact
    C1, S1 = oracle.gemm16(kind, "NT", A, B, M, N, K, sums=True)
    C2, S2 = oracle.gemm16(kind, "NT", A2, B, M, N, K, sums=True)
    assert np.array_equal(S2, 2.0 * S1)
    assert np.array_equal(values_of(C2, kind), 2.0 * values_of(C1, kind))  # RNE commutes with 2x
    # additivity on small integers (every partial sum exact): S(A1 + A2) = S(A1) + S(A2)
    rng = np.random.default_rng(9)
    I1 = rng.integers(-8, 9, (M, K)).astype(np.float64)
    I2 = rng.integers(-8, 9, (M, K)).astype(np.float64)
    Bi = codes_of(rng.integers(-8, 9, (N, K)).astype(np.float64), kind)
    _, Sa = oracle.gemm16(kind, "NT", codes_of(I1, kind), Bi, M, N, K, sums=True)
    _, Sb = oracle.gemm16(kind, "NT", codes_of(I2, kind), Bi, M, N, K, sums=True)
    _, Sab = oracle.gemm16(kind, "NT", codes_of(I1 + I2, kind), Bi, M, N, K, sums=True)
    assert np.array_equal(Sab, Sa + Sb)


def test_degenerate_sizes():
    A = np.zeros((3, 0), np.uint16)
    B = np.zeros((4, 0), np.uint16)
    C, S = oracle.gemm16("bf16", "NT", A, B, 3, 4, 0, sums=True)
    assert np.all(C == 0) and np.all(S == 0)  # K = 0: the empty sum, +0
    C = oracle.gemm16("bf16", "NT", np.zeros((0, 8), np.uint16), np.zeros((4, 8), np.uint16), 0, 4, 8)
    assert C.shape == (0, 4)


# --- an independent library routine --------------------------------------------------------------

@pytest.mark.parametrize("kind,layout", [("bf16", "NT"), ("f16", "NN"), ("bf16", "NN"), ("f16", "NT"),
                                         ("bf16", "TN"), ("f16", "TT"), ("f16", "TN"), ("bf16", "TT")])
def test_matches_torch_float64_matmul(kind, layout):
    # ragged sizes (not multiples of any tile)
    M, N, K = 67, 45, 200
    A, B = workloads.make16(kind, layout, M, N, K, 31)
    C, S = oracle.gemm16(kind, layout, A, B, M, N, K, sums=True)
    At = torch.from_numpy(values_of(A, kind).reshape(oracle.a_shape(layout, M, K)))
    Bt = torch.from_numpy(values_of(B, kind).reshape(oracle.b_shape(layout, N, K)))
    ref = ((At.T if layout[0] == "T" else At) @ (Bt.T if layout[1] == "T" else Bt)).numpy()
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12)
    if kind == "f16":
        assert np.array_equal(C, ref.astype(np.float16).view(np.uint16))  # numpy: direct RNE
    else:
        got = values_of(C, kind)
        # torch's double -> bf16 path rounds through float; compare with a one-ulp allowance
        refb = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()
        ulp = np.abs(refb) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(got - refb) <= ulp)
        assert np.mean(got == refb) > 0.99


def test_sampled_equals_full():
    for kind, layout in (("bf16", "NT"), ("f16", "NN"), ("bf16", "TN"), ("f16", "TT")):
        M, N, K = 33, 29, 130
        A, B = workloads.make16(kind, layout, M, N, K, 41)
        C, S = oracle.gemm16(kind, layout, A, B, M, N, K, sums=True)
        rng = np.random.default_rng(1)
        r = rng.integers(0, M, 50)
        c = rng.integers(0, N, 50)
        Cs, Ss = oracle.gemm16_sampled(kind, layout, A, B, M, N, K, r, c)
        assert np.array_equal(Cs, C[r, c]) and np.array_equal(Ss, S[r, c])


# --- MXFP8 ---------------------------------------------------------------------------------------

def _e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)


def test_mxfp8_unit_scales_reduce_to_plain_e4m3_gemm():
    M, N, K = 40, 36, 384
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, 51)
    sfA[:] = 127
    sfB[:] = 127
    _, S = oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K, sums=True)
    ref = (_e4m3_values(A) @ _e4m3_values(B).T).numpy()
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12)


def test_mxfp8_uniform_exponent_shift_scales_exactly():
    M, N, K = 24, 20, 256
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, 52)
    _, S0 = oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K, sums=True)
    _, S1 = oracle.gemm_mxfp8(A, B, sfA + 3, sfB, M, N, K, sums=True)
    _, S2 = oracle.gemm_mxfp8(A, B, sfA, sfB - 2, M, N, K, sums=True)
    assert np.array_equal(S1, S0 * 8.0) and np.array_equal(S2, S0 * 0.25)


@pytest.mark.parametrize("K", [256, 200, 8])  # whole blocks, a partial last block, K < 128
def test_mxfp8_per_block_scales_equal_premultiplied_operands(K):
    M, N = 30, 26
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, 53)
    C, S = oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K, sums=True)
    kidx = torch.arange(K) // 128
    sa = torch.from_numpy(sfA.astype(np.float64))[:, kidx] - 127
    sb = torch.from_numpy(sfB.astype(np.float64))[:, kidx] - 127
    Aval = _e4m3_values(A) * torch.pow(2.0, sa)
    Bval = _e4m3_values(B) * torch.pow(2.0, sb)
    ref = (Aval @ Bval.T).numpy()
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12)
    r = np.arange(M).repeat(N)
    c = np.tile(np.arange(N), M)
    Cs, Ss = oracle.gemm_mxfp8_sampled(A, B, sfA, sfB, M, N, K, r, c)
    assert np.array_equal(Cs, C.ravel()) and np.array_equal(Ss, S.ravel())


# --- other block-scaled formats: e5m2 elements, 32-element scale blocks ----------------------------

def _fp8_values(codes, fmt):
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(codes)).view(dt).to(torch.float64)


def test_golden_mx_block32_e5m2():
    g = read_golden("mx_1x2_k64_e4m3_e5m2_block32.txt")
    M, N, K = 1, 2, 64
    A = np.zeros((M, K), np.uint8)
    B = np.zeros((N, K), np.uint8)
    for r, k, c in g["A_nz"]:
        A[int(r), int(k)] = int(c, 16)
    for r, k, c in g["B_nz"]:
        B[int(r), int(k)] = int(c, 16)
    sfA = np.array(g["sfA"], dtype=np.uint8)
    sfB = np.array(g["sfB"], dtype=np.uint8)
    C, S = oracle.gemm_mx(A, B, sfA, sfB, M, N, K, a_fmt="e4m3", b_fmt="e5m2", block=32, sums=True)
    assert np.array_equal(S, matrix(g["C"]))
    assert np.array_equal(values_of(C, "bf16"), matrix(g["C"]))


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("block", [32, 128])
@pytest.mark.parametrize("K", [256, 200, 8])  # whole blocks, a partial last block, K < 32
def test_mx_per_block_scales_equal_premultiplied_operands(a_fmt, b_fmt, block, K):
    # an independent routine: torch float64 matmul on torch-decoded, scaled operands
    M, N = 22, 18
    A, B, sfA, sfB = workloads.make_mx(M, N, K, 54, a_fmt, b_fmt, block)
    C, S = oracle.gemm_mx(A, B, sfA, sfB, M, N, K, a_fmt=a_fmt, b_fmt=b_fmt, block=block, sums=True)
    kidx = torch.arange(K) // block
    sa = torch.from_numpy(sfA.astype(np.float64))[:, kidx] - 127
    sb = torch.from_numpy(sfB.astype(np.float64))[:, kidx] - 127
    ref = ((_fp8_values(A, a_fmt) * torch.pow(2.0, sa)) @ (_fp8_values(B, b_fmt) * torch.pow(2.0, sb)).T).numpy()
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12)
    r = np.arange(M).repeat(N)
    c = np.tile(np.arange(N), M)
    Cs, Ss = oracle.gemm_mx_sampled(A, B, sfA, sfB, M, N, K, r, c, a_fmt=a_fmt, b_fmt=b_fmt,
                                    block=block)
    assert np.array_equal(Cs, C.ravel()) and np.array_equal(Ss, S.ravel())


def test_mx_block32_with_repeated_scales_equals_block128():
    # 32-element blocks whose scales repeat 4x along K give exactly the 128-element result
    M, N, K = 20, 24, 384
    A, B, sfA, sfB = workloads.make_mx(M, N, K, 55)
    C128, S128 = oracle.gemm_mx(A, B, sfA, sfB, M, N, K, block=128, sums=True)
    C32, S32 = oracle.gemm_mx(A, B, np.repeat(sfA, 4, axis=1), np.repeat(sfB, 4, axis=1), M, N, K,
                              block=32, sums=True)
    assert np.array_equal(S32, S128) and np.array_equal(C32, C128)


def test_mx_default_formats_are_the_mxfp8_product():
    M, N, K = 16, 12, 256
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, 56)
    assert np.array_equal(oracle.gemm_mx(A, B, sfA, sfB, M, N, K),
                          oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K))


def test_workload_recipe_shapes_and_ranges():
    A, B, sfA, sfB = workloads.make_mxfp8(64, 32, 300, 4)
    assert A.shape == (64, 300) and B.shape == (32, 300) and sfA.shape == (64, 3)
    assert sfA.min() >= 124 and sfA.max() <= 130  # exponents in {-3..3}
    vals = _e4m3_values(A).numpy()
    assert np.isfinite(vals).all() and np.abs(vals).max() < 448
    a16, b16 = workloads.make16("f16", "NN", 8, 6, 4, 1)
    assert a16.shape == (8, 4) and b16.shape == (4, 6)
    assert math.isclose(workloads.WORKLOADS["bf16_nt_4096x4096x8192"].flops, 274877906944)
