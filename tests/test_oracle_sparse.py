"""Pins of the oracle's 2:4 structured-sparse product (CPU only): a hand-derived fixture, equality
with the dense oracle on the decompressed matrix (bit for bit), and torch float64 matmul on a
decompression written here with numpy. Names the sparse GEMM as 05 Blackwell TCGEN05 GEMM tutorial,
"An API-level note" does (gemm_sp), read as the 2:4 pattern along K."""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

T16 = {"bf16": torch.bfloat16, "f16": torch.float16}


def codes(values, kind):
    t = torch.tensor(np.asarray(values, dtype=np.float64)).to(T16[kind])
    return t.view(torch.int16).numpy().view(np.uint16)


def values(codes_, kind):
    return torch.from_numpy(np.ascontiguousarray(codes_).view(np.int16)).view(T16[kind]).to(
        torch.float64).numpy()


def decompress(vals, meta, M, K):
    """Dense [M, K] codes from vals [M, K/2] and meta [M, K/8] (written independently of the
    oracle: unpack the nibbles with numpy, then scatter)."""
    G = K // 4
    nib = np.stack([meta & 0xF, meta >> 4], axis=-1).reshape(M, -1)[:, :G]
    pos = np.stack([nib & 0x3, (nib >> 2) & 0x3], axis=-1)  # [M, G, 2]
    dense = np.zeros((M, K), dtype=np.uint16)
    rows = np.repeat(np.arange(M), G * 2).reshape(M, G, 2)
    cols = 4 * np.arange(G)[None, :, None] + pos
    dense[rows, cols] = vals.reshape(M, G, 2)
    return dense


def random_sparse(rng, kind, M, K):
    """Random 2:4 rows: N(0,1) values at two distinct random positions of every group."""
    G = K // 4
    pos = np.sort(np.stack([rng.permutation(4)[:2] for _ in range(M * G)]), axis=1).reshape(M, G, 2)
    swap = rng.random((M, G)) < 0.5  # both orders of the two fields occur
    pos[swap] = pos[swap][:, ::-1]
    nib = pos[..., 0] | (pos[..., 1] << 2)
    if G % 2:
        nib = np.concatenate([nib, np.zeros((M, 1), nib.dtype)], axis=1)
    meta = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    vals = codes(rng.standard_normal((M, K // 2)), kind)
    return vals, meta


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["NT", "NN"])
def test_golden_sparse_2x2(kind, layout):
    g = read_golden("sp24_2x2_k8.txt")
    M, N, K = (int(g[k][0][0]) for k in ("M", "N", "K"))
    vals = codes([[float(x) for x in row] for row in g["vals"]], kind)
    meta = np.array([[int(x, 16) for x in row] for row in g["meta"]], np.uint8)
    B = codes([[float(x) for x in row] for row in g["B"]], kind)
    if layout == "NN":
        B = np.ascontiguousarray(B.T)
    want = np.array([[float(x) for x in row] for row in g["C"]])
    C, S = oracle.gemm_sp(kind, layout, vals, meta, B, M, N, K, sums=True)
    assert np.array_equal(S, want) and np.array_equal(values(C, kind), want)


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["NT", "NN"])
@pytest.mark.parametrize("M,N,K", [(5, 7, 16), (9, 4, 36), (3, 3, 4)])
def test_equals_dense_oracle_on_the_decompressed_matrix(kind, layout, M, N, K):
    rng = np.random.default_rng(M * N + K)
    vals, meta = random_sparse(rng, kind, M, K)
    dense = decompress(vals, meta, M, K)
    B = codes(rng.standard_normal((N, K) if layout == "NT" else (K, N)), kind)
    C, S = oracle.gemm_sp(kind, layout, vals, meta, B, M, N, K, sums=True)
    Cd, Sd = oracle.gemm16(kind, layout, dense, B, M, N, K, sums=True)
    assert np.array_equal(C, Cd) and np.array_equal(S, Sd)
    bop = values(B, kind) if layout == "NN" else values(B, kind).T
    ref = (torch.from_numpy(values(dense, kind)) @ torch.from_numpy(np.ascontiguousarray(bop))).numpy()
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12)


def test_only_kept_positions_contribute():
    # every group keeps positions 2 and 1 (in that order): B's columns 0 and 3 of every group
    # must not matter
    M, N, K = 2, 3, 16
    rng = np.random.default_rng(0)
    vals = codes(rng.standard_normal((M, K // 2)), "bf16")
    meta = np.full((M, K // 8), (2 | 1 << 2) * 0x11, np.uint8)
    B1 = codes(rng.standard_normal((N, K)), "bf16")
    B2 = B1.copy()
    B2[:, 0::4] = codes(np.full((N, K // 4), 99.0), "bf16")
    B2[:, 3::4] = codes(np.full((N, K // 4), -7.0), "bf16")
    assert np.array_equal(oracle.gemm_sp("bf16", "NT", vals, meta, B1, M, N, K),
                          oracle.gemm_sp("bf16", "NT", vals, meta, B2, M, N, K))


def test_bad_arguments_are_refused():
    v = np.zeros((1, 2), np.uint16)
    m = np.zeros((1, 1), np.uint8)
    B = np.zeros((1, 6), np.uint16)
    with pytest.raises((ValueError, AssertionError)):
        oracle.gemm_sp("bf16", "NT", v, m, B, 1, 1, 6)  # K % 4 != 0
    with pytest.raises(ValueError):
        oracle.gemm_sp("bf16", "TN", np.zeros((1, 2), np.uint16), m, np.zeros((1, 4), np.uint16), 1, 1, 4)
