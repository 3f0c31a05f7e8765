"""GPU parity of the block-scaled product with fp6 and fp4 elements (OCP MX E2M3, E3M2, E2M1) and
E8M0 scales per 32 or 128 K-elements, against the CPU oracle, through the C ABI.

These are the "other block-scaled formats" of 05 Blackwell TCGEN05 GEMM tutorial, "Advanced (not
implemented here)", run by the one-CTA block-scaled kernel with kind::mxf8f6f4: the packed rows
are unpacked by the tensor memory access unit into 16-byte groups (12 or 8 bytes of data, then
padding), the layout the MMA reads for these element types.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tensor_core_gb300 import workloads
from parity import check_close, sample_positions, to_device8, values16, with_packed_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_bs(A, B, sfA, sfB, a_fmt, b_fmt, block, **kw):
    import dense_tensor_core_gb300 as dtc

    K = A.shape[1] * 8 // {"e4m3": 8, "e5m2": 8, "e2m3": 6, "e3m2": 6, "e2m1": 4}[a_fmt]
    kw = with_packed_scales(A.shape[0], B.shape[0], K,
                            dict(kw, a_format=a_fmt, b_format=b_fmt, scale_block=block))
    C = dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), sfA=to_device8(sfA),
                    sfB=to_device8(sfB), **kw)
    dtc.gemm_stream_status()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


def check_bs(M, N, K, a_fmt, b_fmt, block, seed, **kw):
    A, B, sfA, sfB = workloads.make_sub_byte(M, N, K, seed, a_fmt, b_fmt, block)
    C = run_bs(A, B, sfA, sfB, a_fmt, b_fmt, block, **kw)
    ref = oracle.gemm_bs(A, B, sfA, sfB, M, N, K, a_fmt=a_fmt, b_fmt=b_fmt, block=block)
    return check_close(values16(C, "bf16"), values16(ref, "bf16"),
                       f"{a_fmt} x {b_fmt} block {block} {M}x{N}x{K}")


PAIRS = [("e2m1", "e2m1"), ("e2m3", "e3m2"), ("e3m2", "e2m1"), ("e2m1", "e4m3"),
         ("e5m2", "e2m3"), ("e4m3", "e4m3")]


KERNELS = {"1cta": dict(variant=1), "1cta_packed": dict(variant=1, pack=True),
           "pair": dict(variant=2, pack=True)}


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("block", [32, 128])
@pytest.mark.parametrize("a_fmt,b_fmt", PAIRS, ids=lambda p: str(p))
@pytest.mark.parametrize("M,N,K", [(128, 224, 128), (300, 520, 384), (256, 448, 1024), (1, 8, 128),
                                   (640, 904, 256)])
def test_formats_full_parity(M, N, K, a_fmt, b_fmt, block, kernel):
    kw = KERNELS[kernel]
    if kw.get("pack") and kw["variant"] == 1 and block == 128:
        pytest.skip("the one-CTA kernel repacks the scales of 32-element blocks only")
    if kw["variant"] == 2 and block != 128:
        pytest.skip("the pair kernel takes 128-element scale blocks")
    # K = 128 and 384 leave a half-filled 256-deep pair stage; 300 x 520 and 640 x 904 partial
    # tiles (and a partial 256-row pair tile)
    check_bs(M, N, K, a_fmt, b_fmt, block, seed=M + N + K + block, **KERNELS[kernel])


@pytest.mark.parametrize("variant,tile_n,pack", [(1, 0, False), (1, 0, True), (2, 0, True)])
@pytest.mark.parametrize("which", ["A rows", "B rows", "K-blocks"])
@pytest.mark.parametrize("block", [32, 128])
def test_scales_varying_along_one_axis(which, block, variant, tile_n, pack):
    if pack and variant == 1 and block == 128:
        pytest.skip("the one-CTA kernel repacks the scales of 32-element blocks only")
    if variant == 2 and block != 128:
        pytest.skip("the pair kernel takes 128-element scale blocks")
    # fp4 operands with every element code 2 (= 1.0); scales vary along one axis only, so any
    # mixing of rows or blocks in the scale layout changes some output
    M, N, K = 256, 448, 512
    kb = K // block
    A = workloads.pack_rows(np.full((M, K), 0x2, np.uint8), 4)
    B = workloads.pack_rows(np.full((N, K), 0x2, np.uint8), 4)
    sfA = np.full((M, kb), 127, np.uint8)
    sfB = np.full((N, kb), 127, np.uint8)
    rng = np.random.default_rng(block)
    if which == "A rows":
        sfA[:] = rng.integers(124, 131, (M, 1))
    elif which == "B rows":
        sfB[:] = rng.integers(124, 131, (N, 1))
    else:
        sfA[:] = rng.integers(124, 131, (1, kb))
    C = run_bs(A, B, sfA, sfB, "e2m1", "e2m1", block, variant=variant, tile_n=tile_n, pack=pack)
    ref = oracle.gemm_bs(A, B, sfA, sfB, M, N, K, a_fmt="e2m1", b_fmt="e2m1", block=block)
    assert np.array_equal(C, ref), which  # sums of powers of two: exact


def test_rows_of_larger_arrays():
    # packed rows inside wider arrays: the row strides go to the library as leading dimensions
    import dense_tensor_core_gb300 as dtc

    M, N, K = 264, 448, 384
    A, B, sfA, sfB = workloads.make_sub_byte(M, N, K, 21, "e2m1", "e3m2", 32)
    Ab = torch.zeros((M, A.shape[1] + 64), dtype=torch.uint8, device="cuda")
    Bb = torch.zeros((N, B.shape[1] + 96), dtype=torch.uint8, device="cuda")
    Ab[:, : A.shape[1]] = to_device8(A)
    Bb[:, : B.shape[1]] = to_device8(B)
    C = dtc.gemm_ex("mxfp8", Ab[:, : A.shape[1]], Bb[:, : B.shape[1]], sfA=to_device8(sfA),
                    sfB=to_device8(sfB), a_format="e2m1", b_format="e3m2", scale_block=32)
    dtc.gemm_stream_status()
    ref = oracle.gemm_bs(A, B, sfA, sfB, M, N, K, a_fmt="e2m1", b_fmt="e3m2", block=32)
    check_close(values16(C.view(torch.int16).cpu().numpy().view(np.uint16), "bf16"),
                values16(ref, "bf16"), "packed rows of larger arrays")


def test_packed_rule_violations_are_refused():
    import dense_tensor_core_gb300 as dtc

    A, B, sfA, sfB = workloads.make_sub_byte(128, 224, 192, 3, "e2m1", "e2m1", 32)
    with pytest.raises(dtc.GemmError) as e:  # K % 128 != 0
        dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), sfA=to_device8(sfA),
                    sfB=to_device8(sfB), a_format="e2m1", b_format="e2m1", scale_block=32)
    assert e.value.status == 1
    A, B, sfA, sfB = workloads.make_sub_byte(256, 448, 256, 3, "e2m1", "e2m1", 128)
    with pytest.raises(dtc.GemmError) as e:  # the pair kernel needs the workspace for its scales
        dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), sfA=to_device8(sfA),
                    sfB=to_device8(sfB), a_format="e2m1", b_format="e2m1", variant=2)
    assert e.value.status == 2


@pytest.mark.parametrize("variant,pack", [(1, False), (1, True)])
@pytest.mark.parametrize("name", ["mxfp4_b32_nt_4096x4096x8192",
                                  "mxfp6_e2m3_e3m2_b32_nt_4096x4096x8192"])
def test_benchmark_sizes_sampled(name, variant, pack):
    w = workloads.WORKLOADS[name]
    A, B, sfA, sfB = workloads.make(w)
    C = run_bs(A, B, sfA, sfB, w.a_fmt, w.b_fmt, w.block, variant=variant, pack=pack)
    r, c = sample_positions(w.M, w.N, count=3000, seed=w.seed, tile_n=224)
    r = np.concatenate([r, np.full(w.N, w.M // 3), np.arange(w.M)])
    c = np.concatenate([c, np.arange(w.N), np.full(w.M, w.N // 5)])
    ref, _ = oracle.gemm_bs_sampled(A, B, sfA, sfB, w.M, w.N, w.K, r, c, a_fmt=w.a_fmt,
                                    b_fmt=w.b_fmt, block=w.block)
    check_close(values16(C[r, c], "bf16"), values16(ref, "bf16"), name)
