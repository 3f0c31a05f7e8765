"""GPU parity of the NVFP4 product (gemm_nvfp4: e2m1 elements, one UE4M3 scale per 16 K-elements)
against the CPU oracle, through the C ABI: the expansion kernel's bf16 operands value for value,
C for every kernel variant of the bf16 product it runs on, ragged and degenerate shapes, NaN
scales, and sampled outputs of the full 4096 x 4096 x 8192 product. NVFP4 is the fp4 member of
the "other block-scaled formats" of the 05 Blackwell TCGEN05 GEMM tutorial, "Advanced"
(gemm_blockscaled)."""
import numpy as np
import pytest
import torch

import oracle
from dense_tensor_core_gb300 import workloads
from parity import check_close, sample_positions, to_device8, values16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run(A, B, sfA, sfB, workspace=None, **kw):
    import dense_tensor_core_gb300 as dtc

    C = dtc.gemm_nvfp4(to_device8(A), to_device8(B), to_device8(sfA), to_device8(sfB),
                       workspace=workspace, **kw)
    dtc.gemm_stream_status()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


def ref(A, B, sfA, sfB, M, N, K):
    return oracle.gemm_bs(A, B, sfA, sfB, M, N, K, a_fmt="e2m1", b_fmt="e2m1", scale="ue4m3",
                          block=16)


def expanded(codes, sf, rows, K):
    """The oracle's value of every element times its scale (float64; exact in bf16)."""
    nib = np.empty((rows, K), np.uint8)
    nib[:, 0::2] = codes & 15
    nib[:, 1::2] = codes >> 4
    v = oracle.dec_e2m1(nib).reshape(rows, K)
    s = oracle.dec_ue4m3(sf).reshape(rows, K // 16)
    return v * np.repeat(s, 16, axis=1)


def test_expansion_is_exact():
    import dense_tensor_core_gb300 as dtc

    M, N, K = 300, 200, 528
    A, B, sfA, sfB = workloads.make_nvfp4(M, N, K, seed=1)
    # every scale class: zero, the smallest and largest subnormals, the smallest normal, the
    # largest value, and the two kinds of NaN (the e4m3 NaN code and a set sign bit)
    specials = np.array([0x00, 0x01, 0x07, 0x08, 0x7E, 0x7F, 0x80, 0xB5], np.uint8)
    sfA[:8, 0] = specials
    sfB[-8:, -1] = specials
    ws = torch.full((dtc.gemm_nvfp4_workspace_size(M, N, K),), 0xAB, dtype=torch.uint8,
                    device="cuda")
    run(A, B, sfA, sfB, workspace=ws)
    off = (M * K * 2 + 255) // 256 * 256
    raw = ws.cpu().numpy()
    for got_bytes, codes, sf, rows in ((raw[: M * K * 2], A, sfA, M),
                                       (raw[off: off + N * K * 2], B, sfB, N)):
        got = values16(got_bytes.view(np.uint16).reshape(rows, K), "bf16")
        want = expanded(codes, sf, rows, K)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], want[~nan])  # exact: every product fits bf16


VARIANTS = {"auto": {}, "1cta": dict(variant=1), "2cta": dict(variant=2),
            "splitk": dict(variant=3, split_k=2)}


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("M,N,K", [(256, 448, 512), (300, 520, 208), (1, 8, 16), (640, 768, 1024)])
def test_full_parity(M, N, K, variant):
    A, B, sfA, sfB = workloads.make_nvfp4(M, N, K, seed=M + N + K)
    C = run(A, B, sfA, sfB, **VARIANTS[variant])
    check_close(values16(C, "bf16"), values16(ref(A, B, sfA, sfB, M, N, K), "bf16"),
                f"nvfp4 {M}x{N}x{K} {variant}")


def test_equals_the_bf16_product_of_the_expanded_operands():
    import dense_tensor_core_gb300 as dtc

    M, N, K = 512, 384, 1024
    A, B, sfA, sfB = workloads.make_nvfp4(M, N, K, seed=5)
    ws = torch.empty(dtc.gemm_nvfp4_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    C = run(A, B, sfA, sfB, workspace=ws)
    off = (M * K * 2 + 255) // 256 * 256
    Ae = ws[: M * K * 2].view(torch.bfloat16).view(M, K)
    Be = ws[off: off + N * K * 2].view(torch.bfloat16).view(N, K)
    D = dtc.gemm_bf16(Ae, Be)
    dtc.gemm_stream_status()
    assert np.array_equal(C, D.view(torch.int16).cpu().numpy().view(np.uint16))


def test_nan_scales_give_nan_rows_and_columns():
    M, N, K = 128, 256, 256
    A, B, sfA, sfB = workloads.make_nvfp4(M, N, K, seed=3)
    sfA[5, 3] = 0x80   # sign bit set: not a UE4M3 value
    sfB[17, 0] = 0x7F  # the e4m3 NaN code
    C = values16(run(A, B, sfA, sfB), "bf16")
    R = values16(ref(A, B, sfA, sfB, M, N, K), "bf16")
    assert np.isnan(R[5]).all() and np.isnan(R[:, 17]).all()
    assert np.array_equal(np.isnan(C), np.isnan(R))
    ok = ~np.isnan(R)
    check_close(C[ok], R[ok], "nvfp4 with NaN scales")


def test_degenerate_shapes():
    import dense_tensor_core_gb300 as dtc

    A, B, sfA, sfB = workloads.make_nvfp4(64, 32, 0, seed=0)  # K = 0: the empty sum
    C = torch.full((64, 32), 7.0, dtype=torch.bfloat16, device="cuda")
    dtc.gemm_nvfp4(to_device8(A), to_device8(B), to_device8(sfA), to_device8(sfB), C=C)
    dtc.gemm_stream_status()
    assert torch.count_nonzero(C).item() == 0
    A, B, sfA, sfB = workloads.make_nvfp4(0, 32, 64, seed=0)  # M = 0: nothing to do
    out = dtc.gemm_nvfp4(to_device8(A), to_device8(B), to_device8(sfA), to_device8(sfB))
    assert tuple(out.shape) == (0, 32)


def test_full_size_sampled():
    """The benchmark's workload (4096 x 4096 x 8192, the automatic plan, a stream-K workspace as
    the benchmark passes) on outputs the oracle computes one by one."""
    import dense_tensor_core_gb300 as dtc

    w = workloads.WORKLOADS["nvfp4_nt_4096x4096x8192"]
    A, B, sfA, sfB = workloads.make(w)
    sk = torch.zeros(max(1, dtc.gemm_workspace_size("bf16", w.M, w.N, w.K)), dtype=torch.uint8,
                     device="cuda")
    C = run(A, B, sfA, sfB, sk_workspace=sk)
    rows, cols = sample_positions(w.M, w.N, count=1024, seed=12)
    R, _ = oracle.gemm_bs_sampled(A, B, sfA, sfB, w.M, w.N, w.K, rows, cols, a_fmt="e2m1",
                                  b_fmt="e2m1", scale="ue4m3", block=16)
    check_close(values16(C[rows, cols], "bf16"), values16(R, "bf16"), "nvfp4 4096x4096x8192")


def test_argument_errors():
    import dense_tensor_core_gb300 as dtc

    A, B, sfA, sfB = workloads.make_nvfp4(64, 64, 128, seed=2)
    with pytest.raises(dtc.GemmError) as e:  # too small a workspace
        run(A, B, sfA, sfB, workspace=torch.empty(64 * 128, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 1


def test_c_rows_of_a_larger_array():
    # C as a view into a wider row-major array: ldc goes to the bf16 product; the padding columns
    # stay untouched
    import dense_tensor_core_gb300 as dtc

    M, N, K = 200, 264, 320
    A, B, sfA, sfB = workloads.make_nvfp4(M, N, K, seed=9)
    Cb = torch.full((M, N + 40), float("nan"), dtype=torch.bfloat16, device="cuda")
    dtc.gemm_nvfp4(to_device8(A), to_device8(B), to_device8(sfA), to_device8(sfB), C=Cb[:, :N])
    dtc.gemm_stream_status()
    assert torch.isnan(Cb[:, N:].float()).all(), "padding columns of C were written"
    C = Cb[:, :N].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    check_close(values16(C, "bf16"), values16(ref(A, B, sfA, sfB, M, N, K), "bf16"),
                "nvfp4 into rows of a larger C")
