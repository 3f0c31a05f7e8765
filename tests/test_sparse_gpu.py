"""GPU parity of the 2:4 structured-sparse product (gemm_sp) against the CPU oracle, through the C
ABI: the expansion kernel's dense A bit for bit, and C for both layouts of B, both 16-bit types
and every kernel variant of the dense product it runs on. The sparse GEMM is the one 05 Blackwell
TCGEN05 GEMM tutorial names in "An API-level note", read as the 2:4 pattern along K."""
import numpy as np
import pytest
import torch

import oracle
from dense_tensor_core_gb300 import workloads
from parity import check_close, sample_positions, to_device8, to_device16, values16
from test_oracle_sparse import decompress

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_sp(kind, layout, vals, meta, B, M, N, K, workspace=None, **kw):
    import dense_tensor_core_gb300 as dtc

    C = dtc.gemm_sp(kind, to_device16(vals, kind), to_device8(meta), to_device16(B, kind),
                    layout=layout, workspace=workspace, **kw)
    dtc.gemm_stream_status()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


def test_expansion_writes_the_dense_matrix():
    M, N, K = 300, 64, 528
    vals, meta, B = workloads.make_sp24("bf16", "NT", M, N, K, seed=1)
    ws = torch.full((M * K * 2,), 0xAB, dtype=torch.uint8, device="cuda")
    run_sp("bf16", "NT", vals, meta, B, M, N, K, workspace=ws)
    got = ws.cpu().numpy().view(np.uint16).reshape(M, K)
    assert np.array_equal(got, decompress(vals, meta, M, K))


VARIANTS = {"auto": {}, "1cta": dict(variant=1), "2cta": dict(variant=2),
            "splitk": dict(variant=3, split_k=2)}


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["NT", "NN"])
@pytest.mark.parametrize("M,N,K", [(256, 448, 512), (300, 520, 208), (1, 8, 16), (640, 768, 1024)])
def test_full_parity(M, N, K, layout, kind, variant):
    vals, meta, B = workloads.make_sp24(kind, layout, M, N, K, seed=M + N + K)
    C = run_sp(kind, layout, vals, meta, B, M, N, K, **VARIANTS[variant])
    ref = oracle.gemm_sp(kind, layout, vals, meta, B, M, N, K)
    check_close(values16(C, kind), values16(ref, kind), f"sparse {kind} {layout} {M}x{N}x{K}")


def test_equals_the_dense_product_of_the_expanded_matrix():
    import dense_tensor_core_gb300 as dtc

    M, N, K = 512, 512, 1024
    vals, meta, B = workloads.make_sp24("bf16", "NT", M, N, K, seed=7)
    C = run_sp("bf16", "NT", vals, meta, B, M, N, K)
    D = dtc.gemm_bf16(to_device16(decompress(vals, meta, M, K), "bf16"), to_device16(B, "bf16"))
    dtc.gemm_stream_status()
    assert np.array_equal(C, D.view(torch.int16).cpu().numpy().view(np.uint16))


def test_argument_errors():
    import dense_tensor_core_gb300 as dtc

    vals, meta, B = workloads.make_sp24("bf16", "NT", 64, 64, 128, seed=2)
    with pytest.raises(dtc.GemmError) as e:  # too small a workspace
        run_sp("bf16", "NT", vals, meta, B, 64, 64, 128,
               workspace=torch.empty(64 * 128, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 1
    v2, m2, B2 = workloads.make_sp24("bf16", "NT", 64, 64, 136, seed=2)  # K % 16 != 0
    with pytest.raises((dtc.GemmError, ValueError)):
        run_sp("bf16", "NT", v2, m2, B2, 64, 64, 136)


def test_benchmark_size_sampled():
    w = workloads.WORKLOADS["bf16_sp24_nt_4096x4096x8192"]
    vals, meta, B = workloads.make(w)
    C = run_sp("bf16", w.layout, vals, meta, B, w.M, w.N, w.K)
    r, c = sample_positions(w.M, w.N, count=2000, seed=w.seed)
    # a full row and a full column through the oracle's dense path on the decompressed rows
    dense = decompress(vals, meta, w.M, w.K)
    ref, _ = oracle.gemm16_sampled("bf16", w.layout, dense, B, w.M, w.N, w.K, r, c)
    check_close(values16(C[r, c], "bf16"), values16(ref, "bf16"), w.name)
    rows = np.array([w.M // 3])
    full = oracle.gemm_sp("bf16", w.layout, vals[rows], meta[rows], B, 1, w.N, w.K)
    check_close(values16(C[rows], "bf16"), values16(full, "bf16"), w.name + " row")
