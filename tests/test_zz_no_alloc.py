"""gemm_ex_static_workspace, the entry point that allocates nothing (its stream-K workspace is a
region of module memory), against gemm_ex with a workspace the caller allocated: two calls in a
row each, outputs bit for bit equal. Named to be collected last; it also passes alone."""
import pytest
import torch


def allocations():
    """torch's cumulative count of device allocation requests: a call that allocates nothing
    leaves it unchanged, and unlike the bytes in use it does not move when the garbage collector
    frees an earlier test's tensors meanwhile."""
    return torch.cuda.memory_stats().get("allocation.all.allocated", 0)

from dense_tensor_core_gb300 import workloads
from parity import to_device16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("M,N,K,layout,stream_k", [
    (2560, 2560, 1024, "NT", 1),  # 100 pair tiles: one wave, 24 tiles shared out by stream-K
    (2304, 2560, 640, "TN", 1),   # A stored [K,M]; 90 tiles
    (1024, 1024, 512, "NT", 0),   # no stream-K: the plain path, the region unused
])
def test_static_workspace_matches_caller_workspace_two_calls(M, N, K, layout, stream_k):
    import dense_tensor_core_gb300 as dtc

    if stream_k and torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the shapes are chosen for 76 pairs")
    A, B = workloads.make16("bf16", layout, M, N, K, seed=M + N + K)
    At, Bt = to_device16(A, "bf16"), to_device16(B, "bf16")
    nbytes = dtc.gemm_workspace_size("bf16", M, N, K, layout, stream_k=stream_k)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    C_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C_own = torch.empty_like(C_ref)
    for call in range(2):
        C_ref.fill_(float("nan"))
        C_own.fill_(float("nan"))
        dtc.gemm_ex("bf16", At, Bt, C_ref, layout=layout, workspace=ws if nbytes else None,
                    stream_k=stream_k)
        before = allocations()
        dtc.gemm_ex_static_workspace("bf16", At, Bt, C_own, layout=layout, stream_k=stream_k)
        assert allocations() == before  # nothing allocated through torch either
        dtc.gemm_stream_status()
        assert torch.equal(C_ref.view(torch.int16), C_own.view(torch.int16)), f"call {call}"


@pytest.mark.parametrize("variant,block", [(1, 32), (2, 128)])
def test_static_workspace_holds_repacked_scales(variant, block):
    # 32-element scale blocks on the one-CTA kernel, and the pair kernel with 128-element ones:
    # the scales are repacked into the library's region instead of a caller's workspace; bit for
    # bit equal, two calls
    import numpy as np

    import dense_tensor_core_gb300 as dtc
    from parity import to_device8

    M, N, K = 640, 904, 1024
    A, B, sfA, sfB = workloads.make_mx(M, N, K, 12, block=block)
    At, Bt, sAt, sBt = (to_device8(x) for x in (A, B, sfA, sfB))
    nbytes = dtc.gemm_workspace_size("mxfp8", M, N, K, variant=variant, scale_block=block)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert dtc.gemm_plan("mxfp8", M, N, K, variant=variant, scale_block=block, workspace=ws)["sf_packed"] == 1
    C_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C_own = torch.empty_like(C_ref)
    for call in range(2):
        C_ref.fill_(float("nan"))
        C_own.fill_(float("nan"))
        dtc.gemm_ex("mxfp8", At, Bt, C_ref, sfA=sAt, sfB=sBt, scale_block=block, variant=variant,
                    workspace=ws)
        before = allocations()
        dtc.gemm_ex_static_workspace("mxfp8", At, Bt, C_own, sfA=sAt, sfB=sBt, scale_block=block,
                                     variant=variant)
        assert allocations() == before
        dtc.gemm_stream_status()
        assert torch.equal(C_ref.view(torch.int16), C_own.view(torch.int16)), f"call {call}"
    assert not np.isnan(C_own.float().cpu().numpy()).any()
