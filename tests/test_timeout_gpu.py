"""Failure detection on the GPU without a fault: the load producer's test hook skips its first
stage, so nothing ever completes that stage's barrier. The consumer's bounded wait must give up
after the requested limit, the kernel must release its Tensor Memory and return, the status must
read GEMM_ERR_TIMEOUT, and the next normal call on the same context must succeed."""
import time

import numpy as np
import pytest
import torch

import oracle
from dense_tensor_core_gb300 import workloads
from parity import check_close, to_device16, values16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("variant,split_k", [(1, 0), (2, 0), (3, 0), (3, 1)])
def test_wait_that_nothing_completes_reports_timeout_then_recovers(variant, split_k):
    # (3, 1): the split-K kernel's unsplit mode, which tears down without acknowledgements
    import dense_tensor_core_gb300 as dtc

    M, N, K = 512, 512, 512
    A, B = workloads.make16("bf16", "NT", M, N, K, 9)
    At, Bt = to_device16(A, "bf16"), to_device16(B, "bf16")
    dtc.gemm_stream_status()  # start from a clear status word
    t0 = time.time()
    dtc.gemm_ex("bf16", At, Bt, variant=variant, split_k=split_k, timeout_ns=20_000_000,
                fault_inject=1)
    with pytest.raises(dtc.GemmError) as e:
        dtc.gemm_stream_status()
    assert e.value.status == 4  # GEMM_ERR_TIMEOUT
    assert time.time() - t0 < 30
    dtc.gemm_stream_status()  # the status word was cleared by the report
    C = dtc.gemm_ex("bf16", At, Bt, variant=variant, split_k=split_k)
    dtc.gemm_stream_status()
    ref = oracle.gemm16("bf16", "NT", A, B, M, N, K)
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    check_close(values16(got, "bf16"), values16(ref, "bf16"), "after timeout")


def test_stream_k_timeout_reports_and_recovers():
    # a pair that never gets its first stage times out; the pairs waiting for its stream-K piece
    # give up too (bounded), the call reports GEMM_ERR_TIMEOUT, and after the workspace is zeroed
    # the next call is correct
    import dense_tensor_core_gb300 as dtc

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the shape is chosen for 76 pairs")
    M, N, K = 2560, 2560, 512
    nbytes = dtc.gemm_workspace_size("bf16", M, N, K, stream_k=1)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    Ah, Bh = workloads.make16("bf16", "NT", M, N, K, seed=5)
    A, B = to_device16(Ah, "bf16"), to_device16(Bh, "bf16")
    dtc.gemm_stream_status()
    dtc.gemm_ex("bf16", A, B, workspace=ws, stream_k=1, timeout_ns=20_000_000, fault_inject=1)
    with pytest.raises(dtc.GemmError) as e:
        dtc.gemm_stream_status()
    assert e.value.status == 4
    ws.zero_()
    C = dtc.gemm_ex("bf16", A, B, workspace=ws, stream_k=1)
    dtc.gemm_stream_status()
    ref = oracle.gemm16("bf16", "NT", Ah, Bh, M, N, K)
    check_close(values16(C.view(torch.int16).cpu().numpy().view(np.uint16), "bf16"),
                values16(ref, "bf16"), "stream-K after a timeout")
