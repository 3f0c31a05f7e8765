"""Every element of C at the benchmark workloads' full sizes, against the full CPU oracle.

Each product is launched the way the benchmark times it: the library's automatic plan, with the
workspace gemm_workspace_size asks for when it asks for one (block-scaled products also without). The oracle computes every
output (fp64 sums on all host cores, one rounding), so this is the complete parity check at the
sizes the performance figures are quoted on; the sampled checks in the other files cover the
forced kernel variants at these sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tensor_core_gb300 import workloads
from parity import check_close, to_device8, to_device16, values16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bench_launch16(w, A, B):
    import dense_tensor_core_gb300 as dtc

    kw = {}
    ws_bytes = dtc.gemm_workspace_size(w.kind, w.M, w.N, w.K, w.layout)
    if ws_bytes:
        kw = dict(workspace=torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda"))
    C = dtc.gemm_ex(w.kind, to_device16(A, w.kind), to_device16(B, w.kind), layout=w.layout, **kw)
    dtc.gemm_stream_status()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", [n for n, w in workloads.WORKLOADS.items() if w.kind in ("bf16", "f16")])
def test_16bit_workload_every_element(name):
    w = workloads.WORKLOADS[name]
    A, B = workloads.make(w)
    C = bench_launch16(w, A, B)
    ref = oracle.gemm16(w.kind, w.layout, A, B, w.M, w.N, w.K)
    check_close(values16(C, w.kind), values16(ref, w.kind), f"{name}, every element")


@pytest.mark.parametrize("name", [n for n, w in workloads.WORKLOADS.items() if w.kind == "mxfp8"])
def test_block_scaled_workload_every_element(name):
    import dense_tensor_core_gb300 as dtc

    w = workloads.WORKLOADS[name]
    A, B, sfA, sfB = workloads.make(w)
    fmt = dict(a_format=w.a_fmt, b_format=w.b_fmt, scale_block=w.block)
    ref = oracle.gemm_bs(A, B, sfA, sfB, w.M, w.N, w.K, a_fmt=w.a_fmt, b_fmt=w.b_fmt,
                         block=w.block)
    # without a workspace (scale warps) and with the one gemm_workspace_size asks for (repacked
    # scales, the plan the benchmark times)
    ws_bytes = dtc.gemm_workspace_size("mxfp8", w.M, w.N, w.K, **fmt)
    for ws in [None] + ([torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")] if ws_bytes else []):
        C = dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), sfA=to_device8(sfA),
                        sfB=to_device8(sfB), workspace=ws, **fmt)
        dtc.gemm_stream_status()
        C = C.view(torch.int16).cpu().numpy().view(np.uint16)
        check_close(values16(C, "bf16"), values16(ref, "bf16"),
                    f"{name}, every element, {'no workspace' if ws is None else 'workspace'}")


@pytest.mark.parametrize("name", [n for n, w in workloads.WORKLOADS.items() if w.kind.endswith("_sp24")])
def test_sparse_workload_every_element(name):
    import dense_tensor_core_gb300 as dtc

    w = workloads.WORKLOADS[name]
    kind = w.kind[:-5]
    vals, meta, B = workloads.make(w)
    C = dtc.gemm_sp(kind, to_device16(vals, kind), to_device8(meta), to_device16(B, kind),
                    layout=w.layout)
    dtc.gemm_stream_status()
    C = C.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.gemm_sp(kind, w.layout, vals, meta, B, w.M, w.N, w.K)
    check_close(values16(C, kind), values16(ref, kind), f"{name}, every element")
