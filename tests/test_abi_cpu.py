"""The C ABI without a GPU: the library loads, exports every function include/dtc_gemm.h
declares, and rejects bad arguments before making any CUDA call."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = []
    for h in sorted(os.listdir(HEADER_DIR)):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(HEADER_DIR, h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = re.sub(r"typedef[^;]*;", "", src, flags=re.S)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\([^;{]*\)\s*;", src):
            names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def L():
    from dense_tensor_core_gb300 import _binding, build

    build.build()
    return _binding.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gemm_bf16", "gemm_f16", "gemm_mxfp8", "gemm_ex", "gemm_plan", "gemm_last_error",
              "gemm_stream_status", "gemm_nvfp4", "gemm_nvfp4_workspace_size"):
        assert n in names


CITATIONS = ("TileLang SM100 Support", "tilelang (velog)", "05 Blackwell TCGEN05 GEMM",
             "pages have no counterpart")


def test_every_declaration_cites_its_passage():
    # each entry point's comment names the page passage that defines it, or says that the pages
    # have none
    for h in sorted(os.listdir(HEADER_DIR)):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(HEADER_DIR, h)).read()
        for name in declared_functions():
            m = re.search(r"\b(?:int|const char\*)\s+" + name + r"\s*\(", src)
            if not m:
                continue
            start = src.rfind("*/", 0, m.start())
            open_ = src.rfind("/*", 0, start)
            comment = " ".join(re.sub(r"\n\s*\*(?!/)", " ", src[open_:start]).split())
            assert any(c in comment for c in CITATIONS), f"{name}: no citation in {comment[:80]!r}"


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} is declared in include/ but not exported"


def _call16(L, name, A=0x1000, B=0x2000, C=0x3000, M=16, N=16, K=16, layout=0):
    return getattr(L, name)(ctypes.c_void_p(A), ctypes.c_void_p(B), ctypes.c_void_p(C), M, N, K,
                            layout, None)


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("name", ["gemm_bf16", "gemm_f16"])
@pytest.mark.parametrize(
    "kw",
    [
        dict(layout=4),
        dict(layout=-1),
        dict(M=-1),
        dict(K=-8),
        dict(N=2 ** 31),
        dict(A=0),
        dict(B=0),
        dict(C=0),
        dict(A=0x1008),  # 8-byte aligned only
        dict(C=0x3004),
        dict(K=12),  # A rows of 24 bytes
        dict(N=12),  # C rows of 24 bytes
        dict(N=12, layout=1),
        dict(M=12, layout=2),  # TN: A stored [K,M], rows of 24 bytes
        dict(M=12, layout=3),
        dict(N=12, layout=2),  # TN: B stored [K,N]
        dict(K=12, layout=3),  # TT: B stored [N,K]
    ],
)
def test_invalid_arguments_rejected_before_cuda(L, name, kw):
    assert _call16(L, name, **kw) == INVALID
    assert L.gemm_last_error()  # a message is left for the caller


def test_empty_output_is_a_no_op(L):
    assert _call16(L, "gemm_bf16", A=0, B=0, C=0, M=0) == 0
    assert _call16(L, "gemm_f16", A=0, B=0, C=0, N=0, layout=1) == 0


def test_mxfp8_rules(L):
    vp = ctypes.c_void_p
    # K must keep e4m3 rows 16-byte aligned
    assert L.gemm_mxfp8(vp(0x1000), vp(0x2000), vp(0x10), vp(0x20), vp(0x3000), 16, 16, 24, None) == INVALID
    # scale arrays are required
    assert L.gemm_mxfp8(vp(0x1000), vp(0x2000), vp(0), vp(0x20), vp(0x3000), 16, 16, 32, None) == INVALID
    # NN is not offered for the block-scaled product
    rc = L.gemm_ex(2, vp(0x1000), vp(0x2000), vp(0x10), vp(0x20), vp(0x3000), 16, 16, 32, 1, None, None)
    assert rc == UNSUPPORTED


@pytest.mark.parametrize(
    "ld,layout",
    [
        (dict(lda=8), 0),    # below K = 16
        (dict(ldb=8), 0),
        (dict(ldc=8), 0),    # below N = 16
        (dict(lda=20), 0),   # 40-byte rows: not 16-byte aligned
        (dict(ldc=20), 0),
        (dict(ldb=20), 1),
        (dict(lda=-16), 0),
        (dict(lda=2 ** 31), 2),
        (dict(lda=8), 2),    # TN: A rows hold M = 16 elements
    ],
)
def test_leading_dimensions_rejected_before_cuda(L, ld, layout):
    from dense_tensor_core_gb300._binding import gemm_options

    vp = ctypes.c_void_p
    o = gemm_options()
    for k, v in ld.items():
        setattr(o, k, v)
    rc = L.gemm_ex(0, vp(0x1000), vp(0x2000), None, None, vp(0x3000), 16, 16, 16, layout,
                   ctypes.byref(o), None)
    assert rc == INVALID
    assert L.gemm_last_error()


@pytest.mark.parametrize("dtype,opt", [(0, dict(mx_a_format=1)), (1, dict(mx_scale_block=32)),
                                       (2, dict(mx_b_format=2)), (2, dict(mx_scale_block=64)),
                                       (2, dict(mx_a_format=-1))])
def test_block_scaled_options_rejected_before_cuda(L, dtype, opt):
    from dense_tensor_core_gb300._binding import gemm_options

    vp = ctypes.c_void_p
    o = gemm_options()
    for k, v in opt.items():
        setattr(o, k, v)
    rc = L.gemm_ex(dtype, vp(0x1000), vp(0x2000), vp(0x10), vp(0x20), vp(0x3000), 16, 16, 32, 0,
                   ctypes.byref(o), None)
    assert rc == INVALID
    assert L.gemm_last_error()


def _nvfp4(L, A=0x1000, B=0x2000, sfA=0x10, sfB=0x20, C=0x3000, M=16, N=16, K=32, opts=None,
           ws=0x40000, ws_bytes=1 << 20):
    vp = ctypes.c_void_p
    return L.gemm_nvfp4(vp(A), vp(B), vp(sfA), vp(sfB), vp(C), M, N, K,
                        ctypes.byref(opts) if opts is not None else None, vp(ws), ws_bytes, None)


@pytest.mark.parametrize("kw", [
    dict(K=24),             # not whole 16-element scale blocks
    dict(K=-16),
    dict(A=0),
    dict(sfB=0),
    dict(A=0x1008),         # packed rows must start 16-byte aligned
    dict(C=0),
    dict(ws=0),             # no workspace
    dict(ws=0x40008),       # misaligned workspace
    dict(ws_bytes=2047),    # one byte short: 16 x 32 x 2 for A padded to 1024, + 1024 for B
    dict(N=12),             # C rows of 24 bytes
])
def test_nvfp4_rules(L, kw):
    assert _nvfp4(L, **kw) == INVALID
    assert L.gemm_last_error()


@pytest.mark.parametrize("opt", [dict(lda=16), dict(ldb=32), dict(mx_scale_block=16),
                                 dict(mx_a_format=4)])
def test_nvfp4_rejects_options_that_do_not_apply(L, opt):
    from dense_tensor_core_gb300._binding import gemm_options

    o = gemm_options()
    for k, v in opt.items():
        setattr(o, k, v)
    assert _nvfp4(L, opts=o) == INVALID


def test_nvfp4_empty_output_and_workspace_size(L):
    assert _nvfp4(L, A=0, B=0, sfA=0, sfB=0, C=0, M=0, ws=0, ws_bytes=0) == 0
    out = ctypes.c_uint64(0)
    assert L.gemm_nvfp4_workspace_size(16, 16, 32, ctypes.byref(out)) == 0
    assert out.value == 2048  # A: 16 x 32 x 2 = 1024 (already a multiple of 256), B: 1024
    assert L.gemm_nvfp4_workspace_size(3, 5, 16, ctypes.byref(out)) == 0
    assert out.value == 256 + 5 * 16 * 2  # A's 96 bytes padded to 256
    assert L.gemm_nvfp4_workspace_size(-1, 5, 16, ctypes.byref(out)) == INVALID


def test_static_workspace_entry_refuses_a_caller_workspace(L):
    from dense_tensor_core_gb300._binding import gemm_options

    vp = ctypes.c_void_p
    o = gemm_options()
    o.workspace = 0x4000
    o.workspace_bytes = 1 << 20
    rc = L.gemm_ex_static_workspace(0, vp(0x1000), vp(0x2000), None, None, vp(0x3000), 16, 16, 16,
                                    0, ctypes.byref(o), None)
    assert rc == INVALID
    assert L.gemm_last_error()


def test_options_struct_matches_header():
    # the binding's ctypes mirror of gemm_options lists the header's fields in order
    from dense_tensor_core_gb300._binding import gemm_options

    with open(os.path.join(ROOT, "include", "dtc_gemm.h")) as f:
        text = f.read()
    body = text[text.index("typedef struct {", text.index("gemm_variant;")):]
    body = body[: body.index("} gemm_options;")]
    fields = re.findall(r"^\s*(?:int|uint64_t|int64_t|void\*)\s+(\w+);", body, re.M)
    assert fields == [n for n, _ in gemm_options._fields_]


def test_binding_checks_tensors_without_gpu():
    import torch

    import dense_tensor_core_gb300 as dtc

    A = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises((ValueError, TypeError)):
        dtc.gemm_bf16(A, A)  # CPU tensors are refused before any call
    with pytest.raises(TypeError):
        dtc.gemm_f16(A, A)
