"""ctypes binding of libdtc_gemm.so: argument marshalling only.

Each function takes torch CUDA tensors, checks dtype/shape/contiguity/device, passes raw device
pointers, sizes and the current (or given) stream to the C entry point of the same name, and
raises GemmError with the library's message on a non-OK status. Every arithmetic step runs in
the library's kernels.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libdtc_gemm.so")

GEMM_LAYOUT_NT, GEMM_LAYOUT_NN, GEMM_LAYOUT_TN, GEMM_LAYOUT_TT = 0, 1, 2, 3
_LAYOUTS = {"NT": 0, "NN": 1, "TN": 2, "TT": 3}
GEMM_VARIANT_AUTO, GEMM_VARIANT_1CTA, GEMM_VARIANT_2CTA, GEMM_VARIANT_SPLITK = 0, 1, 2, 3
_STATUS = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_UNSUPPORTED", 3: "GEMM_ERR_CUDA",
           4: "GEMM_ERR_TIMEOUT"}
_DTYPE = {"bf16": 0, "f16": 1, "mxfp8": 2}


class GemmError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class gemm_options(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("split_k", ctypes.c_int),
                ("timeout_ns", ctypes.c_uint64), ("fault_inject", ctypes.c_int),
                ("tile_n", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64),
                ("mx_a_format", ctypes.c_int), ("mx_b_format", ctypes.c_int),
                ("mx_scale_block", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_uint64), ("stream_k", ctypes.c_int)]


class gemm_plan_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("variant", "tile_m", "tile_n", "tile_k", "stages", "split_k", "ctas", "tiles",
                 "cluster", "sk_tiles", "sf_packed")]


class gemm_device_model(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("sm_count", "pair_clusters", "split2_clusters", "split4_clusters")]


# GB300: 152 SMs; clusters of 2 fill all 76 pairs; clusters of 4 fit 36 times
GB300_MODEL = dict(sm_count=152, pair_clusters=76, split2_clusters=76, split4_clusters=36)

_lib = None


def library_path():
    return _LIB_PATH


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with dense_tensor_core_gb300.build.build() "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        for name in ("gemm_bf16", "gemm_f16"):
            f = getattr(L, name)
            f.restype = i32
            f.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
        L.gemm_mxfp8.restype = i32
        L.gemm_mxfp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp]
        L.gemm_ex.restype = i32
        L.gemm_ex.argtypes = [i32, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                              ctypes.POINTER(gemm_options), vp]
        L.gemm_plan.restype = i32
        L.gemm_plan.argtypes = [i32, i64, i64, i64, i32, ctypes.POINTER(gemm_options),
                                ctypes.POINTER(gemm_plan_info)]
        L.gemm_plan_model.restype = i32
        L.gemm_plan_model.argtypes = [ctypes.POINTER(gemm_device_model), i32, i64, i64, i64, i32,
                                      ctypes.POINTER(gemm_options), ctypes.POINTER(gemm_plan_info)]
        L.gemm_device_model_query.restype = i32
        L.gemm_device_model_query.argtypes = [ctypes.POINTER(gemm_device_model)]
        L.gemm_ex_static_workspace.restype = i32
        L.gemm_ex_static_workspace.argtypes = [i32, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                               ctypes.POINTER(gemm_options), vp]
        L.gemm_sp.restype = i32
        L.gemm_sp.argtypes = [i32, vp, vp, vp, vp, i64, i64, i64, i32, ctypes.POINTER(gemm_options),
                              vp, ctypes.c_uint64, vp]
        L.gemm_sp_workspace_size.restype = i32
        L.gemm_sp_workspace_size.argtypes = [i32, i64, i64, ctypes.POINTER(ctypes.c_uint64)]
        L.gemm_nvfp4.restype = i32
        L.gemm_nvfp4.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.POINTER(gemm_options),
                                 vp, ctypes.c_uint64, vp]
        L.gemm_nvfp4_workspace_size.restype = i32
        L.gemm_nvfp4_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(ctypes.c_uint64)]
        L.gemm_workspace_size.restype = i32
        L.gemm_workspace_size.argtypes = [i32, i64, i64, i64, i32, ctypes.POINTER(gemm_options),
                                          ctypes.POINTER(ctypes.c_uint64)]
        L.gemm_last_error.restype = ctypes.c_char_p
        L.gemm_last_error.argtypes = []
        L.gemm_stream_status.restype = i32
        L.gemm_stream_status.argtypes = [vp]
        _lib = L
    return _lib


def gemm_last_error():
    return lib().gemm_last_error().decode(errors="replace")


def _check(status):
    if status != 0:
        raise GemmError(status, gemm_last_error())


def _stream_handle(stream, device=None):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _same_device(*tensors):
    """The one CUDA device all given tensors live on (the library works on the current device
    only, so the call is made with that device current)."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one CUDA device, got {sorted(map(str, devs))}")
    return devs.pop()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _layout_code(layout):
    if layout in _LAYOUTS:
        return _LAYOUTS[layout]
    if layout in _LAYOUTS.values():
        return layout
    raise ValueError(f"unknown layout {layout!r}: NT, NN, TN or TT")


def _layout_name(layout):
    code = _layout_code(layout)
    return next(k for k, v in _LAYOUTS.items() if v == code)


def _shapes16(A, B, layout):
    """(M, N, K) from the stored shapes: A is [M,K] or, for TN / TT, [K,M]; B is [N,K] for NT /
    TT, else [K,N]."""
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    name = _layout_name(layout)
    K, M = A.shape if name[0] == "T" else A.shape[::-1]
    N, Kb = B.shape if name[1] == "T" else B.shape[::-1]
    if Kb != K:
        raise ValueError(f"inner sizes differ: A is {tuple(A.shape)}, B is {tuple(B.shape)} ({name})")
    return M, N, K


def _check_tensor(t, dtype, name, rows_of_larger=False):
    """dtype and device checks; the tensor must be dense row-major, or, with rows_of_larger, may
    be rows of a larger row-major array (unit column stride, row stride >= its row length)."""
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.is_contiguous():
        return
    if rows_of_larger and t.dim() == 2 and t.stride(1) == 1 and t.stride(0) >= t.shape[1]:
        return
    raise ValueError(f"{name} must be dense row-major" +
                     (" or rows of a larger row-major array" if rows_of_larger else ""))


def _ld(t):
    """Leading dimension to pass: 0 (dense) unless the rows are further apart than their length."""
    if t is None or t.dim() != 2 or t.shape[0] <= 1 or t.stride(0) == t.shape[1]:
        return 0
    return t.stride(0)


def _out(C, M, N, dtype, device, rows_of_larger=False):
    if C is None:
        return torch.empty((M, N), dtype=dtype, device=device)
    _check_tensor(C, dtype, "C", rows_of_larger)
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    return C


_MX_FORMATS = {"e4m3": 0, "e5m2": 1, "e2m3": 2, "e3m2": 3, "e2m1": 4}
_MX_BITS = {"e4m3": 8, "e5m2": 8, "e2m3": 6, "e3m2": 6, "e2m1": 4}


def _options(variant, split_k, timeout_ns, fault_inject, tile_n=0, tile_k=0,
             lda=0, ldb=0, ldc=0, a_format="e4m3", b_format="e4m3", scale_block=0,
             workspace=None, stream_k=0):
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return gemm_options(variant, split_k, timeout_ns, fault_inject, tile_n, tile_k,
                        lda, ldb, ldc, _MX_FORMATS[a_format], _MX_FORMATS[b_format],
                        scale_block, ws_ptr, ws_bytes, stream_k)


def _gemm16(name, dtype, A, B, C, layout, stream):
    _check_tensor(A, dtype, "A")
    _check_tensor(B, dtype, "B")
    M, N, K = _shapes16(A, B, layout)
    C = _out(C, M, N, dtype, A.device)
    dev = _same_device(A, B, C)
    with torch.cuda.device(dev):
        _check(getattr(lib(), name)(_ptr(A), _ptr(B), _ptr(C), M, N, K, _layout_code(layout),
                                    _stream_handle(stream, dev)))
    return C


def gemm_bf16(A, B, C=None, layout="NT", stream=None):
    """C[M,N] = Aop . Bop; bf16 in/out. A is [M,K] (NT, NN) or [K,M] (TN, TT); B is [N,K] (NT,
    TT) or [K,N] (NN, TN); all dense row-major."""
    return _gemm16("gemm_bf16", torch.bfloat16, A, B, C, layout, stream)


def gemm_f16(A, B, C=None, layout="NT", stream=None):
    """As gemm_bf16 with fp16 operands and output."""
    return _gemm16("gemm_f16", torch.float16, A, B, C, layout, stream)


def _check_mxfp8(A, B, sfA, sfB, rows_of_larger=False, scale_block=128, a_format="e4m3",
                 b_format="e4m3"):
    """Shapes of a block-scaled call: A [M, row bytes] and B [N, row bytes] uint8 rows of element
    codes (fp8: one byte each; fp6 / fp4: packed), scales [rows, ceil(K / scale_block)]."""
    _check_tensor(A, torch.uint8, "A", rows_of_larger)
    _check_tensor(B, torch.uint8, "B", rows_of_larger)
    _check_tensor(sfA, torch.uint8, "sfA")
    _check_tensor(sfB, torch.uint8, "sfB")
    M, a_bytes = A.shape
    N, b_bytes = B.shape
    K = a_bytes * 8 // _MX_BITS[a_format]
    if a_bytes * 8 % _MX_BITS[a_format] or b_bytes * 8 != K * _MX_BITS[b_format]:
        raise ValueError(f"rows of {a_bytes} ({a_format}) and {b_bytes} ({b_format}) bytes do "
                         "not hold the same K")
    kb = (K + scale_block - 1) // scale_block
    if tuple(sfA.shape) != (M, kb) or tuple(sfB.shape) != (N, kb):
        raise ValueError(f"scales must be [M, {kb}] and [N, {kb}]")
    return M, N, K


def _ld_elems(t, fmt):
    """Leading dimension in elements of a uint8 tensor of packed rows (0 = dense)."""
    ld = _ld(t)
    return ld * 8 // _MX_BITS[fmt] if ld else 0


def gemm_mxfp8(A, B, sfA, sfB, C=None, stream=None):
    """Block-scaled e4m3 NT GEMM. A [M,K], B [N,K] e4m3 codes (uint8 tensors), sfA [M,ceil(K/128)],
    sfB [N,ceil(K/128)] E8M0 codes (uint8); C bf16 [M,N]."""
    M, N, K = _check_mxfp8(A, B, sfA, sfB)
    C = _out(C, M, N, torch.bfloat16, A.device)
    dev = _same_device(A, B, sfA, sfB, C)
    with torch.cuda.device(dev):
        _check(lib().gemm_mxfp8(_ptr(A), _ptr(B), _ptr(sfA), _ptr(sfB), _ptr(C), M, N, K,
                                _stream_handle(stream, dev)))
    return C


def gemm_ex(kind, A, B, C=None, layout="NT", sfA=None, sfB=None, variant=0, split_k=0,
            timeout_ns=0, fault_inject=0, tile_n=0, tile_k=0, stream=None,
            a_format="e4m3", b_format="e4m3", scale_block=0, workspace=None, stream_k=0):
    """Any of the three products with options (variant, split_k, wait limit, test hook). A, B
    and C may be rows of larger row-major arrays (e.g. ``big[:, :n]``); their row strides are
    passed as the leading dimensions. For the block-scaled product ("mxfp8") the element formats
    of A and B ("e4m3", "e5m2", "e2m3", "e3m2" or "e2m1"; fp6 / fp4 rows packed, K inferred from
    the row length) and the scale block (128, the default, or 32) may be chosen.
    `workspace` (a CUDA tensor of gemm_workspace_size bytes): for the 16-bit products the
    stream-K workspace (zero-filled before its first use; stream_k: 0 auto, 1 required, 2 off);
    for the block-scaled product the home of the repacked scales, which the pair kernel needs
    and the one-CTA kernel uses with 32-element blocks."""
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if kind == "mxfp8":
        M, N, K = _check_mxfp8(A, B, sfA, sfB, rows_of_larger=True,
                               scale_block=scale_block or 128, a_format=a_format,
                               b_format=b_format)
        C = _out(C, M, N, torch.bfloat16, A.device, rows_of_larger=True)
        lda, ldb = _ld_elems(A, a_format), _ld_elems(B, b_format)
    else:
        dt = torch.bfloat16 if kind == "bf16" else torch.float16
        _check_tensor(A, dt, "A", rows_of_larger=True)
        _check_tensor(B, dt, "B", rows_of_larger=True)
        M, N, K = _shapes16(A, B, layout)
        C = _out(C, M, N, dt, A.device, rows_of_larger=True)
        lda, ldb = _ld(A), _ld(B)
    opts = _options(variant, split_k, timeout_ns, fault_inject, tile_n, tile_k,
                    lda, ldb, _ld(C), a_format, b_format, scale_block, workspace, stream_k)
    dev = _same_device(A, B, C, sfA, sfB, workspace)
    with torch.cuda.device(dev):
        _check(lib().gemm_ex(_DTYPE[kind], _ptr(A), _ptr(B), _ptr(sfA), _ptr(sfB), _ptr(C), M, N,
                             K, _layout_code(layout), ctypes.byref(opts),
                             _stream_handle(stream, dev)))
    return C


def gemm_plan(kind, M, N, K, layout="NT", variant=0, split_k=0, tile_n=0, tile_k=0,
              a_format="e4m3", b_format="e4m3", scale_block=0, workspace=None, stream_k=0,
              model=None):
    """The launch the library would make for these sizes: a dict with variant, tile_m, tile_n,
    tile_k, stages, split_k, ctas, tiles, cluster, sk_tiles, sf_packed (raises GemmError if the
    call would be rejected). With `model` (a dict of gemm_device_model's fields, e.g. GB300_MODEL) the plan
    is made for that device description, without a GPU; otherwise for the current device."""
    opts = _options(variant, split_k, 0, 0, tile_n, tile_k, 0, 0, 0, a_format, b_format,
                    scale_block, workspace, stream_k)
    info = gemm_plan_info()
    if model is not None:
        m = gemm_device_model(**model)
        _check(lib().gemm_plan_model(ctypes.byref(m), _DTYPE[kind], M, N, K, _layout_code(layout),
                                     ctypes.byref(opts), ctypes.byref(info)))
    else:
        _check(lib().gemm_plan(_DTYPE[kind], M, N, K, _layout_code(layout), ctypes.byref(opts),
                               ctypes.byref(info)))
    return {n: getattr(info, n) for n, _ in gemm_plan_info._fields_}


def gemm_device_model_query():
    """The current device as the planner sees it (gemm_device_model's fields, as a dict)."""
    m = gemm_device_model()
    _check(lib().gemm_device_model_query(ctypes.byref(m)))
    return {n: getattr(m, n) for n, _ in gemm_device_model._fields_}


def gemm_stream_status(stream=None):
    """Synchronise the stream and raise GemmError if a device-side wait gave up."""
    _check(lib().gemm_stream_status(_stream_handle(stream)))


def gemm_workspace_size(kind, M, N, K, layout="NT", variant=0, tile_n=0, tile_k=0, stream_k=0,
                        a_format="e4m3", b_format="e4m3", scale_block=0):
    """Bytes of workspace the call can use: for the 16-bit products the stream-K workspace (0 if
    stream-K would not be used); for the block-scaled product the repacked scale arrays when the
    plan would use them (0 otherwise)."""
    opts = _options(variant, 0, 0, 0, tile_n, tile_k, a_format=a_format, b_format=b_format,
                    scale_block=scale_block, stream_k=stream_k)
    out = ctypes.c_uint64(0)
    _check(lib().gemm_workspace_size(_DTYPE[kind], M, N, K, _layout_code(layout),
                                     ctypes.byref(opts), ctypes.byref(out)))
    return out.value


def gemm_ex_static_workspace(kind, A, B, C=None, layout="NT", variant=0, tile_n=0, tile_k=0,
                             stream_k=0, stream=None, sfA=None, sfB=None, a_format="e4m3",
                             b_format="e4m3", scale_block=0):
    """gemm_ex with the library's own workspace (a region of module memory) instead of a caller's:
    allocates nothing. It serves stream-K of the 16-bit products and the repacked scales of the
    block-scaled product ("mxfp8": sfA / sfB and the formats as in gemm_ex). Calls on one device
    must not overlap (they share that region)."""
    if kind == "mxfp8":
        M, N, K = _check_mxfp8(A, B, sfA, sfB, rows_of_larger=True,
                               scale_block=scale_block or 128, a_format=a_format,
                               b_format=b_format)
        C = _out(C, M, N, torch.bfloat16, A.device, rows_of_larger=True)
        lda, ldb = _ld_elems(A, a_format), _ld_elems(B, b_format)
    else:
        dt = torch.bfloat16 if kind == "bf16" else torch.float16
        _check_tensor(A, dt, "A", rows_of_larger=True)
        _check_tensor(B, dt, "B", rows_of_larger=True)
        M, N, K = _shapes16(A, B, layout)
        C = _out(C, M, N, dt, A.device, rows_of_larger=True)
        lda, ldb = _ld(A), _ld(B)
    opts = _options(variant, 0, 0, 0, tile_n, tile_k, lda, ldb, _ld(C), a_format, b_format,
                    scale_block, stream_k=stream_k)
    dev = _same_device(A, B, C, sfA, sfB)
    with torch.cuda.device(dev):
        _check(lib().gemm_ex_static_workspace(_DTYPE[kind], _ptr(A), _ptr(B), _ptr(sfA), _ptr(sfB),
                                              _ptr(C), M, N, K, _layout_code(layout),
                                              ctypes.byref(opts), _stream_handle(stream, dev)))
    return C


def gemm_nvfp4_workspace_size(M, N, K):
    """Bytes of workspace gemm_nvfp4 needs (A and B expanded to bf16, A padded to 256 bytes)."""
    out = ctypes.c_uint64(0)
    _check(lib().gemm_nvfp4_workspace_size(M, N, K, ctypes.byref(out)))
    return out.value


def gemm_nvfp4(A, B, sfA, sfB, C=None, workspace=None, variant=0, split_k=0, tile_n=0, tile_k=0,
               stream_k=0, sk_workspace=None, timeout_ns=0, stream=None):
    """NVFP4 product, NT: A [M, K/2] and B [N, K/2] uint8 (packed e2m1 codes, element k in the
    low nibble of byte k/2 for even k), sfA [M, K/16] and sfB [N, K/16] uint8 (UE4M3 scales).
    `workspace` (gemm_nvfp4_workspace_size bytes of device memory) receives A and B expanded to
    bf16; it is allocated here when not given. `sk_workspace` is the bf16 product's stream-K
    workspace. Returns C [M,N] bf16."""
    for t, name in ((A, "A"), (B, "B"), (sfA, "sfA"), (sfB, "sfB")):
        _check_tensor(t, torch.uint8, name)
        if t.dim() != 2:
            raise ValueError(f"{name} must be 2-D")
    M, K = A.shape[0], 2 * A.shape[1]
    N = B.shape[0]
    if B.shape[1] * 2 != K:
        raise ValueError(f"B {tuple(B.shape)} does not match A {tuple(A.shape)}")
    if K % 16:
        raise ValueError(f"K = {K}: NVFP4 needs whole 16-element scale blocks")
    if tuple(sfA.shape) != (M, K // 16) or tuple(sfB.shape) != (N, K // 16):
        raise ValueError(f"sfA / sfB must be {(M, K // 16)} / {(N, K // 16)}, got "
                         f"{tuple(sfA.shape)} / {tuple(sfB.shape)}")
    C = _out(C, M, N, torch.bfloat16, A.device, rows_of_larger=True)
    if workspace is None:
        workspace = torch.empty(max(1, gemm_nvfp4_workspace_size(M, N, K)), dtype=torch.uint8,
                                device=A.device)
    opts = _options(variant, split_k, timeout_ns, 0, tile_n, tile_k, 0, 0, _ld(C),
                    workspace=sk_workspace, stream_k=stream_k)
    dev = _same_device(A, B, sfA, sfB, C, workspace, sk_workspace)
    with torch.cuda.device(dev):
        _check(lib().gemm_nvfp4(_ptr(A), _ptr(B), _ptr(sfA), _ptr(sfB), _ptr(C), M, N, K,
                                ctypes.byref(opts), _ptr(workspace),
                                workspace.numel() * workspace.element_size(),
                                _stream_handle(stream, dev)))
    return C


def gemm_sp_workspace_size(kind, M, K):
    """Bytes of workspace gemm_sp needs (the dense A it expands: M x K 16-bit elements)."""
    out = ctypes.c_uint64(0)
    _check(lib().gemm_sp_workspace_size(_DTYPE[kind], M, K, ctypes.byref(out)))
    return out.value


def gemm_sp(kind, vals, meta, B, C=None, layout="NT", workspace=None, variant=0, split_k=0,
            tile_n=0, tile_k=0, stream_k=0, sk_workspace=None, stream=None):
    """2:4 structured-sparse A times B: vals [M, K/2] ("bf16" or "f16"), meta [M, K/8] uint8
    (per group of 4 K-elements two 2-bit positions, two groups per byte), B [N,K] ("NT") or
    [K,N] ("NN"). `workspace` (M x K x 2 bytes of device memory) receives the expanded A; it is
    allocated here when not given. `sk_workspace` is the dense product's stream-K workspace."""
    dt = torch.bfloat16 if kind == "bf16" else torch.float16
    _check_tensor(vals, dt, "vals")
    _check_tensor(meta, torch.uint8, "meta")
    _check_tensor(B, dt, "B", rows_of_larger=True)
    if vals.dim() != 2 or meta.dim() != 2:
        raise ValueError("vals and meta must be 2-D")
    M, K = vals.shape[0], 2 * vals.shape[1]
    if tuple(meta.shape) != (M, K // 8):
        raise ValueError(f"meta must be [M, K/8] = {(M, K // 8)}, got {tuple(meta.shape)}")
    name = _layout_name(layout)
    N, Kb = (B.shape if name == "NT" else B.shape[::-1])
    if Kb != K:
        raise ValueError(f"B {tuple(B.shape)} does not match K = {K} ({name})")
    C = _out(C, M, N, dt, vals.device, rows_of_larger=True)
    if workspace is None:
        workspace = torch.empty(max(1, M * K * 2), dtype=torch.uint8, device=vals.device)
    opts = _options(variant, split_k, 0, 0, tile_n, tile_k, 0, _ld(B), _ld(C),
                    workspace=sk_workspace, stream_k=stream_k)
    dev = _same_device(vals, meta, B, C, workspace, sk_workspace)
    with torch.cuda.device(dev):
        _check(lib().gemm_sp(_DTYPE[kind], _ptr(vals), _ptr(meta), _ptr(B), _ptr(C), M, N, K,
                             _layout_code(layout), ctypes.byref(opts), _ptr(workspace),
                             workspace.numel() * workspace.element_size(),
                             _stream_handle(stream, dev)))
    return C
