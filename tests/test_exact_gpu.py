"""GPU parity at the special values and closed forms the oracle is pinned with, through every
16-bit kernel (one-CTA, CTA pair, split-K in 2 and 4, stream-K) and the block-scaled kernel.

* fp16 output overflow: the header promises IEEE round-to-nearest-even with overflow to +-inf (the
  generated kernel of tilelang (velog) section 1.3 casts the fp32 accumulator to half). Operands
  are small integers, so every fp32 partial sum is exact whatever the summation order, and the
  kernels' output must equal the oracle's bit for bit, infinities included: sums of 65504 stay
  finite, 65505..65519 round down to 65504, 65520 (the tie between 65504 and the first value past
  the format, which rounds to even) and beyond become inf.
* Closed forms: all-ones operands give C = K exactly (K a power of two); A = I gives C = Bop
  exactly, in all four storage layouts.
* MXFP8: max |C - ref| against K from 128 to 8192 (one scale per 128 or 32 K-elements), the early
  warning for reduced-precision accumulation inside the block-scaled MMA; set DTC_KSWEEP_OUT to a
  file path to have the curve appended there as JSON lines.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from dense_tensor_core_gb300 import workloads
from parity import check_close, to_device8, to_device16, values16, with_packed_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _codes(values, kind):
    """float64 values (exactly representable) -> uint16 codes of bf16/fp16."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float64)).to(
        torch.bfloat16 if kind == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _run(kind, layout, A, B, M, N, K, **kw):
    import dense_tensor_core_gb300 as dtc

    C = dtc.gemm_ex(kind, to_device16(A, kind), to_device16(B, kind), layout=layout, **kw)
    dtc.gemm_stream_status()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


def _store(op_mk, layout_letter):
    """The stored array of an operand given as [rows, K]: K-major [rows, K] ("N" for A, "T" for
    B) or MN-major [K, rows]."""
    return np.ascontiguousarray(op_mk if layout_letter == "K" else op_mk.T)


def _stored(layout, a_mk, b_nk):
    """A and B as the layout stores them, from A as [M,K] and B as [N,K]."""
    A = _store(a_mk, "M" if layout[0] == "T" else "K")
    B = _store(b_nk, "K" if layout[1] == "T" else "M")
    return A, B


# The kernels under test: (name, gemm_ex options, whether it needs the 152-SM GB300 shapes).
KERNELS = [
    ("1cta", dict(variant=1), False),
    ("2cta", dict(variant=2), False),
    ("splitk2", dict(variant=3, split_k=2), False),
    ("splitk4", dict(variant=3, split_k=4, tile_n=128), False),
    ("streamk", dict(stream_k=1), True),
]


def _kernel_kw(name, kind, M, N, K, layout):
    import dense_tensor_core_gb300 as dtc

    kw = dict(next(k[1] for k in KERNELS if k[0] == name))
    if name == "streamk":
        if torch.cuda.get_device_properties(0).multi_processor_count != 152:
            pytest.skip("the stream-K shape is chosen for 76 pairs")
        nbytes = dtc.gemm_workspace_size(kind, M, N, K, layout, stream_k=1)
        kw["workspace"] = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    return kw


def _shape(name):
    # stream-K needs more pair tiles than pairs, and a part-full last wave (100 tiles of 256 x 256)
    return (2560, 2560, 1024) if name == "streamk" else (256, 520, 2048)


# --- fp16 overflow ------------------------------------------------------------------------------

TARGETS = [65504, 65505, 65511, 65512, 65519, 65520, 65521, 65535, 65536, 70000, 131072, 1000,
           -65504, -65519, -65520, -70000, 12345, 0, 32768, 65488, 65496, 65503]


def _overflow_operands(M, N, K, seed):
    """A [M,K] of +-1 (rows of all +1, all -1, and random signs), B [N,K] of small integers whose
    row n sums to a target near the fp16 limit: C[m,n] is +-target on the uniform rows and an
    integer of either sign elsewhere."""
    rng = np.random.default_rng(seed)
    a = rng.choice([-1.0, 1.0], size=(M, K))
    a[0::4] = 1.0
    a[1::4] = -1.0
    b = np.zeros((N, K))
    for n in range(N):
        t = TARGETS[n % len(TARGETS)] if n < 2 * len(TARGETS) else int(rng.integers(-90000, 90000))
        base, rem = divmod(abs(t), K)  # K parts of base or base + 1
        parts = np.full(K, float(base))
        parts[:rem] += 1.0
        b[n] = np.sign(t) * rng.permutation(parts) if t else 0.0
    assert np.abs(b).max() <= 2048  # integers of at most 2048 are exact in fp16
    return a, b


@pytest.mark.parametrize("layout", ["NT", "NN", "TN", "TT"])
@pytest.mark.parametrize("name", [k[0] for k in KERNELS])
def test_fp16_overflow_to_inf_bit_exact(name, layout):
    M, N, K = _shape(name)
    a, b = _overflow_operands(M, N, K, seed=len(name) + K)
    A, B = _stored(layout, _codes(a, "f16"), _codes(b, "f16"))
    ref = oracle.gemm16("f16", layout, A, B, M, N, K)
    vals = values16(ref, "f16")
    assert np.isposinf(vals).any() and np.isneginf(vals).any() and (vals == 65504).any()
    got = _run("f16", layout, A, B, M, N, K, **_kernel_kw(name, "f16", M, N, K, layout))
    check_close(values16(got, "f16"), vals, f"fp16 overflow, {name} {layout}")
    assert np.array_equal(got, ref), f"{name} {layout}: not bit-equal to the oracle"


# --- closed forms -------------------------------------------------------------------------------

@pytest.mark.parametrize("K", [512, 1024, 8192])
@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("name", [k[0] for k in KERNELS])
def test_all_ones_gives_K_exactly(name, kind, K):
    M, N = (2560, 2560) if name == "streamk" else (256, 520)
    if name == "streamk" and K % 64:
        pytest.skip("stream-K needs K % 64 == 0")
    A = _codes(np.ones((M, K)), kind)
    B = _codes(np.ones((N, K)), kind)
    ref = oracle.gemm16(kind, "NT", A, B, M, N, K)
    assert (values16(ref, kind) == K).all()
    got = _run(kind, "NT", A, B, M, N, K, **_kernel_kw(name, kind, M, N, K, "NT"))
    assert np.array_equal(got, ref), f"{name}: all-ones product is not C = {K} everywhere"


@pytest.mark.parametrize("layout", ["NT", "NN", "TN", "TT"])
@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("name", [k[0] for k in KERNELS])
def test_identity_gives_bop_exactly(name, kind, layout):
    M, N, K = (2560, 2560, 2560) if name == "streamk" else (512, 776, 512)
    eye = _codes(np.eye(M, K), kind)
    _, b = workloads.make16(kind, "NT", 8, N, K, seed=M + N)  # B [N,K], N(0,1) draws
    A, B = _stored(layout, eye, b)
    ref = oracle.gemm16(kind, layout, A, B, M, N, K)
    assert np.array_equal(ref, np.ascontiguousarray(b.T[:M]))  # C = Bop, as the oracle's pin says
    got = _run(kind, layout, A, B, M, N, K, **_kernel_kw(name, kind, M, N, K, layout))
    assert np.array_equal(got, ref), f"{name} {layout}: A = I does not give C = Bop"


# --- MXFP8 error against K ----------------------------------------------------------------------

SWEEP_K = [128, 256, 512, 1024, 2048, 4096, 8192]


@pytest.mark.parametrize("block,variant", [(128, 1), (128, 2), (32, 1)])
def test_mxfp8_error_against_k(block, variant):
    import dense_tensor_core_gb300 as dtc

    M, N = 256, 448
    rows = []
    for K in SWEEP_K:
        A, B, sfA, sfB = workloads.make_mx(M, N, K, seed=K + block, block=block)
        kw = with_packed_scales(M, N, K, dict(scale_block=block if block != 128 else 0,
                                              variant=variant, pack=variant == 2))
        C = dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), sfA=to_device8(sfA),
                        sfB=to_device8(sfB), **kw)
        dtc.gemm_stream_status()
        got = values16(C.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
        ref_codes, exact = oracle.gemm_mx(A, B, sfA, sfB, M, N, K, block=block, sums=True)
        ref = values16(ref_codes, "bf16")
        err = np.abs(got - ref)
        small = np.abs(ref) < 1.0
        # one bf16 rounding step of the reference (8 significant bits), or 2^-8 near zero
        step = np.where(ref != 0, 2.0 ** (np.floor(np.log2(np.abs(ref) + (ref == 0))) - 7), 0.0)
        bound = np.maximum(step, 2.0 ** -8)
        rows.append({"K": K, "block": block, "variant": variant,
                     "max_abs_err": float(err.max()),
                     "max_abs_err_ref_below_1": float(err[small].max()) if small.any() else None,
                     "max_abs_err_vs_exact_sum": float(np.abs(got - exact).max()),
                     "max_err_in_output_steps": float((err / bound).max()),
                     "max_abs_ref": float(np.abs(ref).max())})
        check_close(got, ref, f"MXFP8 K = {K}, block {block}, variant {variant}")
    out = os.environ.get("DTC_KSWEEP_OUT")
    if out:
        with open(out, "a") as f:
            for r in rows:
                f.write(json.dumps(r) + "\n")
    # The early warning the tolerance alone would hide: the kernel's output must stay within one
    # output rounding step of the correctly rounded sum (fp32 accumulation may round a sum that
    # lies near a bf16 midpoint the other way), and within 2^-8 of it near zero, at every K. A
    # reduced-precision accumulation inside the block-scaled MMA would grow past this with K.
    assert all(r["max_err_in_output_steps"] <= 1.0 for r in rows), rows
