"""GPU parity of the MXFP8 block-scaled GEMM (e4m3 x e4m3, E8M0 scale per row per 128 K-elements,
bf16 output) against the CPU oracle, through the C ABI."""
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


_BENCH = []


def _bench_inputs():
    if not _BENCH:
        _BENCH.append(workloads.make(workloads.WORKLOADS["mxfp8_nt_4096x4096x8192"]))
    return _BENCH[0]


def run_mx(A, B, sfA, sfB, **kw):
    import dense_tensor_core_gb300 as dtc

    kw = with_packed_scales(A.shape[0], B.shape[0], _k_of(A, kw), kw)
    C = dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), sfA=to_device8(sfA),
                    sfB=to_device8(sfB), **kw)
    dtc.gemm_stream_status()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


def _k_of(A, kw):
    # K from A's stored row (bytes per row for fp8; fp6 / fp4 rows are packed)
    bits = {"e4m3": 8, "e5m2": 8, "e2m3": 6, "e3m2": 6, "e2m1": 4}[kw.get("a_format", "e4m3")]
    return A.shape[1] * 8 // bits


def check_mx(A, B, sfA, sfB, what, **kw):
    M, K = A.shape
    N = B.shape[0]
    C = run_mx(A, B, sfA, sfB, **kw)
    ref = oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K)
    return check_close(values16(C, "bf16"), values16(ref, "bf16"), what)


@pytest.mark.parametrize("M,N,K", [
    (128, 224, 128),    # one tile, one K-block, one scale group
    (256, 448, 1024),   # 4 tiles, 8 K-blocks = 2 scale groups
    (256, 448, 384),    # 3 K-blocks: with 256-deep stages the last stage is half past K
    (300, 520, 400),    # ragged M and N; K = 3 K-blocks + 16 (partial block and group)
    (1, 8, 16),         # smallest legal product
    (129, 232, 656),    # a row / 8 columns past a tile; 6 K-blocks (one partial group)
    (640, 896, 2048),   # 20 tiles, 16 K-blocks
])
def test_small_shapes_full_parity(M, N, K):
    # the one-CTA kernel: 128-deep stages (2-D boxes, any K with 16-byte rows)
    import dense_tensor_core_gb300 as dtc

    assert dtc.gemm_plan("mxfp8", M, N, K, variant=1)["tile_k"] == 128
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=M + N + K)
    check_mx(A, B, sfA, sfB, f"mxfp8 {M}x{N}x{K}", variant=1)


@pytest.mark.parametrize("M,N,K", [
    (256, 224, 256),    # one pair tile, one 256-deep stage = 2 scale blocks
    (512, 448, 1024),   # 4 pair tiles, 4 stages = 2 scale groups
    (300, 520, 384),    # ragged M and N; the last stage is half padding (K = 3 x 128)
    (1, 8, 128),        # smallest K the pair kernel takes
    (640, 896, 2048),
    (1280, 2240, 640),  # 50 pair tiles, 640 = 2.5 stages of 256 (half-padded last stage)
])
def test_pair_kernel_full_parity(M, N, K):
    # the pair kernel: 256-deep stages, the scales repacked into a workspace (the helper checks
    # through the plan that the call takes them)
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=M + N + K + 1)
    check_mx(A, B, sfA, sfB, f"mxfp8 pair {M}x{N}x{K}", variant=2, pack=True)


def test_unit_scales_reduce_to_plain_e4m3():
    M, N, K = 256, 448, 512
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=3)
    check_mx(A, B, np.full_like(sfA, 127), np.full_like(sfB, 127), "unit scales")


@pytest.mark.parametrize("variant,tile_k,pack", [(1, 128, False), (2, 0, True), (2, 256, True)])
@pytest.mark.parametrize("which", ["a_rows", "b_rows", "k_blocks"])
def test_scales_varying_along_one_axis(which, variant, tile_k, pack):
    # Scales that vary along a single axis: a wrong row / column / K-block mapping of the scale
    # layout in Tensor Memory shows up as a failure of exactly one of these.
    M, N, K = 256, 448, 1024
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=4)
    kb = sfA.shape[1]
    sfA[:] = 127
    sfB[:] = 127
    if which == "a_rows":
        sfA[:] = (120 + (np.arange(M) % 13))[:, None]
    elif which == "b_rows":
        sfB[:] = (121 + (np.arange(N) % 11))[:, None]
    else:
        sfA[:] = (123 + (np.arange(kb) % 7))[None, :]
        sfB[:] = (130 - (np.arange(kb) % 5))[None, :]
    check_mx(A, B, sfA, sfB, f"scales along {which}", variant=variant, tile_k=tile_k, pack=pack)


def test_wide_scale_range():
    M, N, K = 128, 224, 512
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=5)
    rng = np.random.default_rng(0)
    sfA[:] = rng.integers(110, 145, sfA.shape)
    sfB[:] = rng.integers(110, 145, sfB.shape)
    check_mx(A, B, sfA, sfB, "wide scale range")


@pytest.mark.parametrize("variant,pack,tile_k", [(1, False, 0), (2, True, 0), (2, True, 256)])
def test_more_tiles_than_sms(variant, pack, tile_k):
    # 200 one-CTA tiles of 128 x 224 over 152 SMs, or 100 pair tiles over 76 pairs: persistent
    # loop, both accumulators, scale sets reused across tiles
    M, N, K = 2560, 2240, 256
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=6)
    check_mx(A, B, sfA, sfB, "more tiles than SMs", variant=variant, pack=pack, tile_k=tile_k)


@pytest.mark.parametrize("variant,tile_k,pack", [(0, 0, False), (0, 0, True), (1, 128, False),
                                                (2, 256, True)])
def test_benchmark_size_sampled(variant, tile_k, pack):
    w = workloads.WORKLOADS["mxfp8_nt_4096x4096x8192"]
    A, B, sfA, sfB = _bench_inputs()
    C = run_mx(A, B, sfA, sfB, variant=variant, tile_k=tile_k, pack=pack)
    r, c = sample_positions(w.M, w.N, count=3000, seed=w.seed, tile_m=128, tile_n=224)
    r = np.concatenate([r, np.full(w.N, 1000), np.arange(w.M)])
    c = np.concatenate([c, np.arange(w.N), np.full(w.M, 999)])
    ref, _ = oracle.gemm_mxfp8_sampled(A, B, sfA, sfB, w.M, w.N, w.K, r, c)
    check_close(values16(C[r, c], "bf16"), values16(ref, "bf16"), w.name)


def test_k_zero_and_empty():
    import dense_tensor_core_gb300 as dtc

    A = torch.empty((64, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((32, 0), dtype=torch.uint8, device="cuda")
    sf = torch.empty((64, 0), dtype=torch.uint8, device="cuda")
    sfb = torch.empty((32, 0), dtype=torch.uint8, device="cuda")
    C = torch.full((64, 32), float("nan"), dtype=torch.bfloat16, device="cuda")
    dtc.gemm_mxfp8(A, B, sf, sfb, C)
    dtc.gemm_stream_status()
    assert torch.equal(C, torch.zeros_like(C))


@pytest.mark.parametrize("variant,pack,block", [(1, False, 128), (1, True, 32), (2, True, 128)])
def test_timeout_reports_and_recovers(variant, pack, block):
    import dense_tensor_core_gb300 as dtc

    M, N, K = 256, 448, 512
    A, B, sfA, sfB = workloads.make_mx(M, N, K, 7, block=block)
    dtc.gemm_stream_status()
    kw = with_packed_scales(M, N, K, dict(variant=variant, pack=pack, scale_block=block))
    dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), sfA=to_device8(sfA), sfB=to_device8(sfB),
                timeout_ns=20_000_000, fault_inject=1, **kw)
    with pytest.raises(dtc.GemmError) as e:
        dtc.gemm_stream_status()
    assert e.value.status == 4
    C = run_mx_fmt(A, B, sfA, sfB, "e4m3", "e4m3", block, variant=variant, pack=pack)
    ref = oracle.gemm_mx(A, B, sfA, sfB, M, N, K, block=block)
    check_close(values16(C, "bf16"), values16(ref, "bf16"), "after timeout")


def test_automatic_choice():
    import dense_tensor_core_gb300 as dtc

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are worked out for 152 SMs")
    # without a workspace: the one-CTA kernel, 128-deep stages, scales through its scale warps
    p = dtc.gemm_plan("mxfp8", 4096, 4096, 8192)
    assert (p["variant"], p["tile_k"], p["sf_packed"]) == (1, 128, 0)
    # with one: the pair kernel (256-deep stages, repacked scales) where it fills a wave and
    # K % 128 == 0; repacked scales on the one-CTA kernel for 32-element blocks
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    p = dtc.gemm_plan("mxfp8", 4096, 4096, 8192, workspace=ws)
    assert (p["variant"], p["tile_k"], p["stages"], p["sf_packed"]) == (2, 256, 3, 1)
    assert dtc.gemm_plan("mxfp8", 4096, 4096, 8208, workspace=ws)["variant"] == 1
    assert dtc.gemm_plan("mxfp8", 4096, 4096, 8192, workspace=ws, tile_k=128)["variant"] == 1
    p = dtc.gemm_plan("mxfp8", 4096, 4096, 8192, workspace=ws, scale_block=32)
    assert (p["variant"], p["sf_packed"]) == (1, 1)
    p = dtc.gemm_plan("mxfp8", 1024, 1024, 1024, workspace=ws)  # 20 pair tiles: under a wave
    assert (p["variant"], p["sf_packed"]) == (1, 0)
    assert dtc.gemm_plan("mxfp8", 1024, 1024, 1024, workspace=ws, variant=2)["sf_packed"] == 1
    # what the pair kernel does not take
    for kw in (dict(variant=2), dict(variant=2, workspace=ws, scale_block=32),
               dict(variant=2, workspace=ws, tile_k=128), dict(variant=2, workspace=ws, tile_n=256),
               dict(variant=1, tile_k=256)):
        with pytest.raises(dtc.GemmError) as e:
            dtc.gemm_plan("mxfp8", 4096, 4096, 8192, **kw)
        assert e.value.status == 2, kw
    with pytest.raises(dtc.GemmError):
        dtc.gemm_plan("mxfp8", 4096, 4096, 8208, variant=2, workspace=ws)


# --- other block-scaled formats: e5m2 elements, 32-element (OCP MX) scale blocks ---------------

def run_mx_fmt(A, B, sfA, sfB, a_fmt, b_fmt, block, **kw):
    return run_mx(A, B, sfA, sfB, a_format=a_fmt, b_format=b_fmt, scale_block=block, **kw)


@pytest.mark.parametrize("variant,tile_k,pack", [(1, 128, False), (1, 128, True), (2, 0, True)])
@pytest.mark.parametrize("block", [32, 128])
@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3"),
                                         ("e4m3", "e4m3")])
@pytest.mark.parametrize("M,N,K", [(256, 448, 1024), (300, 520, 400), (129, 232, 656),
                                   (256, 224, 384)])
def test_formats_and_blocks_full_parity(M, N, K, a_fmt, b_fmt, block, variant, tile_k, pack):
    if variant == 2 and (block != 128 or K % 128):
        pytest.skip("the pair kernel takes 128-element blocks and K % 128 == 0")
    if pack and variant == 1 and block == 128:
        pytest.skip("the one-CTA kernel repacks the scales of 32-element blocks only")
    A, B, sfA, sfB = workloads.make_mx(M, N, K, M + N + K + block, a_fmt, b_fmt, block)
    C = run_mx_fmt(A, B, sfA, sfB, a_fmt, b_fmt, block, variant=variant, tile_k=tile_k, pack=pack)
    ref = oracle.gemm_mx(A, B, sfA, sfB, M, N, K, a_fmt=a_fmt, b_fmt=b_fmt, block=block)
    check_close(values16(C, "bf16"), values16(ref, "bf16"),
                f"{a_fmt}x{b_fmt} block {block} {M}x{N}x{K} tile_k {tile_k}")


@pytest.mark.parametrize("pack", [False, True])
@pytest.mark.parametrize("which", ["a_rows", "b_rows", "k_blocks"])
def test_block32_scales_varying_along_one_axis(which, pack):
    # with 32-element blocks each MMA of a K-block takes its own scale byte: scales that vary along
    # K by 32-block pin that byte selection
    M, N, K = 256, 448, 1024
    A, B, sfA, sfB = workloads.make_mx(M, N, K, 9, block=32)
    kb = sfA.shape[1]
    sfA[:] = 127
    sfB[:] = 127
    if which == "a_rows":
        sfA[:] = (120 + (np.arange(M) % 13))[:, None]
    elif which == "b_rows":
        sfB[:] = (121 + (np.arange(N) % 11))[:, None]
    else:
        sfA[:] = (123 + (np.arange(kb) % 7))[None, :]
        sfB[:] = (130 - (np.arange(kb) % 5))[None, :]
    C = run_mx_fmt(A, B, sfA, sfB, "e4m3", "e4m3", 32, variant=1, pack=pack)
    ref = oracle.gemm_mx(A, B, sfA, sfB, M, N, K, block=32)
    check_close(values16(C, "bf16"), values16(ref, "bf16"), f"block-32 scales along {which}")


@pytest.mark.parametrize("pack", [False, True])
@pytest.mark.parametrize("name", ["mxfp8_b32_nt_4096x4096x8192", "mx_e5m2_b32_nt_4096x4096x8192"])
def test_format_workloads_sampled(name, pack):
    w = workloads.WORKLOADS[name]
    A, B, sfA, sfB = workloads.make(w)
    C = run_mx_fmt(A, B, sfA, sfB, w.a_fmt, w.b_fmt, w.block, pack=pack)
    r, c = sample_positions(w.M, w.N, count=3000, seed=w.seed, tile_m=128, tile_n=224)
    r = np.concatenate([r, np.full(w.N, 777), np.arange(w.M)])
    c = np.concatenate([c, np.arange(w.N), np.full(w.M, 555)])
    ref, _ = oracle.gemm_mx_sampled(A, B, sfA, sfB, w.M, w.N, w.K, r, c, a_fmt=w.a_fmt,
                                    b_fmt=w.b_fmt, block=w.block)
    check_close(values16(C[r, c], "bf16"), values16(ref, "bf16"), name)


def test_format_options_plan():
    import dense_tensor_core_gb300 as dtc

    p = dtc.gemm_plan("mxfp8", 4096, 4096, 8192, scale_block=32, a_format="e5m2")
    assert (p["variant"], p["tile_k"]) == (1, 128)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    p = dtc.gemm_plan("mxfp8", 4096, 4096, 8192, variant=2, b_format="e2m1", workspace=ws)
    assert (p["variant"], p["tile_m"], p["tile_n"], p["tile_k"]) == (2, 256, 224, 256)


@pytest.mark.parametrize("variant", [1, 2])
def test_rows_of_larger_arrays(variant):
    # A, B and C as views into wider row-major arrays: lda, ldb (bytes of e4m3) and ldc go to the
    # library; C's padding columns stay untouched
    import dense_tensor_core_gb300 as dtc

    M, N, K = 384, 448, 512
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=21)
    Ab = torch.zeros((M, K + 48), dtype=torch.uint8, device="cuda")
    Bb = torch.zeros((N, K + 16), dtype=torch.uint8, device="cuda")
    Ab[:, :K] = to_device8(A)
    Bb[:, :K] = to_device8(B)
    Cb = torch.full((M, N + 24), float("nan"), dtype=torch.bfloat16, device="cuda")
    kw = with_packed_scales(M, N, K, dict(variant=variant, pack=variant == 2))
    dtc.gemm_ex("mxfp8", Ab[:, :K], Bb[:, :K], Cb[:, :N], sfA=to_device8(sfA), sfB=to_device8(sfB),
                **kw)
    dtc.gemm_stream_status()
    assert torch.isnan(Cb[:, N:].float()).all(), "padding columns of C were written"
    C = Cb[:, :N].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K)
    check_close(values16(C, "bf16"), values16(ref, "bf16"), f"strided mxfp8 variant {variant}")


@pytest.mark.parametrize("variant,tile_k", [(1, 128), (2, 0)])
def test_writes_exactly_C(variant, tile_k):
    # C inside a NaN-filled buffer: every element overwritten, nothing around it touched (224-wide
    # tiles end in a 32-column chunk; 520 columns and 300 rows leave partial chunks and bands)
    import dense_tensor_core_gb300 as dtc

    M, N, K = 300, 520, 512
    A, B, sfA, sfB = workloads.make_mxfp8(M, N, K, seed=21)
    guard = 4096
    buf = torch.full((guard * 2 + M * N,), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    kw = with_packed_scales(M, N, K, dict(variant=variant, tile_k=tile_k, pack=variant == 2))
    dtc.gemm_ex("mxfp8", to_device8(A), to_device8(B), C, sfA=to_device8(sfA), sfB=to_device8(sfB),
                **kw)
    dtc.gemm_stream_status()
    h = buf.float().cpu()
    assert torch.isnan(h[:guard]).all() and torch.isnan(h[guard + M * N:]).all()
    got = h[guard:guard + M * N].view(M, N)
    assert not torch.isnan(got).any()
    ref = oracle.gemm_mxfp8(A, B, sfA, sfB, M, N, K)
    check_close(got.double().numpy(), values16(ref, "bf16"), f"mxfp8 variant {variant} in a buffer")
