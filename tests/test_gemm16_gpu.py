"""GPU parity of the bf16/fp16 GEMM (NT and NN) against the CPU oracle, through the C ABI.

Small and medium sizes are compared on every element of C; the benchmark sizes (in the launch
configuration the benchmark times) on sampled elements, which the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tensor_core_gb300 import workloads
from parity import check_close, sample_positions, to_device16, values16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()
    import dense_tensor_core_gb300 as dtc

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return dtc


def run16(kind, layout, A, B, M, N, K, variant=0, **kw):
    import dense_tensor_core_gb300 as dtc

    At, Bt = to_device16(A, kind), to_device16(B, kind)
    C = dtc.gemm_ex(kind, At, Bt, layout=layout, variant=variant, **kw)
    dtc.gemm_stream_status()
    return C.view(torch.int16).cpu().numpy().view(np.uint16)


_INPUT_CACHE = {}


def _cached_inputs(name):
    if name not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        _INPUT_CACHE[name] = workloads.make(workloads.WORKLOADS[name])
    return _INPUT_CACHE[name]


def full_check(kind, layout, M, N, K, seed, variant=0, **kw):
    A, B = workloads.make16(kind, layout, M, N, K, seed)
    C = run16(kind, layout, A, B, M, N, K, variant, **kw)
    ref = oracle.gemm16(kind, layout, A, B, M, N, K)
    return check_close(values16(C, kind), values16(ref, kind), f"{kind} {layout} {M}x{N}x{K}")


SHAPES = [
    (128, 256, 64),    # one tile, one K-block
    (256, 256, 512),   # two tiles, eight K-blocks
    (300, 520, 200),   # ragged in M, N and K (partial tiles and a partial K-block)
    (1, 8, 8),         # smallest legal product
    (129, 264, 72),    # one row / one 8-column group past a tile; K = one block + 8
    (640, 768, 1024),  # 15 tiles, 16 K-blocks
]


VARIANTS = {"1cta": 1, "2cta": 2}


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["NT", "NN"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_full_parity(kind, layout, shape, variant):
    M, N, K = shape
    full_check(kind, layout, M, N, K, seed=M + N + K, variant=VARIANTS[variant])


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("kind,layout", [("bf16", "NT"), ("f16", "NN"), ("f16", "NT")])
def test_more_tiles_than_sms_full_parity(kind, layout, variant):
    # 256 one-CTA tiles or 128-152 pair tiles (more than the resident CTAs / pairs): CTAs loop over
    # several tiles, the two accumulators alternate, and with K = 128 the epilogue of one tile
    # overlaps the short main loop of the next.
    full_check(kind, layout, 4096, 2048, 128, seed=77, variant=VARIANTS[variant])


@pytest.mark.parametrize("tile_n", [256, 224])
@pytest.mark.parametrize("layout", ["NT", "NN"])
@pytest.mark.parametrize("M,N,K", [(640, 520, 200), (384, 264, 136), (1152, 1792, 512)])
def test_one_cta_configurations_full_parity(M, N, K, layout, tile_n):
    # both tile widths; 640 and 384 rows give partial 128-row tiles; K = 200 and 136 end in a
    # partial K-block
    if layout == "NN" and tile_n == 224:
        pytest.skip("224-wide one-CTA tiles are offered for a B stored [N,K] only")
    import dense_tensor_core_gb300 as dtc

    p = dtc.gemm_plan("bf16", M, N, K, layout, variant=1, tile_n=tile_n)
    assert p["cluster"] == 1 and p["tile_n"] == tile_n and p["tile_k"] == 64
    full_check("bf16", layout, M, N, K, seed=M + N, variant=1, tile_n=tile_n)


@pytest.mark.parametrize("tile_n,tile_k", [(128, 0), (128, 64), (256, 0)])
@pytest.mark.parametrize("split_k", [2, 4])
@pytest.mark.parametrize("layout", ["NT", "NN"])
@pytest.mark.parametrize("M,N,K", [(128, 2048, 4096), (300, 520, 1000), (64, 264, 64),
                                   (129, 256, 200), (256, 392, 192)])
def test_split_k_full_parity(M, N, K, layout, split_k, tile_n, tile_k):
    if tile_n == 256 and split_k == 4:
        pytest.skip("256-wide split-K tiles take a split of 2")
    # K split over a cluster of CTAs that push their partial sums into the owning CTA's shared
    # memory; K = 64 is one K-block, so all CTAs but one have an empty K-range and must contribute
    # zeros; 300 x 520 and 129 x 256 leave partial tiles in M and N; K = 192 ends in a half-filled
    # 128-deep stage; K = 1000 and 200 take 64-deep stages (K % 64 != 0)
    import dense_tensor_core_gb300 as dtc

    p = dtc.gemm_plan("bf16", M, N, K, layout, variant=3, split_k=split_k, tile_n=tile_n,
                      tile_k=tile_k)
    want_k = tile_k or (128 if tile_n == 128 and K % 64 == 0 else 64)
    assert (p["variant"], p["split_k"], p["cluster"]) == (3, split_k, split_k)
    assert (p["tile_n"], p["tile_k"]) == (tile_n, want_k)
    kw = dict(variant=3, split_k=split_k, tile_n=tile_n, tile_k=tile_k)
    full_check("bf16", layout, M, N, K, seed=M + K, **kw)
    full_check("f16", layout, M, N, K, seed=M + K + 1, **kw)


@pytest.mark.parametrize("layout", ["NT", "NN", "TN", "TT"])
@pytest.mark.parametrize("M,N,K", [(128, 2048, 4096), (296, 520, 1024), (64, 264, 64),
                                   (136, 200, 192), (256, 392, 640)])
def test_unsplit_mode_full_parity(M, N, K, layout):
    # the split-K kernel with one CTA per 128 x 64 tile and the whole K (no exchange): partial
    # tiles in M and N, one K-block (K = 64), a half-filled last 128-deep stage (K = 192); every
    # stored row a multiple of 16 bytes in all four layouts
    import dense_tensor_core_gb300 as dtc

    p = dtc.gemm_plan("bf16", M, N, K, layout, variant=3, split_k=1)
    assert (p["variant"], p["split_k"], p["cluster"], p["tile_n"], p["tile_k"]) == (3, 1, 1, 64, 128)
    full_check("bf16", layout, M, N, K, seed=M + K + 7, variant=3, split_k=1)
    full_check("f16", layout, M, N, K, seed=M + K + 8, variant=3, split_k=1)


def test_automatic_choice_follows_the_cost_model():
    import dense_tensor_core_gb300 as dtc

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are worked out for 152 SMs")
    p = dtc.gemm_plan("bf16", 4096, 4096, 8192, "NT")  # 304 pair tiles of 256x224 = 4 waves
    assert (p["variant"], p["tile_m"], p["tile_n"], p["tile_k"]) == (2, 256, 224, 128)
    p = dtc.gemm_plan("bf16", 8192, 8192, 8192, "NT")  # 1024 pair tiles of 256x256
    assert (p["variant"], p["tile_m"], p["tile_n"], p["tile_k"]) == (2, 256, 256, 128)
    p = dtc.gemm_plan("bf16", 4096, 4096, 8200, "NT")  # K % 64 != 0: 64-deep stages only
    assert p["tile_k"] == 64
    p = dtc.gemm_plan("bf16", 128, 8192, 8192, "NT")  # 64 tiles of 128x128, K split in 2
    assert (p["variant"], p["split_k"], p["tile_n"], p["tile_k"], p["ctas"]) == (3, 2, 128, 128, 128)
    p = dtc.gemm_plan("bf16", 128, 2048, 8192, "NT")  # 16 tiles: K split in 4
    assert (p["variant"], p["split_k"], p["tile_n"], p["ctas"]) == (3, 4, 128, 64)
    p = dtc.gemm_plan("f16", 1024, 1024, 1000, "NN")  # K % 64 != 0: 64-deep stages
    assert (p["variant"], p["split_k"], p["tile_n"], p["tile_k"]) == (3, 2, 128, 64)
    p = dtc.gemm_plan("bf16", 256, 256, 512, "NT")  # 2 one-CTA tiles, short K: 8 unsplit 128x64
    assert (p["variant"], p["split_k"], p["tile_n"], p["ctas"]) == (3, 1, 64, 8)
    p = dtc.gemm_plan("bf16", 256, 256, 256, "NT")  # 4 K-blocks: too few to split
    assert p["variant"] == 1


@pytest.mark.parametrize("tile_k", [64, 128])
@pytest.mark.parametrize("tile_n", [256, 224])
@pytest.mark.parametrize("layout", ["NT", "NN"])
@pytest.mark.parametrize("M,N,K", [(640, 520, 192), (384, 264, 320), (1280, 1792, 1024)])
def test_pair_kernel_configurations_full_parity(M, N, K, layout, tile_n, tile_k):
    # 128-deep stages load each operand with one 3-D box of two 128-byte K-chunks; K = 192 and
    # 320 end in a half-filled 128-deep stage; 640 and 384 rows leave a partial pair tile. With NN
    # and 224-wide tiles each CTA's 112 columns of B come in two 64-column boxes, the second
    # partly used
    import dense_tensor_core_gb300 as dtc

    p = dtc.gemm_plan("bf16", M, N, K, layout, variant=2, tile_n=tile_n, tile_k=tile_k)
    assert (p["tile_m"], p["tile_n"], p["tile_k"]) == (256, tile_n, tile_k)
    full_check("bf16", layout, M, N, K, seed=M + K, variant=2, tile_n=tile_n, tile_k=tile_k)
    full_check("f16", layout, M, N, K, seed=M + K + 1, variant=2, tile_n=tile_n, tile_k=tile_k)


@pytest.mark.parametrize("tile_n", [128, 64])
@pytest.mark.parametrize("layout", ["NT", "NN", "TN", "TT"])
@pytest.mark.parametrize("M,N,K", [(640, 520, 192), (384, 200, 320), (256, 64, 64), (1280, 1792, 1024)])
def test_pair_kernel_narrow_tiles_full_parity(M, N, K, layout, tile_n):
    # 256 x 128 and 256 x 64 pair tiles (4 stages of 128 K-elements): each CTA holds 64 or 32 rows
    # of B; a B stored [K,N] comes in one 64-column box per CTA, of which the MMA reads the first 32
    # columns when the tile is 64 wide. 520 and 200 columns end in a partial tile
    import dense_tensor_core_gb300 as dtc

    p = dtc.gemm_plan("bf16", M, N, K, layout, variant=2, tile_n=tile_n)
    assert (p["tile_m"], p["tile_n"], p["tile_k"], p["stages"]) == (256, tile_n, 128, 4)
    full_check("bf16", layout, M, N, K, seed=M + K + tile_n, variant=2, tile_n=tile_n)
    full_check("f16", layout, M, N, K, seed=M + K + tile_n + 1, variant=2, tile_n=tile_n)


@pytest.mark.parametrize("M,N,tile_n", [(4096, 4096, 224), (8192, 8192, 256), (512, 448, 224)])
def test_pair_tile_width_choice(M, N, tile_n):
    import dense_tensor_core_gb300 as dtc

    p = dtc.gemm_plan("bf16", M, N, 8192, "NT", variant=2)
    assert p["variant"] == 2 and p["tile_m"] == 256 and p["tile_n"] == tile_n
    assert p["ctas"] % 2 == 0


@pytest.mark.parametrize("M,N,K", [(512, 448, 320), (600, 904, 264), (4096, 4096, 256)])
def test_pair_kernel_224_wide_tiles_full_parity(M, N, K):
    import dense_tensor_core_gb300 as dtc

    assert dtc.gemm_plan("bf16", M, N, K, "NT", variant=2)["tile_n"] == 224
    full_check("bf16", "NT", M, N, K, seed=M + K, variant=2)


def test_config_bf16_nt_256x256x512_full():
    w = workloads.WORKLOADS["bf16_nt_256x256x512"]
    full_check(w.kind, w.layout, w.M, w.N, w.K, w.seed)


def test_config_f16_nn_1024_full():
    w = workloads.WORKLOADS["f16_nn_1024x1024x1024"]
    full_check(w.kind, w.layout, w.M, w.N, w.K, w.seed)


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("name", ["bf16_nt_4096x4096x8192", "bf16_nt_8192x8192x8192",
                                  "bf16_nt_128x8192x8192", "bf16_tn_4096x4096x8192",
                                  "bf16_tt_4096x4096x8192"])
def test_benchmark_sizes_sampled(name, variant):
    # variant 0 is the launch the benchmark times (the library's own choice)
    w = workloads.WORKLOADS[name]
    A, B = _cached_inputs(name)
    C = run16(w.kind, w.layout, A, B, w.M, w.N, w.K, variant=variant)
    r, c = sample_positions(w.M, w.N, count=3000, seed=w.seed)
    # plus one full row and one full column
    r = np.concatenate([r, np.full(w.N, w.M // 3), np.arange(w.M)])
    c = np.concatenate([c, np.arange(w.N), np.full(w.M, w.N // 5)])
    ref, _ = oracle.gemm16_sampled(w.kind, w.layout, A, B, w.M, w.N, w.K, r, c)
    check_close(values16(C[r, c], w.kind), values16(ref, w.kind), name)


def test_k_zero_writes_zeros_and_empty_is_noop():
    import dense_tensor_core_gb300 as dtc

    A = torch.empty((64, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((32, 0), dtype=torch.bfloat16, device="cuda")
    C = torch.full((64, 32), float("nan"), dtype=torch.bfloat16, device="cuda")
    dtc.gemm_bf16(A, B, C)
    dtc.gemm_stream_status()
    assert torch.equal(C, torch.zeros_like(C))
    A0 = torch.empty((0, 16), dtype=torch.float16, device="cuda")
    B0 = torch.empty((16, 16), dtype=torch.float16, device="cuda")
    C0 = dtc.gemm_f16(A0, B0, layout="NN")
    assert C0.shape == (0, 16)


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("layout", ["NT", "NN"])
def test_writes_exactly_C(layout, variant):
    # C sits inside a larger buffer filled with NaN: every element of C must be overwritten and
    # nothing around it touched (the TMA stores clip ragged edges to [M, N]; 264 columns end in a
    # partial 64-column chunk, 200 rows in a partial 32-row band)
    import dense_tensor_core_gb300 as dtc

    M, N, K = 200, 264, 136
    A, B = workloads.make16("bf16", layout, M, N, K, 5)
    guard = 4096
    buf = torch.full((guard * 2 + M * N,), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    kw = dict(split_k=2) if variant == 3 else {}
    dtc.gemm_ex("bf16", to_device16(A, "bf16"), to_device16(B, "bf16"), C, layout=layout,
                variant=variant, **kw)
    dtc.gemm_stream_status()
    h = buf.float().cpu()
    assert torch.isnan(h[:guard]).all() and torch.isnan(h[guard + M * N:]).all()
    assert not torch.isnan(h[guard:guard + M * N]).any()


def test_runs_on_a_side_stream():
    import dense_tensor_core_gb300 as dtc

    M, N, K = 256, 512, 256
    A, B = workloads.make16("f16", "NT", M, N, K, 6)
    s = torch.cuda.Stream()
    At, Bt = to_device16(A, "f16"), to_device16(B, "f16")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        C = dtc.gemm_f16(At, Bt, stream=s)
    dtc.gemm_stream_status(s)
    ref = oracle.gemm16("f16", "NT", A, B, M, N, K)
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    check_close(values16(got, "f16"), values16(ref, "f16"), "side stream")


def test_repeated_calls_are_deterministic():
    import dense_tensor_core_gb300 as dtc

    M, N, K = 512, 512, 1024
    A, B = workloads.make16("bf16", "NT", M, N, K, 8)
    At, Bt = to_device16(A, "bf16"), to_device16(B, "bf16")
    C1 = dtc.gemm_bf16(At, Bt)
    C2 = dtc.gemm_bf16(At, Bt)
    dtc.gemm_stream_status()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


# --- A stored transposed (TN, TT) and rows of larger arrays (leading dimensions) ---------------

@pytest.mark.parametrize("variant,extra", [(1, {}), (1, dict(tile_n=224)),
                                           (2, dict(tile_k=64)), (2, dict(tile_k=128)),
                                           (3, dict(split_k=2)), (3, dict(split_k=4, tile_k=64))])
@pytest.mark.parametrize("layout", ["TN", "TT"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (264, 520, 200), (512, 448, 384), (8, 8, 8)])
def test_transposed_a_full_parity(M, N, K, layout, variant, extra):
    # A stored [K,M] is loaded as 64-column boxes and read through an MN-major descriptor;
    # 264 rows leave a partial tile in M (and a partial 64-column box), K = 200 a partial K-block
    if extra.get("tile_k") == 128 and K % 64:
        pytest.skip("128-deep pair stages need K % 64 == 0")
    if variant == 1 and extra.get("tile_n") == 224 and layout == "TN":
        pytest.skip("224-wide one-CTA tiles are offered for a B stored [N,K] only")
    kind = "bf16" if (M + N) % 2 == 0 else "f16"
    full_check(kind, layout, M, N, K, seed=M + N + K, variant=variant, **extra)
    full_check("f16" if kind == "bf16" else "bf16", layout, M, N, K, seed=M + N + K + 1,
               variant=variant, **extra)


@pytest.mark.parametrize("layout", ["NT", "NN", "TN", "TT"])
@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_rows_of_larger_arrays(layout, variant):
    # A, B and C are views into wider row-major arrays: the row strides go to the library as
    # lda / ldb / ldc; C's padding columns must be left untouched
    import dense_tensor_core_gb300 as dtc

    M, N, K = 264, 392, 320
    A, B = workloads.make16("bf16", layout, M, N, K, seed=77)
    pad = {"A": 24, "B": 40, "C": 16}
    At = torch.full((A.shape[0], A.shape[1] + pad["A"]), 7.0, dtype=torch.bfloat16, device="cuda")
    Bt = torch.full((B.shape[0], B.shape[1] + pad["B"]), 7.0, dtype=torch.bfloat16, device="cuda")
    At[:, : A.shape[1]] = to_device16(A, "bf16")
    Bt[:, : B.shape[1]] = to_device16(B, "bf16")
    Cbig = torch.full((M, N + pad["C"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    kw = dict(split_k=2) if variant == 3 else {}
    dtc.gemm_ex("bf16", At[:, : A.shape[1]], Bt[:, : B.shape[1]], Cbig[:, :N], layout=layout,
                variant=variant, **kw)
    dtc.gemm_stream_status()
    assert torch.isnan(Cbig[:, N:].float()).all(), "padding columns of C were written"
    C = Cbig[:, :N].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.gemm16("bf16", layout, A, B, M, N, K)
    check_close(values16(C, "bf16"), values16(ref, "bf16"), f"strided {layout} variant {variant}")


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_c_view_at_an_offset(variant):
    # C is a window of a larger array starting 8 columns and 3 rows in: its base is 16-byte but not
    # 128-byte aligned, its rows are ldc apart; only the window may be written
    import dense_tensor_core_gb300 as dtc

    M, N, K = 136, 200, 192
    A, B = workloads.make16("f16", "NT", M, N, K, seed=31)
    big = torch.full((M + 6, N + 24), float("nan"), dtype=torch.float16, device="cuda")
    C = big[3:3 + M, 8:8 + N]
    kw = dict(split_k=2) if variant == 3 else {}
    dtc.gemm_ex("f16", to_device16(A, "f16"), to_device16(B, "f16"), C, variant=variant, **kw)
    dtc.gemm_stream_status()
    h = big.float().cpu()
    inside = torch.zeros_like(h, dtype=torch.bool)
    inside[3:3 + M, 8:8 + N] = True
    assert torch.isnan(h[~inside]).all(), "written outside the C window"
    got = C.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.gemm16("f16", "NT", A, B, M, N, K)
    check_close(values16(got, "f16"), values16(ref, "f16"), f"C window, variant {variant}")


def test_k_zero_with_strided_c_writes_only_the_region():
    import dense_tensor_core_gb300 as dtc

    A = torch.empty((64, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((32, 0), dtype=torch.bfloat16, device="cuda")
    Cbig = torch.full((64, 48), float("nan"), dtype=torch.bfloat16, device="cuda")
    dtc.gemm_ex("bf16", A, B, Cbig[:, :32])
    dtc.gemm_stream_status()
    assert torch.equal(Cbig[:, :32], torch.zeros((64, 32), dtype=torch.bfloat16, device="cuda"))
    assert torch.isnan(Cbig[:, 32:].float()).all()


def test_transposed_layout_plans():
    import dense_tensor_core_gb300 as dtc

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are worked out for 152 SMs")
    # 304 pair tiles of 256 x 224 = 4 full waves, whatever the storage of A and B
    for layout in ("TT", "TN", "NN"):
        p = dtc.gemm_plan("bf16", 4096, 4096, 8192, layout)
        assert (p["variant"], p["tile_n"]) == (2, 224), layout
    # one-CTA 224-wide tiles need B stored [N,K]
    with pytest.raises(dtc.GemmError):
        dtc.gemm_plan("bf16", 4096, 4096, 8192, "TN", variant=1, tile_n=224)


# --- stream-K on CTA pairs (the leftover tiles of the last wave shared out over all pairs) ------

def _workspace(kind, M, N, K, layout):
    import dense_tensor_core_gb300 as dtc

    nbytes = dtc.gemm_workspace_size(kind, M, N, K, layout, stream_k=1)
    assert nbytes > 0
    return torch.zeros(nbytes, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("tile_k", [0, 64])
@pytest.mark.parametrize("layout", ["NT", "NN", "TN", "TT"])
@pytest.mark.parametrize("M,N,K", [(2560, 2560, 1024), (2560, 2304, 384), (2304, 2560, 640)])
def test_stream_k_full_parity(M, N, K, layout, tile_k):
    # 100 (or 90) pair tiles of 256 x 256 over 76 pairs: one whole wave, then 24 (or 14) tiles
    # shared out as runs of K-blocks; K = 384 gives fewer K-blocks than pairs, so some pairs have
    # an empty share and tiles are split over up to 3 pairs; every piece, the flags and the fixup
    # are exercised, and the flags must be back at zero afterwards
    import dense_tensor_core_gb300 as dtc

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the shapes are chosen for 76 pairs")
    kind = "bf16" if layout in ("NT", "TN") else "f16"
    # (tile_k 64: 64-deep stages, twice the K-blocks per tile to share out)
    ws = _workspace(kind, M, N, K, layout)
    p = dtc.gemm_plan(kind, M, N, K, layout, workspace=ws, stream_k=1, tile_k=tile_k)
    assert (p["variant"], p["tile_n"], p["tile_k"]) == (2, 256, tile_k or 128) and p["sk_tiles"] > 0
    A, B = workloads.make16(kind, layout, M, N, K, seed=M + K)
    At, Bt = to_device16(A, kind), to_device16(B, kind)
    C1 = dtc.gemm_ex(kind, At, Bt, layout=layout, workspace=ws, stream_k=1, tile_k=tile_k)
    C2 = dtc.gemm_ex(kind, At, Bt, layout=layout, workspace=ws, stream_k=1, tile_k=tile_k)
    dtc.gemm_stream_status()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16)), "two runs differ"
    assert int(ws[:1024].count_nonzero()) == 0, "stream-K flags not back at zero"
    ref = oracle.gemm16(kind, layout, A, B, M, N, K)
    check_close(values16(C1.view(torch.int16).cpu().numpy().view(np.uint16), kind),
                values16(ref, kind), f"stream-K {layout} {M}x{N}x{K}")


def test_stream_k_benchmark_size_sampled():
    import dense_tensor_core_gb300 as dtc

    w = workloads.WORKLOADS["bf16_nt_4096x4096x8192"]
    A, B = _cached_inputs(w.name)
    ws = _workspace(w.kind, w.M, w.N, w.K, w.layout)
    C = dtc.gemm_ex(w.kind, to_device16(A, w.kind), to_device16(B, w.kind), layout=w.layout,
                    workspace=ws, stream_k=1)
    dtc.gemm_stream_status()
    C = C.view(torch.int16).cpu().numpy().view(np.uint16)
    r, c = sample_positions(w.M, w.N, count=3000, seed=w.seed, tile_m=256, tile_n=256)
    r = np.concatenate([r, np.full(w.N, 4000), np.arange(w.M)])  # the stream-K rows are at the end
    c = np.concatenate([c, np.arange(w.N), np.full(w.M, 3333)])
    ref, _ = oracle.gemm16_sampled(w.kind, w.layout, A, B, w.M, w.N, w.K, r, c)
    check_close(values16(C[r, c], w.kind), values16(ref, w.kind), "stream-K 4096x4096x8192")


def test_stream_k_plan_choice():
    import dense_tensor_core_gb300 as dtc

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are worked out for 152 SMs")
    ws = _workspace("bf16", 8192, 8192, 8192, "NT")
    # 1024 pair tiles of 256 x 256 = 13.47 waves: with a workspace, the last 36 are shared out
    p = dtc.gemm_plan("bf16", 8192, 8192, 8192, workspace=ws)
    assert (p["variant"], p["tile_n"], p["sk_tiles"]) == (2, 256, 1024 % 76)
    assert dtc.gemm_plan("bf16", 8192, 8192, 8192)["sk_tiles"] == 0  # no workspace: whole tiles
    assert dtc.gemm_plan("bf16", 8192, 8192, 8192, workspace=ws, stream_k=2)["sk_tiles"] == 0
    # 4096^2 x 8192: 256 tiles of 256 x 256 (3.37 waves) with stream-K, against 304 of 256 x 224
    # in exactly 4 waves: measured within 1 %, stream-K slightly ahead
    p = dtc.gemm_plan("bf16", 4096, 4096, 8192, workspace=ws)
    assert (p["variant"], p["tile_n"], p["sk_tiles"]) == (2, 256, 256 % 76)
    p = dtc.gemm_plan("bf16", 4096, 4096, 8192)  # without a workspace: whole 224-wide tiles
    assert (p["variant"], p["tile_n"], p["sk_tiles"]) == (2, 224, 0)
    # a whole number of waves (76 x 2 tiles) needs no stream-K
    assert dtc.gemm_workspace_size("bf16", 256 * 19, 256 * 8, 8192) == 0
    with pytest.raises(dtc.GemmError):  # too small a workspace when stream-K is required
        dtc.gemm_plan("bf16", 4096, 4096, 8192, workspace=ws[:1024], stream_k=1)


def test_stream_k_with_rows_of_larger_arrays():
    # stream-K pieces and fixup with A stored [K,M] in a wider array and C a view with ldc > N
    import dense_tensor_core_gb300 as dtc

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the shape is chosen for 76 pairs")
    M, N, K = 2560, 2560, 768
    A, B = workloads.make16("bf16", "TN", M, N, K, seed=99)
    Ab = torch.zeros((K, M + 64), dtype=torch.bfloat16, device="cuda")
    Ab[:, :M] = to_device16(A, "bf16")
    Cb = torch.full((M, N + 32), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = _workspace("bf16", M, N, K, "TN")
    dtc.gemm_ex("bf16", Ab[:, :M], to_device16(B, "bf16"), Cb[:, :N], layout="TN", workspace=ws,
                stream_k=1)
    dtc.gemm_stream_status()
    assert torch.isnan(Cb[:, N:].float()).all()
    C = Cb[:, :N].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.gemm16("bf16", "TN", A, B, M, N, K)
    check_close(values16(C, "bf16"), values16(ref, "bf16"), "stream-K, strided")


# --- device-memory checks and the device model ---------------------------------------------------

def test_host_memory_is_refused_before_launch():
    # the kernels read through tensor maps of the current device: a host pointer (pageable or
    # pinned) is refused with GEMM_ERR_INVALID_ARG and nothing is enqueued
    import ctypes

    import dense_tensor_core_gb300 as dtc

    L = dtc.lib()
    M = N = K = 256
    dev_buf = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    pinned = torch.zeros((M, K), dtype=torch.bfloat16).pin_memory()
    pageable = np.zeros((M, K), dtype=np.uint16)
    vp = ctypes.c_void_p
    for name, ptr in (("pinned", pinned.data_ptr()), ("pageable", pageable.ctypes.data)):
        for args in ((ptr, dev_buf.data_ptr(), C.data_ptr()), (dev_buf.data_ptr(), ptr, C.data_ptr()),
                     (dev_buf.data_ptr(), dev_buf.data_ptr(), ptr)):
            rc = L.gemm_bf16(vp(args[0]), vp(args[1]), vp(args[2]), M, N, K, 0, None)
            assert rc == 1, f"{name}: status {rc}"
            assert b"device memory" in L.gemm_last_error()
    dtc.gemm_stream_status()
    assert (C.float() == 7.0).all()  # nothing ran


def test_plan_matches_the_queried_device_model():
    import dense_tensor_core_gb300 as dtc

    m = dtc.gemm_device_model_query()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert m["sm_count"] == sms
    assert 1 <= m["pair_clusters"] <= sms // 2
    assert 1 <= m["split2_clusters"] <= sms // 2 and 1 <= m["split4_clusters"] <= sms // 4
    ws = torch.zeros(32 << 20, dtype=torch.uint8, device="cuda")
    for shape, kw in [((4096, 4096, 8192), {}), ((8192, 8192, 8192), dict(workspace=ws)),
                      ((128, 8192, 8192), {}), ((1024, 1024, 1024), dict(layout="NN")),
                      ((256, 256, 512), {}), ((2560, 2560, 1024), dict(workspace=ws))]:
        assert dtc.gemm_plan("bf16", *shape, **kw) == dtc.gemm_plan("bf16", *shape, model=m, **kw)
