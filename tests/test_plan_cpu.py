"""The planner without a GPU: gemm_plan_model plans for a described device (a pure function of its
arguments), so the automatic kernel choice, stream-K and its residency guard are checked here on
the GB300 model (152 SMs, 76 resident CTA pairs, 36 resident clusters of 4)."""
import pytest
import torch

import dense_tensor_core_gb300 as dtc
from dense_tensor_core_gb300 import GB300_MODEL


@pytest.fixture(scope="module", autouse=True)
def built():
    from dense_tensor_core_gb300 import build

    build.build()


def plan(kind, M, N, K, layout="NT", model=GB300_MODEL, **kw):
    return dtc.gemm_plan(kind, M, N, K, layout, model=model, **kw)


def fake_workspace(nbytes=32 << 20):
    # a host buffer stands in for the caller's device workspace: the planner only reads its
    # address (non-NULL) and size; nothing is launched
    return torch.zeros(nbytes, dtype=torch.uint8)


def test_automatic_choice_on_gb300():
    p = plan("bf16", 4096, 4096, 8192)  # 304 pair tiles of 256 x 224 = 4 waves of 76 pairs
    assert (p["variant"], p["tile_m"], p["tile_n"], p["tile_k"], p["ctas"]) == (2, 256, 224, 128, 152)
    p = plan("bf16", 8192, 8192, 8192)  # 1024 pair tiles of 256 x 256
    assert (p["variant"], p["tile_m"], p["tile_n"], p["tile_k"]) == (2, 256, 256, 128)
    assert plan("bf16", 4096, 4096, 8200)["tile_k"] == 64  # K % 64 != 0: 64-deep stages only
    p = plan("bf16", 128, 8192, 8192)  # 64 tiles of 128 x 128, K split in 2
    assert (p["variant"], p["split_k"], p["tile_n"], p["tile_k"], p["ctas"]) == (3, 2, 128, 128, 128)
    p = plan("bf16", 128, 2048, 8192)  # 16 tiles: K split in 4
    assert (p["variant"], p["split_k"], p["tile_n"], p["ctas"]) == (3, 4, 128, 64)
    p = plan("f16", 1024, 1024, 1000, "NN")  # K % 64 != 0: 64-deep stages
    assert (p["variant"], p["split_k"], p["tile_n"], p["tile_k"]) == (3, 2, 128, 64)
    # 2 one-CTA tiles of 128 x 256 would leave 150 SMs idle; with K this short the 8 tiles of
    # 128 x 64 with the whole K each beat a split in 2 (no exchange)
    p = plan("bf16", 256, 256, 512)
    assert (p["variant"], p["split_k"], p["tile_n"], p["ctas"], p["cluster"]) == (3, 1, 64, 8, 1)
    p = plan("bf16", 256, 256, 1024)  # a longer K: split (in 4 here)
    assert (p["variant"], p["split_k"], p["tile_n"], p["ctas"]) == (3, 4, 128, 16)
    p = plan("bf16", 256, 256, 256)  # 4 K-blocks: too few to split
    assert p["variant"] == 1 and p["cluster"] == 1 and p["tile_k"] == 64
    p = plan("bf16", 1024, 1024, 512)  # 32 one-CTA tiles: a split needs 8 K-blocks per CTA
    assert p["variant"] == 1
    p = plan("mxfp8", 4096, 4096, 8192)
    assert (p["variant"], p["tile_n"], p["tile_k"], p["sf_packed"]) == (1, 224, 128, 0)


def test_block_scaled_repacking_policy():
    # with a workspace the scales are repacked: 128-element blocks go to the pair kernel with
    # 256-deep stages (when K % 128 == 0 and the pair tiles fill a wave), 32-element blocks to the
    # one-CTA kernel; the pair kernel takes nothing else; a workspace too small leaves the scale
    # warps in charge
    ws = fake_workspace()
    p = plan("mxfp8", 4096, 4096, 8192, workspace=ws)
    assert (p["variant"], p["tile_m"], p["tile_n"], p["tile_k"], p["stages"], p["sf_packed"]) == (2, 256, 224, 256, 3, 1)
    assert plan("mxfp8", 4096, 4096, 8192)["variant"] == 1  # no workspace: one-CTA, scale warps
    assert plan("mxfp8", 4096, 4096, 8200, workspace=ws)["variant"] == 1  # K % 128 != 0
    assert plan("mxfp8", 1024, 1024, 1024, workspace=ws)["variant"] == 1  # 20 pair tiles < 76
    assert plan("mxfp8", 4096, 4096, 8192, workspace=ws, tile_k=128)["variant"] == 1
    for kw in (dict(variant=2), dict(variant=2, tile_k=256),  # no workspace for the scales
               dict(variant=2, workspace=ws, scale_block=32), dict(variant=2, workspace=ws, tile_k=128),
               dict(variant=2, workspace=ws, tile_n=256), dict(variant=1, tile_k=256)):
        with pytest.raises(dtc.GemmError) as e:
            plan("mxfp8", 4096, 4096, 8192, **kw)
        assert e.value.status == 2, kw
    with pytest.raises(dtc.GemmError):  # K % 128 != 0
        plan("mxfp8", 4096, 4096, 8200, variant=2, workspace=ws)
    assert plan("mxfp8", 4096, 4096, 8192, workspace=ws, scale_block=32)["variant"] == 1
    assert plan("mxfp8", 4096, 4096, 8192, workspace=ws, scale_block=32)["sf_packed"] == 1
    assert plan("mxfp8", 4096, 4096, 8192, workspace=ws, scale_block=32, b_format="e2m1")["sf_packed"] == 1
    assert plan("mxfp8", 1024, 1024, 1024, workspace=ws, variant=2)["sf_packed"] == 1
    small = fake_workspace(1024)
    assert plan("mxfp8", 4096, 4096, 8192, workspace=small, scale_block=32)["sf_packed"] == 0
    # the chunk layout: 32 groups of 128 A rows and 19 tiles of 224 B rows, 64 sets (K / 128) of
    # 512-byte chunks (B: two per set), B from the first 1 KB boundary after A
    need = (32 * 64 * 512 + 1023) // 1024 * 1024 + 19 * 64 * 2 * 512
    assert plan("mxfp8", 4096, 4096, 8192, workspace=fake_workspace(need), scale_block=32)["sf_packed"] == 1
    assert plan("mxfp8", 4096, 4096, 8192, workspace=fake_workspace(need - 16), scale_block=32)["sf_packed"] == 0


def test_stream_k_on_gb300():
    ws = fake_workspace()
    p = plan("bf16", 8192, 8192, 8192, workspace=ws)  # 1024 tiles = 13 waves + 36
    assert (p["variant"], p["tile_n"], p["sk_tiles"], p["ctas"]) == (2, 256, 1024 % 76, 152)
    p = plan("bf16", 4096, 4096, 8192, workspace=ws)  # 256 tiles = 3 waves + 28
    assert (p["variant"], p["tile_n"], p["sk_tiles"]) == (2, 256, 256 % 76)
    assert plan("bf16", 4096, 4096, 8192)["sk_tiles"] == 0  # no workspace: whole tiles
    assert plan("bf16", 8192, 8192, 8192, workspace=ws, stream_k=2)["sk_tiles"] == 0
    # a whole number of waves needs no stream-K
    assert plan("bf16", 256 * 19, 256 * 8, 8192, workspace=ws)["sk_tiles"] == 0


def test_stream_k_counts_only_resident_pairs():
    # The pair kernel's stream-K pairs wait for pieces other pairs compute, so the launch uses the
    # pairs the device keeps resident, not half the SMs.
    ws = fake_workspace()
    fewer = dict(GB300_MODEL, pair_clusters=70)
    M, N = 256 * 13, 256 * 77  # 1001 pair tiles: 13 waves + 13 of 76 pairs, 14 + 21 of 70
    assert plan("bf16", M, N, 1024, workspace=ws)["sk_tiles"] == 1001 % 76
    p = plan("bf16", M, N, 1024, model=fewer, workspace=ws)
    assert (p["ctas"], p["sk_tiles"]) == (140, 1001 % 70)
    # with 64 resident pairs the 1024 tiles fill whole waves: stream-K is dropped
    p = plan("bf16", 8192, 8192, 8192, model=dict(GB300_MODEL, pair_clusters=64), workspace=ws)
    assert p["sk_tiles"] == 0 and p["ctas"] == 128
    with pytest.raises(dtc.GemmError) as e:
        plan("bf16", 8192, 8192, 8192, model=dict(GB300_MODEL, pair_clusters=64), workspace=ws,
             stream_k=1)
    assert e.value.status == 2
    # whole-tile pair launches are sized to the resident pairs too
    p = plan("bf16", 8192, 8192, 8192, model=fewer)
    assert p["ctas"] == 140


def test_stream_k_flag_capacity():
    # the workspace's 1 KB of flags holds 128 pairs: a device with more resident pairs runs whole
    # tiles, and a call that requires stream-K there is refused
    big = dict(sm_count=300, pair_clusters=150, split2_clusters=150, split4_clusters=75)
    ws = fake_workspace(64 << 20)
    assert plan("bf16", 8192, 8192, 8192, model=big, workspace=ws)["sk_tiles"] == 0
    with pytest.raises(dtc.GemmError):
        plan("bf16", 8192, 8192, 8192, model=big, workspace=ws, stream_k=1)


def test_split_k_respects_resident_clusters():
    # 64 tiles of 128 x 128 split in 2 need 64 resident clusters of 2; with fewer the split is
    # not taken in one wave and the next candidate wins
    p = plan("bf16", 128, 8192, 8192, model=dict(GB300_MODEL, split2_clusters=60))
    assert not (p["variant"] == 3 and p["split_k"] == 2 and p["tile_n"] == 128)


def test_plan_model_rejects_bad_models():
    with pytest.raises(dtc.GemmError) as e:
        plan("bf16", 256, 256, 256, model=dict(GB300_MODEL, sm_count=0))
    assert e.value.status == 1
    with pytest.raises(dtc.GemmError):
        plan("bf16", 256, 256, 256, model=dict(GB300_MODEL, pair_clusters=-1))


def test_removed_options_are_refused():
    # the one-CTA kernel takes 64-deep stages only
    with pytest.raises(dtc.GemmError):
        plan("bf16", 1024, 1024, 1024, variant=1, tile_k=32)


def test_narrow_pair_tiles_for_few_long_tiles():
    # 256 x 128 pair tiles when they give as many CTAs as the best K-split (no exchange of partial
    # sums), fit one wave of 76 pairs and fill their 256 rows
    p = plan("bf16", 512, 4096, 4096)
    assert (p["variant"], p["tile_m"], p["tile_n"], p["tile_k"], p["stages"], p["ctas"]) == (2, 256, 128, 128, 4, 128)
    assert plan("bf16", 1024, 2048, 2048)["tile_n"] == 128
    # half the CTAs of a 128 x 128 split in 2: split-K stays
    assert plan("bf16", 1024, 1024, 1024)["variant"] == 3
    # M = 128 would leave half of every pair tile empty; K % 64 != 0 has no 128-deep stages
    assert plan("bf16", 128, 8192, 8192)["variant"] == 3
    assert plan("bf16", 512, 4096, 4072)["variant"] == 3
    # forced widths and the refusals
    assert plan("bf16", 1024, 1024, 1024, variant=2, tile_n=64)["stages"] == 4
    with pytest.raises(dtc.GemmError):
        plan("bf16", 1024, 1024, 1024, variant=2, tile_n=64, tile_k=64)
    with pytest.raises(dtc.GemmError):
        plan("bf16", 1024, 1024, 1024, variant=1, tile_n=64)
