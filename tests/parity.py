"""Helpers shared by the GPU parity tests: host <-> device bytes and the pages' tolerance.

The tolerance is the pages' own check, torch.testing.assert_close(c, ref_c, rtol=1e-2, atol=1e-2)
(TileLang SM100 Support (Preview), "Compilation and Usage"): element by element,
|C - ref| <= 1e-2 + 1e-2 |ref|, with ref the oracle's rounded output. A NaN anywhere fails;
an infinity must match exactly.
"""
import numpy as np
import torch

RTOL = 1e-2
ATOL = 1e-2

T16 = {"bf16": torch.bfloat16, "f16": torch.float16}


def to_device16(codes, kind, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(T16[kind]).to(device)


def to_device8(codes, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(codes)).to(device)


def values16(codes, kind):
    t = torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(T16[kind])
    return t.to(torch.float64).numpy()


def check_close(got, ref, what=""):
    """got, ref: float64 arrays of the same shape. Raises AssertionError with a summary."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    inf = np.isinf(ref)
    assert np.array_equal(got[inf], ref[inf]), f"{what}: infinities differ"
    fin = ~inf
    err = np.abs(got[fin] - ref[fin])
    bound = ATOL + RTOL * np.abs(ref[fin])
    ok = err <= bound  # NaN compares False
    if not np.all(ok):
        idx = np.flatnonzero(~ok)
        flat_got, flat_ref = got[fin], ref[fin]
        ex = ", ".join(f"[{i}] got {flat_got[i]:.6g} ref {flat_ref[i]:.6g}" for i in idx[:5])
        raise AssertionError(f"{what}: {idx.size} of {ok.size} elements outside "
                             f"{ATOL} + {RTOL}|ref| (max err {np.nanmax(err):.4g}); {ex}")
    return float(err.max()) if err.size else 0.0


def sample_positions(M, N, count=2048, seed=0, tile_m=128, tile_n=256):
    """Positions to check at sizes where the full product is too slow for the oracle: every
    corner of the first/last tiles, tile-boundary rows/columns, and uniform random points."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, M - 1, M - 2, min(tile_m - 1, M - 1), min(tile_m, M - 1), M // 2}
    cols = {0, 1, N - 1, N - 2, min(tile_n - 1, N - 1), min(tile_n, N - 1), N // 2}
    pts = [(r, c) for r in rows for c in cols if 0 <= r < M and 0 <= c < N]
    r = rng.integers(0, M, count)
    c = rng.integers(0, N, count)
    pts += list(zip(r.tolist(), c.tolist()))
    pts = sorted(set(pts))
    return np.array([p[0] for p in pts], np.int64), np.array([p[1] for p in pts], np.int64)


def with_packed_scales(M, N, K, kw):
    """kw for a block-scaled gemm_ex call; `pack=True` in kw is replaced by a workspace of the size
    gemm_workspace_size reports, so the one-CTA kernel takes its scales repacked there (checked
    through the plan)."""
    import dense_tensor_core_gb300 as dtc

    kw = dict(kw)
    if not kw.pop("pack", False):
        return kw
    size_kw = {k: kw[k] for k in ("variant", "tile_n", "tile_k") if k in kw}
    for k_in, k_out in (("a_format", "a_format"), ("b_format", "b_format"), ("scale_block", "scale_block")):
        if k_in in kw:
            size_kw[k_out] = kw[k_in]
    nbytes = dtc.gemm_workspace_size("mxfp8", M, N, K, **size_kw)
    assert nbytes > 0
    kw["workspace"] = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    plan_kw = {k: v for k, v in kw.items() if k in ("variant", "tile_n", "tile_k", "a_format",
                                                    "b_format", "scale_block", "workspace")}
    assert dtc.gemm_plan("mxfp8", M, N, K, **plan_kw)["sf_packed"] == 1
    return kw
