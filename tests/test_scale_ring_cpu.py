"""The scale-set ring of the block-scaled kernels, checked by simulation on the CPU.

The repacked-scale paths copy a scale set into Tensor Memory (tcgen05.cp) before the set's first
MMA. A copy and later MMAs run in issue order, but an MMA and a later copy into the columns it
reads do not, so a set's columns may be refilled only once the MMAs that last read them are done.
The kernels skip the explicit wait for that (and the commit it waits for) when the stage ring
already proves it: passing the full barrier of stage n means the MMAs of every stage up to n -
stages are complete, because stage n was refilled only after the commit that followed them. The
kernels encode this as kSfRingSafe = (sets - 1) * group + 1 >= stages * blocks_per_stage, used
only when every tile's K-blocks are a multiple of the set length. This test replays the copy and
MMA schedule of both kernels, with the ring constants read from their headers, and checks that
whenever the kernels skip the wait no copy can overwrite a set whose MMAs might still run."""
import os
import re

import pytest

from conftest import ROOT

CSRC = os.path.join(ROOT, "dense_tensor_core_gb300", "csrc")


def _const(path, name):
    src = open(os.path.join(CSRC, path)).read()
    m = re.search(r"constexpr int " + name + r" = (\d+);", src)
    assert m, (path, name)
    return int(m.group(1))


def kernels():
    return {
        "one-CTA": dict(sets=_const("gemm_mxfp8.cuh", "kSfSets"),
                        stages=_const("gemm_mxfp8.cuh", "kStages"),
                        blocks=_const("gemm_mxfp8.cuh", "kBlocks"), groups=(1, 4)),
        "pair": dict(sets=_const("gemm_mxfp8_2cta.cuh", "kSfSets"),
                     stages=_const("gemm_mxfp8_2cta.cuh", "kNStages"),
                     blocks=_const("gemm_mxfp8_2cta.cuh", "kBlocks"), groups=(4,)),
    }


def ring_safe(sets, stages, blocks, group):
    return (sets - 1) * group + 1 >= stages * blocks


def violations(sets, stages, blocks, group, num_kb, tiles):
    """Copies that could overwrite a set still read by MMAs not yet proven complete, if the
    kernel issued no explicit wait. Global stage n completes its full barrier only after the MMAs
    of every stage <= n - stages are done."""
    last_stage = {}  # global set index -> global stage of its last MMA
    bad = []
    n = 0
    gs_base = 0
    groups = -(-num_kb // group)
    for _ in range(tiles):
        for st in range(-(-num_kb // blocks)):
            for h in range(blocks):
                kb = st * blocks + h
                if kb >= num_kb:
                    break
                g = gs_base + kb // group
                if kb % group == 0 and g - sets >= 0:
                    prev = last_stage[g - sets]
                    if prev > n - stages:
                        bad.append((g, prev, n))
                last_stage[g] = n
            n += 1
        gs_base += groups
    return bad


@pytest.mark.parametrize("name", ["one-CTA", "pair"])
def test_skipped_waits_are_proven_by_the_ring(name):
    k = kernels()[name]
    for group in k["groups"]:
        safe = ring_safe(k["sets"], k["stages"], k["blocks"], group)
        for num_kb in range(1, 40):
            if not (safe and num_kb % group == 0):
                continue  # the kernel waits explicitly here
            for tiles in (1, 2, 3, 7):
                assert not violations(k["sets"], k["stages"], k["blocks"], group, num_kb, tiles), \
                    (name, group, num_kb, tiles)


def test_the_kernels_skip_the_wait_in_their_benchmark_configurations():
    # 32-element blocks on the one-CTA kernel (a set per K-block) and 128-element blocks on the
    # pair kernel (a set per two 256-deep stages) run without the explicit wait
    k = kernels()
    assert ring_safe(k["one-CTA"]["sets"], k["one-CTA"]["stages"], k["one-CTA"]["blocks"], 1)
    assert ring_safe(k["pair"]["sets"], k["pair"]["stages"], k["pair"]["blocks"], 4)


def test_the_simulation_finds_an_unsafe_ring():
    # a ring one stage deeper than the sets can cover: the condition fails, and so does the replay
    sets, group, blocks = 4, 1, 1
    stages = (sets - 1) * group + 2
    assert not ring_safe(sets, stages, blocks, group)
    assert violations(sets, stages, blocks, group, num_kb=16, tiles=2)
