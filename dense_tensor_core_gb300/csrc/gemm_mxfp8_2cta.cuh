// gemm_mxfp8_2cta.cuh -- persistent block-scaled GEMM on CTA pairs (cluster 2x1, tcgen05
// cta_group::2), NT layout: fp8 / fp6 / fp4 elements (e4m3, e5m2, e2m3, e3m2, e2m1 for A and B
// independently) with one E8M0 scale per row per 128 K-elements, fp32 accumulation in Tensor
// Memory, bf16 output.
//
// The product of gemm_mxfp8.cuh (05 Blackwell TCGEN05 GEMM tutorial, "Advanced": gemm_blockscaled
// with granularity 128 for both operands, and "other block-scaled formats"), on the operand feed
// that keeps the tensor pipe busiest on GB300: a pair computes a 256 x 224 tile; CTA r loads its
// own 128 rows of A and its own 112 rows of B^T, 256 K-elements per stage, each operand in one 3-D
// box {128 bytes, rows, 2} over the array viewed as [K/128][rows][128 bytes] (one 128-byte swizzled
// row per operand row and K-block, whatever the element format: fp6 / fp4 rows are unpacked by the
// tensor memory access unit into 16-byte groups), 32 KB of A and 28 KB of B per CTA per stage, in
// a ring of 3 stages (K % 128 == 0). A TMA instruction that moves more bytes streams faster per
// SM, which the fp8 rate needs: 2-D boxes of one K-block per stage, in a ring of 6, ran 118.8 us
// on 4096 x 4096 x 8192 against 102.4 here. Both CTAs' copies complete on the leader's full
// barrier; the leader's single MMA thread issues
// tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X (M = 256, N = 224, K = 32),
// eight per stage, with descriptors advanced by 32-bit adds, and releases each stage in both CTAs
// with one multicast commit.
//
// Scales, as in the one-CTA kernel: R rows take R/32 Tensor Memory columns (row r in lane r % 32
// of column r / 32, repeated in all four lane quarters); one 32-bit cell packs the scale bytes of
// 4 consecutive 128-element K-blocks of a row, selected by a_sf_id / b_sf_id = K-block % 4. Each
// CTA holds the scales of its own 128 A rows and of all 224 B rows (each CTA's datapath computes
// all 224 columns of its rows). They come repacked by sf_pack_kernel (sf_pack.cuh) into the
// caller's workspace: each CTA's producer loads, beside the stage that holds a scale set's first
// K-block, the 512-byte chunk of its own 128 A rows and the two chunks of the tile's B rows (2-D
// boxes of 512 and 1024 bytes completing on the leader's full barrier), and the leader's MMA
// thread moves them into both CTAs' Tensor Memory with three tcgen05.cp.cta_group::2.32x128b.warpx4
// before the set's first MMA (each CTA copies from its own shared memory). That point, where the
// MMAs change scale set anyway and the stage's operands have landed, is where the copies cost
// least: copies issued a stage earlier (between two MMAs of one set), ahead of the full-barrier
// wait, or from a second thread all measured slower.
//
// Tensor Memory per CTA: accumulators at columns [0,224) and [224,448), scale sets at
// 448 + 12*set (4 columns for A, 8 for B), set = 0..3.
#pragma once

#include "gemm_mxfp8.cuh"

namespace dtc {

namespace gmx2 {
constexpr int kBMc = 128;   // rows of C per CTA
constexpr int kBN = 224;    // columns of C per pair tile
constexpr int kHalfN = kBN / 2;
constexpr int kBK = 128;    // K-elements per K-block: one 128-byte swizzled row per operand row
constexpr int kBlocks = 2;  // K-blocks per stage
constexpr int kNStages = 3;
constexpr int kThreads = 192;  // producer, MMA, 4 epilogue warps
constexpr int kAChunk = kBMc * 128;    // one K-block of the CTA's 128 rows of A
constexpr int kBChunk = kHalfN * 128;  // one K-block of its 112 rows of B
constexpr int kAStg = kAChunk * kBlocks;
constexpr int kBStage = kBChunk * kBlocks;
constexpr int kStageBytes = kAStg + kBStage;
constexpr int kCBytes = 4 * 2 * 4096;  // two 4 KB output staging slots per epilogue warp
constexpr int kTmemCols = 512;
constexpr int kAccStride = kBN;
constexpr int kSfBase = 2 * kBN;       // after the two accumulators
constexpr int kSfSet = 12;
constexpr int kSfSets = 4;
constexpr int kGroup = 4;  // K-blocks per scale set
constexpr int kSlotBytes = gmx::kSfSetBytes;  // a stage starts at most one scale set
constexpr int kSmemBytes = kNStages * (kStageBytes + kSlotBytes) + kCBytes + 1024;
constexpr int kGroupM = 8;
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
constexpr uint64_t kPeerSettleNs = 1000ull * 1000;
static_assert(kBChunk % 1024 == 0, "chunks keep the 1024-byte swizzle alignment");
static_assert(kAStg % 1024 == 0 && kBStage % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
static_assert(kSmemBytes <= 227 * 1024 - 512, "shared memory budget");
static_assert(kSfBase + kSfSets * kSfSet <= kTmemCols, "Tensor Memory budget");
static_assert(kGroup % kBlocks == 0, "scale sets start at stage boundaries");
}  // namespace gmx2

// (A template so that every translation unit that includes this header may define it; the one
// instantiation is the 224-wide tile.)
template <int kTileN = gmx2::kBN>
__global__ void __launch_bounds__(gmx2::kThreads, 1)
    gemm_mxfp8_2cta_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC,
                           const __grid_constant__ CUtensorMap tmC32,
                           const __grid_constant__ CUtensorMap tmSA,
                           const __grid_constant__ CUtensorMap tmSB, const GemmMxArgs args) {
    using namespace gmx2;
    static_assert(kTileN == kBN, "one tile width");
    constexpr int kNS = kNStages;
    constexpr int grp = kGroup;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kNS];
    __shared__ __align__(8) uint64_t bar_empty[kNS];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_sempty[kSfSets];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t sB = base + kNS * kAStg;
    const uint32_t sSF = base + kNS * kStageBytes + kCBytes;  // scale slots
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int total = args.num_m * args.num_n;  // num_m counts 256-row pair tiles
    const int num_st = (args.num_kb + kBlocks - 1) / kBlocks;  // stages per tile
    // Refilling a scale set's columns needs the MMAs that last read them done. Passing a stage's
    // full barrier already proves every MMA of the stages a whole ring earlier done (the stage was
    // refilled only after the commit that followed them), so with full sets (every tile's K-blocks
    // a multiple of the set length) spaced at least a ring apart the explicit wait, and the commit
    // it waits for, are not needed.
    constexpr bool kSfRingSafe = (kSfSets - 1) * grp + 1 >= kNS * kBlocks;
    const bool sf_wait = !(kSfRingSafe && args.num_kb % grp == 0);
    volatile int* abort = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 8);  // 4 epilogue warps in each CTA
        }
        for (int b = 0; b < kSfSets; ++b) mbar_init(smem_u32(&bar_sempty[b]), 1);
        mbar_init(smem_u32(&bar_drain), 1);
        abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc<2>(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish<2>();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any copy or arrival targets them
    tc_fence_after_sync();
    const uint32_t tmem_base = tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer (both CTAs) ------------------------------
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true, chunks_ready = false;
            for (int t = pair; t < total && ok; t += num_pairs) {
                int mt, nt;
                tile_coords(t, args.num_m, args.num_n, kGroupM, mt, nt);
                const int a_row = mt * 256 + (int)rank * kBMc;
                const int b_row = nt * kBN + (int)rank * kHalfN;
                for (int st = 0; st < num_st; ++st, ++it) {
                    const uint32_t s = it % kNS, ph = (it / kNS) & 1u;
                    if (!wait_bounded(smem_u32(&bar_empty[s]), ph ^ 1u, abort, args.timeout_ns,
                                      args.status, 41)) {
                        ok = false;
                        break;
                    }
                    if (args.fault == 1 && it == 0) continue;  // test hook: stage never filled
                    const uint32_t full_local = smem_u32(&bar_full[s]);
                    const uint32_t full_leader = map_to_cta(full_local, 0);
                    const int kb0 = st * kBlocks;
                    const bool set_start = kb0 % grp == 0;  // a scale set starts in this stage
                    if (leader)  // both CTAs' bytes
                        mbar_arrive_expect_tx(full_local,
                                              args.stage_tx + (set_start ? 2 * gmx::kSfSetBytes : 0));
                    // one 3-D box of two 128-byte K-chunks per operand
                    tma_load_3d_pair(sA + s * kAStg, &tmA, full_leader, 0, a_row, st * 2);
                    tma_load_3d_pair(sB + s * kBStage, &tmB, full_leader, 0, b_row, st * 2);
                    if (set_start) {
                        // this CTA's A chunk (its 128-row group) and the tile's two B chunks, as
                        // rows of 128 bytes of the repacked arrays; the kernel that writes them
                        // may still be running (it launched this one early)
                        if (!chunks_ready) {
                            grid_dependency_wait();
                            chunks_ready = true;
                        }
                        const int g = kb0 / grp;
                        const uint32_t slot = sSF + s * kSlotBytes;
                        tma_load_2d_pair(slot, &tmSA, full_leader, 0,
                                         ((mt * 2 + (int)rank) * args.sf_sets + g) * 4);
                        tma_load_2d_pair(slot + kSfChunkBytes, &tmSB, full_leader, 0,
                                         (nt * args.sf_sets + g) * 8);
                    }
                }
            }
            if (!ok && leader) {
                // The leader's full barriers count both CTAs' copies: let those in flight land.
                const uint32_t first = it > (uint32_t)kNS ? it - kNS : 0;
                for (uint32_t i = first; i < it; ++i) {
                    if (args.fault == 1 && i == 0) continue;
                    wait_drain(smem_u32(&bar_full[i % kNS]), (i / kNS) & 1u, kDrainNs);
                }
            } else if (!ok) {
                // The peer's copies complete on the leader's barriers, which it cannot observe:
                // give them a fixed, bounded time to land before this CTA may exit.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < kPeerSettleNs) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer (leader CTA) ------------------------------
        if (lane == 0 && leader) {
            const uint32_t idesc0 = idesc_mxf8(256, kBN, 0, 0) | args.fmt_bits;
            // Operand descriptors: only the start-address field (bits 0-13: address >> 4) changes,
            // by fixed offsets per stage and per K-step (32 bytes), so it is built once and
            // advanced with 32-bit adds (shared addresses stay below 256 KB: no carry out).
            const uint64_t a_desc0 = smem_desc_sw128(sA, 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(sB, 16, 1024);
            const uint32_t a_hi = (uint32_t)(a_desc0 >> 32), b_hi = (uint32_t)(b_desc0 >> 32);
            uint32_t s = 0, ph = 0, acc = 0, sit = 0;
            bool ok = true, issued = false;
            for (int t = pair; t < total && ok; t += num_pairs) {
                const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
                if (!wait_bounded<true>(smem_u32(&bar_tempty[b]), aph ^ 1u, abort, args.timeout_ns,
                                        args.status, 42)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kAccStride;
                for (int st = 0; st < num_st && ok; ++st) {
                    if (!wait_bounded(smem_u32(&bar_full[s]), ph, abort, args.timeout_ns,
                                      args.status, 43)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll
                    for (int h = 0; h < kBlocks; ++h) {
                        const int kb = st * kBlocks + h;
                        if (kb >= args.num_kb) break;  // a K-block past K: zero-filled, skipped
                        const uint32_t set = sit % kSfSets;
                        if (kb % grp == 0) {
                            // the first K-block of a scale set: its columns are free once the
                            // MMAs that last read them are done; then both CTAs copy the set
                            // from the stage's slot
                            if (sf_wait) {
                                if (!wait_bounded(smem_u32(&bar_sempty[set]),
                                                  ((sit / kSfSets) & 1u) ^ 1u, abort,
                                                  args.timeout_ns, args.status, 47)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after_sync();
                            }
                            const uint32_t slot = sSF + s * kSlotBytes;
                            const uint32_t col = tmem_base + kSfBase + set * kSfSet;
                            tmem_cp_32x128b_x4_cta2(col, smem_desc_plain(slot, 128, 128));
                            tmem_cp_32x128b_x4_cta2(
                                col + 4, smem_desc_plain(slot + kSfChunkBytes, 128, 128));
                            tmem_cp_32x128b_x4_cta2(
                                col + 8, smem_desc_plain(slot + 2 * kSfChunkBytes, 128, 128));
                        }
                        // K-block h of the stage: 128-byte chunk h of each operand's box
                        const uint32_t a_lo = (uint32_t)a_desc0 + s * (uint32_t)(kAStg >> 4) +
                                              (uint32_t)h * (uint32_t)(kAChunk >> 4);
                        const uint32_t b_lo = (uint32_t)b_desc0 + s * (uint32_t)(kBStage >> 4) +
                                              (uint32_t)h * (uint32_t)(kBChunk >> 4);
                        const uint32_t sfa = tmem_base + kSfBase + set * kSfSet;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t sf_id = (uint32_t)(kb & 3);
                            const uint32_t idesc = idesc0 | (sf_id << 4) | (sf_id << 29);
                            const uint64_t adesc = ((uint64_t)a_hi << 32) | (a_lo + 2u * kk);
                            const uint64_t bdesc = ((uint64_t)b_hi << 32) | (b_lo + 2u * kk);
                            mma_mxf8_cta2(d_tmem, adesc, bdesc, idesc, sfa, sfa + 4,
                                          (kb | kk) != 0 ? 1u : 0u);
                        }
                        issued = true;
                        if (kb % grp == grp - 1 || kb == args.num_kb - 1) {
                            if (sf_wait)  // set consumed
                                mma_commit_cta2_both(smem_u32(&bar_sempty[set]));
                            ++sit;
                        }
                    }
                    if (!ok) break;
                    mma_commit_cta2_both(smem_u32(&bar_empty[s]));  // stage free in both CTAs
                    if (++s == (uint32_t)kNS) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_cta2_both(smem_u32(&bar_tfull[b]));
                ++acc;
            }
            if (!ok && issued) {
                mma_commit_cta2(smem_u32(&bar_drain));
                wait_drain(smem_u32(&bar_drain), 0, kDrainNs);
            }
        }
    } else {
        // ------------------------------ epilogue (warps 2..5, both CTAs) ---------------------
        const int q = warp & 3;
        const uint32_t my_slots = base + kNS * kStageBytes + (uint32_t)q * 8192u;
        uint32_t acc = 0, stores = 0;
        for (int t = pair; t < total; t += num_pairs, ++acc) {
            int mt, nt;
            tile_coords(t, args.num_m, args.num_n, kGroupM, mt, nt);
            const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded<false, true>(smem_u32(&bar_tfull[b]), aph, abort,
                                               args.timeout_ns, args.status, 44);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * kAccStride;
            drain_tile16<true, kBN>(taddr, &tmC, &tmC32, my_slots, stores, nt * kBN,
                                    mt * 256 + (int)rank * kBMc + q * 32, args.M, args.N, lane,
                                    [&]() {
                                        tc_fence_before_sync();
                                        __syncwarp();
                                        if (lane == 0)
                                            mbar_arrive_cluster(map_to_cta(smem_u32(&bar_tempty[b]), 0));
                                    });
        }
        if (lane == 0) bulk_wait_group_read<0>();  // the C stores have read their slots
        __syncwarp();
    }

    // ------------------------------ teardown ------------------------------
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still signal its barriers
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem_base, kTmemCols);
    }
}

}  // namespace dtc
