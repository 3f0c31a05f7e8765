// gemm16_2cta.cuh -- persistent bf16/fp16 GEMM on CTA pairs (cluster 2x1, tcgen05 cta_group::2).
//
// The 2-CTA variant named by the 05 Blackwell TCGEN05 GEMM tutorial, "Advanced" (use_2cta with
// cluster_dims (2,1,1), the persistent warp-specialised example), written for sm_103a.
//
// A pair computes a 256 x kBN tile of C. CTA r of the pair (r = 0 is the leader):
//   - loads its own 128 rows of A (rows 256*mt + 128*r) and its own kBN/2 rows of B^T
//     (columns kBN*nt + r*kBN/2 of C) into its own shared memory, kBK-deep K-blocks (64, or 128
//     as two 128-byte K-chunks per 3-D box), a kStages ring; either operand K-major or MN-major
//     (kAMN, kNN); both CTAs' copies complete on the LEADER's full barrier (cp.async.bulk.tensor
//     .cta_group::2), which the leader arms with the bytes of both CTAs;
//   - holds rows 128*r..128*r+127 of the accumulator in its own Tensor Memory.
// The leader's single MMA thread issues tcgen05.mma.cta_group::2 (M = 256, N = kBN, K = 16); the
// tensor cores of both SMs read A and B from both CTAs' shared memory at the same offsets. Each of
// its commits arrives on the empty / accumulator-full barrier at the same offset in both CTAs (one
// tcgen05.commit with .multicast::cluster, mask 0b11). Each CTA's epilogue drains its own 128 rows
// through swizzled shared-memory staging and TMA tensor stores, and arrives on the leader's
// accumulator-empty barrier (8 arrivals: 4 warps x 2 CTAs) once it has read the accumulator.
// Compared with one CTA per 128 x 256 tile, every SM loads half as much of B per FLOP, and a stage
// takes 16 + kBN/8 KiB of shared memory, which leaves room for a deeper ring.
//
// Stream-K (kSK and args.sk_tiles > 0): when the tiles do not fill the last wave, sk_tiles tiles are
// shared out as equal runs of K-blocks over all pairs, before the whole tiles (WorkIter). A pair
// whose run starts inside a tile writes that piece's fp32 partial sums to the workspace and raises
// its flag (release, GPU scope); the pair whose run holds the tile's first K-block waits for those
// flags (acquire, bounded), adds the pieces in K order (deterministic), stores C and lowers the
// flags again, while its MMAs go on with the next tile. A pair waits only at the end of its run,
// for pairs that produce their pieces at the start of theirs, so no cycle of waits can form.
#pragma once

#include "gemm_common.cuh"

namespace dtc {

namespace g2 {
constexpr int kBMc = 128;  // rows of C per CTA
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kAccStride = 256;  // column offset of the second accumulator
constexpr int kGroupM = 8;  // M-tiles per rasterisation group (16 ran level, with ~10 % more DRAM reads)
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
constexpr uint64_t kPeerSettleNs = 1000ull * 1000;  // 1 ms

// K-blocks of 64 (one 128-byte swizzle row; one 2-D box per operand) or 128 (two rows; for
// NT one 3-D box {64, rows, 2} per operand). A TMA instruction's cost does not grow much with its
// size, and measured per-SM delivery is highest with the large 3-D boxes: a 128-deep stage feeds
// the tensor pipe better than two 64-deep ones, although fewer stages fit.
// A B stored [K,N] (kBMN) is loaded as 64-column boxes, kBBoxes per CTA; with a 224-wide tile a
// CTA's 112 columns take two boxes, the second only partly used (the MMA reads 112 columns through
// the MN-major descriptor), so its stage holds whole boxes.
// Ring depth: 6 stages of 64-deep K-blocks; of 128-deep ones 3 for 224- and 256-wide tiles and 4
// for the narrow 64- and 128-wide tiles of small products (a CTA of 1024-deep K then has half its
// K range in flight at once).
constexpr int stages_for(int bn, int bk) { return bk == 128 ? (bn <= 128 ? 4 : 3) : 6; }

template <int kBN, int kBK, int kStages, bool kBMN = false>
struct Cfg {
    static constexpr int kHalfN = kBN / 2;
    static constexpr int kBBoxes = (kHalfN + 63) / 64;
    static constexpr int kAStage = kBMc * kBK * 2;
    static constexpr int kBStage = kBMN ? kBBoxes * 64 * kBK * 2 : kHalfN * kBK * 2;
    static_assert(kBK == 64 || kBK == 128, "K-block of 64 or 128");
    static constexpr int kStageBytes = kAStage + kBStage;
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    // output staging: two 4 KB slots (32 rows x 64 columns of 16-bit C) per epilogue warp
    static constexpr int kCBytes = 4 * 2 * 4096;
    static constexpr int kSmemBytes = kStages * kStageBytes + kCBytes + 1024;
    static_assert(kBN % 32 == 0 && kBN >= 64 && kBN <= 256, "pair tile N must be 64..256, /32");
    static_assert(kSmemBytes <= 227 * 1024 - 256, "shared memory budget");
};
}  // namespace g2

template <bool kBF16, bool kAMN, bool kNN, int kBN, int kBK, int kStages, bool kSK = false>
__global__ void __launch_bounds__(g2::kThreads, 1)
    gemm16_2cta_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC,
                       const __grid_constant__ CUtensorMap tmC32, const Gemm16Args args) {
    using namespace g2;
    using C_ = Cfg<kBN, kBK, kStages, kNN>;
    constexpr int kChunks = kBK / 64;  // 128-byte K-chunks per stage
    static_assert(!kNN || C_::kHalfN % 16 == 0, "B stored [K,N]: 16-column steps per CTA");
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ __align__(8) uint64_t bar_ep;  // stream-K: the epilogue threads are done with a piece
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * C_::kAStage;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int total = args.num_m * args.num_n;  // num_m counts 256-row pair tiles
    const int sk_tiles = kSK ? args.sk_tiles : 0;  // whole tiles only unless built for stream-K
    volatile int* abort = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 8);  // 4 epilogue warps in each CTA
        }
        mbar_init(smem_u32(&bar_drain), 1);
        mbar_init(smem_u32(&bar_ep), 128);
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
            bool ok = true;
            WorkIter wi(pair, num_pairs, total, sk_tiles, args.num_kb);
            WorkItem w;
            int whole = 0;  // whole tiles this pair has loaded
            while (ok && wi.next(w)) {
                int mt, nt;
                tile_coords(w.tile, args.num_m, args.num_n, kGroupM, mt, nt);
                const int a_row = mt * 256 + (int)rank * kBMc;
                const int b_row = nt * kBN + (int)rank * C_::kHalfN;
                // Every other whole tile reads its K-blocks last to first: the pairs move through
                // their tiles in waves, so a wave then starts on the K-slices of the operand panels
                // the wave before read last, which are still in the L2 (4096 x 4096 x 8192: DRAM
                // reads 249 MB against 291, ~1 % faster; 8192^3: 918 MB against 1057). The MMA
                // thread is unaffected: it accumulates whatever K-block a stage holds.
                const bool reverse = w.kind == kWhole && (whole++ & 1);
                for (int kbi = w.k0; kbi < w.k1; ++kbi, ++it) {
                    const int kb = reverse ? w.k0 + w.k1 - 1 - kbi : kbi;
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!wait_bounded(smem_u32(&bar_empty[s]), ph ^ 1u, abort, args.timeout_ns,
                                      args.status, 11)) {
                        ok = false;
                        break;
                    }
                    if (args.fault == 1 && it == 0) continue;  // test hook: stage never filled
                    const uint32_t full_local = smem_u32(&bar_full[s]);
                    const uint32_t full_leader = map_to_cta(full_local, 0);
                    if (leader) mbar_arrive_expect_tx(full_local, 2 * C_::kStageBytes);
                    if constexpr (kAMN) {
                        // A stored [K,M]: two 64-column boxes of kBK K-rows (128-byte swizzle)
                        tma_load_2d_pair(sA + s * C_::kAStage, &tmA, full_leader, a_row, kb * kBK);
                        tma_load_2d_pair(sA + s * C_::kAStage + 64 * kBK * 2, &tmA, full_leader,
                                         a_row + 64, kb * kBK);
                    } else if constexpr (kChunks == 2) {
                        tma_load_3d_pair(sA + s * C_::kAStage, &tmA, full_leader, 0, a_row, kb * 2);
                    } else {
                        tma_load_2d_pair(sA + s * C_::kAStage, &tmA, full_leader, kb * kBK, a_row);
                    }
                    if constexpr (!kNN) {
                        if constexpr (kChunks == 2)
                            tma_load_3d_pair(sB + s * C_::kBStage, &tmB, full_leader, 0, b_row,
                                             kb * 2);
                        else
                            tma_load_2d_pair(sB + s * C_::kBStage, &tmB, full_leader, kb * kBK,
                                             b_row);
                    } else {
#pragma unroll
                        for (int j = 0; j < C_::kBBoxes; ++j)
                            tma_load_2d_pair(sB + s * C_::kBStage + j * (64 * kBK * 2), &tmB,
                                             full_leader, b_row + j * 64, kb * kBK);
                    }
                }
            }
            if (!ok && leader) {
                // The leader's full barriers count both CTAs' copies: let those in flight land.
                const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
                for (uint32_t i = first; i < it; ++i) {
                    if (args.fault == 1 && i == 0) continue;
                    wait_drain(smem_u32(&bar_full[i % kStages]), (i / kStages) & 1u, kDrainNs);
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
            constexpr uint32_t idesc = idesc_f16(kBF16, kNN, 256, kBN, kAMN);
            // Operand descriptors: only the start-address field (bits 0-13: address >> 4)
            // changes, by fixed offsets per stage and per K-step, so it is built once and
            // advanced with 32-bit adds (shared addresses stay below 256 KB: no carry out).
            const uint64_t a_desc0 = smem_desc_sw128(sA, kAMN ? 64 * kBK * 2 : 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(sB, kNN ? 64 * kBK * 2 : 16, 1024);
            const uint32_t a_hi = (uint32_t)(a_desc0 >> 32), b_hi = (uint32_t)(b_desc0 >> 32);
            uint32_t s = 0, ph = 0, acc = 0;
            bool ok = true, issued = false;
            WorkIter wi(pair, num_pairs, total, sk_tiles, args.num_kb);
            WorkItem w;
            while (ok && wi.next(w)) {
                const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
                if (!wait_bounded(smem_u32(&bar_tempty[b]), aph ^ 1u, abort, args.timeout_ns,
                                  args.status, 12)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kAccStride;
                for (int kb = w.k0; kb < w.k1; ++kb) {
                    if (!wait_bounded(smem_u32(&bar_full[s]), ph, abort, args.timeout_ns,
                                      args.status, 13)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_lo = (uint32_t)a_desc0 + s * (uint32_t)(C_::kAStage >> 4);
                    const uint32_t b_lo = (uint32_t)b_desc0 + s * (uint32_t)(C_::kBStage >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // K-major: K-chunk kk/4 of the stage, 32-byte step kk%4 inside its
                        // swizzle row; MN-major: 16 K-rows of 128 bytes per step
                        constexpr int kRowsA = kBMc, kRowsB = C_::kHalfN;
                        const uint32_t a_off =
                            kAMN ? kk * 16 * 128 : (kk / 4) * (kRowsA * 128) + (kk % 4) * 32;
                        const uint32_t b_off =
                            kNN ? kk * 16 * 128 : (kk / 4) * (kRowsB * 128) + (kk % 4) * 32;
                        const uint64_t adesc = ((uint64_t)a_hi << 32) | (a_lo + (a_off >> 4));
                        const uint64_t bdesc = ((uint64_t)b_hi << 32) | (b_lo + (b_off >> 4));
                        mma_f16_cta2(d_tmem, adesc, bdesc, idesc, (kb != w.k0 || kk != 0) ? 1u : 0u);
                    }
                    issued = true;
                    mma_commit_cta2_both(smem_u32(&bar_empty[s]));  // stage free in both CTAs
                    if (++s == (uint32_t)kStages) {
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
        const uint32_t my_slots = base + kStages * C_::kStageBytes + (uint32_t)q * 8192u;
        uint32_t acc = 0, ep_phase = 0, stores = 0;
        WorkIter wi(pair, num_pairs, total, sk_tiles, args.num_kb);
        WorkItem w;
        while (wi.next(w)) {
            int mt, nt;
            tile_coords(w.tile, args.num_m, args.num_n, kGroupM, mt, nt);
            const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
            ++acc;
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded<false, true>(smem_u32(&bar_tfull[b]), aph, abort,
                                               args.timeout_ns, args.status, 14);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            // stream-K: this CTA's workspace slot; for a first piece, the later units whose runs
            // hold the rest of the tile (units pair+1 .. last_unit with a non-empty run)
            int last_unit = pair;
            auto sk_run_empty = [&](int u) {
                return sk_start(u + 1, num_pairs, sk_tiles, args.num_kb) ==
                       sk_start(u, num_pairs, sk_tiles, args.num_kb);
            };
            if (kSK && w.kind == kFirst) {
                const int64_t tile_end = (int64_t)(w.tile + 1) * args.num_kb;
                while (last_unit + 1 < num_pairs &&
                       sk_start(last_unit + 1, num_pairs, sk_tiles, args.num_kb) < tile_end)
                    ++last_unit;
                for (int u = pair + 1; u <= last_unit && ok; ++u) {
                    if (sk_run_empty(u)) continue;  // a unit with no K-blocks wrote nothing
                    const uint32_t* f = args.sk_flags + u * 2 + (int)rank;
                    if (lane == 0) ok = wait_flag_bounded(f, abort, args.timeout_ns, args.status, 15);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok) (void)ld_acquire_gpu_u32(f);  // every lane takes its own acquire
                }
            }
            const int band_y = mt * 256 + (int)rank * kBMc + q * 32;  // C row of lane 0
            const int x0 = nt * kBN;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * kAccStride;
            auto hand_back = [&]() {  // accumulator fully read: back to the MMA issuer
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&bar_tempty[b]), 0));
            };
            // 64-column chunks (and a last 32-column one for 224-wide tiles): TMEM -> registers
            // -> 16-bit in a staging slot -> TMA store
            constexpr int kFull = kBN / 64;
            if (!kSK || w.kind == kWhole) {
                drain_tile16<kBF16, kBN>(taddr, &tmC, &tmC32, my_slots, stores, x0, band_y, args.M,
                                         args.N, lane, hand_back);
            } else if constexpr (kSK) {
                // Pieces of shared tiles, 64-column chunks. The workspace slot of a CTA holds its
                // 128 x 256 fp32 partial sums warp-interleaved (float4 number ((c*4 + q)*16 + g)*32
                // + lane = columns 64c + 4g .. +3 of row 32q + lane), so every warp-wide access
                // moves 512 contiguous bytes.
                static_assert(kBN % 64 == 0, "stream-K tiles are 64-column multiples");
                float4* const mine4 = reinterpret_cast<float4*>(
                    args.sk_partial + (size_t)(pair * 2 + (int)rank) * kBMc * kBN);
                auto piece4 = [&](int u, int c, int g) -> const float4* {
                    return mine4 + (size_t)(u - pair) * 2 * kBMc * kBN / 4 +
                           ((c * 4 + q) * 16 + g) * 32 + lane;
                };
#pragma unroll 1
                for (int c = 0; c < kFull; ++c) {
                    uint32_t v[64];
                    tmem_load_64cols(taddr + c * 64, v);
                    if (c == kFull - 1) hand_back();
                    if (!ok) continue;
                    if (w.kind == kOther) {  // partial sums of a piece another unit finishes
#pragma unroll
                        for (int g = 0; g < 16; ++g)
                            mine4[((c * 4 + q) * 16 + g) * 32 + lane] =
                                make_float4(__uint_as_float(v[g * 4 + 0]), __uint_as_float(v[g * 4 + 1]),
                                            __uint_as_float(v[g * 4 + 2]), __uint_as_float(v[g * 4 + 3]));
                        continue;
                    }
                    // the later pieces, added in K order, two pieces' loads in flight at a time
                    int u = pair + 1;
                    while (true) {
                        while (u <= last_unit && sk_run_empty(u)) ++u;
                        if (u > last_unit) break;
                        int u2 = u + 1;
                        while (u2 <= last_unit && sk_run_empty(u2)) ++u2;
                        const bool two = u2 <= last_unit;
                        float4 pa[16], pb[16];
#pragma unroll
                        for (int g = 0; g < 16; ++g) pa[g] = ld_global_cg_f4(piece4(u, c, g));
                        if (two) {
#pragma unroll
                            for (int g = 0; g < 16; ++g) pb[g] = ld_global_cg_f4(piece4(u2, c, g));
                        }
#pragma unroll
                        for (int g = 0; g < 16; ++g) {
                            v[g * 4 + 0] = __float_as_uint(__uint_as_float(v[g * 4 + 0]) + pa[g].x);
                            v[g * 4 + 1] = __float_as_uint(__uint_as_float(v[g * 4 + 1]) + pa[g].y);
                            v[g * 4 + 2] = __float_as_uint(__uint_as_float(v[g * 4 + 2]) + pa[g].z);
                            v[g * 4 + 3] = __float_as_uint(__uint_as_float(v[g * 4 + 3]) + pa[g].w);
                        }
                        if (two) {
#pragma unroll
                            for (int g = 0; g < 16; ++g) {
                                v[g * 4 + 0] = __float_as_uint(__uint_as_float(v[g * 4 + 0]) + pb[g].x);
                                v[g * 4 + 1] = __float_as_uint(__uint_as_float(v[g * 4 + 1]) + pb[g].y);
                                v[g * 4 + 2] = __float_as_uint(__uint_as_float(v[g * 4 + 2]) + pb[g].z);
                                v[g * 4 + 3] = __float_as_uint(__uint_as_float(v[g * 4 + 3]) + pb[g].w);
                            }
                        }
                        u = u2 + 1;
                    }
                    store_chunk16<kBF16, 64>(&tmC, my_slots, stores, v, x0 + c * 64, band_y,
                                             args.M, args.N, lane);
                }
            }
            if (kSK && w.kind != kWhole) {
                // every epilogue thread of this CTA is done with the piece (an mbarrier, so a
                // thread that gave up cannot leave the others waiting without a bound)
                mbar_arrive(smem_u32(&bar_ep));
                if (warp == 2 && lane == 0) {
                    const bool all = wait_bounded(smem_u32(&bar_ep), ep_phase, abort,
                                                  args.timeout_ns, args.status, 16);
                    if (all && ok) {
                        if (w.kind == kOther) {
                            __threadfence();
                            st_release_gpu_u32(args.sk_flags + pair * 2 + (int)rank, 1u);
                        } else {
                            for (int u = pair + 1; u <= last_unit; ++u)  // consumed: back to zero
                                if (!sk_run_empty(u)) args.sk_flags[u * 2 + (int)rank] = 0u;
                        }
                    }
                }
                ep_phase ^= 1u;
            }
            if (!ok) break;
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
