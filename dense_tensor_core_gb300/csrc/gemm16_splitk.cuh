// gemm16_splitk.cuh -- bf16/fp16 GEMM with K split across the CTAs of a cluster, for products
// with too few output tiles to occupy the GPU (the skinny, memory-bound M = 128 case, and small
// M x N with a long K).
//
// C[M,N] = A[M,K] . Bop as in the one-CTA kernel (128 x kBN tiles, kBK-deep K-blocks, TMA producer
// warp, single-thread tcgen05.mma issuer, Tensor Memory accumulator), but a cluster of kS CTAs
// computes one tile: CTA r accumulates the r-th of kS contiguous K-ranges. The partial sums are
// reduced on chip, without a global workspace. Split in 2, CTA r owns columns
// [r*kBN/2, (r+1)*kBN/2) of the tile (all 128 rows): each epilogue warp copies its 32 rows of the
// peer's columns into the peer's exchange area, then sums its rows of its own columns with the
// copy it received and stores them, so all four warps share the reduction. Split in 4, CTA r owns
// rows [r*32, (r+1)*32) (one 32-lane quarter of the accumulator):
//   1. an epilogue warp whose quarter another CTA owns reads it from Tensor Memory, 64 columns
//      per round trip, into a staging copy in its own ring (idle once the last MMA has
//      completed), laid out as the owner's exchange area is, and hands each 64-column piece to
//      the copy engine as soon as it is staged: one bulk shared-memory copy into the owner's
//      exchange area, counted in bytes on the owner's barrier for that piece (the owner armed it
//      with the bytes it expects);
//   2. an epilogue warp whose quarter this CTA owns takes the pieces in order: once a piece's
//      barrier completes it sums its own accumulator columns with the kS - 1 copies in the
//      fixed order 0..kS-1 (the result does not depend on which CTA finished first), rounds once
//      to the output type into a swizzled staging slot over the idle ring and stores it with a
//      TMA tensor store, while later pieces are still in flight;
//   3. cluster barrier (no CTA leaves while a copy into it, or out of it, may be in flight).
// The exchange area is a region of its own, not the ring, so no CTA waits for a peer's main loop
// to end before copying into it. The exchange is laid out piece-major ([piece][row][64 floats],
// the 16-byte chunk j of row r stored at chunk position j ^ (r % 8), so that a warp's lanes,
// one row each, hit distinct banks) so that each copy is one contiguous range; whole-piece bulk copies move full 32-byte
// sectors over the cluster network, where per-lane 16-byte remote stores to 32 different rows
// would move half-filled ones. The start-up cluster barrier is split: every thread arrives after
// the set-up, and a thread waits only before its first copy into a peer (or at the end), so the
// main loop does not wait for the other CTAs to start.
// One cluster per tile, not persistent: a product of T tiles launches T * kS CTAs. With kS = 1 (64-
// wide tiles) a CTA takes the whole K of its tile and stores it itself: no exchange, no reduction
// (the skinny product: 128 CTAs, each streaming its 64 rows of B once with all of A from the L2).
#pragma once

#include "gemm_common.cuh"

namespace dtc {

namespace gsk {
constexpr int kBM = 128;
constexpr int kThreads = 192;
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;

// Ring depth: as many stages as fit beside the exchange area, at most 6.
constexpr int stages_for(int bn, int bk, int s) {
    const int room = 227 * 1024 - 256 - 1024 - (s - 1) * (kBM / s) * (bn * 4);
    const int n = room / (kBM * bk * 2 + bn * bk * 2);
    return n < 6 ? n : 6;
}

// K-blocks of 64 (one 128-byte swizzle row, one 2-D box per operand) or 128 (two rows; for A and
// for B in NT one 3-D box {64, rows, 2}).
template <int kBN, int kBK, int kStages, int kS>
struct Cfg {
    static constexpr int kAStage = kBM * kBK * 2;
    static constexpr int kBStage = kBN * kBK * 2;
    static constexpr int kStageBytes = kAStage + kBStage;
    static constexpr int kRing = kStages * kStageBytes;
    static constexpr int kPieces = kBN / 64;             // 64-column pieces of a row
    static constexpr int kXPitch = 64 * 4;               // fp32 piece row (16-byte chunks swizzled)
    static constexpr int kBandRows = kBM / kS;           // rows of the tile one CTA owns
    static constexpr int kXSlot = kPieces * kBandRows * kXPitch;  // one peer's band
    static constexpr int kXBytes = (kS - 1) * kXSlot;             // one band from each peer
    static constexpr int kXPieceBytes = (kS - 1) * kBandRows * kXPitch;  // expected per piece
    static constexpr int kSmemBytes = kRing + kXBytes + 1024;
    static constexpr int kTmemCols = kBN <= 128 ? 128 : 256;
    static constexpr int kQPieceBytes = 32 * kXPitch;                   // one quarter's piece
    static constexpr int kStaging = (4 - 4 / kS) * kPieces * kQPieceBytes;  // all pushed quarters
    // Split in 2: each CTA owns half of the tile's columns (kOwnPieces 64-column pieces, all 128
    // rows), so every epilogue warp pushes and reduces alike; split in 4: each owns 32 rows.
    static constexpr bool kColOwn = kS == 2;
    static constexpr int kOwnPieces = kPieces / 2;
    static constexpr int kColPieceBytes = kBM * kXPitch;  // one owned piece, all 128 rows
    static_assert(!kColOwn || kOwnPieces * kColPieceBytes == kXBytes, "same exchange area");
    // the owner warps' output staging (two 4 KB slots each) follows the pushed pieces
    static constexpr int kCStaging = kStaging + (kColOwn ? 4 : 4 / kS) * 2 * 4096;
    static_assert(kCStaging <= kRing, "the staging copies must fit over the ring");
    static_assert(kBK == 64 || kBK == 128, "K-block of 64 or 128");
    static_assert(kS == 1 || kS == 2 || kS == 4, "K split over 1, 2 or 4 CTAs");
    static_assert(kBN % 64 == 0 && kBN <= 256, "the accumulator is read 64 columns at a time");
    static_assert(kSmemBytes <= 227 * 1024 - 256, "shared memory budget");
};
}  // namespace gsk

// One arrival on bar_ack of every other CTA of the cluster (release at cluster scope).
template <int kS>
__device__ __forceinline__ void ack_peers_n(uint32_t rank, uint32_t bar_ack) {
#pragma unroll
    for (uint32_t r = 0; r < (uint32_t)kS; ++r)
        if (r != rank) mbar_arrive_cluster(map_to_cta(bar_ack, r));
}

template <bool kBF16, bool kAMN, bool kNN, int kBN, int kBK, int kStages, int kS>
__global__ void __launch_bounds__(gsk::kThreads, 1)
    gemm16_splitk_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const Gemm16Args args) {
    using namespace gsk;
    using C_ = Cfg<kBN, kBK, kStages, kS>;
    constexpr int kChunks = kBK / 64;    // 128-byte K-chunks per stage
    constexpr int kQPerBand = 4 / kS;    // accumulator quarters per owned band
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull;
    __shared__ __align__(8) uint64_t bar_xchg[C_::kPieces];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ __align__(8) uint64_t bar_ack;  // every owner this CTA copied into has seen it land
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * C_::kAStage;
    const uint32_t sX = base + C_::kRing;  // exchange area: peers' partial sums of owned rows
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int tile = blockIdx.x / kS;
    const int mt = tile / args.num_n;
    const int nt = tile - mt * args.num_n;
    const int kb0 = (int)((int64_t)rank * args.num_kb / kS);
    const int kb1 = (int)((int64_t)(rank + 1) * args.num_kb / kS);
    volatile int* abort = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        mbar_init(smem_u32(&bar_tfull), 1);
        // each armed once with every byte the peers will copy into its piece
        for (int c = 0; c < C_::kPieces; ++c) {
            mbar_init(smem_u32(&bar_xchg[c]), 1);
            if (!C_::kColOwn)
                mbar_arrive_expect_tx(smem_u32(&bar_xchg[c]), C_::kXPieceBytes);
            else if (c < C_::kOwnPieces)
                mbar_arrive_expect_tx(smem_u32(&bar_xchg[c]), C_::kColPieceBytes);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        if constexpr (kS > 1) mbar_init(smem_u32(&bar_ack), kS - 1);  // one from each other CTA
        abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(&tmem_slot), C_::kTmemCols);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_arrive();  // this CTA's exchange barriers exist (a peer waits before copying in)
    bool cluster_waited = false;
    tc_fence_after_sync();
    const uint32_t tmem_base = tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!wait_bounded(smem_u32(&bar_empty[s]), ph ^ 1u, abort, args.timeout_ns,
                                  args.status, 21)) {
                    ok = false;
                    break;
                }
                if (args.fault == 1 && it == 0) continue;  // test hook: stage never filled
                const uint32_t full = smem_u32(&bar_full[s]);
                mbar_arrive_expect_tx(full, C_::kStageBytes);
                if constexpr (kAMN) {
                    // A stored [K,M]: two 64-column boxes of kBK K-rows (128-byte swizzle)
                    tma_load_2d(sA + s * C_::kAStage, &tmA, full, mt * kBM, kb * kBK);
                    tma_load_2d(sA + s * C_::kAStage + 64 * kBK * 2, &tmA, full, mt * kBM + 64,
                                kb * kBK);
                } else if constexpr (kChunks == 2) {
                    tma_load_3d(sA + s * C_::kAStage, &tmA, full, 0, mt * kBM, kb * 2);
                } else {
                    tma_load_2d(sA + s * C_::kAStage, &tmA, full, kb * kBK, mt * kBM);
                }
                if constexpr (!kNN) {
                    if constexpr (kChunks == 2)
                        tma_load_3d(sB + s * C_::kBStage, &tmB, full, 0, nt * kBN, kb * 2);
                    else
                        tma_load_2d(sB + s * C_::kBStage, &tmB, full, kb * kBK, nt * kBN);
                } else {
#pragma unroll
                    for (int j = 0; j < kBN / 64; ++j)
                        tma_load_2d(sB + s * C_::kBStage + j * (64 * kBK * 2), &tmB, full,
                                    nt * kBN + j * 64, kb * kBK);
                }
            }
            if (!ok) {
                const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
                for (uint32_t i = first; i < it; ++i) {
                    if (args.fault == 1 && i == 0) continue;
                    wait_drain(smem_u32(&bar_full[i % kStages]), (i / kStages) & 1u, kDrainNs);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kBF16, kNN, kBM, kBN, kAMN);
            uint32_t it = 0;
            bool ok = true, issued = false;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!wait_bounded(smem_u32(&bar_full[s]), ph, abort, args.timeout_ns,
                                  args.status, 23)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a0 = sA + s * C_::kAStage, b0 = sB + s * C_::kBStage;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    // K-chunk kk/4 of the stage, 32-byte step kk%4 inside its swizzle row
                    const uint32_t koff = (kk % 4) * 32;
                    const uint64_t adesc =
                        kAMN ? smem_desc_sw128(a0 + kk * 16 * 128, 64 * kBK * 2, 1024)
                                  : smem_desc_sw128(a0 + (kk / 4) * (kBM * 128) + koff, 16, 1024);
                    const uint64_t bdesc =
                        kNN ? smem_desc_sw128(b0 + kk * 16 * 128, 64 * kBK * 2, 1024)
                            : smem_desc_sw128(b0 + (kk / 4) * (kBN * 128) + koff, 16, 1024);
                    mma_f16_cta1(tmem_base, adesc, bdesc, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                }
                issued = true;
                mma_commit_cta1(smem_u32(&bar_empty[s]));
            }
            if (ok) {
                mma_commit_cta1(smem_u32(&bar_tfull));  // with no K-blocks this arrives at once
            } else if (issued) {
                mma_commit_cta1(smem_u32(&bar_drain));
                wait_drain(smem_u32(&bar_drain), 0, kDrainNs);
            }
        }
    } else {
        // ------------------------------ epilogue (warps 2..5) ------------------------------
        const int q = warp & 3;  // Tensor Memory lane quarter this warp may access
        if constexpr (C_::kColOwn) {
            // Split in 2, column ownership: CTA r owns pieces [r*kOwnPieces, (r+1)*kOwnPieces).
            // Every warp first copies its 32 rows of the peer's pieces into the peer's exchange
            // area (piece j of the peer at rows 32q..32q+31, the bytes counted on the peer's
            // bar_xchg[j]), then sums its rows of its own pieces with the peer's copies, in rank
            // order, and stores them.
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
            const bool empty_slice = kb1 <= kb0;  // no K-blocks: this CTA's share is zero
            const uint32_t peer = rank ^ 1u;
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_u32(&bar_tfull), 0, abort, args.timeout_ns, args.status, 24);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) tc_fence_after_sync();
            cluster_wait();  // the peer's barriers exist
            cluster_waited = true;
            if (ok) {
                const uint32_t stage = sA + (uint32_t)q * (C_::kOwnPieces * C_::kQPieceBytes);
#pragma unroll 1
                for (int j = 0; j < C_::kOwnPieces; ++j) {
                    uint32_t v[64];
                    tmem_load_64cols(taddr + (peer * C_::kOwnPieces + j) * 64, v);
                    const uint32_t spiece = stage + j * C_::kQPieceBytes;
                    const uint32_t srow = spiece + lane * C_::kXPitch;
#pragma unroll
                    for (int g = 0; g < 16; ++g) {
                        const uint32_t a = srow + ((g ^ (lane & 7)) << 4);
                        if (empty_slice)
                            st_shared_u4(a, 0u, 0u, 0u, 0u);
                        else
                            st_shared_u4(a, v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]);
                    }
                    fence_proxy_async_smem();  // the staging writes, before the copy engine reads
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t dst = sX + (j * kBM + q * 32) * C_::kXPitch;
                        bulk_copy_smem_to_cta(map_to_cta(dst, peer), spiece, C_::kQPieceBytes,
                                              map_to_cta(smem_u32(&bar_xchg[j]), peer));
                    }
                }
                const uint32_t my_slots = sA + C_::kStaging + (uint32_t)q * 8192u;
                uint32_t stores = 0;
#pragma unroll 1
                for (int j = 0; j < C_::kOwnPieces; ++j) {
                    const int gp = (int)rank * C_::kOwnPieces + j;  // piece index within the tile
                    uint32_t v[64];
                    tmem_load_64cols(taddr + gp * 64, v);  // own partial sums, ready since tfull
                    int xok = 1;
                    if (lane == 0)
                        xok = wait_bounded<true>(smem_u32(&bar_xchg[j]), 0, abort, args.timeout_ns,
                                                 args.status, 25);
                    xok = __shfl_sync(0xffffffffu, xok, 0);
                    if (!xok) break;
                    // the phase has completed: every lane takes its own acquire of it
                    (void)mbar_try_wait_cluster(smem_u32(&bar_xchg[j]), 0);
                    if (j == C_::kOwnPieces - 1 && q == 0 && lane == 0)
                        ack_peers_n<kS>(rank, smem_u32(&bar_ack));  // every copy into this CTA landed
                    const uint32_t xrow = sX + (j * kBM + q * 32 + lane) * C_::kXPitch;
                    float acc[64];
#pragma unroll
                    for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
#pragma unroll
                    for (int src = 0; src < 2; ++src) {  // rank order: the same sum either way
                        if (src == (int)rank) {
#pragma unroll
                            for (int i = 0; i < 64; ++i)
                                acc[i] += empty_slice ? 0.0f : __uint_as_float(v[i]);
                        } else {
#pragma unroll
                            for (int g = 0; g < 16; ++g) {
                                const float4 pp = ld_shared_f4(xrow + ((g ^ (lane & 7)) << 4));
                                acc[g * 4 + 0] += pp.x;
                                acc[g * 4 + 1] += pp.y;
                                acc[g * 4 + 2] += pp.z;
                                acc[g * 4 + 3] += pp.w;
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = __float_as_uint(acc[i]);
                    store_chunk16<kBF16, 64>(&tmC, my_slots, stores, v, nt * kBN + gp * 64,
                                             mt * kBM + q * 32, args.M, args.N, lane);
                }
                if (lane == 0) bulk_wait_group_read<0>();  // the C stores have read their slots
                __syncwarp();
            }
        } else {
            const uint32_t owner = (uint32_t)(q / kQPerBand);
            const int qb = q % kQPerBand;  // quarter within the owner's band
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
            const bool empty_slice = kb1 <= kb0;  // no K-blocks: this CTA's share is zero
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_u32(&bar_tfull), 0, abort, args.timeout_ns, args.status, 24);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) tc_fence_after_sync();
            if (owner != rank) {
                // stage this quarter piece by piece in the ring and copy each piece into the owner's
                // exchange area, in the slot of source rank `rank`
                const uint32_t slot = rank < owner ? rank : rank - 1;
                const uint32_t first_own = rank * kQPerBand;
                const uint32_t pidx = (uint32_t)q < first_own ? (uint32_t)q : (uint32_t)q - kQPerBand;
                const uint32_t stage = sA + pidx * (C_::kPieces * C_::kQPieceBytes);
                cluster_wait();  // the owner's barriers exist
                cluster_waited = true;
                if (ok) {
    #pragma unroll 1
                    for (int c = 0; c < C_::kPieces; ++c) {
                        uint32_t v[64];
                        tmem_load_64cols(taddr + c * 64, v);
                        const uint32_t spiece = stage + c * C_::kQPieceBytes;
                        const uint32_t srow = spiece + lane * C_::kXPitch;
    #pragma unroll
                        for (int g = 0; g < 16; ++g) {
                            const uint32_t a = srow + ((g ^ (lane & 7)) << 4);
                            if (empty_slice)
                                st_shared_u4(a, 0u, 0u, 0u, 0u);
                            else
                                st_shared_u4(a, v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]);
                        }
                        fence_proxy_async_smem();  // the staging writes, before the copy engine reads
                        __syncwarp();
                        if (lane == 0) {
                            const uint32_t dst = sX + slot * C_::kXSlot +
                                                 (c * C_::kBandRows + qb * 32) * C_::kXPitch;
                            bulk_copy_smem_to_cta(map_to_cta(dst, owner), spiece, C_::kQPieceBytes,
                                                  map_to_cta(smem_u32(&bar_xchg[c]), owner));
                        }
                    }
                }
            } else if (ok) {
                // C through two staging slots over the idle ring (after the pushed quarters' copies)
                const uint32_t my_slots = sA + C_::kStaging + (uint32_t)qb * 8192u;
                uint32_t stores = 0;
    #pragma unroll 1
                for (int c = 0; c < C_::kPieces; ++c) {
                    uint32_t v[64];
                    tmem_load_64cols(taddr + c * 64, v);  // own partial sums, ready since tfull
                    int xok = 1;
                    if (lane == 0)
                        xok = wait_bounded<true>(smem_u32(&bar_xchg[c]), 0, abort, args.timeout_ns,
                                                 args.status, 25);
                    xok = __shfl_sync(0xffffffffu, xok, 0);
                    if (!xok) break;
                    // the phase has completed: every lane takes its own acquire of it
                    (void)mbar_try_wait_cluster(smem_u32(&bar_xchg[c]), 0);
                    if (c == C_::kPieces - 1 && qb == 0 && lane == 0)
                        ack_peers_n<kS>(rank, smem_u32(&bar_ack));  // every copy into this CTA landed
                    float acc[64];
                    // sum over source ranks 0..kS-1 in that order (own rows from Tensor Memory)
    #pragma unroll
                    for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
    #pragma unroll
                    for (int src = 0; src < kS; ++src) {
                        if (src == (int)rank) {
    #pragma unroll
                            for (int i = 0; i < 64; ++i)
                                acc[i] += empty_slice ? 0.0f : __uint_as_float(v[i]);
                        } else {
                            const int slot = src < (int)rank ? src : src - 1;
                            const uint32_t xrow = sX + slot * C_::kXSlot +
                                                  (c * C_::kBandRows + qb * 32 + lane) * C_::kXPitch;
    #pragma unroll
                            for (int g = 0; g < 16; ++g) {
                                const float4 p = ld_shared_f4(xrow + ((g ^ (lane & 7)) << 4));
                                acc[g * 4 + 0] += p.x;
                                acc[g * 4 + 1] += p.y;
                                acc[g * 4 + 2] += p.z;
                                acc[g * 4 + 3] += p.w;
                            }
                        }
                    }
    #pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = __float_as_uint(acc[i]);
                    store_chunk16<kBF16, 64>(&tmC, my_slots, stores, v, nt * kBN + c * 64,
                                             mt * kBM + q * 32, args.M, args.N, lane);
                }
                if (lane == 0) bulk_wait_group_read<0>();  // the C stores have read their slots
                __syncwarp();
            }
        }
    }

    // ------------------------------ teardown ------------------------------
    if (!cluster_waited) cluster_wait();  // complete the start-up cluster barrier
    tc_fence_before_sync();
    __syncthreads();
    // Every copy into this CTA has landed (its owners waited for them); the copies out of it read
    // its shared memory until they land: each other CTA acknowledges when all of them have, so the
    // CTA (and its shared memory) stays until then. No cluster-wide barrier at exit.
    if constexpr (kS > 1)
        if (threadIdx.x == 0 && !*abort)
            (void)wait_bounded<true>(smem_u32(&bar_ack), 0, abort, args.timeout_ns, args.status, 26);
    if (*abort && threadIdx.x == 0) {
        // After a timeout an owner may have stopped waiting: give copies still in flight a
        // fixed, bounded time to land before the CTAs' shared memory is released.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000ull * 1000) __nanosleep(1000);
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, C_::kTmemCols);
    }
}

}  // namespace dtc
