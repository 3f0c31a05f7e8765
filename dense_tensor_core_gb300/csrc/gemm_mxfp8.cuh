// gemm_mxfp8.cuh -- persistent MXFP8 block-scaled GEMM (e4m3 x e4m3, one E8M0 scale per row per
// 128 K-elements for A and for B, fp32 accumulation in Tensor Memory, bf16 output), NT layout.
//
// C[m,n] = bf16( sum_k e4m3(A[m,k]) 2^(sfA[m,k/128]-127) * e4m3(B[n,k]) 2^(sfB[n,k/128]-127) ):
// the block-scaled GEMM of the 05 Blackwell TCGEN05 GEMM tutorial, "Advanced" (gemm_blockscaled
// with sf_a_granularity_k = sf_b_granularity_k = 128, the "1d1d" example), on sm_103a tensor cores:
// tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X, M = 128, N = 224, K = 32.
//
// The instruction takes one scale per row per 32 K-elements. With granularity 128 the four MMAs
// of a 128-deep K-block all use the same scales. A K-block of 128 e4m3 = 128 bytes per row = one
// 128-byte swizzle row, and the shared-memory descriptors are those of the bf16 kernels (32 bytes
// per MMA step). A pipeline stage is one K-block (2-D boxes, any K), in a ring of 4. (Stages of two
// K-blocks, one 3-D box per operand, fit only twice beside the output staging and measured level
// or slower here -- 110.9 against 112.7 us, fp6 110.9 against 122.6 on 4096 x 4096 x 8192 -- so
// this kernel does not take them; the pair kernel does.)
//
// Scales live in Tensor Memory. For an operand of R rows (128 for A, 224 for B) they take R/32
// columns: row r sits in lane r % 32 of column r / 32, repeated in each of the four 32-lane
// quarters (each quarter of the datapath reads the scales it needs from its own lanes). One
// 32-bit cell holds 4 consecutive scale bytes of the row: with 128-element scale blocks those of 4
// consecutive K-blocks, and the instruction descriptor's scale byte selectors (a_sf_id, b_sf_id)
// pick K-block kb % 4; with 32-element blocks (the OCP MX block size) the 4 bytes of one K-block,
// one per MMA, and the selectors pick MMA kk of the K-block. Either way one scale set is one
// 32-bit word per row, and the elements may be e4m3 or e5m2 (the descriptor's format fields). Four "scale" warps (6..9, one per lane
// quarter) gather the bytes from global memory (one 32-bit load per row when the scale rows are
// 4-byte aligned) and write them with tcgen05.st, one group of 4 K-blocks at a time, into a ring
// of kSfSets scale sets; the gather for the next group is issued before the wait for a free set,
// so its latency overlaps the MMAs. The MMA thread waits for a group before its first MMA and
// releases it with a commit after its last.
//
// Roles: warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer, warps 2..5 epilogue (as in the
// bf16 kernels), warps 6..9 scale writers. Tensor Memory: accumulators at columns [0,224) and
// [224,448), scale sets at 448 + 12*set (4 columns for A, 8 for B), set = 0..3.
//
// With kTmaSf the scales come instead from a copy of the scale arrays repacked by sf_pack_kernel
// (sf_pack.cuh) into 512-byte chunks, one per (128-row group, set): the producer loads a set's
// chunks (A: one, B: two) with bulk copies into a slot beside the stage holding the set's first
// K-block, on that stage's full barrier, and the MMA thread moves them into the set's columns with
// three tcgen05.cp.32x128b.warpx4 before the set's first MMA. A copy and the MMAs after it form a
// tcgen05 pipeline (they run in issue order); an MMA and a later copy into columns it reads do
// not, so the MMA thread reuses a set only after the commit that follows its last MMA
// (bar_sempty). No scale warps, no cross-warp hand-off: 6 warps.
#pragma once

#include "gemm_common.cuh"
#include "sf_pack.cuh"

namespace dtc {

struct GemmMxArgs {
    void* C;
    int64_t ldc;  // elements between rows of C (>= N)
    const uint8_t* sfA;
    const uint8_t* sfB;
    int M, N, K;
    int num_m, num_n, num_kb;  // num_kb: 128-element K-blocks
    int sf_cols;               // bytes per scale row: ceil(K / scale block)
    uint32_t fmt_bits;         // instruction-descriptor element formats of A (bits 7-9), B (10-12)
    uint32_t stage_tx;         // bytes one stage's copies write (fp6 / fp4: the packed data only;
                               // the padding of each 16-byte group is not written)
    const uint8_t* sfA_pack;   // kTmaSf: scale chunks of A (128-row groups) and of B (tile_n-row
    const uint8_t* sfB_pack;   // groups, two 128-row halves each), sf_pack.cuh
    int sf_sets;               // scale sets per row: ceil(sf_cols / 4)
    uint64_t timeout_ns;
    int fault;
    int* status;  // device status word: the first wait that gives up records its site here
};

namespace gmx {
constexpr int kBM = 128;
constexpr int kBN = 224;
constexpr int kBK = 128;  // e4m3 elements (= bytes) per K-block, one 128-byte swizzle row
constexpr int kThreads = 320;
constexpr int kTmemCols = 512;
constexpr int kAccStride = 224;
constexpr int kSfBase = 448;   // first scale column
constexpr int kSfSet = 12;     // columns per scale set: 4 (A) + 8 (B)
constexpr int kSfSets = 4;     // scale sets in flight
constexpr int kGroup = 4;      // K-blocks per scale set (one byte each per 32-bit cell)
constexpr int kGroupM = 8;
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
static_assert(kSfBase + kSfSets * kSfSet <= kTmemCols, "Tensor Memory budget");
constexpr int kSfSetBytes = 3 * kSfChunkBytes;  // one set's chunks: A (128 rows), B (2 x 128 rows)
static_assert(kBN <= 256, "a B tile's scales fit two 128-row chunks");

constexpr int threads_for(bool tma_sf) { return tma_sf ? 192 : kThreads; }

// Stage geometry: one K-block per stage (2-D boxes), 4 stages.
// With kTmaSf each stage has a slot for the chunks of the sets that start in it (at most one per
// K-block).
template <bool kTmaSf = false>
struct Cfg {
    static constexpr int kBlocks = 1;
    static constexpr int kStages = 4;
    static constexpr int kAStage = kBM * kBK * kBlocks;
    static constexpr int kBStage = kBN * kBK * kBlocks;
    static constexpr int kStageBytes = kAStage + kBStage;
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static constexpr int kCBytes = 4 * 2 * 4096;  // two 4 KB output staging slots per epilogue warp
    static constexpr int kSlotBytes = kTmaSf ? kBlocks * kSfSetBytes : 0;
    static constexpr int kSmemBytes = kStages * (kStageBytes + kSlotBytes) + kCBytes + 1024;
    static_assert(kSmemBytes <= 227 * 1024 - 256, "shared memory budget");
};
}  // namespace gmx

// Scale word of row `row` for K-block group g: the E8M0 bytes of K-blocks 4g..4g+3 (byte j =
// K-block 4g+j), zero past the end of the row or past the last row.
__device__ __forceinline__ uint32_t sf_word(const uint8_t* sf, int rows, int cols, int row, int g) {
    if (row >= rows) return 0u;
    const uint8_t* p = sf + (int64_t)row * cols;
    if ((cols & 3) == 0 && (reinterpret_cast<uintptr_t>(sf) & 3) == 0)
        return __ldg(reinterpret_cast<const uint32_t*>(p + g * 4));  // 4 whole bytes in range
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = g * 4 + j;
        if (c < cols) w |= (uint32_t)__ldg(p + c) << (8 * j);
    }
    return w;
}

template <bool kB32, bool kTmaSf = false>
__global__ void __launch_bounds__(gmx::threads_for(kTmaSf), 1)
    gemm_mxfp8_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmC32, const GemmMxArgs args) {
    using namespace gmx;
    using C_ = Cfg<kTmaSf>;
    constexpr int kStages = C_::kStages;
    constexpr int kAStage = C_::kAStage;
    constexpr int kBStage = C_::kBStage;
    constexpr int kBlocks = C_::kBlocks;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_sfull[gmx::kSfSets];
    __shared__ __align__(8) uint64_t bar_sempty[gmx::kSfSets];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * kAStage;
    const uint32_t sSF = base + kStages * C_::kStageBytes + C_::kCBytes;  // kTmaSf: scale slots
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = args.num_m * args.num_n;
    constexpr int grp = kB32 ? 1 : kGroup;  // K-blocks per scale set
    const int groups = (args.num_kb + grp - 1) / grp;
    const int num_st = (args.num_kb + kBlocks - 1) / kBlocks;  // stages per tile
    // Refilling a scale set's columns needs the MMAs that last read them done. Passing a stage's
    // full barrier already proves every MMA of the stages a whole ring earlier done (the stage was
    // refilled only after the commit that followed them), so with full sets (every tile's K-blocks
    // a multiple of the set length) spaced at least a ring apart the explicit wait, and the commit
    // it waits for, are not needed.
    constexpr bool kSfRingSafe = (kSfSets - 1) * grp + 1 >= kStages * kBlocks;
    const bool sf_wait = kTmaSf && !(kSfRingSafe && args.num_kb % grp == 0);
    volatile int* abort = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 4);
        }
        for (int b = 0; b < kSfSets; ++b) {
            mbar_init(smem_u32(&bar_sfull[b]), 4);  // one arrival per scale warp
            mbar_init(smem_u32(&bar_sempty[b]), 1);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true, chunks_ready = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int mt, nt;
                tile_coords(t, args.num_m, args.num_n, kGroupM, mt, nt);
                for (int st = 0; st < num_st; ++st, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!wait_bounded(smem_u32(&bar_empty[s]), ph ^ 1u, abort, args.timeout_ns,
                                      args.status, 31)) {
                        ok = false;
                        break;
                    }
                    if (args.fault == 1 && it == 0) continue;  // test hook: stage never filled
                    const uint32_t full = smem_u32(&bar_full[s]);
                    uint32_t tx = args.stage_tx;
                    if constexpr (kTmaSf) {
#pragma unroll
                        for (int h = 0; h < kBlocks; ++h) {
                            const int kb = st * kBlocks + h;
                            if (kb < args.num_kb && kb % grp == 0) tx += kSfSetBytes;
                        }
                    }
                    mbar_arrive_expect_tx(full, tx);
                    tma_load_2d(sA + s * kAStage, &tmA, full, st * kBK, mt * kBM);
                    tma_load_2d(sB + s * kBStage, &tmB, full, st * kBK, nt * kBN);
                    if constexpr (kTmaSf) {
                        // the chunks of each set that starts in this stage, into slot h; the
                        // kernel that writes them may still be running (it launched this one
                        // early): wait for it before the first chunk copy
                        if (!chunks_ready) {
                            grid_dependency_wait();
                            chunks_ready = true;
                        }
#pragma unroll
                        for (int h = 0; h < kBlocks; ++h) {
                            const int kb = st * kBlocks + h;
                            if (kb >= args.num_kb || kb % grp != 0) continue;
                            const int g = kb / grp;
                            const uint32_t slot = sSF + s * C_::kSlotBytes + h * kSfSetBytes;
                            bulk_load_g2s(slot, args.sfA_pack + ((int64_t)mt * args.sf_sets + g) * kSfChunkBytes,
                                          kSfChunkBytes, full);
                            bulk_load_g2s(slot + kSfChunkBytes,
                                          args.sfB_pack + ((int64_t)nt * args.sf_sets + g) * 2 * kSfChunkBytes,
                                          2 * kSfChunkBytes, full);
                        }
                    }
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
            const uint32_t idesc0 = idesc_mxf8(kBM, kBN, 0, 0) | args.fmt_bits;
            uint32_t it = 0, acc = 0, sit = 0;
            bool ok = true, issued = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
                if (!wait_bounded(smem_u32(&bar_tempty[b]), aph ^ 1u, abort, args.timeout_ns,
                                  args.status, 32)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kAccStride;
                for (int st = 0; st < num_st && ok; ++st, ++it) {
                    const int kb0 = st * kBlocks;  // first K-block of the stage
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!wait_bounded(smem_u32(&bar_full[s]), ph, abort, args.timeout_ns,
                                      args.status, 33)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll
                    for (int h = 0; h < kBlocks; ++h) {
                        const int kb = kb0 + h;
                        if (kb >= args.num_kb) break;  // a K-block past K: zero-filled, skipped
                        const uint32_t set = sit % kSfSets;
                        if (kb % grp == 0) {  // the first K-block of a scale set
                            if constexpr (kTmaSf) {
                                // the set's columns are free once the MMAs that last read them
                                // are done; then copy the set from the stage's slot
                                if (sf_wait) {
                                    if (!wait_bounded(smem_u32(&bar_sempty[set]),
                                                      ((sit / kSfSets) & 1u) ^ 1u, abort,
                                                      args.timeout_ns, args.status, 37)) {
                                        ok = false;
                                        break;
                                    }
                                    tc_fence_after_sync();
                                }
                                const uint32_t slot = sSF + s * C_::kSlotBytes + h * kSfSetBytes;
                                const uint32_t col = tmem_base + kSfBase + set * kSfSet;
                                tmem_cp_32x128b_x4(col, smem_desc_plain(slot, 128, 128));
                                tmem_cp_32x128b_x4(col + 4, smem_desc_plain(slot + kSfChunkBytes, 128, 128));
                                tmem_cp_32x128b_x4(col + 8,
                                                   smem_desc_plain(slot + 2 * kSfChunkBytes, 128, 128));
                            } else {
                                if (!wait_bounded(smem_u32(&bar_sfull[set]), (sit / kSfSets) & 1u,
                                                  abort, args.timeout_ns, args.status, 35)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after_sync();
                            }
                        }
                        // K-block h of the stage: 128-byte chunk h of each operand's box
                        const uint32_t a0 = sA + s * kAStage + h * (kBM * kBK);
                        const uint32_t b0 = sB + s * kBStage + h * (kBN * kBK);
                        const uint32_t sfa = tmem_base + kSfBase + set * kSfSet;
                        const uint32_t sfb = sfa + 4;
#pragma unroll
                        for (int kk = 0; kk < kBK / 32; ++kk) {
                            const uint32_t sf_id = kB32 ? (uint32_t)kk : (uint32_t)(kb % kGroup);
                            const uint32_t idesc = idesc0 | (sf_id << 4) | (sf_id << 29);
                            const uint64_t adesc = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                            const uint64_t bdesc = smem_desc_sw128(b0 + kk * 32, 16, 1024);
                            mma_mxf8_cta1(d_tmem, adesc, bdesc, idesc, sfa, sfb,
                                          (kb | kk) != 0 ? 1u : 0u);
                        }
                        issued = true;
                        if (kb % grp == grp - 1 || kb == args.num_kb - 1) {
                            if (!kTmaSf || sf_wait)  // scale set consumed
                                mma_commit_cta1(smem_u32(&bar_sempty[set]));
                            ++sit;
                        }
                    }
                    if (!ok) break;
                    mma_commit_cta1(smem_u32(&bar_empty[s]));
                }
                if (!ok) break;
                mma_commit_cta1(smem_u32(&bar_tfull[b]));
                ++acc;
            }
            if (!ok && issued) {
                mma_commit_cta1(smem_u32(&bar_drain));
                wait_drain(smem_u32(&bar_drain), 0, kDrainNs);
            }
        }
    } else if (warp < 6) {
        // ------------------------------ epilogue (warps 2..5) ------------------------------
        const int q = warp & 3;
        const uint32_t my_slots = base + kStages * C_::kStageBytes + (uint32_t)q * 8192u;
        uint32_t acc = 0, stores = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++acc) {
            int mt, nt;
            tile_coords(t, args.num_m, args.num_n, kGroupM, mt, nt);
            const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded<false, true>(smem_u32(&bar_tfull[b]), aph, abort,
                                               args.timeout_ns, args.status, 34);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * kAccStride;
            drain_tile16<true, kBN>(taddr, &tmC, &tmC32, my_slots, stores, nt * kBN, mt * kBM + q * 32,
                                    args.M, args.N, lane, [&]() {
                                        tc_fence_before_sync();
                                        __syncwarp();
                                        if (lane == 0) mbar_arrive(smem_u32(&bar_tempty[b]));
                                    });
        }
        if (lane == 0) bulk_wait_group_read<0>();  // the C stores have read their slots
        __syncwarp();
    } else if constexpr (!kTmaSf) {
        // ------------------------------ scale writers (warps 6..9) ------------------------------
        // The (tile, group) sequence of this CTA, flattened so the gather of the next group
        // (possibly of the next tile) is in flight while the current one waits for a free set.
        const int q = warp & 3;  // the Tensor Memory lane quarter this warp writes
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const int my_tiles =
            (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        const int steps = my_tiles * groups;
        auto gather = [&](int step, uint32_t (&ga)[4], uint32_t (&gb)[8]) {
            const int t = (int)blockIdx.x + (step / groups) * (int)gridDim.x;
            const int g = step % groups;
            int mt, nt;
            tile_coords(t, args.num_m, args.num_n, kGroupM, mt, nt);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                ga[j] = sf_word(args.sfA, args.M, args.sf_cols, mt * kBM + lane + 32 * j, g);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                gb[j] = j < kBN / 32
                            ? sf_word(args.sfB, args.N, args.sf_cols, nt * kBN + lane + 32 * j, g)
                            : 0u;
        };
        uint32_t wa[4], wb[8];
        if (steps > 0) gather(0, wa, wb);
        for (int step = 0; step < steps; ++step) {
            uint32_t na[4], nb[8];
            if (step + 1 < steps) gather(step + 1, na, nb);
            const uint32_t sit = (uint32_t)step;
            const uint32_t set = sit % kSfSets;
            int w_ok = 1;
            if (lane == 0)
                w_ok = wait_bounded<false, true>(smem_u32(&bar_sempty[set]),
                                                 ((sit / kSfSets) & 1u) ^ 1u, abort,
                                                 args.timeout_ns, args.status, 36);
            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
            if (!w_ok) break;
            tc_fence_after_sync();
            const uint32_t col = tmem_base + kSfBase + set * kSfSet;
            tmem_store_4cols(col + lane_addr, wa[0], wa[1], wa[2], wa[3]);
            tmem_store_8cols(col + 4 + lane_addr, wb);
            tmem_store_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_sfull[set]));
            if (step + 1 < steps) {
#pragma unroll
                for (int j = 0; j < 4; ++j) wa[j] = na[j];
#pragma unroll
                for (int j = 0; j < 8; ++j) wb[j] = nb[j];
            }
        }
    }

    // ------------------------------ teardown ------------------------------
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, kTmemCols);
    }
}

}  // namespace dtc
