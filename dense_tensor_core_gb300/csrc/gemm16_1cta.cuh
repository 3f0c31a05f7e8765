// gemm16_1cta.cuh -- persistent, warp-specialised bf16/fp16 GEMM, one CTA per 128 x kBN tile.
//
// C[M,N] = A[M,K] . Bop, fp32 accumulation in Tensor Memory, bf16/fp16 output.
// The tile (128 x 256, K-blocks of 64) follows the example shape of TileLang SM100 Support
// (Preview), "Compilation and Usage" (block 128 x 256 x 128: two of our 64-deep stages per
// 128-deep K-block), and its accumulate/clear rule ("Code Example": clear_accum = (k == 0)) is the
// enable-input-d flag of the first MMA of each tile.
//
// Differences from the pages' kernels: there the SM100 preview ran without TMA and without warp
// specialisation, one stage, and waited for each MMA (TileLang SM100 Support (Preview),
// "Compilation and Usage" pass configs and "Code Example"); here
//   warp 0      : TMA producer (one lane) filling a kStages ring of 128B-swizzled A/B tiles,
//   warp 1      : Tensor Memory allocator and single-thread tcgen05.mma issuer,
//   warps 2..5  : epilogue (tcgen05.ld -> cvt -> swizzled shared-memory staging -> TMA store),
// with full/empty barriers per stage (the producer waits on the inverted parity, as in the
// 3-stage ring of tilelang (velog) section 1.3) and a double-buffered accumulator (2 x 256
// columns) so the epilogue of one tile overlaps the main loop of the next. CTAs are persistent:
// CTA i takes tiles i, i + grid, ... in a grouped order that keeps A and B panels in L2.
//
// Every TMA load goes to the issuing CTA's own shared memory (no cluster multicast).
#pragma once

#include "gemm_common.cuh"

namespace dtc {

namespace g16 {
constexpr int kBM = 128;
constexpr int kBK = 64;                 // K-elements per stage: one 128-byte swizzle row
constexpr int kTmemCols = 512;          // two fp32 accumulators
constexpr int kAccStride = 256;         // column offset of the second accumulator
constexpr int kThreads = 192;
constexpr int kGroupM = 8;              // M-tiles per rasterisation group
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;

// As many 64-deep stages as fit beside the 32 KB of output staging.
template <int kBN, int kStages>
struct Cfg {
    static constexpr int kAStage = kBM * kBK * 2;
    static constexpr int kBStage = kBN * kBK * 2;
    static constexpr int kStageBytes = kAStage + kBStage;
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static constexpr int kCBytes = 4 * 2 * 4096;  // two 4 KB output staging slots per epilogue warp
    static constexpr int kSmemBytes = kStages * kStageBytes + kCBytes + 1024;  // + alignment slack
    static_assert(kBN % 16 == 0 && kBN <= 256, "UMMA N for M = 128");
    static_assert(kSmemBytes <= 227 * 1024 - 256, "shared memory budget");
};
}  // namespace g16

template <bool kBF16, bool kAMN, bool kNN, int kBN, int kStages>
__global__ void __launch_bounds__(g16::kThreads, 1)
    gemm16_1cta_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC,
                       const __grid_constant__ CUtensorMap tmC32, const Gemm16Args args) {
    using namespace g16;
    using C_ = Cfg<kBN, kStages>;
    constexpr int kAStage = C_::kAStage;
    static_assert(!kNN || kBN % 64 == 0, "B stored [K,N] is loaded as 64-column boxes");

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sA = base;                      // kStages x kAStage
    const uint32_t sB = base + kStages * kAStage;  // kStages x kBStage
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = args.num_m * args.num_n;
    volatile int* abort = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 4);  // one arrival per epilogue warp
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
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int mt, nt;
                tile_coords(t, args.num_m, args.num_n, kGroupM, mt, nt);
                for (int kb = 0; kb < args.num_kb; ++kb, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!wait_bounded(smem_u32(&bar_empty[s]), ph ^ 1u, abort, args.timeout_ns,
                                      args.status, 1)) {
                        ok = false;
                        break;
                    }
                    if (args.fault == 1 && it == 0) continue;  // test hook: stage never filled
                    const uint32_t full = smem_u32(&bar_full[s]);
                    mbar_arrive_expect_tx(full, C_::kStageBytes);
                    if constexpr (kAMN) {
                        // A stored [K,M]: two 64-column boxes of kBK K-rows (128-byte swizzle)
                        tma_load_2d(sA + s * kAStage, &tmA, full, mt * kBM, kb * kBK);
                        tma_load_2d(sA + s * kAStage + 64 * kBK * 2, &tmA, full, mt * kBM + 64,
                                    kb * kBK);
                    } else {
                        tma_load_2d(sA + s * kAStage, &tmA, full, kb * kBK, mt * kBM);
                    }
                    const uint32_t bdst = sB + s * C_::kBStage;
                    if constexpr (!kNN) {
                        tma_load_2d(bdst, &tmB, full, kb * kBK, nt * kBN);
                    } else {
#pragma unroll
                        for (int j = 0; j < kBN / 64; ++j)  // 64-column boxes of kBK K-rows
                            tma_load_2d(bdst + j * (64 * kBK * 2), &tmB, full, nt * kBN + j * 64,
                                        kb * kBK);
                    }
                }
            }
            if (!ok) {
                // Let the copies already issued land before the CTA may exit.
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
            uint32_t it = 0, acc = 0;
            bool ok = true, issued = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
                if (!wait_bounded(smem_u32(&bar_tempty[b]), aph ^ 1u, abort, args.timeout_ns,
                                  args.status, 2)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kAccStride;
                for (int kb = 0; kb < args.num_kb; ++kb, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!wait_bounded(smem_u32(&bar_full[s]), ph, abort, args.timeout_ns,
                                      args.status, 3)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a0 = sA + s * kAStage, b0 = sB + s * C_::kBStage;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t adesc =
                            kAMN ? smem_desc<128>(a0 + kk * 16 * 128, 64 * kBK * 2, 1024)
                                 : smem_desc<128>(a0 + kk * 32, 16, 1024);
                        const uint64_t bdesc =
                            kNN ? smem_desc<128>(b0 + kk * 16 * 128, 64 * kBK * 2, 1024)
                                : smem_desc<128>(b0 + kk * 32, 16, 1024);
                        mma_f16_cta1(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    mma_commit_cta1(smem_u32(&bar_empty[s]));
                }
                if (!ok) break;
                mma_commit_cta1(smem_u32(&bar_tfull[b]));
                ++acc;
            }
            if (!ok && issued) {
                // Wait for the MMAs in flight before Tensor Memory is released.
                mma_commit_cta1(smem_u32(&bar_drain));
                wait_drain(smem_u32(&bar_drain), 0, kDrainNs);
            }
        }
    } else {
        // ------------------------------ epilogue (warps 2..5) ------------------------------
        const int q = warp & 3;  // Tensor Memory lane quarter this warp may access
        const uint32_t my_slots = base + kStages * C_::kStageBytes + (uint32_t)q * 8192u;
        uint32_t acc = 0, stores = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++acc) {
            int mt, nt;
            tile_coords(t, args.num_m, args.num_n, kGroupM, mt, nt);
            const uint32_t b = acc & 1u, aph = (acc >> 1) & 1u;
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_u32(&bar_tfull[b]), aph, abort, args.timeout_ns,
                                  args.status, 4);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * kAccStride;
            // accumulator -> 16-bit staging -> TMA store; the buffer goes back to the MMA issuer
            // once fully read
            drain_tile16<kBF16, kBN>(taddr, &tmC, &tmC32, my_slots, stores, nt * kBN,
                                     mt * kBM + q * 32, args.M, args.N, lane, [&]() {
                                         tc_fence_before_sync();
                                         __syncwarp();
                                         if (lane == 0) mbar_arrive(smem_u32(&bar_tempty[b]));
                                     });
        }
        if (lane == 0) bulk_wait_group_read<0>();  // the C stores have read their slots
        __syncwarp();
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
