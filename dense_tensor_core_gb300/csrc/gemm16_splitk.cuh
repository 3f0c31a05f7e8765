// gemm16_splitk.cuh -- bf16/fp16 GEMM with K split across the CTAs of a cluster, for products
// with too few output tiles to occupy the GPU (the skinny, memory-bound M = 128 case).
//
// C[M,N] = A[M,K] . Bop as in the one-CTA kernel (128 x kBN tiles, 64-deep K-blocks, TMA producer
// warp, single-thread tcgen05.mma issuer, Tensor Memory accumulator), but a cluster of kS CTAs
// computes one tile: CTA r accumulates the r-th of kS contiguous K-ranges. The partial sums are
// reduced on chip, without a global workspace:
//   1. each CTA's epilogue copies its fp32 accumulator (tcgen05.ld, 64 columns per round trip)
//      into its own shared memory, over the ring buffers, which are idle once the tile's last
//      MMA has completed;
//   2. cluster barrier;
//   3. CTA r sums rows [r*128/kS, (r+1)*128/kS) of the tile over the kS CTAs' copies, reading
//      them through distributed shared memory in the fixed order 0..kS-1 (so the result does not
//      depend on which CTA finished first; each thread keeps 4 column groups x kS loads in
//      flight), rounds once to the output type and stores;
//   4. cluster barrier (no CTA leaves while a peer may still read its copy).
// One cluster per tile, not persistent: a product of T tiles launches T * kS CTAs.
#pragma once

#include "gemm_common.cuh"

namespace dtc {

namespace gsk {
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;

template <int kBN, int kStages>
struct Cfg {
    static constexpr int kAStage = kBM * kBK * 2;
    static constexpr int kBStage = kBN * kBK * 2;
    static constexpr int kStageBytes = kAStage + kBStage;
    static constexpr int kRing = kStages * kStageBytes;
    static constexpr int kXPitch = kBN * 4 + 16;  // fp32 row + 16 bytes: conflict-free v4 stores
    static constexpr int kXBytes = kBM * kXPitch;
    static constexpr int kSmemBytes = kRing + 1024;
    static_assert(kXBytes <= kRing, "the partial-sum copy must fit over the ring");
    static_assert(kSmemBytes <= 227 * 1024 - 256, "shared memory budget");
};
}  // namespace gsk

template <bool kBF16, bool kNN, int kBN, int kStages, int kS>
__global__ void __launch_bounds__(gsk::kThreads, 1)
    gemm16_splitk_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const Gemm16Args args) {
    using namespace gsk;
    using C_ = Cfg<kBN, kStages>;
    static_assert(kS == 2 || kS == 4, "K split over 2 or 4 CTAs");
    static_assert(kBN % 64 == 0, "the accumulator is read 64 columns at a time");
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull;
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t sB = base + kStages * C_::kAStage;
    const uint32_t sX = base;  // partial-sum copy, over the ring after the main loop
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
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!wait_bounded(smem_u32(&bar_empty[s]), ph ^ 1u, abort, args.timeout_ns,
                                  &g_dtc_status, 21)) {
                    ok = false;
                    break;
                }
                if (args.fault == 1 && it == 0) continue;  // test hook: stage never filled
                const uint32_t full = smem_u32(&bar_full[s]);
                mbar_arrive_expect_tx(full, C_::kStageBytes);
                tma_load_2d(sA + s * C_::kAStage, &tmA, full, kb * kBK, mt * kBM);
                if constexpr (!kNN) {
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
            constexpr uint32_t idesc = idesc_f16(kBF16, kNN, kBM, kBN);
            uint32_t it = 0;
            bool ok = true, issued = false;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!wait_bounded(smem_u32(&bar_full[s]), ph, abort, args.timeout_ns,
                                  &g_dtc_status, 23)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a0 = sA + s * C_::kAStage, b0 = sB + s * C_::kBStage;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t adesc = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                    const uint64_t bdesc = kNN ? smem_desc_sw128(b0 + kk * 16 * 128, 64 * kBK * 2, 1024)
                                               : smem_desc_sw128(b0 + kk * 32, 16, 1024);
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
    }
    if (warp >= 2) {
        // -------------------- epilogue part 1: accumulator -> own shared memory --------------
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int ok = 1;
        if (lane == 0)
            ok = wait_bounded(smem_u32(&bar_tfull), 0, abort, args.timeout_ns, &g_dtc_status, 24);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
            const uint32_t xrow = sX + row * C_::kXPitch;
            const bool empty_slice = kb1 <= kb0;  // no K-blocks: this CTA's share is zero
#pragma unroll 1
            for (int c = 0; c < kBN / 64; ++c) {
                uint32_t v[64];
                tmem_load_64cols(taddr + c * 64, v);
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                    const uint32_t a = xrow + (c * 64 + g * 4) * 4;
                    if (empty_slice)
                        st_shared_u4(a, 0u, 0u, 0u, 0u);
                    else
                        st_shared_u4(a, v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]);
                }
            }
        }
    }

    // -------------------- epilogue part 2: reduce the band of rows this CTA owns ------------
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // every CTA's partial sums are in its shared memory
    {
        constexpr int kRows = kBM / kS;   // rows of the tile this CTA reduces
        constexpr int kGroups = kBN / 4;  // 4-column groups per row
        constexpr int kItems = kRows * kGroups;
        constexpr int kUnroll = 4;        // column groups per thread per round
        uint32_t peer[kS];
#pragma unroll
        for (int s = 0; s < kS; ++s) peer[s] = map_to_cta(sX, (uint32_t)s);
        for (int i0 = threadIdx.x; i0 < kItems; i0 += kThreads * kUnroll) {
            float4 acc[kUnroll];
            uint32_t off[kUnroll];
            bool live[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * kThreads;
                live[u] = i < kItems;
                const int r = (int)rank * kRows + (live[u] ? i / kGroups : 0);
                const int g = live[u] ? i % kGroups : 0;
                off[u] = r * C_::kXPitch + g * 16;
                acc[u] = live[u] ? ld_shared_cluster_f4(peer[0] + off[u]) : make_float4(0, 0, 0, 0);
            }
#pragma unroll
            for (int s = 1; s < kS; ++s) {
                float4 v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    v[u] = live[u] ? ld_shared_cluster_f4(peer[s] + off[u]) : make_float4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    acc[u].x += v[u].x;
                    acc[u].y += v[u].y;
                    acc[u].z += v[u].z;
                    acc[u].w += v[u].w;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * kThreads;
                if (!live[u]) continue;
                const int64_t grow = (int64_t)mt * kBM + (int64_t)rank * kRows + i / kGroups;
                const int gcol = nt * kBN + (i % kGroups) * 4;
                if (grow >= args.M || gcol >= args.N) continue;
                uint2 out;
                out.x = pack2<kBF16>(__float_as_uint(acc[u].x), __float_as_uint(acc[u].y));
                out.y = pack2<kBF16>(__float_as_uint(acc[u].z), __float_as_uint(acc[u].w));
                *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(args.C) + grow * args.N +
                                          gcol) = out;
            }
        }
    }
    cluster_sync();  // peers are done reading this CTA's copy
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, kTmemCols);
    }
}

}  // namespace dtc
