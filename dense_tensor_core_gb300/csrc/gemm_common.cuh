// gemm_common.cuh -- pieces shared by the GEMM kernels: the kernel argument block, the
// persistent tile order and the fp32 -> 16-bit output packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace dtc {

struct Gemm16Args {
    void* C;
    int64_t ldc;  // elements between rows of C (>= N)
    int M, N, K;
    int num_m, num_n, num_kb;
    uint64_t timeout_ns;
    int fault;
    int* status;  // device status word: the first wait that gives up records its site here
    // Stream-K (pair kernel): the last sk_tiles tiles are shared out as equal runs of K-blocks
    // over all units; 0 = every tile whole. Partial sums go through the caller's workspace.
    int sk_tiles;
    uint32_t* sk_flags;  // one per (unit, CTA of the pair): 1 = that CTA's partial is written
    float* sk_partial;   // per (unit, CTA): 128 rows x tile width fp32
};

// One unit of a persistent kernel's work: K-blocks [k0, k1) of tile `tile`.
//   kind kWhole: the whole K range; kOther: a later piece of a tile another unit finishes (its
//   partial sums go to the workspace); kFirst: the first piece, finished here with the pieces of
//   units unit+1 .. unit+contrib.
struct WorkItem {
    int tile, k0, k1, kind;
};
constexpr int kWhole = 0, kOther = 1, kFirst = 2;

// The work of `unit` of `units`: first its equal share [s0, s1) of the sk_tiles * kiters K-blocks
// of tiles 0 .. sk_tiles-1 in (tile, K-block) order, then tiles sk_tiles + unit, + units, ...
// whole. Shared tiles come first so that finishing them (waiting for other units' pieces, adding
// them) overlaps the main loops of whole tiles instead of trailing the kernel. Every role of the
// kernel walks the same sequence.
struct WorkIter {
    int t, total, units, kiters, sk_tiles;
    int64_t i, s1;
    __device__ WorkIter(int unit, int units_, int total_, int sk_tiles_, int kiters_)
        : t(sk_tiles_ + unit), total(total_), units(units_), kiters(kiters_), sk_tiles(sk_tiles_) {
        const int64_t S = (int64_t)sk_tiles_ * kiters_;
        i = (int64_t)unit * S / units_;
        s1 = (int64_t)(unit + 1) * S / units_;
    }
    __device__ bool next(WorkItem& w) {
        if (i < s1) {
            const int j = (int)(i / kiters);
            w.tile = j;
            w.k0 = (int)(i - (int64_t)j * kiters);
            w.k1 = (int)min((int64_t)kiters, (int64_t)w.k0 + (s1 - i));
            w.kind = w.k0 > 0 ? kOther : (w.k1 < kiters ? kFirst : kWhole);
            i += w.k1 - w.k0;
            return true;
        }
        if (t < total) {
            w.tile = t;
            w.k0 = 0;
            w.k1 = kiters;
            w.kind = kWhole;
            t += units;
            return true;
        }
        return false;
    }
};

// First K-block of `unit`'s stream-K share (the start of its range).
__device__ __forceinline__ int64_t sk_start(int unit, int units, int sk_tiles, int kiters) {
    return (int64_t)unit * ((int64_t)sk_tiles * kiters) / units;
}

// Grouped rasterisation: tiles are numbered down groups of kGroupM M-tiles, N-tile by N-tile.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int& mt,
                                            int& nt) {
    const int per_group = group_m * num_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gm = min(num_m - first_m, group_m);
    const int r = t - g * per_group;
    mt = first_m + r % gm;
    nt = r / gm;
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) {
    const float a = __uint_as_float(lo), b = __uint_as_float(hi);
    if constexpr (kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Staged 16-bit output: one warp's 32 rows (lane = row) x W fp32 accumulator columns, converted
// to 16-bit and written into a shared-memory slot in the layout a TMA store with the matching
// swizzle reads: W = 64 -> 128-byte rows, 16-byte chunk j of row r at chunk j ^ (r % 8) (128-byte
// swizzle, slot 1024-byte aligned); W = 32 -> 64-byte rows, chunk j at j ^ ((r / 2) % 4) (64-byte
// swizzle, slot 512-byte aligned). Eight consecutive lanes cover every 16-byte position of a
// 128-byte line, so each warp-wide 16-byte store takes the minimum four shared-memory wavefronts.
template <bool kBF16, int W>
__device__ __forceinline__ void stage_rows16(uint32_t slot, const uint32_t (&v)[W], int lane) {
    static_assert(W == 64 || W == 32, "64 or 32 columns per staged chunk");
#pragma unroll
    for (int j = 0; j < W / 8; ++j) {
        const uint32_t off = W == 64 ? (uint32_t)lane * 128u + ((uint32_t)(j ^ (lane & 7)) << 4)
                                     : (uint32_t)lane * 64u + ((uint32_t)(j ^ ((lane >> 1) & 3)) << 4);
        st_shared_u4(slot + off, pack2<kBF16>(v[j * 8 + 0], v[j * 8 + 1]),
                     pack2<kBF16>(v[j * 8 + 2], v[j * 8 + 3]), pack2<kBF16>(v[j * 8 + 4], v[j * 8 + 5]),
                     pack2<kBF16>(v[j * 8 + 6], v[j * 8 + 7]));
    }
}

// One warp's path from registers to C through two 4 KB staging slots: wait until the store issued
// two chunks ago has read the slot, stage the chunk, and let lane 0 issue the TMA store of the
// box {W columns, 32 rows} at C column x, row y (a box that starts past C's last row or column is
// skipped; one that only overlaps the edge is clipped by the TMA). Call with the whole warp;
// `count` is the warp's running chunk number (it picks the slot).
template <bool kBF16, int W>
__device__ __forceinline__ void store_chunk16(const CUtensorMap* tmC, uint32_t slots,
                                              uint32_t& count, const uint32_t (&v)[W], int x,
                                              int y, int M, int N, int lane) {
    if (x >= N || y >= M) return;
    const uint32_t slot = slots + (count & 1u) * 4096u;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    stage_rows16<kBF16, W>(slot, v, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmC, slot, x, y);
        bulk_commit_group();
    }
    ++count;
}

// Drains one warp's 32 accumulator rows x kBN columns (Tensor Memory address `taddr`) into C
// rows y0.., columns x0.. through its staging slots: 64-column chunks, and a last 32-column chunk
// (through tmC32) when kBN % 64 == 32. `hand_back` runs right after the last Tensor Memory load,
// from which point the accumulator may be overwritten.
template <bool kBF16, int kBN, typename HandBack>
__device__ __forceinline__ void drain_tile16(uint32_t taddr, const CUtensorMap* tmC,
                                             const CUtensorMap* tmC32, uint32_t slots,
                                             uint32_t& count, int x0, int y0, int M, int N,
                                             int lane, HandBack hand_back) {
    static_assert(kBN % 32 == 0, "tile width in 32-column steps");
    constexpr int kFull = kBN / 64;
    constexpr bool kTail = (kBN % 64) != 0;
#pragma unroll 1
    for (int c = 0; c < kFull; ++c) {
        uint32_t v[64];
        tmem_load_64cols(taddr + c * 64, v);
        if (!kTail && c == kFull - 1) hand_back();
        store_chunk16<kBF16, 64>(tmC, slots, count, v, x0 + c * 64, y0, M, N, lane);
    }
    if constexpr (kTail) {
        uint32_t v[32];
        tmem_load_32cols(taddr + kFull * 64, v);
        hand_back();
        store_chunk16<kBF16, 32>(tmC32, slots, count, v, x0 + kFull * 64, y0, M, N, lane);
    }
}

}  // namespace dtc
