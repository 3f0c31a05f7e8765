// gemm_common.cuh -- pieces shared by the GEMM kernels: the device status word, the kernel
// argument block, the persistent tile order and the fp32 -> 16-bit output packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace dtc {

__device__ int g_dtc_status;  // first device-side wait that gave up (0 = none)

// Scratch of gemm_ex_static_workspace: the stream-K workspace (flags, then the pieces' partial
// sums) in module memory, zero at load, so that entry point allocates nothing. 20 MiB holds the
// stream-K workspace of 76 CTA pairs (152 SMs) with 256-wide tiles: 1 KB of flags + 76 x 2 x 128
// x 256 fp32.
constexpr uint64_t kStaticWsBytes = 20ull << 20;
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];


struct Gemm16Args {
    void* C;
    int64_t ldc;  // elements between rows of C (>= N)
    int M, N, K;
    int num_m, num_n, num_kb;
    uint64_t timeout_ns;
    int fault;
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

}  // namespace dtc
