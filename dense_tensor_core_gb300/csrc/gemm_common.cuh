// gemm_common.cuh -- pieces shared by the GEMM kernels: the device status word, the kernel
// argument block, the persistent tile order and the fp32 -> 16-bit output packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace dtc {

__device__ int g_dtc_status;  // first device-side wait that gave up (0 = none)


struct Gemm16Args {
    void* C;
    int64_t ldc;  // elements between rows of C (>= N)
    int M, N, K;
    int num_m, num_n, num_kb;
    uint64_t timeout_ns;
    int fault;
};

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
