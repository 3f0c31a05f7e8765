// sp24_expand.cuh -- expansion of a 2:4 structured-sparse A into a dense 16-bit A, on the GPU.
//
// The sparse GEMM (gemm_sp) that the 05 Blackwell TCGEN05 GEMM tutorial names in "An API-level
// note", read as the 2:4 pattern along K: each group of 4 consecutive K-elements of a row of A keeps
// two values, vals [M, K/2] (16-bit, in order), at two positions given by the metadata, meta
// [M, K/8] bytes (group g's nibble at bits 4*(g % 2) of byte g/2; its bits 0-1 hold the position of
// vals[m, 2g], bits 2-3 that of vals[m, 2g+1]). The product then runs on the dense tensor cores:
// this kernel writes A [M, K] (the kept values at their positions, zeros elsewhere) into the
// caller's workspace, and the dense GEMM reads it. (The sparse tensor-core form would take the
// metadata from Tensor Memory in a layout that no document on this machine fixes, so it is not
// used.)
//
// HBM-bound: per row it reads K bytes of values and K/8 of metadata and writes 2K bytes. One
// thread per metadata byte (two groups): one 8-byte load of 4 values, one 1-byte load, one 16-byte
// store of 8 elements; consecutive threads take consecutive bytes of a row, so every warp-wide
// access is contiguous. Grid-stride loop over M * K/8 units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dtc {

constexpr int kSpThreads = 256;

// Sum of two 16-bit codes rounded to the same format (only for a group whose two positions are
// equal, which the 2:4 pattern excludes).
template <bool kBF16>
__device__ __forceinline__ uint16_t add16(uint16_t a, uint16_t b) {
    if constexpr (kBF16) {
        const float s = __bfloat162float(__ushort_as_bfloat16(a)) + __bfloat162float(__ushort_as_bfloat16(b));
        return __bfloat16_as_ushort(__float2bfloat16_rn(s));
    } else {
        const float s = __half2float(__ushort_as_half(a)) + __half2float(__ushort_as_half(b));
        return __half_as_ushort(__float2half_rn(s));
    }
}

template <bool kBF16>
__global__ void __launch_bounds__(kSpThreads)
    sp24_expand_kernel(const uint16_t* __restrict__ vals, const uint8_t* __restrict__ meta,
                       uint16_t* __restrict__ dense, int64_t M, int64_t K) {
    const int64_t per_row = K / 8;  // metadata bytes (= 16-byte output chunks) per row
    const int64_t units = M * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < units;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / per_row;
        const int64_t u = i - m * per_row;
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(vals + m * (K / 2) + 4 * u));
        const uint32_t e = __ldg(meta + m * per_row + u);
        const uint16_t val[4] = {(uint16_t)(v.x & 0xffffu), (uint16_t)(v.x >> 16),
                                 (uint16_t)(v.y & 0xffffu), (uint16_t)(v.y >> 16)};
        uint16_t out[8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // the two groups of this byte
            const uint32_t nib = (e >> (4 * j)) & 0xfu;
            const uint32_t p0 = nib & 3u, p1 = (nib >> 2) & 3u;
            const uint16_t second = p1 == p0 ? add16<kBF16>(val[2 * j], val[2 * j + 1]) : val[2 * j + 1];
#pragma unroll
            for (uint32_t q = 0; q < 4; ++q)  // constant indices: the slots stay in registers
                out[4 * j + q] = q == p1 ? second : (q == p0 ? val[2 * j] : (uint16_t)0);
        }
        uint4 w;
        w.x = (uint32_t)out[0] | ((uint32_t)out[1] << 16);
        w.y = (uint32_t)out[2] | ((uint32_t)out[3] << 16);
        w.z = (uint32_t)out[4] | ((uint32_t)out[5] << 16);
        w.w = (uint32_t)out[6] | ((uint32_t)out[7] << 16);
        *reinterpret_cast<uint4*>(dense + m * K + 8 * u) = w;
    }
}

}  // namespace dtc
