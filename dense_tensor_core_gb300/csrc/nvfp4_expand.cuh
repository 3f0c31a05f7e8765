// nvfp4_expand.cuh -- exact expansion of NVFP4 operands (e2m1 elements, one UE4M3 scale per 16
// K-elements) into bf16, on the GPU.
//
// The block-scaled product of the 05 Blackwell TCGEN05 GEMM tutorial, "Advanced" (gemm_blockscaled,
// "MXFP8 and other block-scaled formats"), for the NVFP4 member of that family:
//   C[m,n] = bf16( sum_k e2m1(A[m,k]) ue4m3(sfA[m,k/16]) * e2m1(B[n,k]) ue4m3(sfB[n,k/16]) )
// The tensor-core kind that takes UE4M3 scales per 16 elements is not used (no document on this
// machine fixes its instruction-descriptor codes or where its scale vectors sit in Tensor Memory).
// Instead each element is multiplied by its scale here and written as bf16, and the bf16 tensor-
// core product runs on the result. The multiplication is exact: an e2m1 value has at most 2
// significant bits and a UE4M3 value at most 4, so their product has at most 5 (bf16 holds 8),
// and its magnitude lies in [2^-10, 2688] (bf16 normals reach 2^-126 and 3.4e38). The product
// C = A' B'^T of the expanded operands is then the NVFP4 product up to the order of the fp32
// accumulation.
//
// Formats (OCP Microscaling Formats (MX) v1.0 for e2m1; UE4M3 is an e4m3 code with the sign bit
// clear):
//   e2m1  : 4 bits s.ee.m, bias 1: e = 0 -> m * 0.5 (0 or 0.5); else (1 + m/2) * 2^(e-1).
//           Packed two per byte along a row, element k in the low nibble of byte k/2 for even k.
//   UE4M3 : 8 bits 0.eeee.mmm, bias 7: e = 0 -> m/8 * 2^-6; else (1 + m/8) * 2^(e-7);
//           e = 15 and m = 7 is NaN, and so is any code with the sign bit set (not a UE4M3 code).
//
// HBM traffic per 16 elements: 8 bytes of codes and one scale byte read, 32 bytes written. One
// thread per 8 elements (half a scale block): one 4-byte load of codes, one 1-byte load of the
// scale, one 16-byte store; consecutive threads take consecutive halves (the operand's rows are
// contiguous), so a warp's stores cover 512 contiguous bytes. blockIdx.y selects the operand (0 =
// A, 1 = B); grid-stride loop over rows x K/8 halves. The decode is kept to a few integer
// instructions per element (byte lookups, then one bf16 multiply per two elements): with a float
// decode and conversion per element the kernel was instruction-bound (~45 us for 4096 x 4096 x
// 8192, ~3.8 TB/s; 34 us now, ~5.0 TB/s).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace dtc {

constexpr int kNvfp4Threads = 256;

struct Nvfp4Operand {
    const uint8_t* codes;  // [rows, K/2] packed e2m1
    const uint8_t* sf;     // [rows, K/16] UE4M3
    uint16_t* out;         // [rows, K] bf16
    int64_t rows;
};

// bf16 bits of a UE4M3 scale code (exact): a normal code 0.eeee.mmm (e >= 1) has exponent e + 120
// and mantissa mmm << 4, by integer arithmetic; the subnormal codes (e = 0, m / 8 * 2^-6) go
// through fp32; a code with the sign bit set, or the NaN code 0x7F, gives a bf16 NaN.
__device__ __forceinline__ uint32_t ue4m3_bf16_bits(uint32_t c) {
    if ((c & 0x80u) || c == 0x7Fu) return 0x7FC0u;
    if ((c & 0x78u) == 0)
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((float)(c & 7u) * 0x1p-9f));
    return ((c & 0x7Fu) << 4) + 0x3C00u;
}

// e2m1 -> bf16 by byte lookup: the bf16 of magnitude code n (0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6) is
// 0xHHLL with HH byte n of {kHi0, kHi1} and LL byte n of {kLo0, kLo1} (little-endian byte order).
constexpr uint32_t kLo0 = 0xC0800000u, kLo1 = 0xC0804000u;  // 00 00 80 C0 | 00 40 80 C0
constexpr uint32_t kHi0 = 0x3F3F3F00u, kHi1 = 0x40404040u;  // 00 3F 3F 3F | 40 40 40 40

// 8 packed e2m1 codes (element 2j in the low nibble of byte j) times the scale pair s2, as 4
// words of two bf16 (element 2j in the low half of word j). The magnitudes of elements 2j and
// 2j + 1 become the selectors of two byte permutations (one into the low-byte table, one into
// the high-byte table, the unused selector nibbles picking the zero entry 0; a permutation reads
// only the low 16 bits of its selector). A third permutation takes byte j of the sign bits, once
// shifted left by 4 (element 2j's sign to bit 7) into byte 1 and once as they are (element
// 2j + 1's) into byte 3, i.e. to bits 15 and 31. The products are exact (at most 5 significant
// bits), so the bf16 multiply rounds nothing.
__device__ __forceinline__ void e2m1x8_times(uint32_t c, __nv_bfloat162 s2, uint32_t (&out)[4]) {
    const uint32_t lo_mag = c & 0x07070707u;         // even elements' magnitudes, one per byte
    const uint32_t hi_mag = (c >> 4) & 0x07070707u;  // odd elements'
    const uint32_t i01 = __byte_perm(lo_mag, hi_mag, 0x5140);  // m0 m1 m2 m3
    const uint32_t i23 = __byte_perm(lo_mag, hi_mag, 0x7362);  // m4 m5 m6 m7
    const uint32_t sel[4] = {i01, i01 >> 16, i23, i23 >> 16};
    const uint32_t sgn = c & 0x88888888u;
    const uint32_t sgn4 = sgn << 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t sign = __byte_perm(sgn4, sgn, (j << 4) | ((4 + j) << 12)) & 0x80008000u;
        uint32_t w = __byte_perm(kLo0, kLo1, sel[j]) | __byte_perm(kHi0, kHi1, sel[j] << 4) | sign;
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
        v = __hmul2(v, s2);
        out[j] = *reinterpret_cast<uint32_t*>(&v);
    }
}

// Each thread takes kUnroll halves of 16-element blocks per pass, kThreads apart, and issues all
// their loads before converting any; a warp's 16-byte stores then cover 512 contiguous bytes.
template <int kThreads = kNvfp4Threads, int kUnroll = 4>
__global__ void __launch_bounds__(kThreads)
    nvfp4_expand_kernel(const Nvfp4Operand opA, const Nvfp4Operand opB, int64_t K) {
    const Nvfp4Operand& op = blockIdx.y == 0 ? opA : opB;
    const int64_t units = op.rows * (K / 8);  // halves of 16-element scale blocks
    const uint32_t* codes = reinterpret_cast<const uint32_t*>(op.codes);
    const int64_t stride = (int64_t)gridDim.x * kThreads * kUnroll;
    for (int64_t base = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; base < units;
         base += stride) {
        uint32_t v[kUnroll], sc[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i < units) {
                v[u] = __ldg(codes + i);
                sc[u] = __ldg(op.sf + (i >> 1));  // two halves share a scale
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + (int64_t)u * kThreads;
            if (i >= units) continue;
            uint32_t sb = ue4m3_bf16_bits(sc[u]);
            sb |= sb << 16;
            const __nv_bfloat162 s2 = *reinterpret_cast<__nv_bfloat162*>(&sb);
            uint32_t w[4];
            e2m1x8_times(v[u], s2, w);
            *reinterpret_cast<uint4*>(op.out + i * 8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

}  // namespace dtc
