// sf_pack.cuh -- repacking of the block-scaled product's scale arrays into the order in which the
// GEMM kernel copies them into Tensor Memory.
//
// The caller's scale arrays are row-major bytes, sf[row][c] = the E8M0 scale of K-block c of the
// row (c < cols = ceil(K / scale block)). The kernel's Tensor Memory holds a scale set as one
// 32-bit cell per row: 4 consecutive scale bytes of the row (with 128-element blocks those of 4
// consecutive 128-deep K-blocks; with 32-element blocks those of the 4 MMAs of one K-block), row r
// of a 128-row group in lane r % 32 of column r / 32. A tcgen05.cp of shape 32x128b.warpx4 writes
// 4 such columns from a 32 x 16-byte matrix whose row i is the cells of rows i, 32 + i, 64 + i and
// 96 + i. This kernel writes those 512-byte matrices ("chunks"), so that the GEMM kernel moves one
// set of one 128-row group with a single 512-byte bulk copy and a single tcgen05.cp:
//
//   chunk (g, s, h) at byte ((g * sets + s) * halves + h) * 512; its byte 16 i + 4 j + b is
//   sf[g * tile_rows + 128 h + 32 j + i][4 s + b]
//
// g = group of tile_rows rows (the 128 rows of an A tile, or the 224 / 256 rows of a B tile),
// h = 128-row half of the group (halves = ceil(tile_rows / 128)), s = scale set (sets =
// ceil(cols / 4)). Bytes past the last row, past the group or past the last scale column are 127
// (a scale of 1; the elements they would scale are zero or never read). One thread per 16 bytes.
#pragma once

#include <stdint.h>

#include "sm103_ptx.cuh"

namespace dtc {

constexpr int kSfChunkBytes = 512;
constexpr int kSfPackThreads = 256;

struct SfPackOperand {
    const uint8_t* sf;  // [rows, cols] row-major
    uint8_t* dst;       // groups * sets * halves chunks
    int rows, cols, sets, tile_rows, halves, groups;
};

// blockIdx.y selects the operand (0 = A, 1 = B); grid-stride over its chunks' 16-byte rows.
// (A template so that every translation unit that includes this header may define it.)
template <int kThreads = kSfPackThreads>
__global__ void __launch_bounds__(kThreads)
    sf_pack_kernel(const SfPackOperand opA, const SfPackOperand opB) {
    // the product kernel may start its set-up and operand loads now; it reads the chunks only
    // after waiting for this grid to complete
    grid_launch_dependents();
    const SfPackOperand& op = blockIdx.y == 0 ? opA : opB;
    const int64_t units = (int64_t)op.groups * op.sets * op.halves * 32;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(u & 31);
        int64_t rest = u >> 5;
        const int h = (int)(rest % op.halves);
        rest /= op.halves;
        const int s = (int)(rest % op.sets);
        const int g = (int)(rest / op.sets);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r_in = 128 * h + 32 * j + i;  // row within the group
            const int64_t row = (int64_t)g * op.tile_rows + r_in;
            uint32_t cell = 0x7F7F7F7Fu;
            if (r_in < op.tile_rows && row < op.rows) {
                const uint8_t* p = op.sf + row * op.cols;
                cell = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int c = 4 * s + b;
                    const uint32_t v = c < op.cols ? (uint32_t)__ldg(p + c) : 0x7Fu;
                    cell |= v << (8 * b);
                }
            }
            w[j] = cell;
        }
        uint4 out;
        out.x = w[0];
        out.y = w[1];
        out.z = w[2];
        out.w = w[3];
        *reinterpret_cast<uint4*>(op.dst + u * 16) = out;
    }
}

}  // namespace dtc
