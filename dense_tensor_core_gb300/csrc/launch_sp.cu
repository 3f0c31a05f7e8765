// launch_sp.cu -- launchers of the expansion kernels that feed the dense tensor-core product: the
// 2:4 sparse-A expansion (sp24_expand.cuh) and the NVFP4 dequantisation (nvfp4_expand.cuh).
#include "host.h"
#include "nvfp4_expand.cuh"
#include "sp24_expand.cuh"

namespace dtc_host {

int launch_sp24_expand(bool bf16, const void* vals, const void* meta, void* dense, int64_t M,
                       int64_t K, DeviceInfo* dev, cudaStream_t stream) {
    const int64_t units = M * (K / 8);
    if (units == 0) return GEMM_OK;
    // a grid-stride loop over the units: a few waves of 8 blocks per SM at most
    const int64_t want = (units + dtc::kSpThreads - 1) / dtc::kSpThreads;
    const int grid = (int)std::min<int64_t>(want, (int64_t)dev->model.sms * 8);
    if (bf16)
        dtc::sp24_expand_kernel<true><<<grid, dtc::kSpThreads, 0, stream>>>(
            static_cast<const uint16_t*>(vals), static_cast<const uint8_t*>(meta),
            static_cast<uint16_t*>(dense), M, K);
    else
        dtc::sp24_expand_kernel<false><<<grid, dtc::kSpThreads, 0, stream>>>(
            static_cast<const uint16_t*>(vals), static_cast<const uint8_t*>(meta),
            static_cast<uint16_t*>(dense), M, K);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sparse expansion launch");
    return GEMM_OK;
}

int launch_nvfp4_expand(const void* A, const void* sfA, const void* B, const void* sfB,
                        void* a_out, void* b_out, int64_t M, int64_t N, int64_t K,
                        DeviceInfo* dev, cudaStream_t stream) {
    const int64_t units = std::max(M, N) * (K / 8);
    if (units == 0) return GEMM_OK;
    // one wave: 8 blocks of 256 threads per SM for the two operands together (the SM's 2048
    // threads), each thread looping over 4 halves of 16-element blocks per pass
    const int64_t want = (units + dtc::kNvfp4Threads * 4 - 1) / (dtc::kNvfp4Threads * 4);
    const int grid = (int)std::min<int64_t>(want, (int64_t)dev->model.sms * 4);
    const dtc::Nvfp4Operand a{static_cast<const uint8_t*>(A), static_cast<const uint8_t*>(sfA),
                              static_cast<uint16_t*>(a_out), M};
    const dtc::Nvfp4Operand b{static_cast<const uint8_t*>(B), static_cast<const uint8_t*>(sfB),
                              static_cast<uint16_t*>(b_out), N};
    dtc::nvfp4_expand_kernel<><<<dim3(grid, 2), dtc::kNvfp4Threads, 0, stream>>>(a, b, K);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "NVFP4 expansion launch");
    return GEMM_OK;
}

}  // namespace dtc_host
