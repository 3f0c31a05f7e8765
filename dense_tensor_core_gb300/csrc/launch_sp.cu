// launch_sp.cu -- launcher of the 2:4 sparse-A expansion kernel (sp24_expand.cuh).
#include "host.h"
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

}  // namespace dtc_host
