// dtc_gemm.cu -- host side of the C ABI declared in include/dtc_gemm.h: argument checks, variant
// choice, TMA descriptor encoding and kernel launches.
//
// The host-side checks mirror what the generated host function of tilelang (velog) section 1.2
// (Host IRModule) asserts before launching: 2-D operands of the expected dtype and shape, unit
// inner stride, non-null data, and row lengths divisible by 8 elements (16 bytes). Tensor maps are
// encoded per call, as the generated call() of section 1.3 does with cuTensorMapEncodeTiled
// (there: fp16, rank 2, a 128-byte inner box, L2 promotion, zero fill out of bounds), and passed
// to the kernel as __grid_constant__ parameters.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "dtc_gemm.h"
#include "gemm16_1cta.cuh"

namespace {

using dtc::Gemm16Args;

thread_local char g_err[1024];

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(GEMM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr uint64_t kDefaultTimeoutNs = 2ull * 1000 * 1000 * 1000;
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    int major = 0, minor = 0;
    bool attr_set[8] = {};
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Looks up (once per device) the SM count and compute capability of the current device.
int current_device(int* dev_out, DeviceInfo** info_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GEMM_ERR_UNSUPPORTED, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.probed) {
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.supported = (d.major == 10 && d.minor == 3);
        d.probed = true;
    }
    if (!d.supported)
        return fail(GEMM_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, d.major, d.minor);
    *dev_out = dev;
    *info_out = &d;
    return GEMM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major 2-D tensor [outer, inner] with dense rows; box [box_outer, box_inner]; 128-byte
// swizzle (box_inner * element size must be 128 bytes); out-of-bounds elements read as zero.
int make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
              uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz, const char* name) {
    auto fn = encode_fn();
    if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
    return GEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared argument rules of every entry point. Returns GEMM_OK or an error (message set).
int validate(int dtype, const void* A, const void* B, const void* sfA, const void* sfB,
             const void* C, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o) {
    const int64_t kMax = 2147483647;
    if (dtype < 0 || dtype > 2) return fail(GEMM_ERR_INVALID_ARG, "dtype %d is not 0, 1 or 2", dtype);
    if (layout != GEMM_LAYOUT_NT && layout != GEMM_LAYOUT_NN)
        return fail(GEMM_ERR_INVALID_ARG, "layout %d is not NT (0) or NN (1)", layout);
    if (dtype == 2 && layout != GEMM_LAYOUT_NT)
        return fail(GEMM_ERR_UNSUPPORTED, "the MXFP8 GEMM supports the NT layout only");
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax)
        return fail(GEMM_ERR_INVALID_ARG, "sizes M=%lld N=%lld K=%lld must be in [0, 2^31-1]",
                    (long long)M, (long long)N, (long long)K);
    if (o && (o->variant < 0 || o->variant > 3))
        return fail(GEMM_ERR_INVALID_ARG, "unknown variant %d", o->variant);
    if (o && o->split_k < 0) return fail(GEMM_ERR_INVALID_ARG, "split_k must be >= 0");
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return fail(GEMM_ERR_INVALID_ARG, "C is NULL");
    if (!aligned16(C)) return fail(GEMM_ERR_INVALID_ARG, "C is not 16-byte aligned");
    if (N % 8) return fail(GEMM_ERR_INVALID_ARG, "N=%lld: C rows must be a multiple of 16 bytes (N %% 8 == 0)", (long long)N);
    if (K == 0) return GEMM_OK;
    if (!A || !B) return fail(GEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (!aligned16(A) || !aligned16(B)) return fail(GEMM_ERR_INVALID_ARG, "A or B is not 16-byte aligned");
    if (dtype == 2) {
        if (!sfA || !sfB) return fail(GEMM_ERR_INVALID_ARG, "sfA or sfB is NULL");
        if (K % 16)
            return fail(GEMM_ERR_INVALID_ARG, "K=%lld: e4m3 rows must be a multiple of 16 bytes", (long long)K);
    } else {
        if (K % 8)
            return fail(GEMM_ERR_INVALID_ARG, "K=%lld: A rows must be a multiple of 16 bytes (K %% 8 == 0)", (long long)K);
        if (layout == GEMM_LAYOUT_NN && N % 8)
            return fail(GEMM_ERR_INVALID_ARG, "N=%lld: B rows must be a multiple of 16 bytes", (long long)N);
    }
    return GEMM_OK;
}

int choose_variant(int dtype, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o,
                   int sms) {
    (void)M; (void)N; (void)K; (void)layout; (void)sms;
    const int v = o ? o->variant : GEMM_VARIANT_AUTO;
    if (v != GEMM_VARIANT_AUTO) return v;
    if (dtype == 2) return GEMM_VARIANT_1CTA;
    return GEMM_VARIANT_1CTA;
}

template <bool kBF16, bool kNN>
int launch_gemm16_1cta(const void* A, const void* B, void* C, int M, int N, int K,
                       const gemm_options* o, DeviceInfo* dev, int attr_slot, cudaStream_t stream) {
    using namespace dtc::g16;
    const CUtensorMapDataType dt = kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tA, tB;
    int rc = make_tmap(&tA, dt, 2, A, (uint64_t)K, (uint64_t)M, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B, "A");
    if (rc) return rc;
    if (!kNN)
        rc = make_tmap(&tB, dt, 2, B, (uint64_t)K, (uint64_t)N, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B, "B");
    else
        rc = make_tmap(&tB, dt, 2, B, (uint64_t)N, (uint64_t)K, 64, kBK, CU_TENSOR_MAP_SWIZZLE_128B, "B");
    if (rc) return rc;

    auto kern = dtc::gemm16_1cta_kernel<kBF16, kNN>;
    if (!dev->attr_set[attr_slot]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        dev->attr_set[attr_slot] = true;
    }
    Gemm16Args args;
    args.C = C;
    args.M = M;
    args.N = N;
    args.K = K;
    args.num_m = (M + kBM - 1) / kBM;
    args.num_n = (N + kBN - 1) / kBN;
    args.num_kb = (K + kBK - 1) / kBK;
    args.timeout_ns = (o && o->timeout_ns) ? o->timeout_ns : kDefaultTimeoutNs;
    args.fault = o ? o->fault_inject : 0;
    const int tiles = args.num_m * args.num_n;
    const int grid = std::min(tiles, dev->sms);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(tA, tB, args);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return GEMM_OK;
}

int run(int dtype, const void* A, const void* B, const void* sfA, const void* sfB, void* C,
        int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o, cudaStream_t stream) {
    g_err[0] = '\0';
    int rc = validate(dtype, A, B, sfA, sfB, C, M, N, K, layout, o);
    if (rc) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev;
    DeviceInfo* info;
    if ((rc = current_device(&dev, &info))) return rc;
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(C, 0, (size_t)M * (size_t)N * 2, stream);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    const int v = choose_variant(dtype, M, N, K, layout, o, info->sms);
    if (dtype == 2)
        return fail(GEMM_ERR_UNSUPPORTED, "the MXFP8 kernel is not available in this build");
    if (v != GEMM_VARIANT_1CTA)
        return fail(GEMM_ERR_UNSUPPORTED, "variant %d is not available in this build", v);
    const int m = (int)M, n = (int)N, k = (int)K;
    if (dtype == 0)
        return layout == GEMM_LAYOUT_NT
                   ? launch_gemm16_1cta<true, false>(A, B, C, m, n, k, o, info, 0, stream)
                   : launch_gemm16_1cta<true, true>(A, B, C, m, n, k, o, info, 1, stream);
    return layout == GEMM_LAYOUT_NT
               ? launch_gemm16_1cta<false, false>(A, B, C, m, n, k, o, info, 2, stream)
               : launch_gemm16_1cta<false, true>(A, B, C, m, n, k, o, info, 3, stream);
}

}  // namespace

extern "C" {

int gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int layout,
              dtc_stream_t stream) {
    return run(0, A, B, nullptr, nullptr, C, M, N, K, layout, nullptr, (cudaStream_t)stream);
}

int gemm_f16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int layout,
             dtc_stream_t stream) {
    return run(1, A, B, nullptr, nullptr, C, M, N, K, layout, nullptr, (cudaStream_t)stream);
}

int gemm_mxfp8(const void* A, const void* B, const void* sfA, const void* sfB, void* C, int64_t M,
               int64_t N, int64_t K, dtc_stream_t stream) {
    return run(2, A, B, sfA, sfB, C, M, N, K, GEMM_LAYOUT_NT, nullptr, (cudaStream_t)stream);
}

int gemm_ex(int dtype, const void* A, const void* B, const void* sfA, const void* sfB, void* C,
            int64_t M, int64_t N, int64_t K, int layout, const gemm_options* opts,
            dtc_stream_t stream) {
    return run(dtype, A, B, sfA, sfB, C, M, N, K, layout, opts, (cudaStream_t)stream);
}

int gemm_plan(int dtype, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* opts) {
    g_err[0] = '\0';
    // Sizes only: pointer rules are not part of the plan.
    const int64_t kMax = 2147483647;
    if (dtype < 0 || dtype > 2) return -fail(GEMM_ERR_INVALID_ARG, "dtype %d is not 0, 1 or 2", dtype);
    if (layout != GEMM_LAYOUT_NT && layout != GEMM_LAYOUT_NN)
        return -fail(GEMM_ERR_INVALID_ARG, "layout %d is not NT (0) or NN (1)", layout);
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax)
        return -fail(GEMM_ERR_INVALID_ARG, "sizes must be in [0, 2^31-1]");
    int dev;
    DeviceInfo* info;
    int rc = current_device(&dev, &info);
    if (rc) return -rc;
    return choose_variant(dtype, M, N, K, layout, opts, info->sms);
}

const char* gemm_last_error(void) { return g_err; }

int gemm_stream_status(dtc_stream_t stream) {
    g_err[0] = '\0';
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int status = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&status, dtc::g_dtc_status, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (status == 0) return GEMM_OK;
    e = cudaMemcpyToSymbol(dtc::g_dtc_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    return fail(GEMM_ERR_TIMEOUT, "a device-side wait gave up (status 0x%x, site %d)", status,
                status & 0xff);
}

}  // extern "C"
