// dtc_gemm.cu -- host side of the C ABI declared in include/dtc_gemm.h: argument checks, variant
// choice, TMA descriptor encoding and the entry points. The kernels' launchers live in the
// launch_*.cu translation units.
//
// The host-side checks mirror what the generated host function of tilelang (velog) section 1.2
// (Host IRModule) asserts before launching: 2-D operands of the expected dtype and shape, unit
// inner stride, non-null data, and row lengths divisible by 8 elements (16 bytes). Tensor maps are
// encoded per call, as the generated call() of section 1.3 does with cuTensorMapEncodeTiled
// (there: fp16, rank 2, a 128-byte inner box, L2 promotion, zero fill out of bounds), and passed
// to the kernel as __grid_constant__ parameters. That call() returns an int status and keeps the
// message of its last CUDA error in a static buffer; gemm_last_error / gemm_stream_status follow
// the same convention (a per-thread buffer here).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "gemm16_2cta.cuh"
#include "gemm16_splitk.cuh"
#include "gemm_mxfp8_2cta.cuh"
#include "host.h"

namespace dtc_host {

namespace {
thread_local char g_err[1024];
}

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

std::mutex g_dev_mu;

}  // namespace dtc_host

namespace {

using namespace dtc_host;

// First device-side wait that gave up (0 = none); each kernel receives its address.
__device__ int g_dtc_status;

// Scratch of gemm_ex_static_workspace: the stream-K workspace (flags, then the pieces' partial
// sums) in module memory, zero at load, so that entry point allocates nothing. 20 MiB holds the
// stream-K workspace of up to 79 CTA pairs (158 SMs) with 256-wide tiles: 1 KB of flags + 79 x 2 x
// 128 x 256 fp32.
constexpr uint64_t kStaticWsBytes = 20ull << 20;
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];

// Looks up (once per device) the compute capability, the SM count and the status word's address
// on the current device.
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
            (e = cudaDeviceGetAttribute(&d.model.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.supported = (d.major == 10 && d.minor == 3);
        if (d.supported) {
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_dtc_status)) != cudaSuccess)
                return cuda_fail(e, "cudaGetSymbolAddress(status word)");
            d.status = static_cast<int*>(p);
        }
        d.probed = true;
    }
    if (!d.supported)
        return fail(GEMM_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, d.major, d.minor);
    *dev_out = dev;
    *info_out = &d;
    return GEMM_OK;
}

// The device model of the planner: resident clusters are asked once per device, on first use.
const DevModel& device_model(DeviceInfo* d) {
    bool need;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        need = !d->clusters_probed;
    }
    if (need) {
        // (the queries take the lock themselves to raise the kernels' shared-memory limits)
        const int pairs = query_pair_clusters(d);
        const int c2 = query_splitk_clusters(2, d);
        const int c4 = query_splitk_clusters(4, d);
        std::lock_guard<std::mutex> lk(g_dev_mu);
        d->model.pairs = pairs;
        d->model.clusters2 = c2;
        d->model.clusters4 = c4;
        d->clusters_probed = true;
    }
    return d->model;
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

}  // namespace

namespace dtc_host {

// Row-major 2-D tensor [outer, inner] with rows `ld` elements apart; box [box_outer, box_inner];
// with a swizzle the box's inner extent is the swizzle width (128 or 64 bytes); out-of-bounds
// elements read as zero.
int make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
              uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz, const char* name) {
    auto fn = encode_fn();
    if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * (uint64_t)elem_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
    return GEMM_OK;
}

// A K-major row-major [rows, K] operand (rows `ld` elements apart) seen as the 3-D tensor
// {E, rows, ceil(K/E)}, E = the elements in 128 bytes, with strides (row, 128 bytes): a box
// {E, box_rows, 2} is two 128-byte K-chunks of box_rows rows in one instruction. Requires
// K % E == 0 (a partial last chunk would read past the row's K elements).
int make_tmap_kchunks(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
                      uint64_t K, uint64_t rows, uint64_t ld, uint32_t box_rows, const char* name) {
    auto fn = encode_fn();
    if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    const uint64_t e = 128 / elem_bytes;
    cuuint64_t dims[3] = {e, rows, (K + e - 1) / e};
    cuuint64_t strides[2] = {ld * (uint64_t)elem_bytes, 128};
    cuuint32_t box[3] = {(cuuint32_t)e, box_rows, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled(%s, 3-D) failed with CUresult %d", name, (int)r);
    return GEMM_OK;
}

// Tensor map of a block-scaled operand stored as K-major rows of `bits`-bit elements (8: one byte
// each; 6 or 4: packed, which the tensor memory access unit unpacks into 16-byte groups of 16
// elements, 12 or 8 bytes of data then 4 or 8 bytes of padding: the layout the block-scaled MMA
// reads for these types). A 128-element K-block takes one 128-byte swizzled row in shared memory
// whatever the format. 2-D boxes {128, box_rows}, or with `deep` one 3-D box {128, box_rows, 2}
// of two K-blocks (K % 128 == 0).
int tmap_block_scaled(CUtensorMap* m, int bits, const void* ptr, uint64_t K, uint64_t rows,
                      uint64_t row_bytes, uint32_t box_rows, bool deep, const char* name) {
    auto fn = encode_fn();
    if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    const CUtensorMapDataType dt = bits == 8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : bits == 6 ? CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B
                                               : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
    CUresult r;
    if (deep) {
        cuuint64_t dims[3] = {128, rows, (K + 127) / 128};
        cuuint64_t strides[2] = {row_bytes, (cuuint64_t)(128 * bits / 8)};
        cuuint32_t box[3] = {128, box_rows, 2};
        cuuint32_t estr[3] = {1, 1, 1};
        r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[2] = {K, rows};
        cuuint64_t strides[1] = {row_bytes};
        cuuint32_t box[2] = {128, box_rows};
        cuuint32_t estr[2] = {1, 1};
        r = fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS)
        return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled(%s, %d-bit elements) failed with CUresult %d",
                    name, bits, (int)r);
    return GEMM_OK;
}

// Tensor map of a 16-bit operand with `mn` elements along M (or N) and K along the reduction:
// MN-major storage [K, mn] -> 2-D boxes {64, kBK} (128-byte swizzle); K-major storage [mn, K] ->
// one 3-D box {64, box_rows, 2} per 128-deep stage, or a 2-D box {64, box_rows} per 64-deep one.
int tmap_operand16(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, int64_t ld, bool mn_major,
                   int64_t mn, int64_t K, int kBK, uint32_t box_rows, const char* name) {
    if (mn_major)
        return make_tmap(m, dt, 2, ptr, (uint64_t)mn, (uint64_t)K, (uint64_t)ld, 64, (uint32_t)kBK,
                         CU_TENSOR_MAP_SWIZZLE_128B, name);
    if (kBK == 128)
        return make_tmap_kchunks(m, dt, 2, ptr, (uint64_t)K, (uint64_t)mn, (uint64_t)ld, box_rows, name);
    return make_tmap(m, dt, 2, ptr, (uint64_t)K, (uint64_t)mn, (uint64_t)ld, 64, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B, name);
}

// Tensor maps of a 16-bit C [M, N] (rows ldc elements apart) for the TMA-store epilogues: boxes
// of 32 rows x 64 columns with the 128-byte swizzle, and of 32 rows x 32 columns with the 64-byte
// swizzle (the last chunk of a 224-wide tile).
int tmap_c16(CUtensorMap* c64, CUtensorMap* c32, CUtensorMapDataType dt, const Operands& ops,
             int64_t M, int64_t N) {
    int rc = make_tmap(c64, dt, 2, ops.C, (uint64_t)N, (uint64_t)M, (uint64_t)ops.ldc, 64, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B, "C");
    if (rc) return rc;
    return make_tmap(c32, dt, 2, ops.C, (uint64_t)N, (uint64_t)M, (uint64_t)ops.ldc, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B, "C");
}

dtc::Gemm16Args make_args(const Launch& L, int tile_m, int tile_n, int tile_k) {
    const gemm_options* o = L.o;
    const int sk = L.p->sk_tiles;
    dtc::Gemm16Args a;
    a.sk_tiles = sk;
    a.sk_flags = sk ? static_cast<uint32_t*>(o->workspace) : nullptr;
    a.sk_partial = sk ? reinterpret_cast<float*>(static_cast<char*>(o->workspace) + kSkFlagBytes)
                      : nullptr;
    a.C = L.ops->C;
    a.ldc = L.ops->ldc;
    a.M = L.M;
    a.N = L.N;
    a.K = L.K;
    a.num_m = ceil_div(L.M, tile_m);
    a.num_n = ceil_div(L.N, tile_n);
    a.num_kb = ceil_div(L.K, tile_k);
    a.timeout_ns = (o && o->timeout_ns) ? o->timeout_ns : kDefaultTimeoutNs;
    a.fault = o ? o->fault_inject : 0;
    a.status = L.dev->status;
    return a;
}

// Bits per element of a block-scaled element format (gemm_options.mx_a_format / mx_b_format).
int mx_bits(int fmt) { return fmt <= 1 ? 8 : fmt <= 3 ? 6 : 4; }

// Instruction-descriptor element format of kind::mxf8f6f4 for a gemm_options format: e4m3 0,
// e5m2 1, e2m3 3, e3m2 4, e2m1 5 (the PTX ISA's table of the block-scaled kinds' atype / btype).
uint32_t mx_format_code(int fmt) {
    static const uint32_t kCode[5] = {0u, 1u, 3u, 4u, 5u};
    return kCode[fmt];
}

dtc::GemmMxArgs mx_args(const Launch& L, int tile_m, int tile_n, int tile_k) {
    const gemm_options* o = L.o;
    dtc::GemmMxArgs a;
    a.C = L.ops->C;
    a.ldc = L.ops->ldc;
    a.sfA = static_cast<const uint8_t*>(L.ops->sfA);
    a.sfB = static_cast<const uint8_t*>(L.ops->sfB);
    a.M = L.M;
    a.N = L.N;
    a.K = L.K;
    a.num_m = ceil_div(L.M, tile_m);
    a.num_n = ceil_div(L.N, tile_n);
    a.num_kb = ceil_div(L.K, tile_k);
    const int block = (o && o->mx_scale_block) ? o->mx_scale_block : 128;
    a.sf_cols = ceil_div(L.K, block);
    a.fmt_bits = o ? (mx_format_code(o->mx_a_format) << 7) | (mx_format_code(o->mx_b_format) << 10) : 0u;
    // one stage's copies: tile_k K-elements of tile_m rows of A and tile_n rows of B, counted as
    // the bytes the tensor memory access unit writes (packed data only for fp6 / fp4)
    const int a_bits = mx_bits(o ? o->mx_a_format : 0), b_bits = mx_bits(o ? o->mx_b_format : 0);
    a.stage_tx = (uint32_t)((int64_t)tile_k * (tile_m * a_bits + tile_n * b_bits) / 8);
    a.timeout_ns = (o && o->timeout_ns) ? o->timeout_ns : kDefaultTimeoutNs;
    a.fault = o ? o->fault_inject : 0;
    a.status = L.dev->status;
    a.sfA_pack = nullptr;  // set by the launcher when the plan repacks the scales
    a.sfB_pack = nullptr;
    a.sf_sets = 0;
    return a;
}

}  // namespace dtc_host

namespace {

bool layout_a_mn(int layout) { return layout == GEMM_LAYOUT_TN || layout == GEMM_LAYOUT_TT; }
bool layout_b_mn(int layout) { return layout == GEMM_LAYOUT_NN || layout == GEMM_LAYOUT_TN; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Argument rules that need no CUDA call (every entry point, and the planner).
int check_shape(int dtype, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o) {
    const int64_t kMax = 2147483647;
    if (dtype < 0 || dtype > 2) return fail(GEMM_ERR_INVALID_ARG, "dtype %d is not 0, 1 or 2", dtype);
    if (layout < GEMM_LAYOUT_NT || layout > GEMM_LAYOUT_TT)
        return fail(GEMM_ERR_INVALID_ARG, "layout %d is not NT (0), NN (1), TN (2) or TT (3)", layout);
    if (dtype == 2 && layout != GEMM_LAYOUT_NT)
        return fail(GEMM_ERR_UNSUPPORTED, "the MXFP8 GEMM supports the NT layout only");
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax)
        return fail(GEMM_ERR_INVALID_ARG, "sizes M=%lld N=%lld K=%lld must be in [0, 2^31-1]",
                    (long long)M, (long long)N, (long long)K);
    if (o && (o->variant < 0 || o->variant > 3))
        return fail(GEMM_ERR_INVALID_ARG, "unknown variant %d", o->variant);
    if (o && o->split_k < 0) return fail(GEMM_ERR_INVALID_ARG, "split_k must be >= 0");
    if (o && o->tile_n < 0) return fail(GEMM_ERR_INVALID_ARG, "tile_n must be >= 0");
    if (o && (o->mx_a_format < 0 || o->mx_a_format > 4 || o->mx_b_format < 0 || o->mx_b_format > 4))
        return fail(GEMM_ERR_INVALID_ARG, "mx formats must be 0 (e4m3), 1 (e5m2), 2 (e2m3), 3 (e3m2) or 4 (e2m1)");
    if (o && o->mx_scale_block != 0 && o->mx_scale_block != 32 && o->mx_scale_block != 128)
        return fail(GEMM_ERR_INVALID_ARG, "mx_scale_block %d is not 32 or 128", o->mx_scale_block);
    if (dtype != 2 && o && (o->mx_a_format || o->mx_b_format || o->mx_scale_block))
        return fail(GEMM_ERR_INVALID_ARG, "the mx options apply to the block-scaled product only");
    if (o && (o->stream_k < 0 || o->stream_k > 2))
        return fail(GEMM_ERR_INVALID_ARG, "stream_k %d is not 0 (auto), 1 (required) or 2 (off)", o->stream_k);
    return GEMM_OK;
}

// Shared argument rules of every entry point; on success fills `ops` (defaults applied).
// Returns GEMM_OK or an error (message set). Makes no CUDA call.
int validate(int dtype, const void* A, const void* B, const void* sfA, const void* sfB,
             void* C, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o,
             Operands* ops) {
    const int64_t kMax = 2147483647;
    int rc = check_shape(dtype, M, N, K, layout, o);
    if (rc) return rc;
    if (o && (o->lda < 0 || o->ldb < 0 || o->ldc < 0))
        return fail(GEMM_ERR_INVALID_ARG, "lda, ldb and ldc must be >= 0");
    if (o && o->workspace && !aligned16(o->workspace))
        return fail(GEMM_ERR_INVALID_ARG, "the workspace is not 16-byte aligned");
    // operand element bits; the sub-byte block-scaled formats are packed rows, read by the tensor
    // memory access unit's packed types (rows of a multiple of 128 elements and 32 bytes, 32-byte
    // aligned base)
    const int a_bits = dtype == 2 ? mx_bits(o ? o->mx_a_format : 0) : 16;
    const int b_bits = dtype == 2 ? mx_bits(o ? o->mx_b_format : 0) : 16;
    ops->A = A;
    ops->B = B;
    ops->sfA = sfA;
    ops->sfB = sfB;
    ops->C = C;
    ops->a_mn = layout_a_mn(layout);
    ops->b_mn = layout_b_mn(layout);
    const int64_t a_inner = ops->a_mn ? M : K, b_inner = ops->b_mn ? N : K;
    ops->lda = (o && o->lda) ? o->lda : a_inner;
    ops->ldb = (o && o->ldb) ? o->ldb : b_inner;
    ops->ldc = (o && o->ldc) ? o->ldc : N;
    if (ops->lda < a_inner || ops->ldb < b_inner || ops->ldc < N)
        return fail(GEMM_ERR_INVALID_ARG,
                    "lda=%lld ldb=%lld ldc=%lld: a leading dimension is below its row length "
                    "(A %lld, B %lld, C %lld elements)", (long long)ops->lda, (long long)ops->ldb,
                    (long long)ops->ldc, (long long)a_inner, (long long)b_inner, (long long)N);
    if (ops->lda > kMax || ops->ldb > kMax || ops->ldc > kMax)
        return fail(GEMM_ERR_INVALID_ARG, "leading dimensions must be at most 2^31-1");
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return fail(GEMM_ERR_INVALID_ARG, "C is NULL");
    if (!aligned16(C)) return fail(GEMM_ERR_INVALID_ARG, "C is not 16-byte aligned");
    if (ops->ldc % 8)
        return fail(GEMM_ERR_INVALID_ARG, "ldc=%lld: C rows must start 16 bytes apart (a multiple of 8 elements)",
                    (long long)ops->ldc);
    if (K == 0) return GEMM_OK;
    if (!A || !B) return fail(GEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (!aligned16(A) || !aligned16(B)) return fail(GEMM_ERR_INVALID_ARG, "A or B is not 16-byte aligned");
    if (dtype == 2 && (!sfA || !sfB)) return fail(GEMM_ERR_INVALID_ARG, "sfA or sfB is NULL");
    const int64_t a_row = ops->lda * a_bits, b_row = ops->ldb * b_bits;  // bits between rows
    if (a_row % 128)
        return fail(GEMM_ERR_INVALID_ARG, "lda=%lld: rows of A must start 16 bytes apart", (long long)ops->lda);
    if (b_row % 128)
        return fail(GEMM_ERR_INVALID_ARG, "ldb=%lld: rows of B must start 16 bytes apart", (long long)ops->ldb);
    if (a_bits < 8 || b_bits < 8) {
        if (K % 128)
            return fail(GEMM_ERR_INVALID_ARG, "K=%lld: the fp6/fp4 formats need K %% 128 == 0", (long long)K);
        if ((a_bits < 8 && (a_row % 256 || (reinterpret_cast<uintptr_t>(A) & 31))) ||
            (b_bits < 8 && (b_row % 256 || (reinterpret_cast<uintptr_t>(B) & 31))))
            return fail(GEMM_ERR_INVALID_ARG, "fp6/fp4 operands need a 32-byte aligned base and rows "
                        "32 bytes apart");
    }
    return GEMM_OK;
}

// The kernels read and write through tensor maps of the current device: every buffer must be
// device memory of that device (or managed memory). A pointer into another GPU's memory, or into
// host memory, is refused here rather than read over a link.
int check_device_ptr(const void* p, int dev, const char* name) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(GEMM_ERR_INVALID_ARG, "%s (%p) is not memory CUDA knows: %s", name, p,
                    cudaGetErrorName(e));
    }
    if (a.type == cudaMemoryTypeManaged || (a.type == cudaMemoryTypeDevice && a.device == dev))
        return GEMM_OK;
    if (a.type == cudaMemoryTypeDevice)
        return fail(GEMM_ERR_INVALID_ARG, "%s is memory of device %d, not of the current device %d",
                    name, a.device, dev);
    return fail(GEMM_ERR_INVALID_ARG, "%s is not device memory (memory type %d)", name, (int)a.type);
}

// Busy time of the slowest cluster, in tile-width units, when every tile costs time proportional
// to its width: (waves of tiles over the resident units) x (tile width).
int64_t wave_cost(int64_t tiles, int units, int bn) { return (int64_t)ceil_div(tiles, units) * bn; }

// Sustained fraction of tensor peak that one busy unit (an SM running 128 x BN tiles, or a CTA
// pair running 256 x BN tiles) reaches in the main loop, measured on GB300 with bf16 NT operands
// at K = 8192 (4096 x 4096 and 8192 x 8192 products, L2 flushed). The kernels are bound by operand
// delivery from L2 into shared memory, which is fastest with few, large TMA instructions: the
// pair kernel's 128-deep stages (one 3-D box of two K-chunks per operand, needs K % 64 == 0)
// beat its 64-deep ones, and the wider, taller tiles need fewer bytes per flop.
struct TileChoice {
    int variant, tile_n, tile_k;
    double efficiency;
};
constexpr TileChoice kChoices[] = {
    {GEMM_VARIANT_1CTA, 256, 64, 0.61},
    {GEMM_VARIANT_1CTA, 224, 64, 0.585},
    {GEMM_VARIANT_2CTA, 256, 128, 0.70},
    {GEMM_VARIANT_2CTA, 224, 128, 0.635},
    {GEMM_VARIANT_2CTA, 256, 64, 0.64},
    {GEMM_VARIANT_2CTA, 224, 64, 0.56},
};

// Pairs a persistent pair-kernel launch may count on: half the SMs, or fewer when fewer pairs can
// be resident at once.
int resident_pairs(const DevModel& d) {
    const int half = std::max(1, d.sms / 2);
    return d.pairs > 0 ? std::min(half, d.pairs) : half;
}

// Busy time of the slowest SM, in units of (128 x 1 x K) MMA work at full rate: waves of tiles
// over the resident units x per-SM tile width / efficiency.
double plan_cost(int variant, int bn, double eff, int64_t M, int64_t N, const DevModel& d) {
    const int units = variant == GEMM_VARIANT_2CTA ? resident_pairs(d) : std::max(1, d.sms);
    const int64_t rows = variant == GEMM_VARIANT_2CTA ? ceil_div(M, 256) : ceil_div(M, 128);
    const int64_t tiles = rows * ceil_div(N, bn);
    return (double)ceil_div(tiles, units) * bn / eff;
}

double choice_efficiency(int variant, int bn, int bk) {
    for (const TileChoice& c : kChoices)
        if (c.variant == variant && c.tile_n == bn && c.tile_k == bk) return c.efficiency;
    return 0.5;
}

// Stream-K on CTA pairs (256 x 256 tiles, 128-deep stages; 64-deep on request): when the tiles
// leave the last wave part-empty, the leftover tiles are shared out over all pairs as equal runs of
// K-blocks, their pieces summed through the caller's workspace. A pair waits for the pieces of
// later pairs, so every pair of the launch must be resident at once: the units are the pairs the
// device keeps resident (at most 128, the flags' capacity). Taken when a large enough workspace is
// given, the request allows the pair kernel with these tiles, and the cost model beats the plan
// already made: work per pair / efficiency, plus 0.4 of a tile's time for the pieces' exchange and
// the shorter runs (measured on GB300: +2-4 % on 8192^3; on 4096^2 x 8192 within 1 % of 224-wide
// whole tiles, on average slightly ahead, which this constant encodes). Sharing a whole wave more
// (longer runs, fewer splits) measured worse on both. Required or refused with opts->stream_k.
int plan_stream_k(int64_t M, int64_t N, int64_t K, const gemm_options* o, const DevModel& d, Plan* p) {
    const int mode = o ? o->stream_k : 0;
    if (mode == 2) return GEMM_OK;
    const int units = resident_pairs(d);
    const int64_t tiles = (int64_t)ceil_div(M, 256) * ceil_div(N, 256);
    const int req_v = o ? o->variant : GEMM_VARIANT_AUTO;
    const bool allowed = (req_v == GEMM_VARIANT_AUTO || req_v == GEMM_VARIANT_2CTA) &&
                         (!o || o->tile_n == 0 || o->tile_n == 256) &&
                         (!o || o->tile_k == 0 || o->tile_k == 128 || o->tile_k == 64) &&
                         (!o || o->split_k == 0) && units <= kSkMaxUnits &&
                         K % 64 == 0 && p->variant != GEMM_VARIANT_SPLITK && tiles >= units &&
                         tiles % units != 0;
    const bool ws_ok = o && o->workspace && o->workspace_bytes >= sk_workspace_bytes(units, 256);
    if (mode == 1 && !allowed)
        return fail(GEMM_ERR_UNSUPPORTED, "stream-K needs the pair kernel with 256 x 256 tiles, "
                    "K %% 64 == 0, at most %d resident pairs and a tile count that is not a whole "
                    "number of waves of the %d resident pairs", kSkMaxUnits, units);
    if (mode == 1 && !ws_ok)
        return fail(GEMM_ERR_INVALID_ARG, "stream-K needs a workspace of %llu bytes",
                    (unsigned long long)sk_workspace_bytes(units, 256));
    if (!allowed || !ws_ok) return GEMM_OK;
    const double eff = choice_efficiency(GEMM_VARIANT_2CTA, 256, 128);
    const double sk_cost = ((double)tiles / units + 0.4) * 256 / eff;
    const double dp_cost = plan_cost(p->variant, p->tile_n,
                                     choice_efficiency(p->variant, p->tile_n, p->tile_k), M, N, d);
    if (mode == 0 && sk_cost >= dp_cost) return GEMM_OK;
    p->variant = GEMM_VARIANT_2CTA;
    p->cluster = 2;
    p->tile_m = 256;
    p->tile_n = 256;
    p->tile_k = (o && o->tile_k == 64) ? 64 : 128;
    p->stages = p->tile_k == 128 ? 3 : 6;
    p->split_k = 1;
    p->tiles = (int)tiles;
    p->sk_tiles = (int)(tiles % units);
    p->ctas = 2 * units;
    return GEMM_OK;
}

// The launch for these sizes and options on a device described by `d`: a pure function (no CUDA
// call), so it can be asked for any device model.
int make_plan(int dtype, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o,
              const DevModel& d, Plan* p) {
    int v = o ? o->variant : GEMM_VARIANT_AUTO;
    const int want_n = o ? o->tile_n : 0;
    const bool b_mn = layout_b_mn(layout);  // B stored [K,N]: 64-column boxes
    const int sms = std::max(1, d.sms);
    const int pairs = resident_pairs(d);
    if (want_n && want_n != 256 && want_n != 128 && want_n != 224 && want_n != 64)
        return fail(GEMM_ERR_UNSUPPORTED, "tile width %d is not offered", want_n);
    if (want_n == 224 && b_mn && v == GEMM_VARIANT_1CTA)
        return fail(GEMM_ERR_UNSUPPORTED, "224-wide one-CTA tiles need B stored [N,K]");
    if (dtype == 2) {
        if (v != GEMM_VARIANT_AUTO && v != GEMM_VARIANT_1CTA && v != GEMM_VARIANT_2CTA)
            return fail(GEMM_ERR_UNSUPPORTED, "the MXFP8 product has one-CTA and pair kernels");
        if (want_n && want_n != 224)
            return fail(GEMM_ERR_UNSUPPORTED, "the block-scaled kernels use 224-wide tiles");
        const int bk_want = o ? o->tile_k : 0;
        if (bk_want && bk_want != 128 && bk_want != 256)
            return fail(GEMM_ERR_INVALID_ARG, "tile_k %d is not 128 or 256 for the block-scaled kernels", bk_want);
        const int block = (o && o->mx_scale_block) ? o->mx_scale_block : 128;
        const uint64_t need = sf_pack_layout(M, N, (K + block - 1) / block, 224).bytes;
        const bool ws = o && o->workspace && o->workspace_bytes >= need;
        // Two kernels. The pair kernel (256 x 224 tiles, 3 stages of 256 K-elements, scales
        // repacked into the workspace) takes 128-element scale blocks with K % 128 == 0; AUTO
        // takes it when a workspace holds the repacked scales and the pair tiles fill at least
        // one wave with most of their 256 rows (GB300, 4096 x 4096 x 8192: e4m3 102.4 us against
        // 108.8 on the one-CTA kernel, fp4 and fp6 100.4 against 106.8 and 108.8). The one-CTA
        // kernel (128 x 224 tiles, 4 stages of 128 K-elements) takes everything else.
        if (v == GEMM_VARIANT_AUTO) {
            const bool pair = block == 128 && ws && K % 128 == 0 && bk_want != 128 &&
                              (M % 256 == 0 || M % 256 > 128) &&
                              (int64_t)ceil_div(M, 256) * ceil_div(N, 224) >= pairs;
            v = pair ? GEMM_VARIANT_2CTA : GEMM_VARIANT_1CTA;
        }
        if (v == GEMM_VARIANT_2CTA) {
            if (block != 128 || K % 128 || !ws || bk_want == 128)
                return fail(GEMM_ERR_UNSUPPORTED, "the block-scaled pair kernel takes 128-element "
                            "scale blocks, K %% 128 == 0, 256-deep stages and a workspace of %llu "
                            "bytes for the repacked scales", (unsigned long long)need);
            p->variant = v;
            p->cluster = 2;
            p->tile_m = 256;
            p->tile_n = dtc::gmx2::kBN;
            p->tile_k = dtc::gmx2::kBlocks * dtc::gmx2::kBK;
            p->stages = dtc::gmx2::kNStages;
            p->tiles = ceil_div(M, 256) * ceil_div(N, p->tile_n);
            p->ctas = 2 * std::min(p->tiles, pairs);
            p->sf_pack = true;
            return GEMM_OK;
        }
        if (bk_want == 256)
            return fail(GEMM_ERR_UNSUPPORTED, "the one-CTA block-scaled kernel takes 128-deep "
                        "stages (256-deep ones are the pair kernel's)");
        p->variant = GEMM_VARIANT_1CTA;
        p->tile_m = dtc::gmx::kBM;
        p->tile_n = dtc::gmx::kBN;
        p->tile_k = dtc::gmx::kBK;
        p->stages = dtc::gmx::Cfg<>::kStages;
        p->tiles = ceil_div(M, p->tile_m) * ceil_div(N, p->tile_n);
        p->ctas = std::min(p->tiles, sms);
        // With 32-element scale blocks and a large enough workspace the scales are repacked
        // there and reach Tensor Memory by bulk copy and tcgen05.cp instead of through the
        // kernel's scale warps: 4096 x 4096 x 8192 e4m3 ran 115.7 us against 307. With
        // 128-element blocks the scale warps keep up (108.8 us against 109.6 repacked, the
        // repacking included), so they stay.
        p->sf_pack = block == 32 && ws;
        return GEMM_OK;
    }
    const int num_kb = ceil_div(K, 64);
    const int64_t tiles256 = (int64_t)ceil_div(M, 128) * ceil_div(N, 256);
    const int64_t tiles128 = (int64_t)ceil_div(M, 128) * ceil_div(N, 128);
    int split = o ? o->split_k : 0;
    if (split != 0 && split != 1 && split != 2 && split != 4)
        return fail(GEMM_ERR_INVALID_ARG, "split_k %d is not 1, 2 or 4", split);
    if (split == 1 && v == GEMM_VARIANT_AUTO) v = GEMM_VARIANT_SPLITK;
    int split_n = want_n;
    int auto_n = 0;
    if (v == GEMM_VARIANT_AUTO && split == 0 && want_n != 224 && tiles256 * 2 <= sms) {
        // Fewer 128 x 256 tiles than half the SMs: split K over a cluster of 2 or 4 CTAs per
        // 128 x 128 or 128 x 256 tile. Take the (width, split) that occupies the most SMs in one
        // wave; on a tie the smaller split (less to reduce), then the narrower tile (a smaller
        // exchange). Each CTA keeps at least 8 K-blocks of 64, or 4 when one-CTA tiles would
        // leave all but a few SMs idle (at most one 128 x 256 tile per 8 SMs): the on-chip
        // exchange of the partial sums costs ~2 us, which a split pays back only when it halves
        // a long K loop or spreads a product that would otherwise run on a handful of SMs
        // (GB300, L2 flushed: 256 x 256 x 512 split in 2 10.2 us against 10.5-10.7 one-CTA;
        // 384 x 640 x 768 10.2 against 12.7; 1024 x 1024 x 512, 32 one-CTA tiles, 10.9 split
        // against 10.7).
        const int min_kb = tiles256 * 8 <= sms ? 4 : 8;
        struct Cand { int bn, s; };
        const Cand cands[3] = {{128, 2}, {128, 4}, {256, 2}};
        int64_t best_ctas = 0;
        for (const Cand& c : cands) {
            if (want_n && c.bn != want_n) continue;
            const int64_t tl = c.bn == 128 ? tiles128 : tiles256;
            const int64_t ctas = tl * c.s;
            const int resident = c.s == 2 ? (d.clusters2 > 0 ? d.clusters2 : sms / 2)
                                          : (d.clusters4 > 0 ? d.clusters4 : sms / 4);
            if (num_kb < min_kb * c.s || ctas > (int64_t)resident * c.s) continue;
            if (ctas > best_ctas || (ctas == best_ctas && c.s < split)) {
                best_ctas = ctas;
                split = c.s;
                split_n = c.bn;
            }
        }
        // A short K (at most 8 K-blocks of 64): one CTA per 128 x 64 tile with the whole K, no
        // exchange, where that gives at least as many CTAs as the split (256 x 256 x 512: 9.2 us
        // against 10.3 split in 2; 1024^3 level at 12.2; the skinny 128 x 8192 x 8192, K = 8192,
        // 37.0 against 31.4, so not there)
        const int64_t tiles64 = (int64_t)ceil_div(M, 128) * ceil_div(N, 64);
        if (split && !want_n && K <= 512 && K % 64 == 0 && tiles64 >= best_ctas && tiles64 <= sms) {
            split = 1;
            split_n = 64;
        }
        // 256 x 128 pair tiles (4 stages of 128 K-elements) load as many bytes per CTA as 128 x 256
        // tiles split in 2 and need no exchange of partial sums: taken when they give at least as
        // many CTAs as the best split, fit in one wave and fill most of their 256 rows (512 x 4096 x
        // 4096: 22.6 us against 24.6 split; 1024 x 2048 x 2048: 16.4 against 16.5; 1024^3, with
        // half the CTAs of a 128 x 128 split: 12.7 against 12.3, so not taken there)
        const int64_t pair128 = (int64_t)ceil_div(M, 256) * ceil_div(N, 128);
        const bool rows_filled = M >= 256 && (M % 256 == 0 || M % 256 > 128);
        if (!want_n && rows_filled && K % 64 == 0 && pair128 <= pairs && 2 * pair128 >= best_ctas &&
            best_ctas > 0) {
            v = GEMM_VARIANT_2CTA;
            auto_n = 128;
            split = 0;
        }
        if (split) v = GEMM_VARIANT_SPLITK;
    }
    if (v == GEMM_VARIANT_SPLITK && split == 1) {
        // one CTA per 128 x 64 tile with the whole K (128-deep stages): no exchange
        if (split_n && split_n != 64)
            return fail(GEMM_ERR_UNSUPPORTED, "the split-K kernel's unsplit mode uses 64-wide tiles");
        if (K % 64 || (o && o->tile_k && o->tile_k != 128))
            return fail(GEMM_ERR_UNSUPPORTED, "the unsplit split-K mode takes 128-deep stages (K %% 64 == 0)");
        p->variant = v;
        p->split_k = 1;
        p->cluster = 1;
        p->tile_m = 128;
        p->tile_n = 64;
        p->tile_k = 128;
        p->stages = dtc::gsk::stages_for(64, 128, 1);
        p->tiles = (int)((int64_t)ceil_div(M, 128) * ceil_div(N, 64));
        p->ctas = p->tiles;
        return GEMM_OK;
    }
    if (v == GEMM_VARIANT_SPLITK) {
        if (split_n && split_n != 256 && split_n != 128)
            return fail(GEMM_ERR_UNSUPPORTED, "the split-K kernel uses 128- or 256-wide tiles");
        if (split_n == 256 && split == 4)
            return fail(GEMM_ERR_UNSUPPORTED, "256-wide split-K tiles take a split of 2");
        const int bk_want = o ? o->tile_k : 0;
        if (bk_want && bk_want != 64 && bk_want != 128)
            return fail(GEMM_ERR_INVALID_ARG, "tile_k %d is not 64 or 128 for the split-K kernel", bk_want);
        p->variant = v;
        p->split_k = split ? split : 2;
        p->cluster = p->split_k;
        p->tile_m = 128;
        p->tile_n = split_n ? split_n : 128;
        // 128-deep stages (3-D boxes over 128-byte K-chunks) need K % 64 == 0; 256-wide tiles
        // keep 64-deep stages, or too few stages would fit beside the exchange area
        p->tile_k = bk_want ? bk_want : (p->tile_n == 128 && K % 64 == 0 ? 128 : 64);
        if (p->tile_k == 128 && (K % 64 || p->tile_n != 128))
            return fail(GEMM_ERR_UNSUPPORTED, "128-deep split-K stages need K %% 64 == 0 and 128-wide tiles");
        p->stages = dtc::gsk::stages_for(p->tile_n, p->tile_k, p->split_k);
        p->tiles = (int)(p->tile_n == 128 ? tiles128 : tiles256);
        p->ctas = p->tiles * p->split_k;
        return GEMM_OK;
    }
    if ((want_n == 128 || want_n == 64) && v != GEMM_VARIANT_2CTA)
        return fail(GEMM_ERR_UNSUPPORTED, "%d-wide tiles are offered by the split-K (128) and pair kernels only", want_n);
    if (v == GEMM_VARIANT_AUTO) {
        // Cheapest (variant, width) by the cost model; 224-wide tiles exist for a K-major B (NT,
        // TT) only. Below one wave of tiles either way, the one-CTA kernel (shorter ring fill)
        // is preferred.
        double best = -1.0;
        int best_v = GEMM_VARIANT_1CTA, best_n = 256;
        for (const TileChoice& c : kChoices) {
            if (c.tile_n == 224 && b_mn && c.variant == GEMM_VARIANT_1CTA) continue;
            if (want_n && c.tile_n != want_n) continue;
            if (c.variant == GEMM_VARIANT_2CTA && (c.tile_k == 128) != (K % 64 == 0)) continue;
            double cost = plan_cost(c.variant, c.tile_n, c.efficiency, M, N, d);
            if (c.variant == GEMM_VARIANT_2CTA && ceil_div(M, 256) * ceil_div(N, c.tile_n) < pairs)
                cost *= 1.25;
            if (best < 0 || cost < best) {
                best = cost;
                best_v = c.variant;
                best_n = c.tile_n;
            }
        }
        v = best_v;
        auto_n = best_n;
    }
    p->variant = v;
    if (v == GEMM_VARIANT_1CTA) {
        const int bk = o ? o->tile_k : 0;
        if (bk != 0 && bk != 64)
            return fail(GEMM_ERR_INVALID_ARG, "tile_k %d is not 64 for the one-CTA kernel", bk);
        int best = auto_n ? auto_n : 256;
        if (want_n == 224 && b_mn)
            return fail(GEMM_ERR_UNSUPPORTED, "224-wide one-CTA tiles need B stored [N,K]");
        const int64_t rows = ceil_div(M, 128);
        if (want_n) {
            best = want_n;
        } else if (!auto_n && !b_mn) {
            if (wave_cost(rows * ceil_div(N, 224), sms, 224) < wave_cost(rows * ceil_div(N, 256), sms, 256))
                best = 224;
        }
        p->cluster = 1;
        p->tile_m = 128;
        p->tile_n = best;
        p->tile_k = 64;
        p->stages = 4;
        p->tiles = (int)rows * ceil_div(N, best);
        p->ctas = std::min(p->tiles, sms);
    } else {
        p->cluster = 2;
        p->tile_m = 256;
        if (want_n) {
            p->tile_n = want_n;
        } else if (auto_n) {
            p->tile_n = auto_n;
        } else {
            const int64_t rows = ceil_div(M, 256);
            p->tile_n = wave_cost(rows * ceil_div(N, 224), pairs, 224) <
                                wave_cost(rows * ceil_div(N, 256), pairs, 256)
                            ? 224
                            : 256;
        }
        int bk = o ? o->tile_k : 0;
        if (bk != 0 && bk != 64 && bk != 128)
            return fail(GEMM_ERR_INVALID_ARG, "tile_k %d is not 64 or 128 for the pair kernel", bk);
        if (bk == 128 && K % 64)
            return fail(GEMM_ERR_UNSUPPORTED, "128-deep pair stages need K %% 64 == 0");
        if (bk == 0) bk = K % 64 == 0 ? 128 : 64;
        if (p->tile_n <= 128 && bk != 128)
            return fail(GEMM_ERR_UNSUPPORTED, "%d-wide pair tiles take 128-deep stages (K %% 64 == 0)", p->tile_n);
        p->tile_k = bk;
        p->stages = dtc::g2::stages_for(p->tile_n, bk);
        p->tiles = ceil_div(M, 256) * ceil_div(N, p->tile_n);
        p->ctas = 2 * std::min(p->tiles, pairs);
    }
    return plan_stream_k(M, N, K, o, d, p);
}

// A call made ready to launch: checked arguments, the device and the plan.
struct Prepared {
    Operands ops;
    Plan p;
    int dev = -1;
    DeviceInfo* info = nullptr;
    bool noop = false;    // M == 0 or N == 0
    bool zero_k = false;  // K == 0: C = 0
};

int prepare(int dtype, const void* A, const void* B, const void* sfA, const void* sfB, void* C,
            int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o, Prepared* r) {
    int rc = validate(dtype, A, B, sfA, sfB, C, M, N, K, layout, o, &r->ops);
    if (rc) return rc;
    if (M == 0 || N == 0) {
        r->noop = true;
        return GEMM_OK;
    }
    if ((rc = current_device(&r->dev, &r->info))) return rc;
    if ((rc = check_device_ptr(C, r->dev, "C"))) return rc;
    if (K == 0) {
        r->zero_k = true;
        return GEMM_OK;
    }
    if ((rc = check_device_ptr(A, r->dev, "A")) || (rc = check_device_ptr(B, r->dev, "B"))) return rc;
    if (dtype == 2 &&
        ((rc = check_device_ptr(sfA, r->dev, "sfA")) || (rc = check_device_ptr(sfB, r->dev, "sfB"))))
        return rc;
    if ((rc = make_plan(dtype, M, N, K, layout, o, device_model(r->info), &r->p))) return rc;
    if ((r->p.sk_tiles || r->p.sf_pack) && (rc = check_device_ptr(o->workspace, r->dev, "the workspace")))
        return rc;
    return GEMM_OK;
}

int launch_prepared(const Prepared& r, int dtype, int64_t M, int64_t N, int64_t K,
                    const gemm_options* o, cudaStream_t stream) {
    if (r.noop) return GEMM_OK;
    if (r.zero_k) {  // the empty sum: C = 0 (only the M x N region of a strided C)
        cudaError_t e = cudaMemset2DAsync(r.ops.C, (size_t)r.ops.ldc * 2, 0, (size_t)N * 2, (size_t)M, stream);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "cudaMemset2DAsync");
    }
    const Launch L{&r.ops, (int)M, (int)N, (int)K, o, r.info, &r.p, stream};
    if (dtype == 2) return launch_mx(L);
    if (r.p.variant == GEMM_VARIANT_SPLITK) return launch16_splitk(dtype == 0, L);
    if (r.p.variant == GEMM_VARIANT_1CTA) return launch16_1cta(dtype == 0, L);
    return dtype == 0 ? launch16_2cta_bf16(L) : launch16_2cta_f16(L);
}

int run(int dtype, const void* A, const void* B, const void* sfA, const void* sfB, void* C,
        int64_t M, int64_t N, int64_t K, int layout, const gemm_options* o, cudaStream_t stream) {
    g_err[0] = '\0';
    Prepared r;
    int rc = prepare(dtype, A, B, sfA, sfB, C, M, N, K, layout, o, &r);
    if (rc) return rc;
    return launch_prepared(r, dtype, M, N, K, o, stream);
}

void fill_info(const Plan& p, gemm_plan_info* info) {
    info->variant = p.variant;
    info->tile_m = p.tile_m;
    info->tile_n = p.tile_n;
    info->tile_k = p.tile_k;
    info->stages = p.stages;
    info->split_k = p.split_k;
    info->ctas = p.ctas;
    info->tiles = p.tiles;
    info->cluster = p.cluster;
    info->sk_tiles = p.sk_tiles;
    info->sf_packed = p.sf_pack ? 1 : 0;
}

DevModel to_model(const gemm_device_model& m) {
    DevModel d;
    d.sms = m.sm_count;
    d.pairs = m.pair_clusters;
    d.clusters2 = m.split2_clusters;
    d.clusters4 = m.split4_clusters;
    return d;
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

int gemm_ex_static_workspace(int dtype, const void* A, const void* B, const void* sfA,
                             const void* sfB, void* C, int64_t M, int64_t N, int64_t K,
                             int layout, const gemm_options* opts, dtc_stream_t stream) {
    g_err[0] = '\0';
    if (opts && opts->workspace)
        return fail(GEMM_ERR_INVALID_ARG, "this entry point supplies its own workspace: leave opts->workspace NULL");
    int dev;
    DeviceInfo* info;
    int rc = current_device(&dev, &info);
    if (rc) return rc;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!info->static_ws) {  // once per device (a synchronous call: not inside stream capture)
            void* p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
            info->static_ws = p;
        }
    }
    gemm_options o = {};
    if (opts) o = *opts;
    o.workspace = info->static_ws;
    o.workspace_bytes = kStaticWsBytes;
    Prepared r;
    if ((rc = prepare(dtype, A, B, sfA, sfB, C, M, N, K, layout, &o, &r))) return rc;
    if (r.p.sk_tiles) {
        // the flags must be zero when a launch starts: every completed call leaves them zero, but
        // a call that gave up (GEMM_ERR_TIMEOUT) may not, so clear them, in stream order, before
        // each launch that uses them
        cudaError_t e = cudaMemsetAsync(info->static_ws, 0, kSkFlagBytes, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static workspace flags)");
    }
    return launch_prepared(r, dtype, M, N, K, &o, (cudaStream_t)stream);
}

int gemm_sp_workspace_size(int dtype, int64_t M, int64_t K, uint64_t* bytes) {
    g_err[0] = '\0';
    if (!bytes) return fail(GEMM_ERR_INVALID_ARG, "bytes is NULL");
    if (dtype != 0 && dtype != 1) return fail(GEMM_ERR_INVALID_ARG, "dtype %d is not 0 (bf16) or 1 (fp16)", dtype);
    if (M < 0 || K < 0 || M > 2147483647 || K > 2147483647)
        return fail(GEMM_ERR_INVALID_ARG, "sizes must be in [0, 2^31-1]");
    *bytes = (uint64_t)M * (uint64_t)K * 2;
    return GEMM_OK;
}

int gemm_sp(int dtype, const void* vals, const void* meta, const void* B, void* C, int64_t M,
            int64_t N, int64_t K, int layout, const gemm_options* opts, void* workspace,
            uint64_t workspace_bytes, dtc_stream_t stream) {
    g_err[0] = '\0';
    if (dtype != 0 && dtype != 1)
        return fail(GEMM_ERR_INVALID_ARG, "dtype %d is not 0 (bf16) or 1 (fp16)", dtype);
    if (layout != GEMM_LAYOUT_NT && layout != GEMM_LAYOUT_NN)
        return fail(GEMM_ERR_INVALID_ARG, "the sparse product takes layout NT (0) or NN (1)");
    if (opts && opts->lda)
        return fail(GEMM_ERR_INVALID_ARG, "the sparse product's A rows are dense (lda must be 0)");
    if (K % 16)
        return fail(GEMM_ERR_INVALID_ARG, "K=%lld: the sparse product needs K %% 16 == 0", (long long)K);
    const bool work = M > 0 && N > 0 && K > 0;
    if (work) {
        if (!vals || !meta) return fail(GEMM_ERR_INVALID_ARG, "vals or meta is NULL");
        if (!aligned16(vals)) return fail(GEMM_ERR_INVALID_ARG, "vals is not 16-byte aligned");
        if (!workspace || workspace_bytes < (uint64_t)M * (uint64_t)K * 2)
            return fail(GEMM_ERR_INVALID_ARG, "the sparse product needs a workspace of %llu bytes "
                        "(M x K 16-bit elements)", (unsigned long long)((uint64_t)M * (uint64_t)K * 2));
    }
    // the dense call on the expanded A (checks B, C, the workspace, the sizes and the options)
    Prepared r;
    int rc = prepare(dtype, work ? workspace : nullptr, B, nullptr, nullptr, C, M, N, K, layout,
                     opts, &r);
    if (rc) return rc;
    if (work) {
        if ((rc = check_device_ptr(vals, r.dev, "vals")) || (rc = check_device_ptr(meta, r.dev, "meta")))
            return rc;
        if ((rc = launch_sp24_expand(dtype == 0, vals, meta, workspace, M, K, r.info,
                                     (cudaStream_t)stream)))
            return rc;
    }
    return launch_prepared(r, dtype, M, N, K, opts, (cudaStream_t)stream);
}

// NVFP4 workspace: the expanded A (bf16 [M,K]) at offset 0, the expanded B (bf16 [N,K]) at the
// next 256-byte boundary.
uint64_t nvfp4_b_offset(int64_t M, int64_t K) {
    return ((uint64_t)M * (uint64_t)K * 2 + 255) & ~(uint64_t)255;
}

int gemm_nvfp4_workspace_size(int64_t M, int64_t N, int64_t K, uint64_t* bytes) {
    g_err[0] = '\0';
    if (!bytes) return fail(GEMM_ERR_INVALID_ARG, "bytes is NULL");
    if (M < 0 || N < 0 || K < 0 || M > 2147483647 || N > 2147483647 || K > 2147483647)
        return fail(GEMM_ERR_INVALID_ARG, "sizes must be in [0, 2^31-1]");
    *bytes = nvfp4_b_offset(M, K) + (uint64_t)N * (uint64_t)K * 2;
    return GEMM_OK;
}

int gemm_nvfp4(const void* A, const void* B, const void* sfA, const void* sfB, void* C, int64_t M,
               int64_t N, int64_t K, const gemm_options* opts, void* workspace,
               uint64_t workspace_bytes, dtc_stream_t stream) {
    g_err[0] = '\0';
    if (K % 16)
        return fail(GEMM_ERR_INVALID_ARG, "K=%lld: NVFP4 needs K %% 16 == 0 (whole scale blocks)",
                    (long long)K);
    if (opts && (opts->lda || opts->ldb))
        return fail(GEMM_ERR_INVALID_ARG, "NVFP4 rows are dense (lda and ldb must be 0)");
    if (opts && (opts->mx_a_format || opts->mx_b_format || opts->mx_scale_block))
        return fail(GEMM_ERR_INVALID_ARG, "NVFP4 fixes the element formats and the scale block "
                    "(mx_a_format, mx_b_format and mx_scale_block must be 0)");
    const bool work = M > 0 && N > 0 && K > 0;
    uint64_t need = 0;
    if (M >= 0 && N >= 0 && K >= 0 && M <= 2147483647 && N <= 2147483647 && K <= 2147483647)
        need = nvfp4_b_offset(M, K) + (uint64_t)N * (uint64_t)K * 2;
    char* ws = static_cast<char*>(workspace);
    if (work) {
        if (!A || !B || !sfA || !sfB) return fail(GEMM_ERR_INVALID_ARG, "A, B, sfA or sfB is NULL");
        if (!aligned16(A) || !aligned16(B))
            return fail(GEMM_ERR_INVALID_ARG, "A and B must be 16-byte aligned");
        if (!workspace || !aligned16(workspace) || workspace_bytes < need)
            return fail(GEMM_ERR_INVALID_ARG, "NVFP4 needs a 16-byte aligned workspace of %llu bytes "
                        "(the operands expanded to bf16)", (unsigned long long)need);
    }
    // the bf16 product of the expanded operands (checks C, the sizes and the other options)
    Prepared r;
    int rc = prepare(0, work ? ws : nullptr, work ? ws + nvfp4_b_offset(M, K) : nullptr, nullptr,
                     nullptr, C, M, N, K, GEMM_LAYOUT_NT, opts, &r);
    if (rc) return rc;
    if (work) {
        if ((rc = check_device_ptr(A, r.dev, "A")) || (rc = check_device_ptr(B, r.dev, "B")) ||
            (rc = check_device_ptr(sfA, r.dev, "sfA")) || (rc = check_device_ptr(sfB, r.dev, "sfB")))
            return rc;
        if ((rc = launch_nvfp4_expand(A, sfA, B, sfB, ws, ws + nvfp4_b_offset(M, K), M, N, K, r.info,
                                      (cudaStream_t)stream)))
            return rc;
    }
    return launch_prepared(r, 0, M, N, K, opts, (cudaStream_t)stream);
}

int gemm_device_model_query(gemm_device_model* out) {
    g_err[0] = '\0';
    if (!out) return fail(GEMM_ERR_INVALID_ARG, "out is NULL");
    int dev;
    DeviceInfo* d;
    int rc = current_device(&dev, &d);
    if (rc) return rc;
    const DevModel& m = device_model(d);
    out->sm_count = m.sms;
    out->pair_clusters = m.pairs;
    out->split2_clusters = m.clusters2;
    out->split4_clusters = m.clusters4;
    return GEMM_OK;
}

int gemm_plan_model(const gemm_device_model* model, int dtype, int64_t M, int64_t N, int64_t K,
                    int layout, const gemm_options* opts, gemm_plan_info* info) {
    g_err[0] = '\0';
    if (!model || !info) return fail(GEMM_ERR_INVALID_ARG, "model or info is NULL");
    if (model->sm_count < 1 || model->pair_clusters < 0 || model->split2_clusters < 0 ||
        model->split4_clusters < 0)
        return fail(GEMM_ERR_INVALID_ARG, "the device model needs sm_count >= 1 and cluster counts >= 0");
    int rc = check_shape(dtype, M, N, K, layout, opts);
    if (rc) return rc;
    Plan p;
    if ((rc = make_plan(dtype, M, N, K, layout, opts, to_model(*model), &p))) return rc;
    fill_info(p, info);
    return GEMM_OK;
}

int gemm_plan(int dtype, int64_t M, int64_t N, int64_t K, int layout, const gemm_options* opts,
              gemm_plan_info* info) {
    g_err[0] = '\0';
    if (!info) return fail(GEMM_ERR_INVALID_ARG, "info is NULL");
    int rc = check_shape(dtype, M, N, K, layout, opts);
    if (rc) return rc;
    int dev;
    DeviceInfo* d;
    if ((rc = current_device(&dev, &d))) return rc;
    Plan p;
    if ((rc = make_plan(dtype, M, N, K, layout, opts, device_model(d), &p))) return rc;
    fill_info(p, info);
    return GEMM_OK;
}

int gemm_workspace_size(int dtype, int64_t M, int64_t N, int64_t K, int layout,
                        const gemm_options* opts, uint64_t* bytes) {
    g_err[0] = '\0';
    if (!bytes) return fail(GEMM_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = 0;
    gemm_options o = {};
    if (opts) o = *opts;
    if (o.stream_k == 2 && dtype != 2) return GEMM_OK;
    o.workspace = reinterpret_cast<void*>(uintptr_t(256));  // stands for "large enough"
    o.workspace_bytes = ~0ull;
    int rc = check_shape(dtype, M, N, K, layout, &o);
    if (rc) return rc;
    int dev;
    DeviceInfo* d;
    if ((rc = current_device(&dev, &d))) return rc;
    const DevModel& m = device_model(d);
    Plan p;
    if ((rc = make_plan(dtype, M, N, K, layout, &o, m, &p))) return rc;
    if (p.sk_tiles) *bytes = sk_workspace_bytes(resident_pairs(m), 256);
    if (p.sf_pack) {
        const int block = o.mx_scale_block ? o.mx_scale_block : 128;
        *bytes = sf_pack_layout(M, N, (K + block - 1) / block, p.tile_n).bytes;
    }
    return GEMM_OK;
}

const char* gemm_last_error(void) { return g_err; }

int gemm_stream_status(dtc_stream_t stream) {
    g_err[0] = '\0';
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int status = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&status, g_dtc_status, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (status == 0) return GEMM_OK;
    e = cudaMemcpyToSymbol(g_dtc_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    return fail(GEMM_ERR_TIMEOUT, "a device-side wait gave up (status 0x%x, site %d)", status,
                status & 0xff);
}

}  // extern "C"
