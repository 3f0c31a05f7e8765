// host.h -- host-side pieces shared by the library's translation units: error reporting, the
// per-device state, operand descriptions, the launch plan, tensor-map encoding and the launchers
// of each kernel family (each family is compiled in its own translation unit).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <unordered_set>

#include "dtc_gemm.h"
#include "gemm_common.cuh"
#include "gemm_mxfp8.cuh"

namespace dtc_host {

// Leaves a message for the calling thread (gemm_last_error) and returns `code`.
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);

constexpr uint64_t kDefaultTimeoutNs = 2ull * 1000 * 1000 * 1000;

// What the planner needs to know about a device: the SM count and how many clusters of each
// kernel can be resident at once (all of the library's kernels take about 200 KB of shared memory,
// so one CTA per SM; clusters may not fill every SM of a GPC).
struct DevModel {
    int sms = 0;
    int pairs = 0;      // clusters of 2 CTAs of the pair kernel
    int clusters2 = 0;  // clusters of 2 split-K CTAs
    int clusters4 = 0;  // clusters of 4 split-K CTAs
};

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int major = 0, minor = 0;
    DevModel model;                                 // sms set at probe, clusters on first plan
    bool clusters_probed = false;
    std::unordered_set<const void*> smem_attr_set;  // kernels whose smem limit was raised
    int* status = nullptr;                          // device address of the status word
    void* static_ws = nullptr;                      // address of the static workspace
};
extern std::mutex g_dev_mu;

// Where the operands live, after the defaults are applied: storage order and row pitch.
struct Operands {
    const void* A;
    const void* B;
    const void* sfA;
    const void* sfB;
    void* C;
    int64_t lda, ldb, ldc;  // elements between consecutive stored rows
    bool a_mn;              // A stored [K,M] (layouts TN, TT); else [M,K]
    bool b_mn;              // B stored [K,N] (layouts NN, TN); else [N,K]
};

struct Plan {
    int variant = 0, tile_m = 0, tile_n = 0, tile_k = 64, stages = 0, split_k = 1, ctas = 0,
        tiles = 0, cluster = 1, sk_tiles = 0;
    bool sf_pack = false;  // block-scaled one-CTA kernel: scales repacked into the workspace
};

// Repacked scale arrays of the block-scaled product in a workspace (sf_pack.cuh): the chunks of A
// (128-row groups, one 128-row half) from byte 0, those of B (tile_n-row groups, two halves) from
// the next 1 KB boundary.
struct SfPackLayout {
    int sets = 0, groups_a = 0, groups_b = 0;
    uint64_t b_offset = 0, bytes = 0;
};
inline SfPackLayout sf_pack_layout(int64_t M, int64_t N, int64_t sf_cols, int tile_n) {
    SfPackLayout l;
    l.sets = (int)((sf_cols + 3) / 4);
    l.groups_a = (int)((M + 127) / 128);
    l.groups_b = (int)((N + tile_n - 1) / tile_n);
    const uint64_t a = (uint64_t)l.groups_a * l.sets * 512;
    l.b_offset = (a + 1023) / 1024 * 1024;
    l.bytes = l.b_offset + (uint64_t)l.groups_b * l.sets * 2 * 512;
    return l;
}

// Stream-K workspace of the pair kernel for `units` pairs and tile width bn: the flags (one
// 32-bit word per CTA, padded to 1 KB, so at most 128 pairs), then one 128 x bn fp32 slot per CTA.
constexpr uint64_t kSkFlagBytes = 1024;
constexpr int kSkMaxUnits = (int)(kSkFlagBytes / 4 / 2);
inline uint64_t sk_workspace_bytes(int units, int bn) {
    return kSkFlagBytes + (uint64_t)units * 2 * 128 * (uint64_t)bn * 4;
}

inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Everything a launcher needs.
struct Launch {
    const Operands* ops;
    int M, N, K;
    const gemm_options* o;
    DeviceInfo* dev;
    const Plan* p;
    cudaStream_t stream;
};

// Tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry point).
int make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
              uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz, const char* name);
int make_tmap_kchunks(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
                      uint64_t K, uint64_t rows, uint64_t ld, uint32_t box_rows, const char* name);
int tmap_block_scaled(CUtensorMap* m, int bits, const void* ptr, uint64_t K, uint64_t rows,
                      uint64_t row_bytes, uint32_t box_rows, bool deep, const char* name);
int mx_bits(int fmt);
int tmap_operand16(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, int64_t ld,
                   bool mn_major, int64_t mn, int64_t K, int kBK, uint32_t box_rows,
                   const char* name);
int tmap_c16(CUtensorMap* c64, CUtensorMap* c32, CUtensorMapDataType dt, const Operands& ops,
             int64_t M, int64_t N);

dtc::Gemm16Args make_args(const Launch& L, int tile_m, int tile_n, int tile_k);
dtc::GemmMxArgs mx_args(const Launch& L, int tile_m, int tile_n, int tile_k);

// Raises a kernel's dynamic shared-memory limit once per device.
template <typename Kern>
int ensure_smem_attr(Kern kern, int bytes, DeviceInfo* dev) {
    const void* key = reinterpret_cast<const void*>(kern);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!dev->smem_attr_set.count(key)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        dev->smem_attr_set.insert(key);
    }
    return GEMM_OK;
}

inline cudaLaunchConfig_t cluster_config(int grid, int threads, int smem, int cluster,
                                         cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 1 : 0;
    return cfg;
}

template <typename Kern, typename... Params>
int launch_cluster(Kern kern, int grid, int threads, int smem, int cluster, cudaStream_t stream,
                   const Params&... params) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(grid, threads, smem, cluster, stream, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, params...);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return GEMM_OK;
}

// As launch_cluster (one CTA per cluster), for a kernel that depends on the stream's previous
// kernel only through data it reads after griddepcontrol.wait: the launch may begin while that
// kernel still runs (programmatic stream serialisation), so its set-up overlaps the other's tail.
template <typename Kern, typename... Params>
int launch_dependent(Kern kern, int grid, int threads, int smem, cudaStream_t stream,
                     const Params&... params) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(grid, threads, smem, 1, stream, attr);
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, params...);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return GEMM_OK;
}

// How many clusters of `cluster` CTAs of `kern` (with `smem` bytes of dynamic shared memory) the
// device keeps resident at once; `fallback` if the query fails.
template <typename Kern>
int max_active_clusters(Kern kern, int threads, int smem, int cluster, int fallback,
                        DeviceInfo* dev) {
    if (ensure_smem_attr(kern, smem, dev) != GEMM_OK) return fallback;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(cluster * fallback, threads, smem, cluster, nullptr, attr);
    cfg.numAttrs = 1;
    int q = 0;
    if (cudaOccupancyMaxActiveClusters(&q, kern, &cfg) == cudaSuccess && q > 0) return q;
    cudaGetLastError();
    return fallback;
}

// Kernel families, one translation unit each. Each returns GEMM_OK or an error (message set).
int launch16_1cta(bool bf16, const Launch& L);
int launch16_2cta_bf16(const Launch& L);
int launch16_2cta_f16(const Launch& L);
int launch16_splitk(bool bf16, const Launch& L);
int launch_mx(const Launch& L);
// 2:4 sparse A: writes the dense [M, K] 16-bit A into `dense` (stream-ordered).
int launch_sp24_expand(bool bf16, const void* vals, const void* meta, void* dense, int64_t M,
                       int64_t K, DeviceInfo* dev, cudaStream_t stream);
// NVFP4 operands (packed e2m1 rows, UE4M3 scales per 16) to bf16 [M,K] / [N,K] (nvfp4_expand.cuh).
int launch_nvfp4_expand(const void* A, const void* sfA, const void* B, const void* sfB,
                        void* a_out, void* b_out, int64_t M, int64_t N, int64_t K,
                        DeviceInfo* dev, cudaStream_t stream);

// Resident clusters of the pair kernel and of the split-K kernels (clusters of 2 and 4).
int query_pair_clusters(DeviceInfo* dev);
int query_splitk_clusters(int split, DeviceInfo* dev);

}  // namespace dtc_host
