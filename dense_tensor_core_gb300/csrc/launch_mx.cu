// launch_mx.cu -- launchers of the block-scaled kernels: the one-CTA kernel (gemm_mxfp8.cuh; 128-
// or 32-element scale blocks, e4m3 / e5m2 / e2m3 / e3m2 / e2m1 elements; scales through its scale
// warps, or, for 32-element blocks, repacked into the workspace by sf_pack_kernel first) and the
// CTA-pair kernel (gemm_mxfp8_2cta.cuh: the same formats, 128-element blocks, repacked scales).
#include "gemm_mxfp8.cuh"
#include "gemm_mxfp8_2cta.cuh"
#include "host.h"

namespace dtc_host {
namespace {

// The scale arrays of both operands repacked into the workspace (sf_pack.cuh), one launch.
int launch_sf_pack(const Launch& L, const SfPackLayout& l) {
    uint8_t* ws = static_cast<uint8_t*>(L.o->workspace);
    const int cols = ceil_div(L.K, L.o->mx_scale_block ? L.o->mx_scale_block : 128);
    dtc::SfPackOperand a{static_cast<const uint8_t*>(L.ops->sfA), ws, L.M, cols, l.sets, 128, 1,
                         l.groups_a};
    dtc::SfPackOperand b{static_cast<const uint8_t*>(L.ops->sfB), ws + l.b_offset, L.N, cols,
                         l.sets, L.p->tile_n, 2, l.groups_b};
    const int64_t units = std::max((int64_t)l.groups_a * l.sets, (int64_t)l.groups_b * l.sets * 2) * 32;
    const int blocks = (int)std::min<int64_t>((units + dtc::kSfPackThreads - 1) / dtc::kSfPackThreads,
                                              (int64_t)L.dev->model.sms * 8);
    dtc::sf_pack_kernel<><<<dim3(blocks, 2), dtc::kSfPackThreads, 0, L.stream>>>(a, b);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scale repacking launch");
    return GEMM_OK;
}

// The pair kernel: 256 x 224 tiles, 256-deep stages, 128-element scale blocks repacked into the
// workspace (the plan checked the conditions).
int launch_pair(const Launch& L) {
    using namespace dtc::gmx2;
    const Operands& ops = *L.ops;
    const int a_bits = mx_bits(L.o ? L.o->mx_a_format : 0);
    const int b_bits = mx_bits(L.o ? L.o->mx_b_format : 0);
    CUtensorMap tA, tB, tC, tC32, tSA, tSB;
    // 3-D maps over [K/128][rows][128 bytes]: one box {128 bytes, rows, 2} per operand and stage
    int rc = tmap_block_scaled(&tA, a_bits, ops.A, (uint64_t)L.K, (uint64_t)L.M,
                               (uint64_t)ops.lda * a_bits / 8, kBMc, true, "A");
    if (rc) return rc;
    if ((rc = tmap_block_scaled(&tB, b_bits, ops.B, (uint64_t)L.K, (uint64_t)L.N,
                                (uint64_t)ops.ldb * b_bits / 8, kHalfN, true, "B")))
        return rc;
    if ((rc = tmap_c16(&tC, &tC32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm_mxfp8_2cta_kernel<>;
    if ((rc = ensure_smem_attr(kern, kSmemBytes, L.dev))) return rc;
    // 256 rows of A and 224 of B per K-block: both CTAs' copies, armed on the leader's barrier
    dtc::GemmMxArgs a = mx_args(L, 256, kBN, kBK);
    a.stage_tx *= kBlocks;  // a stage holds two K-blocks
    // the repacked arrays as rows of 128 bytes: a chunk is 4 rows (A) or 8 (B's two halves)
    const SfPackLayout l = sf_pack_layout(L.M, L.N, a.sf_cols, kBN);
    uint8_t* ws = static_cast<uint8_t*>(L.o->workspace);
    if ((rc = make_tmap(&tSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ws, 128,
                        (uint64_t)l.groups_a * l.sets * 4, 128, 128, 4, CU_TENSOR_MAP_SWIZZLE_NONE,
                        "repacked sfA")))
        return rc;
    if ((rc = make_tmap(&tSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ws + l.b_offset, 128,
                        (uint64_t)l.groups_b * l.sets * 8, 128, 128, 8, CU_TENSOR_MAP_SWIZZLE_NONE,
                        "repacked sfB")))
        return rc;
    if ((rc = launch_sf_pack(L, l))) return rc;
    a.sf_sets = l.sets;
    // starts while the repacking kernel runs: its producers wait for it before the first chunk
    // copy
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config(L.p->ctas, kThreads, kSmemBytes, 2, L.stream, attr);
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tA, tB, tC, tC32, tSA, tSB, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return GEMM_OK;
}

template <bool kB32, bool kTmaSf>
int launch_one(const Launch& L) {
    using namespace dtc::gmx;
    using C_ = Cfg<kTmaSf>;
    const Operands& ops = *L.ops;
    CUtensorMap tA, tB, tC, tC32;
    // element bits of each operand (fp8: bytes; fp6 / fp4: packed rows the TMA unpacks)
    const int a_bits = mx_bits(L.o ? L.o->mx_a_format : 0);
    const int b_bits = mx_bits(L.o ? L.o->mx_b_format : 0);
    int rc = tmap_block_scaled(&tA, a_bits, ops.A, (uint64_t)L.K, (uint64_t)L.M,
                               (uint64_t)ops.lda * a_bits / 8, kBM, false, "A");
    if (rc) return rc;
    if ((rc = tmap_block_scaled(&tB, b_bits, ops.B, (uint64_t)L.K, (uint64_t)L.N,
                                (uint64_t)ops.ldb * b_bits / 8, kBN, false, "B")))
        return rc;
    if ((rc = tmap_c16(&tC, &tC32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm_mxfp8_kernel<kB32, kTmaSf>;
    if ((rc = ensure_smem_attr(kern, C_::kSmemBytes, L.dev))) return rc;
    dtc::GemmMxArgs a = mx_args(L, kBM, kBN, kBK);
    if constexpr (kTmaSf) {
        const SfPackLayout l = sf_pack_layout(L.M, L.N, a.sf_cols, kBN);
        if ((rc = launch_sf_pack(L, l))) return rc;
        a.sfA_pack = static_cast<const uint8_t*>(L.o->workspace);
        a.sfB_pack = static_cast<const uint8_t*>(L.o->workspace) + l.b_offset;
        a.sf_sets = l.sets;
        // starts while the repacking kernel runs (see the producer)
        return launch_dependent(kern, L.p->ctas, threads_for(kTmaSf), C_::kSmemBytes, L.stream,
                                tA, tB, tC, tC32, a);
    }
    return launch_cluster(kern, L.p->ctas, threads_for(kTmaSf), C_::kSmemBytes, 1, L.stream, tA,
                          tB, tC, tC32, a);
}

}  // namespace

int launch_mx(const Launch& L) {
    if (L.p->variant == GEMM_VARIANT_2CTA) return launch_pair(L);
    if (L.o && L.o->mx_scale_block == 32)  // the planner repacks the scales for 32-element blocks
        return L.p->sf_pack ? launch_one<true, true>(L) : launch_one<true, false>(L);
    return launch_one<false, false>(L);
}

}  // namespace dtc_host
