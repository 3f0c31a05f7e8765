// launch_mx.cu -- launchers of the block-scaled kernels: the one-CTA kernel (gemm_mxfp8.cuh; 128-
// or 256-deep stages, 128- or 32-element scale blocks, e4m3 / e5m2 / e2m3 / e3m2 / e2m1 elements;
// scales through its scale warps, or repacked into the workspace by sf_pack_kernel first) and the
// CTA-pair kernel (gemm_mxfp8_2cta.cuh, the same formats and blocks).
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

template <bool kB32, int kBN, bool kTmaSf, bool kDeep = false>
int launch_pair(const Launch& L) {
    using namespace dtc::gmx2;
    using C_ = Cfg<kBN, kTmaSf, kDeep>;
    const Operands& ops = *L.ops;
    const int a_bits = mx_bits(L.o ? L.o->mx_a_format : 0);
    const int b_bits = mx_bits(L.o ? L.o->mx_b_format : 0);
    CUtensorMap tA, tB, tC, tC32;
    int rc = tmap_block_scaled(&tA, a_bits, ops.A, (uint64_t)L.K, (uint64_t)L.M,
                               (uint64_t)ops.lda * a_bits / 8, kBMc, kDeep, "A");
    if (rc) return rc;
    if ((rc = tmap_block_scaled(&tB, b_bits, ops.B, (uint64_t)L.K, (uint64_t)L.N,
                                (uint64_t)ops.ldb * b_bits / 8, C_::kHalfN, kDeep, "B")))
        return rc;
    if ((rc = tmap_c16(&tC, &tC32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm_mxfp8_2cta_kernel<kB32, kBN, kTmaSf, kDeep>;
    if ((rc = ensure_smem_attr(kern, C_::kSmemBytes, L.dev))) return rc;
    // 256 rows of A and kBN of B per K-block: both CTAs' copies, armed on the leader's barrier
    dtc::GemmMxArgs a = mx_args(L, 256, kBN, kBK);
    a.stage_tx *= C_::kBlocks;  // a 256-deep stage holds two K-blocks
    CUtensorMap tSA = tA, tSB = tA;  // (unused without repacked scales)
    if constexpr (kTmaSf) {
        // the repacked arrays as rows of 128 bytes: a chunk is 4 rows (A) or 8 (B's two halves)
        const SfPackLayout l = sf_pack_layout(L.M, L.N, a.sf_cols, kBN);
        uint8_t* ws = static_cast<uint8_t*>(L.o->workspace);
        if ((rc = make_tmap(&tSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ws, 128,
                            (uint64_t)l.groups_a * l.sets * 4, 128, 128, 4,
                            CU_TENSOR_MAP_SWIZZLE_NONE, "repacked sfA")))
            return rc;
        if ((rc = make_tmap(&tSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ws + l.b_offset, 128,
                            (uint64_t)l.groups_b * l.sets * 8, 128, 128, 8,
                            CU_TENSOR_MAP_SWIZZLE_NONE, "repacked sfB")))
            return rc;
        if ((rc = launch_sf_pack(L, l))) return rc;
        a.sf_sets = l.sets;
        // starts while the repacking kernel runs: its producers wait for it before the first
        // chunk copy
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = cluster_config(L.p->ctas, threads_for(true), C_::kSmemBytes, 2,
                                                L.stream, attr);
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tA, tB, tC, tC32, tSA, tSB, a);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        return GEMM_OK;
    }
    return launch_cluster(kern, L.p->ctas, kThreads, C_::kSmemBytes, 2, L.stream, tA, tB, tC, tC32,
                          tSA, tSB, a);
}

template <bool kDeep, bool kB32, bool kTmaSf>
int launch_one(const Launch& L) {
    using namespace dtc::gmx;
    using C_ = Cfg<kDeep, kTmaSf>;
    const Operands& ops = *L.ops;
    CUtensorMap tA, tB, tC, tC32;
    // element bits of each operand (fp8: bytes; fp6 / fp4: packed rows the TMA unpacks)
    const int a_bits = mx_bits(L.o ? L.o->mx_a_format : 0);
    const int b_bits = mx_bits(L.o ? L.o->mx_b_format : 0);
    int rc = tmap_block_scaled(&tA, a_bits, ops.A, (uint64_t)L.K, (uint64_t)L.M,
                               (uint64_t)ops.lda * a_bits / 8, kBM, kDeep, "A");
    if (rc) return rc;
    if ((rc = tmap_block_scaled(&tB, b_bits, ops.B, (uint64_t)L.K, (uint64_t)L.N,
                                (uint64_t)ops.ldb * b_bits / 8, kBN, kDeep, "B")))
        return rc;
    if ((rc = tmap_c16(&tC, &tC32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm_mxfp8_kernel<kDeep, kB32, kTmaSf>;
    if ((rc = ensure_smem_attr(kern, C_::kSmemBytes, L.dev))) return rc;
    dtc::GemmMxArgs a = mx_args(L, kBM, kBN, kBK);
    a.stage_tx *= C_::kBlocks;  // a 256-deep stage holds two K-blocks
    if constexpr (kTmaSf) {
        const SfPackLayout l = sf_pack_layout(L.M, L.N, a.sf_cols, kBN);
        if ((rc = launch_sf_pack(L, l))) return rc;
        a.sfA_pack = static_cast<const uint8_t*>(L.o->workspace);
        a.sfB_pack = static_cast<const uint8_t*>(L.o->workspace) + l.b_offset;
        a.sf_sets = l.sets;
    }
    if constexpr (kTmaSf)  // starts while the repacking kernel runs (see the producer)
        return launch_dependent(kern, L.p->ctas, threads_for(kTmaSf), C_::kSmemBytes, L.stream,
                                tA, tB, tC, tC32, a);
    return launch_cluster(kern, L.p->ctas, threads_for(kTmaSf), C_::kSmemBytes, 1, L.stream, tA,
                          tB, tC, tC32, a);
}

template <bool kDeep, bool kB32>
int launch_one_any(const Launch& L) {
    if constexpr (kB32)  // the planner repacks the scales for 32-element blocks only
        if (L.p->sf_pack) return launch_one<kDeep, true, true>(L);
    return launch_one<kDeep, kB32, false>(L);
}

}  // namespace

int launch_mx(const Launch& L) {
    const bool b32 = L.o && L.o->mx_scale_block == 32;
    if (L.p->variant == GEMM_VARIANT_2CTA) {
        if (L.p->tile_n == 256)
            return b32 ? launch_pair<true, 256, false>(L) : launch_pair<false, 256, false>(L);
        if (L.p->sf_pack && L.p->tile_k == 2 * dtc::gmx2::kBK)
            return b32 ? launch_pair<true, 224, true, true>(L) : launch_pair<false, 224, true, true>(L);
        if (L.p->sf_pack)
            return b32 ? launch_pair<true, 224, true>(L) : launch_pair<false, 224, true>(L);
        return b32 ? launch_pair<true, 224, false>(L) : launch_pair<false, 224, false>(L);
    }
    if (L.p->tile_k == 2 * dtc::gmx::kBK)
        return b32 ? launch_one_any<true, true>(L) : launch_one_any<true, false>(L);
    return b32 ? launch_one_any<false, true>(L) : launch_one_any<false, false>(L);
}

}  // namespace dtc_host
