// launch_mx.cu -- launchers of the block-scaled kernels: the one-CTA kernel (gemm_mxfp8.cuh; 128-
// or 256-deep stages, 128- or 32-element scale blocks, e4m3/e5m2 elements) and the CTA-pair option
// (gemm_mxfp8_2cta.cuh).
#include "gemm_mxfp8.cuh"
#include "gemm_mxfp8_2cta.cuh"
#include "host.h"

namespace dtc_host {
namespace {

int launch_pair(const Launch& L) {
    using namespace dtc::gmx2;
    const Operands& ops = *L.ops;
    CUtensorMap tA, tB, tC, tC32;
    int rc = make_tmap_kchunks(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ops.A, (uint64_t)L.K,
                               (uint64_t)L.M, (uint64_t)ops.lda, kBMc, "A");
    if (rc) return rc;
    rc = make_tmap_kchunks(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ops.B, (uint64_t)L.K, (uint64_t)L.N,
                           (uint64_t)ops.ldb, kHalfN, "B");
    if (rc) return rc;
    if ((rc = tmap_c16(&tC, &tC32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm_mxfp8_2cta_kernel<0>;
    if ((rc = ensure_smem_attr(kern, kSmemBytes, L.dev))) return rc;
    const dtc::GemmMxArgs a = mx_args(L, 256, kBN, kBK);
    return launch_cluster(kern, L.p->ctas, kThreads, kSmemBytes, 2, L.stream, tA, tB, tC, tC32, a);
}

template <bool kDeep, bool kB32>
int launch_one(const Launch& L) {
    using namespace dtc::gmx;
    using C_ = Cfg<kDeep>;
    const Operands& ops = *L.ops;
    CUtensorMap tA, tB, tC, tC32;
    int rc;
    if (kDeep) {  // one 3-D box {128, rows, 2} per operand and stage (K % 128 == 0)
        if ((rc = make_tmap_kchunks(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ops.A, (uint64_t)L.K,
                                    (uint64_t)L.M, (uint64_t)ops.lda, kBM, "A")))
            return rc;
        if ((rc = make_tmap_kchunks(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ops.B, (uint64_t)L.K,
                                    (uint64_t)L.N, (uint64_t)ops.ldb, kBN, "B")))
            return rc;
    } else {
        if ((rc = make_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ops.A, (uint64_t)L.K, (uint64_t)L.M,
                            (uint64_t)ops.lda, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B, "A")))
            return rc;
        if ((rc = make_tmap(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ops.B, (uint64_t)L.K, (uint64_t)L.N,
                            (uint64_t)ops.ldb, kBK, kBN, CU_TENSOR_MAP_SWIZZLE_128B, "B")))
            return rc;
    }
    if ((rc = tmap_c16(&tC, &tC32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm_mxfp8_kernel<kDeep, kB32>;
    if ((rc = ensure_smem_attr(kern, C_::kSmemBytes, L.dev))) return rc;
    const dtc::GemmMxArgs a = mx_args(L, kBM, kBN, kBK);
    return launch_cluster(kern, L.p->ctas, kThreads, C_::kSmemBytes, 1, L.stream, tA, tB, tC, tC32, a);
}

}  // namespace

int launch_mx(const Launch& L) {
    if (L.p->variant == GEMM_VARIANT_2CTA) return launch_pair(L);
    const bool b32 = L.o && L.o->mx_scale_block == 32;
    if (L.p->tile_k == 2 * dtc::gmx::kBK)
        return b32 ? launch_one<true, true>(L) : launch_one<true, false>(L);
    return b32 ? launch_one<false, true>(L) : launch_one<false, false>(L);
}

}  // namespace dtc_host
