// launch_mx.cu -- launchers of the block-scaled kernels: the one-CTA kernel (gemm_mxfp8.cuh; 128-
// or 256-deep stages, 128- or 32-element scale blocks, e4m3 / e5m2 / e2m3 / e3m2 / e2m1 elements)
// and the CTA-pair kernel (gemm_mxfp8_2cta.cuh, the same formats and blocks).
#include "gemm_mxfp8.cuh"
#include "gemm_mxfp8_2cta.cuh"
#include "host.h"

namespace dtc_host {
namespace {

template <bool kB32, int kBN>
int launch_pair(const Launch& L) {
    using namespace dtc::gmx2;
    using C_ = Cfg<kBN>;
    const Operands& ops = *L.ops;
    const int a_bits = mx_bits(L.o ? L.o->mx_a_format : 0);
    const int b_bits = mx_bits(L.o ? L.o->mx_b_format : 0);
    CUtensorMap tA, tB, tC, tC32;
    int rc = tmap_block_scaled(&tA, a_bits, ops.A, (uint64_t)L.K, (uint64_t)L.M,
                               (uint64_t)ops.lda * a_bits / 8, kBMc, false, "A");
    if (rc) return rc;
    if ((rc = tmap_block_scaled(&tB, b_bits, ops.B, (uint64_t)L.K, (uint64_t)L.N,
                                (uint64_t)ops.ldb * b_bits / 8, C_::kHalfN, false, "B")))
        return rc;
    if ((rc = tmap_c16(&tC, &tC32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm_mxfp8_2cta_kernel<kB32, kBN>;
    if ((rc = ensure_smem_attr(kern, C_::kSmemBytes, L.dev))) return rc;
    // 256 rows of A and kBN of B per stage: both CTAs' copies, armed on the leader's barrier
    const dtc::GemmMxArgs a = mx_args(L, 256, kBN, kBK);
    return launch_cluster(kern, L.p->ctas, kThreads, C_::kSmemBytes, 2, L.stream, tA, tB, tC, tC32, a);
}

template <bool kDeep, bool kB32>
int launch_one(const Launch& L) {
    using namespace dtc::gmx;
    using C_ = Cfg<kDeep>;
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
    auto kern = dtc::gemm_mxfp8_kernel<kDeep, kB32>;
    if ((rc = ensure_smem_attr(kern, C_::kSmemBytes, L.dev))) return rc;
    dtc::GemmMxArgs a = mx_args(L, kBM, kBN, kBK);
    a.stage_tx *= C_::kBlocks;  // a 256-deep stage holds two K-blocks
    return launch_cluster(kern, L.p->ctas, kThreads, C_::kSmemBytes, 1, L.stream, tA, tB, tC, tC32, a);
}

}  // namespace

int launch_mx(const Launch& L) {
    const bool b32 = L.o && L.o->mx_scale_block == 32;
    if (L.p->variant == GEMM_VARIANT_2CTA) {
        if (L.p->tile_n == 256) return b32 ? launch_pair<true, 256>(L) : launch_pair<false, 256>(L);
        return b32 ? launch_pair<true, 224>(L) : launch_pair<false, 224>(L);
    }
    if (L.p->tile_k == 2 * dtc::gmx::kBK)
        return b32 ? launch_one<true, true>(L) : launch_one<true, false>(L);
    return b32 ? launch_one<false, true>(L) : launch_one<false, false>(L);
}

}  // namespace dtc_host
