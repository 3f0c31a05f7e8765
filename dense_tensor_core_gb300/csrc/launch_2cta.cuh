// launch_2cta.cuh -- launcher of the CTA-pair 16-bit kernel (gemm16_2cta.cuh), instantiated once
// per operand type in launch_2cta_bf16.cu and launch_2cta_f16.cu (two translation units compile in
// parallel).
#pragma once

#include "gemm16_2cta.cuh"
#include "host.h"

namespace dtc_host {
namespace pair16 {

template <bool kBF16, bool kAMN, bool kNN, int kBN, int kBK, bool kSK = false>
int launch(const Launch& L) {
    constexpr int kStages = dtc::g2::stages_for(kBN, kBK);
    using Cfg = dtc::g2::Cfg<kBN, kBK, kStages, kNN>;
    const Operands& ops = *L.ops;
    const CUtensorMapDataType dt = kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tA, tB, tC, tC32;
    int rc = tmap_operand16(&tA, dt, ops.A, ops.lda, kAMN, L.M, L.K, kBK, 128, "A");
    if (rc) return rc;
    if ((rc = tmap_operand16(&tB, dt, ops.B, ops.ldb, kNN, L.N, L.K, kBK, Cfg::kHalfN, "B"))) return rc;
    if ((rc = tmap_c16(&tC, &tC32, dt, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm16_2cta_kernel<kBF16, kAMN, kNN, kBN, kBK, kStages, kSK>;
    if ((rc = ensure_smem_attr(kern, Cfg::kSmemBytes, L.dev))) return rc;
    const dtc::Gemm16Args args = make_args(L, 256, kBN, kBK);
    return launch_cluster(kern, L.p->ctas, dtc::g2::kThreads, Cfg::kSmemBytes, 2, L.stream, tA, tB,
                          tC, tC32, args);
}

template <bool kBF16, bool kAMN, bool kNN>
int by_shape(const Launch& L) {
    const Plan& p = *L.p;
    if (p.sk_tiles) {  // stream-K plans are 256 wide, 128- or 64-deep
        if (p.tile_k == 64) return launch<kBF16, kAMN, kNN, 256, 64, true>(L);
        return launch<kBF16, kAMN, kNN, 256, 128, true>(L);
    }
    if (p.tile_k == 128) {
        if (p.tile_n == 224) return launch<kBF16, kAMN, kNN, 224, 128>(L);
        if (p.tile_n == 128) return launch<kBF16, kAMN, kNN, 128, 128>(L);
        if (p.tile_n == 64) return launch<kBF16, kAMN, kNN, 64, 128>(L);
        return launch<kBF16, kAMN, kNN, 256, 128>(L);
    }
    if (p.tile_n == 224) return launch<kBF16, kAMN, kNN, 224, 64>(L);
    return launch<kBF16, kAMN, kNN, 256, 64>(L);
}

template <bool kBF16>
int launch_any(const Launch& L) {
    const bool amn = L.ops->a_mn, bmn = L.ops->b_mn;
    if (amn) return bmn ? by_shape<kBF16, true, true>(L) : by_shape<kBF16, true, false>(L);
    return bmn ? by_shape<kBF16, false, true>(L) : by_shape<kBF16, false, false>(L);
}

}  // namespace pair16
}  // namespace dtc_host
