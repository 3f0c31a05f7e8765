// launch_1cta.cu -- launcher of the one-CTA 16-bit kernel (gemm16_1cta.cuh): tensor maps, shared
// memory limit and the persistent launch, for every (dtype, A storage, B storage, tile width).
#include "gemm16_1cta.cuh"
#include "host.h"

namespace dtc_host {
namespace {

// Ring depth: as many 64-deep stages as fit beside the 32 KB of output staging.
constexpr int kStages1 = 4;

template <bool kBF16, bool kAMN, bool kNN, int kBN>
int launch(const Launch& L) {
    using namespace dtc::g16;
    using Cfg = Cfg<kBN, kStages1>;
    const Operands& ops = *L.ops;
    const CUtensorMapDataType dt = kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tA, tB, tC, tC32;
    int rc = tmap_operand16(&tA, dt, ops.A, ops.lda, kAMN, L.M, L.K, kBK, kBM, "A");
    if (rc) return rc;
    if ((rc = tmap_operand16(&tB, dt, ops.B, ops.ldb, kNN, L.N, L.K, kBK, kBN, "B"))) return rc;
    if ((rc = tmap_c16(&tC, &tC32, dt, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm16_1cta_kernel<kBF16, kAMN, kNN, kBN, kStages1>;
    if ((rc = ensure_smem_attr(kern, Cfg::kSmemBytes, L.dev))) return rc;
    const dtc::Gemm16Args args = make_args(L, kBM, kBN, kBK);
    return launch_cluster(kern, L.p->ctas, kThreads, Cfg::kSmemBytes, 1, L.stream, tA, tB, tC,
                          tC32, args);
}

template <bool kBF16, bool kAMN>
int by_width(const Launch& L) {
    if (L.ops->b_mn) return launch<kBF16, kAMN, true, 256>(L);  // B [K,N]: 256-wide tiles only
    if (L.p->tile_n == 224) return launch<kBF16, kAMN, false, 224>(L);
    return launch<kBF16, kAMN, false, 256>(L);
}

}  // namespace

int launch16_1cta(bool bf16, const Launch& L) {
    if (bf16) return L.ops->a_mn ? by_width<true, true>(L) : by_width<true, false>(L);
    return L.ops->a_mn ? by_width<false, true>(L) : by_width<false, false>(L);
}

}  // namespace dtc_host
