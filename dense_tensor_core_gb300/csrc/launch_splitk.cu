// launch_splitk.cu -- launcher of the split-K 16-bit kernel (gemm16_splitk.cuh): one cluster of 2
// or 4 CTAs per output tile, K split over the cluster, the partial sums reduced on chip.
#include "gemm16_splitk.cuh"
#include "host.h"

namespace dtc_host {
namespace {

template <bool kBF16, bool kAMN, bool kNN, int kBN, int kBK, int kS>
int launch(const Launch& L) {
    constexpr int kStages = dtc::gsk::stages_for(kBN, kBK, kS);
    using Cfg = dtc::gsk::Cfg<kBN, kBK, kStages, kS>;
    const Operands& ops = *L.ops;
    const CUtensorMapDataType dt = kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tA, tB, tC, tC32;
    int rc = tmap_operand16(&tA, dt, ops.A, ops.lda, kAMN, L.M, L.K, kBK, 128, "A");
    if (rc) return rc;
    if ((rc = tmap_operand16(&tB, dt, ops.B, ops.ldb, kNN, L.N, L.K, kBK, kBN, "B"))) return rc;
    if ((rc = tmap_c16(&tC, &tC32, dt, ops, L.M, L.N))) return rc;
    auto kern = dtc::gemm16_splitk_kernel<kBF16, kAMN, kNN, kBN, kBK, kStages, kS>;
    if ((rc = ensure_smem_attr(kern, Cfg::kSmemBytes, L.dev))) return rc;
    const dtc::Gemm16Args args = make_args(L, 128, kBN, kBK);
    return launch_cluster(kern, L.p->ctas, dtc::gsk::kThreads, Cfg::kSmemBytes, kS, L.stream, tA,
                          tB, tC, args);
}

template <bool kBF16, bool kAMN, bool kNN>
int by_shape(const Launch& L) {
    const Plan& p = *L.p;
    if (p.split_k == 1) return launch<kBF16, kAMN, kNN, 64, 128, 1>(L);  // whole K, 64-wide tiles
    if (p.tile_n == 128) {
        if (p.tile_k == 128)
            return p.split_k == 2 ? launch<kBF16, kAMN, kNN, 128, 128, 2>(L)
                                  : launch<kBF16, kAMN, kNN, 128, 128, 4>(L);
        return p.split_k == 2 ? launch<kBF16, kAMN, kNN, 128, 64, 2>(L)
                              : launch<kBF16, kAMN, kNN, 128, 64, 4>(L);
    }
    return launch<kBF16, kAMN, kNN, 256, 64, 2>(L);
}

template <bool kBF16>
int by_layout(const Launch& L) {
    const bool amn = L.ops->a_mn, bmn = L.ops->b_mn;
    if (amn) return bmn ? by_shape<kBF16, true, true>(L) : by_shape<kBF16, true, false>(L);
    return bmn ? by_shape<kBF16, false, true>(L) : by_shape<kBF16, false, false>(L);
}

}  // namespace

int launch16_splitk(bool bf16, const Launch& L) {
    return bf16 ? by_layout<true>(L) : by_layout<false>(L);
}

int query_splitk_clusters(int split, DeviceInfo* dev) {
    // the largest shared memory of each split: 128-wide tiles, 128-deep stages
    if (split == 4) {
        constexpr int kStages = dtc::gsk::stages_for(128, 128, 4);
        using Cfg = dtc::gsk::Cfg<128, 128, kStages, 4>;
        auto kern = dtc::gemm16_splitk_kernel<true, false, false, 128, 128, kStages, 4>;
        return max_active_clusters(kern, dtc::gsk::kThreads, Cfg::kSmemBytes, 4,
                                   dev->model.sms / 4, dev);
    }
    constexpr int kStages = dtc::gsk::stages_for(128, 128, 2);
    using Cfg = dtc::gsk::Cfg<128, 128, kStages, 2>;
    auto kern = dtc::gemm16_splitk_kernel<true, false, false, 128, 128, kStages, 2>;
    return max_active_clusters(kern, dtc::gsk::kThreads, Cfg::kSmemBytes, 2, dev->model.sms / 2,
                               dev);
}

}  // namespace dtc_host
