// launch_2cta_bf16.cu -- the CTA-pair kernel with bf16 operands, and the residency query that
// bounds the number of pairs a persistent launch (and stream-K) may count on.
#include "launch_2cta.cuh"

namespace dtc_host {

int launch16_2cta_bf16(const Launch& L) { return pair16::launch_any<true>(L); }

int query_pair_clusters(DeviceInfo* dev) {
    // the stream-K instantiation: the largest shared memory of the pair kernels
    constexpr int kStages = dtc::g2::stages_for(256, 128);
    using Cfg = dtc::g2::Cfg<256, 128, kStages, false>;
    auto kern = dtc::gemm16_2cta_kernel<true, false, false, 256, 128, kStages, true>;
    return max_active_clusters(kern, dtc::g2::kThreads, Cfg::kSmemBytes, 2,
                               dev->model.sms / 2, dev);
}

}  // namespace dtc_host
