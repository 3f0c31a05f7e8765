// launch_2cta_f16.cu -- the CTA-pair kernel with fp16 operands.
#include "launch_2cta.cuh"

namespace dtc_host {

int launch16_2cta_f16(const Launch& L) { return pair16::launch_any<false>(L); }

}  // namespace dtc_host
