// rmsq_fp8.cu -- instantiations of the fused row kernel for MODE_FP8 without a residual, and
// their dispatch (rmsq_fp8_res.cu has the ones with a residual).
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_fp8_plain, MODE_FP8, false)
}  // namespace rmsq
