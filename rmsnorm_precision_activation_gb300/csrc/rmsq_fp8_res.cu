// rmsq_fp8_res.cu -- instantiations of the fused row kernel for MODE_FP8 with a residual, and
// their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_fp8_res, MODE_FP8, true)
}  // namespace rmsq
