// rmsq_amax_res.cu -- instantiations of the fused row kernel for MODE_AMAX with a residual, and
// their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_amax_res, MODE_AMAX, true)
}  // namespace rmsq
