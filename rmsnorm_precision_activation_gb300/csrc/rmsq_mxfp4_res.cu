// rmsq_mxfp4_res.cu -- instantiations of the fused row kernel for MODE_MXFP4 with a residual, and
// their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_mxfp4_res, MODE_MXFP4, true)
}  // namespace rmsq
