// rmsq_mxfp4.cu -- instantiations of the fused row kernel for MODE_MXFP4 without a residual, and
// their dispatch (rmsq_mxfp4_res.cu has the ones with a residual).
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_mxfp4_plain, MODE_MXFP4, false)
}  // namespace rmsq
