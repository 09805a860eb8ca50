// rmsq_nvfp4_res.cu -- instantiations of the fused row kernel for MODE_NVFP4 with a residual, and
// their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_nvfp4_res, MODE_NVFP4, true)
}  // namespace rmsq
