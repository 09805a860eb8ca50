// rmsq_nvfp4.cu -- instantiations of the fused row kernel for MODE_NVFP4 without a residual, and
// their dispatch (rmsq_nvfp4_res.cu has the ones with a residual).
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_nvfp4_plain, MODE_NVFP4, false)
}  // namespace rmsq
