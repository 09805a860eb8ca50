// rmsq_amax.cu -- instantiations of the fused row kernel for MODE_AMAX (the NVFP4 global-scale
// pre-pass) without a residual, and their dispatch (rmsq_amax_res.cu has the ones with one).
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH_FOR(dispatch_amax_plain, MODE_AMAX, false)
}  // namespace rmsq
