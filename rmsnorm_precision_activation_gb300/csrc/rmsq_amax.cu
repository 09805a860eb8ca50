// rmsq_amax.cu -- instantiations of the fused row kernel for MODE_AMAX and their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH(dispatch_amax, MODE_AMAX)
}  // namespace rmsq
