// rmsq_fp8.cu -- instantiations of the fused row kernel for MODE_FP8 and their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH(dispatch_fp8, MODE_FP8)
}  // namespace rmsq
