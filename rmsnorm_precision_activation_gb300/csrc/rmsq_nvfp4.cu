// rmsq_nvfp4.cu -- instantiations of the fused row kernel for MODE_NVFP4 and their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH(dispatch_nvfp4, MODE_NVFP4)
}  // namespace rmsq
