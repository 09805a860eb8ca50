// rmsq_mxfp4.cu -- instantiations of the fused row kernel for MODE_MXFP4 and their dispatch.
#include "rmsq_host.h"

namespace rmsq {
RMSQ_DEFINE_DISPATCH(dispatch_mxfp4, MODE_MXFP4)
}  // namespace rmsq
