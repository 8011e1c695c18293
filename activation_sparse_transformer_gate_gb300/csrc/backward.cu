// backward.cu -- sparse backward of the TwELL FFN (not built yet).
#include "common.cuh"
#include "kernels.h"

namespace twell {

cudaError_t launch_backward(const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace twell
