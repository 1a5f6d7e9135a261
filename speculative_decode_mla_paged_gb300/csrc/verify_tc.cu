// Tensor-core (tcgen05 / TMEM) split kernel for sm_103a -- placeholder until
// the kernel lands; tc_supported() is false so verify_attn_run uses the
// CUDA-core kernel.
#include "va_internal.cuh"

namespace va {

cudaError_t tc_init() { return cudaSuccess; }

bool tc_supported(const Params &) { return false; }

cudaError_t launch_tc_split(const Params &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace va
