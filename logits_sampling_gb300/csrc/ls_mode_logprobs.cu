// ls_mode_logprobs.cu -- instantiates the sampler kernels for MODE_LOGPROBS.
#include "ls_kernel.cuh"

namespace lsg {
template ls_status dispatch<MODE_LOGPROBS>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
}  // namespace lsg
