// ls_mode_sample.cu -- instantiates the sampler kernels for MODE_SAMPLE.
#include "ls_kernel.cuh"

namespace lsg {
template ls_status dispatch<MODE_SAMPLE>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
}  // namespace lsg
