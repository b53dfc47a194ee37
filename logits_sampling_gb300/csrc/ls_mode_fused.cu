// ls_mode_fused.cu -- instantiates the sampler kernels for MODE_BOTH (ids plus
// log-prob rows and/or the selected token's log-prob from one pass).
#include "ls_kernel.cuh"

namespace lsg {
template ls_status dispatch<MODE_BOTH>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
}  // namespace lsg
