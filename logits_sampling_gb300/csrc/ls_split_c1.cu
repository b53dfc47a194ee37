// ls_split_c1.cu -- instantiates the streaming sampler for rows owned by one
// CTA each (one translation unit per cluster size, compiled in parallel).
#include "ls_split.cuh"

namespace lsg {
template ls_status dispatch_split<1>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
}  // namespace lsg
