// ls_split_c2.cu -- instantiates the streaming sampler for rows owned by
// clusters of 2 CTA(s) (one translation unit per cluster size, compiled in
// parallel).
#include "ls_split.cuh"

namespace lsg {
template ls_status dispatch_split<2>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
}  // namespace lsg
