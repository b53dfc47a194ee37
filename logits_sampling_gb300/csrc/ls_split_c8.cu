// ls_split_c8.cu -- instantiates the streaming sampler for rows owned by
// clusters of 8 CTA(s) (one translation unit per cluster size, compiled in
// parallel).
#include "ls_split.cuh"

namespace lsg {
template ls_status dispatch_split<8>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
}  // namespace lsg
