// ls_argmax.cu -- the all-greedy fast path: the lowest index of each row's
// maximum from one streaming read of the row, with no candidate phases.
//
// Follows the TokenSpeed "backends/triton.py" page (TritonSamplingBackend.
// sample: when every request of the batch is greedy the backend takes the
// argmax of the logits instead of a sampling kernel) with the sampler's rules
// for special values: NaN is read as -inf, ties go to the lowest index, a row
// with no entry above -inf is an error row.
#include "ls_kernel.cuh"

namespace lsg {

struct ArgmaxArgs {
  const void* logits;
  int64_t logits_rows, vocab, stride;
  const int32_t* gather;
  int32_t* out_ids;
  int32_t* error_word;
};

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 2) argmax_row_kernel(const ArgmaxArgs a) {
  using RV = RowView<TIn>;
  __shared__ float red_v[kWarps];
  __shared__ unsigned int red_j[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t i = blockIdx.x;
  int64_t src = i;
  if (a.gather) {
    src = a.gather[i];
    if (src < 0 || src >= a.logits_rows) {
      if (tid == 0) {
        a.out_ids[i] = -1;
        if (a.error_word) atomicOr(a.error_word, LS_ROW_ERR_BAD_GATHER);
      }
      return;
    }
  }
  RV rv;
  rv.init(a.logits, src, a.stride, a.vocab);
  // Each thread walks its groups in increasing order and keeps the first
  // group holding its running maximum (strict >: the lowest group): its words
  // for bf16, only its index for fp32 (re-read from L2 at the end, which keeps
  // two fp32 groups in flight within the register budget).
  constexpr bool kKeep = RV::kWords <= 8;
  constexpr int U = kKeep ? 4 : 2;  // groups in flight per thread
  float m = kNegInf;
  int gbest = -1;
  uint32_t wb[RV::kWords];
  for (int g0 = tid; g0 < rv.NG; g0 += U * kThreads) {
    uint32_t w[U][RV::kWords];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (rv.full(g0 + u * kThreads)) rv.load_words(g0 + u * kThreads, w[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = g0 + u * kThreads;
      if (g < rv.NG) {
        if (!rv.full(g)) rv.load_words_partial(g, w[u]);
        const float gm = RV::group_max(w[u]);
        if (gm > m) {
          m = gm;
          gbest = g;
          if (kKeep) {
#pragma unroll
            for (int q = 0; q < RV::kWords; ++q) wb[q] = w[u][q];
          }
        }
      }
    }
  }
  // lowest entry of the best group equal to the maximum (NaN never equal)
  unsigned int j = 0xFFFFFFFFu;
  if (!kKeep && gbest >= 0) {
    if (rv.full(gbest))
      rv.load_words(gbest, wb);
    else
      rv.load_words_partial(gbest, wb);
  }
  if (gbest >= 0) {
#pragma unroll
    for (int e = kGroup - 1; e >= 0; --e)
      if (RV::element_at(wb, e) == m) j = (unsigned int)rv.index(gbest, e);
  }
  const float mw = warp_max(m);
  const unsigned int jw = __reduce_min_sync(0xFFFFFFFFu, m == mw ? j : 0xFFFFFFFFu);
  if (lane == 0) {
    red_v[warp] = mw;
    red_j[warp] = jw;
  }
  __syncthreads();
  if (warp == 0) {
    const float mq = lane < kWarps ? red_v[lane] : kNegInf;
    const float M = warp_max(mq);
    const unsigned int J = __reduce_min_sync(0xFFFFFFFFu, lane < kWarps && mq == M ? red_j[lane] : 0xFFFFFFFFu);
    if (lane == 0) {
      if (M == kNegInf) {
        a.out_ids[i] = -1;
        if (a.error_word) atomicOr(a.error_word, LS_ROW_ERR_NO_FINITE);
      } else {
        a.out_ids[i] = (int32_t)J;
      }
    }
  }
}

ls_status launch_argmax(const ArgmaxArgs& a, ls_dtype dtype, int32_t n, cudaStream_t stream) {
  if (dtype == LS_DTYPE_BF16)
    argmax_row_kernel<bf16_tag><<<dim3((unsigned)n), dim3(kThreads), 0, stream>>>(a);
  else
    argmax_row_kernel<float><<<dim3((unsigned)n), dim3(kThreads), 0, stream>>>(a);
  return cudaPeekAtLastError() == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}

}  // namespace lsg

extern "C" ls_status ls_argmax(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                               int64_t row_stride, int32_t n, const int32_t* gather_indices, int32_t* out_ids,
                               int32_t* error_word, void* stream) {
  using namespace lsg;
  if (n < 0) return LS_ERR_INVALID_ARG;
  if (n == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !out_ids) return LS_ERR_INVALID_ARG;
  if (!gather_indices && (int64_t)n > logits_rows) return LS_ERR_INVALID_ARG;
  ArgmaxArgs a{logits, logits_rows, vocab, row_stride, gather_indices, out_ids, error_word};
  return launch_argmax(a, dtype, n, static_cast<cudaStream_t>(stream));
}
