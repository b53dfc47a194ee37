// ls_verify.cu -- speculative chain verification against the target's sampled
// tokens, alone or right after sampling the verify rows.
//
// Follows the TokenSpeed "backends/triton.py" page (TritonSamplingBackend.
// verify: target_sampled from the sampling kernels over the verify rows, then
// verify_chain_target_sampled(predicts, accept_index, accept_token_num,
// candidates, target_sampled)).  The pages print only that call; the rule
// implemented is the plain chain rule documented in include/ls_sampler.h.
#include "ls_kernel.cuh"

namespace lsg {

// the sampling calls' kernel choice (ls_sampler.cu)
ls_status dispatch_sample(const KernelArgs& a, ls_dtype dtype, int route, int32_t n, cudaStream_t stream);

// One thread per request: walk the positions while the drafts match.
__global__ void verify_chain_kernel(const int32_t* candidates, const int32_t* target_sampled, int32_t bs, int32_t n,
                                    int32_t* predicts, int32_t* accept_index, int32_t* accept_token_num) {
  const int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= bs) return;
  const int64_t base = (int64_t)b * n;
  int32_t acc = 0;
  bool on = true;
  for (int32_t j = 0; j < n; ++j) {
    const int64_t r = base + j;
    if (j > 0 && on && candidates[r] != target_sampled[r - 1]) on = false;
    if (on) {
      accept_index[r] = (int32_t)r;
      predicts[r] = target_sampled[r];
      acc += j > 0;
    } else {
      accept_index[r] = -1;
    }
  }
  accept_token_num[b] = acc;
}

static ls_status launch_verify(const int32_t* candidates, const int32_t* target_sampled, int32_t bs, int32_t n,
                               int32_t* predicts, int32_t* accept_index, int32_t* accept_token_num,
                               cudaStream_t stream) {
  verify_chain_kernel<<<dim3((unsigned)((bs + 255) / 256)), dim3(256), 0, stream>>>(
      candidates, target_sampled, bs, n, predicts, accept_index, accept_token_num);
  return cudaPeekAtLastError() == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}

}  // namespace lsg

using namespace lsg;

extern "C" {

ls_status ls_verify_chain(const int32_t* candidates, const int32_t* target_sampled, int32_t bs,
                          int32_t num_tokens, int32_t* predicts, int32_t* accept_index, int32_t* accept_token_num,
                          void* stream) {
  if (bs < 0 || num_tokens < 1) return LS_ERR_INVALID_ARG;
  if (bs == 0) return LS_OK;
  if (!candidates || !target_sampled || !predicts || !accept_index || !accept_token_num) return LS_ERR_INVALID_ARG;
  if ((int64_t)bs * num_tokens > 0x7FFFFFFFll) return LS_ERR_INVALID_ARG;
  return launch_verify(candidates, target_sampled, bs, num_tokens, predicts, accept_index, accept_token_num,
                       static_cast<cudaStream_t>(stream));
}

ls_status ls_sample_verify(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                           int32_t bs, int32_t num_tokens, const int32_t* gather_indices, const ls_params* params,
                           uint64_t step, int no_top_k, int no_top_p, const int32_t* candidates,
                           int32_t* out_target_sampled, int32_t* predicts, int32_t* accept_index,
                           int32_t* accept_token_num, int32_t* error_word, void* stream) {
  if (bs < 0 || num_tokens < 1) return LS_ERR_INVALID_ARG;
  const int64_t n64 = (int64_t)bs * num_tokens;
  if (n64 > 0x7FFFFFFFll) return LS_ERR_INVALID_ARG;
  if (bs == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, true) ||
      !out_target_sampled || !candidates || !predicts || !accept_index || !accept_token_num)
    return LS_ERR_INVALID_ARG;
  if (!gather_indices && n64 > logits_rows) return LS_ERR_INVALID_ARG;
  if (bs > params->num_requests) return LS_ERR_INVALID_ARG;
  KernelArgs a = make_args(logits, logits_rows, vocab, row_stride, gather_indices, params, step, error_word);
  a.map_mode = MAP_SPEC;  // request b owns rows b * num_tokens ... b * num_tokens + num_tokens - 1
  a.spec_decode_rows = (int32_t)n64;
  a.spec_per_req = num_tokens;
  a.spec_num_decode = bs;
  a.out_ids = out_target_sampled;
  const int route = (no_top_k ? 0 : ROUTE_K) | (no_top_p ? 0 : ROUTE_P);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ls_status rc = dispatch_sample(a, dtype, route, (int32_t)n64, st);
  if (rc != LS_OK) return rc;
  return launch_verify(candidates, out_target_sampled, bs, num_tokens, predicts, accept_index, accept_token_num, st);
}

}  // extern "C"
