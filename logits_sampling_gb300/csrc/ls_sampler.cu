// ls_sampler.cu -- C ABI of the token sampler (include/ls_sampler.h).
//
// Host-side argument checks and the route/mode dispatch; the kernels are in
// ls_kernel.cuh and are instantiated per mode in ls_mode_*.cu.
#include "ls_kernel.cuh"

namespace lsg {
extern template ls_status dispatch<MODE_SAMPLE>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
extern template ls_status dispatch<MODE_LOGPROBS>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
extern template ls_status dispatch<MODE_BOTH>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);

// Advances a device-resident Philox step word after the sampler that read it
// (stream order: every CTA of the sampler has read the word before this runs).
__global__ void advance_step_kernel(uint64_t* step) { *step += 1ull; }
}  // namespace lsg

using namespace lsg;

extern "C" {

ls_status ls_sample(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                    int32_t n, const int32_t* gather_indices, const int32_t* token_to_request_index,
                    const ls_params* params, uint64_t step, int no_top_k, int no_top_p, int32_t* out_ids,
                    int32_t* error_word, void* stream) {
  if (n < 0) return LS_ERR_INVALID_ARG;
  if (n == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, true) || !out_ids)
    return LS_ERR_INVALID_ARG;
  if (!gather_indices && (int64_t)n > logits_rows) return LS_ERR_INVALID_ARG;
  if (!token_to_request_index && n > params->num_requests) return LS_ERR_INVALID_ARG;
  KernelArgs a = make_args(logits, logits_rows, vocab, row_stride, gather_indices, params, step, error_word);
  a.t2r = token_to_request_index;
  a.map_mode = token_to_request_index ? MAP_T2R : MAP_IDENTITY;
  a.out_ids = out_ids;
  const int route = (no_top_k ? 0 : ROUTE_K) | (no_top_p ? 0 : ROUTE_P);
  return dispatch<MODE_SAMPLE>(a, dtype, route, n, static_cast<cudaStream_t>(stream));
}

ls_status ls_sample_speculative(const void* required_logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                                int64_t row_stride, int32_t num_decode, int32_t num_prefill,
                                int32_t num_speculative_tokens, const int32_t* gather_indices,
                                const ls_params* params, uint64_t step, int no_top_k, int no_top_p,
                                int32_t* out_ids, int32_t* out_token_to_request_index, int32_t* error_word,
                                void* stream) {
  if (num_decode < 0 || num_prefill < 0 || num_speculative_tokens < 0) return LS_ERR_INVALID_ARG;
  const int64_t per = 1 + (int64_t)num_speculative_tokens;
  const int64_t n64 = (int64_t)num_decode * per + num_prefill;
  if (n64 > 0x7FFFFFFFll) return LS_ERR_INVALID_ARG;
  const int32_t n = (int32_t)n64;
  if (n == 0) return LS_OK;
  if (!common_ok(required_logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, true) || !out_ids)
    return LS_ERR_INVALID_ARG;
  if (!gather_indices && n64 > logits_rows) return LS_ERR_INVALID_ARG;
  if ((int64_t)num_decode + num_prefill > params->num_requests) return LS_ERR_INVALID_ARG;
  KernelArgs a = make_args(required_logits, logits_rows, vocab, row_stride, gather_indices, params, step,
                           error_word);
  a.map_mode = MAP_SPEC;
  a.spec_decode_rows = (int32_t)((int64_t)num_decode * per);
  a.spec_per_req = (int32_t)per;
  a.spec_num_decode = num_decode;
  a.out_ids = out_ids;
  a.out_t2r = out_token_to_request_index;
  const int route = (no_top_k ? 0 : ROUTE_K) | (no_top_p ? 0 : ROUTE_P);
  return dispatch<MODE_SAMPLE>(a, dtype, route, n, static_cast<cudaStream_t>(stream));
}

ls_status ls_log_probs(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                       int32_t num_rows, const int32_t* gather_indices, const int32_t* token_to_request_index,
                       const ls_params* params, float* out_log_probs, int32_t* error_word, void* stream) {
  if (num_rows < 0) return LS_ERR_INVALID_ARG;
  if (num_rows == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, false) || !out_log_probs)
    return LS_ERR_INVALID_ARG;
  if (!gather_indices && (int64_t)num_rows > logits_rows) return LS_ERR_INVALID_ARG;
  if (!token_to_request_index && num_rows > params->num_requests) return LS_ERR_INVALID_ARG;
  KernelArgs a = make_args(logits, logits_rows, vocab, row_stride, gather_indices, params, 0, error_word);
  a.t2r = token_to_request_index;
  a.map_mode = token_to_request_index ? MAP_T2R : MAP_IDENTITY;
  a.out_lp = out_log_probs;
  return dispatch<MODE_LOGPROBS>(a, dtype, ROUTE_KP, num_rows, static_cast<cudaStream_t>(stream));
}

ls_status ls_sample_device_step(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                                int64_t row_stride, int32_t n, const int32_t* gather_indices,
                                const int32_t* token_to_request_index, const ls_params* params, uint64_t* step,
                                int no_top_k, int no_top_p, int32_t* out_ids, int32_t* error_word, void* stream) {
  if (n < 0 || !step) return LS_ERR_INVALID_ARG;
  if (n == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, true) || !out_ids)
    return LS_ERR_INVALID_ARG;
  if (!gather_indices && (int64_t)n > logits_rows) return LS_ERR_INVALID_ARG;
  if (!token_to_request_index && n > params->num_requests) return LS_ERR_INVALID_ARG;
  KernelArgs a = make_args(logits, logits_rows, vocab, row_stride, gather_indices, params, 0, error_word);
  a.step_ptr = step;
  a.t2r = token_to_request_index;
  a.map_mode = token_to_request_index ? MAP_T2R : MAP_IDENTITY;
  a.out_ids = out_ids;
  const int route = (no_top_k ? 0 : ROUTE_K) | (no_top_p ? 0 : ROUTE_P);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ls_status rc = dispatch<MODE_SAMPLE>(a, dtype, route, n, st);
  if (rc != LS_OK) return rc;
  advance_step_kernel<<<1, 1, 0, st>>>(step);
  return cudaGetLastError() == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}

ls_status ls_sample_log_probs(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                              int64_t row_stride, int32_t n, const int32_t* gather_indices,
                              const int32_t* token_to_request_index, const ls_params* params, uint64_t step,
                              int no_top_k, int no_top_p, int32_t* out_ids, float* out_log_probs,
                              float* out_selected_log_probs, int32_t* error_word, void* stream) {
  if (n < 0) return LS_ERR_INVALID_ARG;
  if (n == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, true) || !out_ids)
    return LS_ERR_INVALID_ARG;
  if (!gather_indices && (int64_t)n > logits_rows) return LS_ERR_INVALID_ARG;
  if (!token_to_request_index && n > params->num_requests) return LS_ERR_INVALID_ARG;
  KernelArgs a = make_args(logits, logits_rows, vocab, row_stride, gather_indices, params, step, error_word);
  a.t2r = token_to_request_index;
  a.map_mode = token_to_request_index ? MAP_T2R : MAP_IDENTITY;
  a.out_ids = out_ids;
  a.out_lp = out_log_probs;
  a.out_sel = out_selected_log_probs;
  const int route = (no_top_k ? 0 : ROUTE_K) | (no_top_p ? 0 : ROUTE_P);
  if (!out_log_probs && !out_selected_log_probs)  // ids only: the sampling kernels
    return dispatch<MODE_SAMPLE>(a, dtype, route, n, static_cast<cudaStream_t>(stream));
  return dispatch<MODE_BOTH>(a, dtype, route, n, static_cast<cudaStream_t>(stream));
}

const char* ls_status_string(ls_status s) {
  switch (s) {
    case LS_OK: return "LS_OK";
    case LS_ERR_INVALID_ARG: return "LS_ERR_INVALID_ARG: invalid argument (nothing launched)";
    case LS_ERR_UNSUPPORTED: return "LS_ERR_UNSUPPORTED: vocab beyond the shared-memory limit of this device";
    case LS_ERR_CUDA: return "LS_ERR_CUDA: CUDA launch failed";
    default: return "unknown ls_status";
  }
}

int64_t ls_max_vocab(ls_dtype dtype) {
  (void)dtype;  // the limit is the same for both dtypes: 4 bytes of shared memory per 16 logits
  const int lim = max_dyn_smem();
  if (lim <= 0) return 0;
  const int64_t ng = ((int64_t)lim - (int64_t)smem_bytes(0, 256)) / (int64_t)sizeof(float) + 1;
  return ng * kGroup - (2 * kGroup - 1);
}

}  // extern "C"
