// ls_sampler.cu -- C ABI of the token sampler (include/ls_sampler.h).
//
// Host-side argument checks and the route/mode dispatch; the kernels are in
// ls_kernel.cuh and are instantiated per mode in ls_mode_*.cu.
#include "ls_kernel.cuh"

namespace lsg {
extern template ls_status dispatch<MODE_SAMPLE>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
extern template ls_status dispatch<MODE_LOGPROBS>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
extern template ls_status dispatch<MODE_BOTH>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
template <int C>
ls_status dispatch_split(KernelArgs a, ls_dtype dtype, int route, int32_t n, cudaStream_t stream);
extern template ls_status dispatch_split<1>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
extern template ls_status dispatch_split<2>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
extern template ls_status dispatch_split<4>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);
extern template ls_status dispatch_split<8>(KernelArgs, ls_dtype, int, int32_t, cudaStream_t);

// Which sampling kernel runs (ls_set_split_policy): 0 = chosen per call from
// the batch shape; 1, 2, 4, 8 = the streaming sampler with that many CTAs per
// row; -1 = the one-CTA row kernel without in-stream collection.
static std::atomic<int> g_split_policy{0};

static int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && (v = cache[dev].load(std::memory_order_relaxed)) > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Kernel from the batch shape alone (host values, no device read).  A batch
// of at least one and a half times the SM count keeps every SM streaming with
// one CTA per row: the row kernel.  A smaller batch with rows long enough to
// split runs the streaming sampler, doubling the CTAs per row while that
// leaves fewer than two per SM and slices of at least 2048 entries; short rows
// of a small batch take the row kernel.
static int split_for(int32_t n, int64_t vocab) {
  const int pol = g_split_policy.load(std::memory_order_relaxed);
  if (pol == -1 || pol == 1 || pol == 2 || pol == 4 || pol == 8) return pol;
  const int sms = sm_count();
  if (sms <= 0 || (int64_t)n * 2 >= (int64_t)sms * 3) return -1;
  int c = 1;
  while (c < 8 && (int64_t)n * c < 2 * (int64_t)sms && vocab / (2 * c) >= 2048) c *= 2;
  return c > 1 ? c : -1;
}

// The largest vocab every kernel accepts on the current device: the one-CTA
// row kernel's (4 bytes of shared memory per 16 logits) is the smallest.
static int64_t max_vocab_all() {
  const int lim = max_dyn_smem();
  if (lim <= 0) return 0;
  const int64_t ng = ((int64_t)lim - (int64_t)smem_bytes(0, 256)) / (int64_t)sizeof(float) + 1;
  return ng * kGroup - (2 * kGroup - 1);
}

// The sampling calls' kernel (ids only).  Every call accepts the same
// vocabularies (ls_max_vocab), whichever kernel runs.
ls_status dispatch_sample(const KernelArgs& a, ls_dtype dtype, int route, int32_t n, cudaStream_t stream) {
  const int64_t vmax = max_vocab_all();
  if (vmax <= 0) return LS_ERR_CUDA;
  if (a.vocab > vmax) return LS_ERR_UNSUPPORTED;
  switch (split_for(n, a.vocab)) {
    case -1: return dispatch<MODE_SAMPLE>(a, dtype, route, n, stream);
    case 2: return dispatch_split<2>(a, dtype, route, n, stream);
    case 4: return dispatch_split<4>(a, dtype, route, n, stream);
    case 8: return dispatch_split<8>(a, dtype, route, n, stream);
    default: return dispatch_split<1>(a, dtype, route, n, stream);
  }
}

// L2 size of the current device in bytes (cached per device), 0 if unknown.
static int64_t l2_bytes() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && (v = cache[dev].load(std::memory_order_relaxed)) > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Which write the log-prob calls with a workspace take
// (ls_set_log_prob_write_policy): 0 = from the batch shape; 1 = the tiled
// write kernel; -1 = the row kernel's own write pass.
static std::atomic<int> g_lp_write_policy{0};

// Whether a log-prob call with a workspace writes its rows through
// lp_write_kernel.  Measured on top_p-shaped rows (bf16, 128256 entries): the
// tiled write wins while the batch leaves SMs idle (8 rows: 20.5 against
// 28.7 us; 96 rows: 27.9 against 30.9) and loses once every SM holds a row
// (152 rows: 35.9 against 33.0; 256 rows: 52.1 against 49.3), because the row
// kernel then overlaps its early rows' writes with the other rows' streaming.
// So: at most 3/4 of the SM count of rows, rows of at least 16384 entries
// (shorter rows write faster than a second launch costs), and logits that
// fit in 60% of L2 (the write finds them there).
static bool lp_deferred(int32_t n, int64_t vocab, ls_dtype dtype) {
  const int pol = g_lp_write_policy.load(std::memory_order_relaxed);
  if (pol != 0) return pol > 0;
  const int64_t l2 = l2_bytes();
  const int sms = sm_count();
  const int64_t bytes = (int64_t)n * vocab * (dtype == LS_DTYPE_BF16 ? 2 : 4);
  return l2 > 0 && sms > 0 && (int64_t)n * 4 <= (int64_t)sms * 3 && vocab >= 16384 && bytes * 5 <= l2 * 3;
}

// A workspace is absent, or large enough and 16-byte aligned.
static bool workspace_ok(const void* ws, size_t bytes, int32_t n) {
  return !ws || (bytes >= (size_t)n * sizeof(LpRow) && (reinterpret_cast<uintptr_t>(ws) & 15u) == 0u);
}

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
  return dispatch_sample(a, dtype, route, n, static_cast<cudaStream_t>(stream));
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
  return dispatch_sample(a, dtype, route, n, static_cast<cudaStream_t>(stream));
}

size_t ls_log_probs_workspace_bytes(int32_t num_rows) {
  return num_rows > 0 ? (size_t)num_rows * sizeof(LpRow) : 0u;
}

ls_status ls_log_probs(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                       int32_t num_rows, const int32_t* gather_indices, const int32_t* token_to_request_index,
                       const ls_params* params, float* out_log_probs, void* workspace, size_t workspace_bytes,
                       int32_t* error_word, void* stream) {
  if (num_rows < 0) return LS_ERR_INVALID_ARG;
  if (num_rows == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, false) || !out_log_probs ||
      !workspace_ok(workspace, workspace_bytes, num_rows))
    return LS_ERR_INVALID_ARG;
  if (!gather_indices && (int64_t)num_rows > logits_rows) return LS_ERR_INVALID_ARG;
  if (!token_to_request_index && num_rows > params->num_requests) return LS_ERR_INVALID_ARG;
  KernelArgs a = make_args(logits, logits_rows, vocab, row_stride, gather_indices, params, 0, error_word);
  a.t2r = token_to_request_index;
  a.map_mode = token_to_request_index ? MAP_T2R : MAP_IDENTITY;
  a.out_lp = out_log_probs;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (workspace && lp_deferred(num_rows, vocab, dtype)) a.lp_rows = static_cast<LpRow*>(workspace);
  const ls_status rc = dispatch<MODE_LOGPROBS>(a, dtype, ROUTE_KP, num_rows, st);
  if (rc != LS_OK || !a.lp_rows) return rc;
  return dispatch_lp_write(a, dtype, num_rows, st);
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
  const ls_status rc = dispatch_sample(a, dtype, route, n, st);
  if (rc != LS_OK) return rc;
  advance_step_kernel<<<1, 1, 0, st>>>(step);
  return cudaGetLastError() == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}

ls_status ls_sample_log_probs(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                              int64_t row_stride, int32_t n, const int32_t* gather_indices,
                              const int32_t* token_to_request_index, const ls_params* params, uint64_t step,
                              int no_top_k, int no_top_p, int32_t* out_ids, float* out_log_probs,
                              float* out_selected_log_probs, void* workspace, size_t workspace_bytes,
                              int32_t* error_word, void* stream) {
  if (n < 0) return LS_ERR_INVALID_ARG;
  if (n == 0) return LS_OK;
  if (!common_ok(logits, dtype, logits_rows, vocab, row_stride) || !params_ok(params, true) || !out_ids ||
      !workspace_ok(workspace, workspace_bytes, n))
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
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!out_log_probs && !out_selected_log_probs)  // ids only: the sampling kernels
    return dispatch_sample(a, dtype, route, n, st);
  if (out_log_probs && workspace && lp_deferred(n, vocab, dtype)) a.lp_rows = static_cast<LpRow*>(workspace);
  const ls_status rc = dispatch<MODE_BOTH>(a, dtype, route, n, st);
  if (rc != LS_OK || !a.lp_rows) return rc;
  return dispatch_lp_write(a, dtype, n, st);
}

int ls_set_log_prob_write_policy(int policy) {
  if (policy != 0 && policy != 1 && policy != -1) return (int)LS_ERR_INVALID_ARG;
  g_lp_write_policy.store(policy, std::memory_order_relaxed);
  return (int)LS_OK;
}

int ls_set_split_policy(int ctas_per_row) {
  if (ctas_per_row != 0 && ctas_per_row != -1 && ctas_per_row != 1 && ctas_per_row != 2 && ctas_per_row != 4 &&
      ctas_per_row != 8)
    return (int)LS_ERR_INVALID_ARG;
  g_split_policy.store(ctas_per_row, std::memory_order_relaxed);
  return (int)LS_OK;
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
  (void)dtype;  // the limit is the same for both dtypes
  return max_vocab_all();
}

}  // extern "C"
