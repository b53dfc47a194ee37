/*
 * ls_sampler.h -- C ABI of the GB300 token sampler (libls_sampler.so).
 *
 * The library samples one token id per row of a [rows, vocab] logits matrix
 * and computes the per-row log-probs of the processed distribution
 * (temperature, exact top-k, exact top-p).  Every call is asynchronous on the
 * caller's CUDA stream, allocates nothing, never synchronises with the host
 * and launches one kernel (ls_sample_device_step and ls_sample_verify: two).
 * The sampling calls split a row over a thread-block cluster of 2, 4 or 8
 * CTAs when the batch is small (ls_set_split_policy).
 *
 * Conventions shared by all entry points
 * --------------------------------------
 * - Pointers: every buffer argument is a DEVICE pointer (cudaMalloc /
 *   cudaMallocManaged / a device view of pinned host memory) owned by the
 *   caller, except `params`, which points to a small HOST struct whose fields
 *   are device pointers.  Results are valid once `stream` has reached the
 *   call's completion.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 * - Layout: logits row r starts at element r * row_stride; vocab <= row_stride.
 *   Rows need no particular alignment.
 * - Sampling parameters (struct ls_params) are indexed by request; row i uses
 *   request token_to_request_index[i] when that array is given, else request i.
 *     temperature  T < 1e-5 (or NaN) -> greedy row: the id is the lowest index
 *                  of the row maximum, no noise.
 *     top_k        k <= 0 or k >= vocab -> top-k off for that row.  Kept set:
 *                  entries >= the k-th largest logit (ties at the cut kept).
 *     top_p        p >= 0.99999 (or NaN) -> top-p off.  Kept set: walking the
 *                  distinct values downwards, the first value at which the
 *                  cumulative probability reaches p; everything at or above it
 *                  is kept.  p <= 0 keeps the maximum and its ties.
 *     seed         Philox4x32-10 key (lo32, hi32) of the request.
 *   Joint filtering applies top-k first, then top-p on the renormalised top-k
 *   distribution.
 * - Noise: entry j of output row i at step s gets the word (j mod 4) of
 *   Philox4x32-10(counter = (j/4, i, lo32 s, hi32 s), key = seed), mapped to
 *   u = (2*(x>>9)+1) * 2^-24 and g = -ln(-ln u).  The id is the argmax of
 *   z_j + g_j over the kept set (z = logit / T), lowest index on an exact tie.
 *   The same (seed, step, row) always gives the same id; a new step gives
 *   fresh noise.
 * - Special values: NaN logits are read as -inf; -inf entries are never kept.
 *   A row whose maximum is +inf samples uniformly among its +inf entries.
 * - Errors found on the host (bad arguments) return a status before any launch.
 *   Errors found per row on the device (index out of range, a row with no
 *   entry above -inf) write id -1 (log-probs NaN) for that row and OR a bit
 *   into *error_word when error_word is not NULL:
 *     LS_ROW_ERR_BAD_GATHER  gather_indices[i] outside [0, logits_rows)
 *     LS_ROW_ERR_BAD_REQUEST request index outside [0, params->num_requests)
 *     LS_ROW_ERR_NO_FINITE   every entry of the row is -inf or NaN
 *   The library never clears *error_word.
 */
#ifndef LS_SAMPLER_H
#define LS_SAMPLER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LS_OK = 0,
  LS_ERR_INVALID_ARG = 1, /* a host-checkable argument is wrong; nothing launched */
  LS_ERR_UNSUPPORTED = 2, /* valid but beyond this build's limits (e.g. vocab too large) */
  LS_ERR_CUDA = 3         /* the launch failed; cudaGetLastError() holds the reason */
} ls_status;

typedef enum { LS_DTYPE_F32 = 0, LS_DTYPE_BF16 = 1 } ls_dtype;

enum { LS_ROW_ERR_BAD_GATHER = 1, LS_ROW_ERR_BAD_REQUEST = 2, LS_ROW_ERR_NO_FINITE = 4 };

/* Per-request sampling parameters: device arrays of length num_requests, owned
 * by the caller (the per-request sampling metadata a serving controller keeps
 * on the GPU). */
typedef struct {
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const uint64_t* seed;
  int32_t num_requests;
} ls_params;

/*
 * ls_sample -- sample n token ids.
 *
 * Follows "core.inference.sampling.base" (Sampling.sample_kernel) and
 * "core.inference.sampling.flashinfer_sampling" (FlashInferSampling.
 * sample_kernel): sample n tokens from logits[>= n, vocab]; with
 * gather_indices, row i reads logits[gather_indices[i]]; with
 * token_to_request_index, parameters are gathered per token.  The batch flags
 * no_top_k / no_top_p (computed by the caller from host-side metadata) pick
 * the route -- no filter, top-k only, top-p only or joint -- with no device
 * read and no sync.  A set flag switches that filter off for every row.
 *
 *   logits          device, dtype elements, logits_rows x row_stride
 *   logits_rows     rows addressable in logits (>= n when gather_indices is NULL)
 *   vocab           entries per row, 1 <= vocab <= row_stride
 *   n               rows to sample, >= 0 (0: nothing launched, LS_OK)
 *   gather_indices  device int32[n] or NULL
 *   token_to_request_index  device int32[n] or NULL (NULL: row i -> request i)
 *   params          host pointer to device parameter arrays
 *   step            Philox step word (advance it every decoding step)
 *   out_ids         device int32[n], written by the call
 *   error_word      device int32 or NULL
 *   stream          cudaStream_t
 */
ls_status ls_sample(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                    int32_t n, const int32_t* gather_indices, const int32_t* token_to_request_index,
                    const ls_params* params, uint64_t step, int no_top_k, int no_top_p, int32_t* out_ids,
                    int32_t* error_word, void* stream);

/*
 * ls_sample_speculative -- sample the speculative-verify rows.
 *
 * Follows "core.inference.sampling.base" (Sampling.sample_speculative): decode
 * requests contribute 1 + num_speculative_tokens rows and prefill requests 1,
 * so n = num_decode * (1 + S) + num_prefill.  Row r belongs to request
 * r / (1 + S) when r < num_decode * (1 + S), else to request
 * num_decode + (r - num_decode * (1 + S)) (decode rows first).  With
 * gather_indices, row r reads logits[gather_indices[r]]; without, logits are
 * already in that layout (logits_rows >= n).  Requires
 * params->num_requests >= num_decode + num_prefill.
 *
 *   out_ids                       device int32[n]
 *   out_token_to_request_index    device int32[n] or NULL: the mapping above
 * Other arguments as for ls_sample.
 */
ls_status ls_sample_speculative(const void* required_logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                                int64_t row_stride, int32_t num_decode, int32_t num_prefill,
                                int32_t num_speculative_tokens, const int32_t* gather_indices,
                                const ls_params* params, uint64_t step, int no_top_k, int no_top_p,
                                int32_t* out_ids, int32_t* out_token_to_request_index, int32_t* error_word,
                                void* stream);

/*
 * ls_log_probs -- per-row log-probs of the processed distribution.
 *
 * Follows "core.inference.sampling.flashinfer_sampling" (FlashInferSampling.
 * log_probs_kernel): raw logits [num_rows, vocab], optional row -> request
 * mapping; output = log-probs of the distribution the sampler draws from
 * (every row's own temperature, top-k and top-p; no route flags).
 * out[i, j] = z_j - max_K z - ln sum_K exp(z - max_K z) for j in the kept set
 * K, -inf elsewhere (z = logit / T; greedy rows: -ln(#ties) on the maximum's
 * ties).  gather_indices is an extension the page does not have (NULL: row i
 * reads logits row i).
 *
 *   out_log_probs   device float[num_rows * vocab], row-major, written fully
 *   workspace       NULL, or device memory of at least
 *                   ls_log_probs_workspace_bytes(num_rows) bytes, 16-byte
 *                   aligned, owned by the caller and not used by other calls
 *                   in flight (otherwise LS_ERR_INVALID_ARG).  With a
 *                   workspace, a batch of at most 3/4 of the SM count of rows,
 *                   of at least 16384 entries each, whose logits fit in 60% of
 *                   L2, takes two launches: the row kernel leaves 16 bytes of
 *                   scalars per row there, and a second kernel writes the rows
 *                   in tiles spread over every SM (the same values;
 *                   ls_set_log_prob_write_policy overrides the choice).
 *                   Otherwise the row kernel writes each row itself.
 *   workspace_bytes size of workspace (ignored when it is NULL)
 * Other arguments as for ls_sample.
 */
ls_status ls_log_probs(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                       int32_t num_rows, const int32_t* gather_indices, const int32_t* token_to_request_index,
                       const ls_params* params, float* out_log_probs, void* workspace, size_t workspace_bytes,
                       int32_t* error_word, void* stream);

/* Bytes of the optional workspace of ls_log_probs and ls_sample_log_probs for
 * num_rows rows (16 per row; 0 when num_rows <= 0). */
size_t ls_log_probs_workspace_bytes(int32_t num_rows);

/*
 * ls_sample_device_step -- ls_sample with the Philox step word in device
 * memory, advanced on the device after the call, so that a CUDA graph that
 * captured the call draws fresh noise at every replay.
 *
 * The "core.inference.sampling.flashinfer_sampling" page (FlashInferSampling
 * class description) runs its sampler eagerly because FlashInfer bakes the
 * Philox state into a captured graph as a by-value constant, so a captured
 * sampler replays identical random numbers.  Here the kernel reads *step when
 * it starts and a second one-thread kernel adds 1 to *step after it on the same
 * stream (two launches per call).  Rows, ids and errors are exactly those of
 * ls_sample(..., step = the value *step held, ...).
 *
 *   step    device uint64[1], read by the call and left at its value + 1
 *           (n == 0: nothing is launched and *step is unchanged)
 * Other arguments as for ls_sample.
 */
ls_status ls_sample_device_step(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                                int64_t row_stride, int32_t n, const int32_t* gather_indices,
                                const int32_t* token_to_request_index, const ls_params* params, uint64_t* step,
                                int no_top_k, int no_top_p, int32_t* out_ids, int32_t* error_word, void* stream);

/*
 * ls_sample_log_probs -- sample n token ids and, from the same single read of
 * the logits, their log-probs.
 *
 * Follows "core.inference.sampling.flashinfer_sampling" (FlashInferSampling.
 * sample_kernel and log_probs_kernel) and the TokenSpeed "backends/triton.py"
 * page (TritonSamplingBackend.sample followed by _write_logprob_outputs,
 * which fills next_token_logprobs with selected_token_logprobs(logits,
 * sampled)): what ls_sample followed by ls_log_probs and a selected-token
 * log-prob would compute, with the logits read from HBM once instead of
 * twice.
 *
 *   out_ids                device int32[n]: exactly the ids ls_sample returns
 *                          for the same arguments
 *   out_log_probs          device float[n * vocab] or NULL: log-probs of the
 *                          processed distribution, as ls_log_probs writes them
 *                          (the route flags switch filters off as for ls_sample)
 *   out_selected_log_probs device float[n] or NULL: log-probability of the
 *                          sampled id under the raw logits (no temperature, no
 *                          filter): l_id - ln sum_j exp(l_j) over the row, NaN
 *                          logits read as -inf; a row whose maximum is +inf
 *                          gives -ln(#(+inf entries)) for a +inf id
 *   workspace, workspace_bytes
 *                          as for ls_log_probs (used only with out_log_probs)
 * With both optional outputs NULL the call is ls_sample.  Error rows: id -1,
 * NaN log-probs.  Other arguments as for ls_sample.
 */
ls_status ls_sample_log_probs(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                              int64_t row_stride, int32_t n, const int32_t* gather_indices,
                              const int32_t* token_to_request_index, const ls_params* params, uint64_t step,
                              int no_top_k, int no_top_p, int32_t* out_ids, float* out_log_probs,
                              float* out_selected_log_probs, void* workspace, size_t workspace_bytes,
                              int32_t* error_word, void* stream);

/* Rows ls_sample_log_probs_noalloc accepts (its fixed scratch: 16 bytes per row). */
#define LS_NOALLOC_MAX_ROWS 4096

/*
 * ls_sample_log_probs_noalloc -- ls_sample_log_probs without a caller
 * workspace and without any allocation: the per-row scalars of the tiled
 * log-prob write go to a fixed device array of this library
 * (LS_NOALLOC_MAX_ROWS rows, 64 KB, located once per device).
 *
 * Results are exactly those of ls_sample_log_probs with a workspace.  n above
 * LS_NOALLOC_MAX_ROWS returns LS_ERR_UNSUPPORTED with nothing launched.  Calls
 * in flight at the same time on one device (other streams, other host
 * threads) share that array and race; issue them one after another on one
 * stream.  Nothing in the array has to start at zero.
 * Arguments as for ls_sample_log_probs, without workspace and workspace_bytes.
 */
ls_status ls_sample_log_probs_noalloc(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab,
                                      int64_t row_stride, int32_t n, const int32_t* gather_indices,
                                      const int32_t* token_to_request_index, const ls_params* params,
                                      uint64_t step, int no_top_k, int no_top_p, int32_t* out_ids,
                                      float* out_log_probs, float* out_selected_log_probs, int32_t* error_word,
                                      void* stream);

/*
 * ls_argmax -- the all-greedy fast path: out_ids[i] = the lowest index of the
 * maximum of logits row i (row gather_indices[i] when given).
 *
 * Follows the TokenSpeed "backends/triton.py" page (TritonSamplingBackend.
 * sample and verify: when every request of the batch is greedy, the argmax of
 * the logits replaces the sampling kernels).  The ids are the ones ls_sample
 * returns for greedy rows (T < 1e-5): NaN read as -inf, ties to the lowest
 * index; a row with no entry above -inf gives -1 and LS_ROW_ERR_NO_FINITE, a
 * gather index out of range -1 and LS_ROW_ERR_BAD_GATHER.  No parameters, no
 * noise; one streaming read of each row.
 *
 *   out_ids   device int32[n]
 * Other arguments as for ls_sample.
 */
ls_status ls_argmax(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                    int32_t n, const int32_t* gather_indices, int32_t* out_ids, int32_t* error_word, void* stream);

/*
 * ls_verify_chain -- speculative chain verification against the target
 * model's sampled tokens.
 *
 * Follows the TokenSpeed "backends/triton.py" page (TritonSamplingBackend.
 * verify: verify_chain_target_sampled(predicts, accept_index,
 * accept_token_num, candidates, target_sampled), then accept_length += 1).
 * The pages print only the call; the rule implemented (the plain chain rule):
 * request b has n = num_tokens positions; candidates[b, 0] is the token the
 * drafts extend, candidates[b, j] (j >= 1) the j-th draft, and
 * target_sampled[b*n + j] the target's token after position j.  Position 0 is
 * always accepted; position j >= 1 is accepted while every earlier position
 * was and candidates[b, j] == target_sampled[b*n + j - 1].  For an accepted
 * position accept_index[b, j] = b*n + j and predicts[b*n + j] =
 * target_sampled[b*n + j]; other accept_index entries are -1 and other
 * predicts are left unchanged.  accept_token_num[b] = the number of accepted
 * drafts (the page's accept_length is that + 1: the bonus token).
 *
 *   candidates        device int32[bs * num_tokens] (row-major [bs, n])
 *   target_sampled    device int32[bs * num_tokens]
 *   predicts          device int32[bs * num_tokens]
 *   accept_index      device int32[bs * num_tokens]
 *   accept_token_num  device int32[bs]
 * bs = 0: nothing launched.  num_tokens >= 1.
 */
ls_status ls_verify_chain(const int32_t* candidates, const int32_t* target_sampled, int32_t bs,
                          int32_t num_tokens, int32_t* predicts, int32_t* accept_index, int32_t* accept_token_num,
                          void* stream);

/*
 * ls_sample_verify -- sample the verify rows of bs decode requests
 * (num_tokens rows each: ls_sample_speculative with num_decode = bs,
 * num_prefill = 0, num_speculative_tokens = num_tokens - 1) into
 * out_target_sampled, then ls_verify_chain on them: two launches, no host
 * round trip between the target's sampling and the acceptance.
 *
 *   out_target_sampled  device int32[bs * num_tokens]: the sampled verify rows
 * Other arguments as for ls_sample_speculative and ls_verify_chain.
 */
ls_status ls_sample_verify(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                           int32_t bs, int32_t num_tokens, const int32_t* gather_indices, const ls_params* params,
                           uint64_t step, int no_top_k, int no_top_p, const int32_t* candidates,
                           int32_t* out_target_sampled, int32_t* predicts, int32_t* accept_index,
                           int32_t* accept_token_num, int32_t* error_word, void* stream);

/*
 * ls_set_split_policy -- which kernel the sampling calls that return ids only
 * (ls_sample, ls_sample_speculative, ls_sample_device_step, ls_sample_verify,
 * and ls_sample_log_probs with both optional outputs NULL) launch, for every
 * later call in the process.  For tests and tuning: every choice computes the
 * same sampler (ids may differ only where the parity exemption allows, since
 * the row's mass is summed in another order).
 *   0           chosen per call from the batch shape on the host (default):
 *               one CTA per row for batches of at least 1.5x the SM count,
 *               else 2, 4 or 8 CTAs per row (a thread-block cluster) while
 *               that leaves fewer than two CTAs per SM and slices of at least
 *               2048 entries
 *   1, 2, 4, 8  the streaming sampler (candidates collected during the read
 *               of the row) with that many CTAs per row
 *   -1          the one-CTA row kernel that re-reads candidate groups after
 *               the read of the row
 * Returns LS_OK, or LS_ERR_INVALID_ARG for any other value (unchanged).
 * Not synchronised with calls in flight on other host threads.
 */
int ls_set_split_policy(int ctas_per_row);

/*
 * ls_set_log_prob_write_policy -- which write the log-prob calls given a
 * workspace take, for every later call in the process (tests and tuning; both
 * write the same values):
 *   0   chosen from the batch shape (default; see ls_log_probs)
 *   1   the tiled write kernel
 *   -1  the row kernel's own write pass
 * Returns LS_OK, or LS_ERR_INVALID_ARG for any other value (unchanged).
 * Not synchronised with calls in flight on other host threads.
 */
int ls_set_log_prob_write_policy(int policy);

/* Human-readable name of a status code (static storage). */
const char* ls_status_string(ls_status s);

/* Largest vocab the kernels accept for a dtype on the current device (shared
 * memory bound), or 0 when no CUDA device is available. */
int64_t ls_max_vocab(ls_dtype dtype);

#ifdef __cplusplus
}
#endif

#endif /* LS_SAMPLER_H */
