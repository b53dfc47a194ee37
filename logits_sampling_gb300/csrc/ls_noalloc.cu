// ls_noalloc.cu -- ls_sample_log_probs without a caller workspace: the
// per-row scalars of the tiled log-prob write live in a fixed device array of
// this library (LS_NOALLOC_MAX_ROWS rows), so the call needs no allocation by
// anyone.  Everything else is ls_sample_log_probs itself.
#include "ls_kernel.cuh"

namespace lsg {

// Scratch of ls_sample_log_probs_noalloc: one LpRow per row.  No entry has to
// start at zero (the row kernel writes each row's record before the write
// kernel reads it), so nothing is cleared.
static __device__ __align__(256) LpRow g_noalloc_rows[LS_NOALLOC_MAX_ROWS];

// The array's device address, looked up once per device.
static void* noalloc_scratch() {
  static std::atomic<void*> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  if (cudaGetSymbolAddress(&p, g_noalloc_rows) != cudaSuccess) return nullptr;
  cache[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace lsg

extern "C" ls_status ls_sample_log_probs_noalloc(const void* logits, ls_dtype dtype, int64_t logits_rows,
                                                 int64_t vocab, int64_t row_stride, int32_t n,
                                                 const int32_t* gather_indices,
                                                 const int32_t* token_to_request_index, const ls_params* params,
                                                 uint64_t step, int no_top_k, int no_top_p, int32_t* out_ids,
                                                 float* out_log_probs, float* out_selected_log_probs,
                                                 int32_t* error_word, void* stream) {
  if (n > LS_NOALLOC_MAX_ROWS) return LS_ERR_UNSUPPORTED;  // the fixed scratch holds fewer rows
  void* ws = n > 0 ? lsg::noalloc_scratch() : nullptr;
  if (n > 0 && !ws) return LS_ERR_CUDA;
  return ls_sample_log_probs(logits, dtype, logits_rows, vocab, row_stride, n, gather_indices,
                             token_to_request_index, params, step, no_top_k, no_top_p, out_ids, out_log_probs,
                             out_selected_log_probs, ws, ws ? sizeof(lsg::LpRow) * (size_t)LS_NOALLOC_MAX_ROWS : 0u,
                             error_word, stream);
}
