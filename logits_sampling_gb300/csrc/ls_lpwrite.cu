// ls_lpwrite.cu -- the deferred write of log-prob rows.
//
// When the caller gives a workspace and the batch's logits fit in L2, the
// row kernel leaves each row's scalars (LpRow: maximum, temperature,
// normaliser, cut) instead of writing the row itself, and this kernel writes
// every row.  One CTA per row would leave the writes as unevenly spread as
// the rows are over the SMs (a 256-row batch puts two rows on most SMs and
// one on the rest) and with few loads in flight per SM; here the rows are cut
// into tiles of kLpTileEntries entries that every SM shares.  The row is read
// again, normally from L2 (the row kernel loaded it with an evict-last
// policy).  Values are the row kernel's own (LpValue): the same kept test and
// the same arithmetic per entry.
#include "ls_kernel.cuh"

namespace lsg {

constexpr int kLpThreads = 256;
constexpr int kLpTileEntries = 8192;
constexpr int kLpQuads = kLpTileEntries / 4 / kLpThreads;     // quads of 4 entries per thread and tile
constexpr int kLpPer = kLpTileEntries / kGroup / kLpThreads;  // groups per thread and tile (unaligned rows)

template <typename TIn>
__global__ void __launch_bounds__(kLpThreads) lp_write_kernel(const KernelArgs a, int tiles) {
  using RVT = RowView<TIn>;
  constexpr int E = RVT::kBytes;      // bytes per logit
  constexpr int QW = E == 2 ? 2 : 4;  // words per quad
  // the row kernel's scalars are visible once it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t i = (int64_t)(blockIdx.x / (unsigned)tiles);
  const int tile = (int)(blockIdx.x % (unsigned)tiles);
  const LpRow r = a.lp_rows[i];
  float* out = a.out_lp + i * a.vocab;
  const bool bad = !(r.M == r.M);  // error row: NaN throughout (its gather index may be out of range)
  const int64_t src = bad ? 0 : (a.gather ? (int64_t)a.gather[i] : i);
  const int64_t V = a.vocab;
  const uint64_t pol = l2_evict_first_policy();  // the row's last use
  const float lo = r.lo, lnS = r.lnS;
  const bool tie = r.T == 0.f;  // the maximum's ties share the probability exp(-lnS)
  const LpValue val = lp_value(r.M, tie ? 1.f : r.T, lnS);
  auto value = [&](float v) {
    if (bad) return __uint_as_float(0x7FC00000u);
    if (!(v >= lo)) return kNegInf;
    return tie ? -lnS : val(v);
  };
  const unsigned char* row = static_cast<const unsigned char*>(a.logits) + src * a.stride * E;
  const bool aligned =
      (reinterpret_cast<uintptr_t>(row) & (4 * E - 1)) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  if (aligned) {
    // Entries 4 at a time: a warp's loads and stores cover consecutive
    // addresses; all of a thread's loads are in flight before its first store.
    const int64_t q0 = (int64_t)tile * (kLpTileEntries / 4) + threadIdx.x;
    uint32_t w[kLpQuads][QW];
#pragma unroll
    for (int u = 0; u < kLpQuads; ++u) {
      const int64_t j = 4 * (q0 + (int64_t)u * kLpThreads);
      if (!bad && j + 4 <= V) ld_quad(row + j * E, w[u], pol);
    }
#pragma unroll
    for (int u = 0; u < kLpQuads; ++u) {
      const int64_t j = 4 * (q0 + (int64_t)u * kLpThreads);
      if (j + 4 <= V) {
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = value(bad ? 0.f : quad_at(w[u], e));
        st_stream4(out + j, o[0], o[1], o[2], o[3]);
      } else if (j < V) {  // the row's last 1-3 entries
        RVT rv;
        rv.init(a.logits, src, a.stride, V);
        for (int64_t jj = j; jj < V; ++jj) out[jj] = value(bad ? 0.f : rv.at(jj));
      }
    }
    return;
  }
  // Unaligned rows: groups of 16 as the row kernel writes them.
  RVT rv;
  rv.init(a.logits, src, a.stride, V);
  const bool vec = out_vec(rv, out);
  const int g_lo = tile * (kLpTileEntries / kGroup);
  uint32_t w[kLpPer][RVT::kWords];
#pragma unroll
  for (int u = 0; u < kLpPer; ++u) {
    const int g = g_lo + (int)threadIdx.x + u * kLpThreads;
    if (!bad && g < rv.NG && rv.full(g)) rv.load_words(g, w[u], pol);
  }
#pragma unroll
  for (int u = 0; u < kLpPer; ++u) {
    const int g = g_lo + (int)threadIdx.x + u * kLpThreads;
    if (g < rv.NG) write_group(rv, out, vec, g, w[u], [](float) { return true; }, value);
  }
}

template <typename TIn>
static ls_status launch_lp_write(const KernelArgs& a, int32_t n, cudaStream_t stream) {
  // tiles per row: enough for the entries, and for the groups a row of this
  // vocab can span (up to 31 entries of alignment before it)
  const int tiles = (int)((a.vocab + 31 + kLpTileEntries - 1) / kLpTileEntries);
  if ((int64_t)n * tiles > 0x7FFFFFFFll) return LS_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)n * tiles));
  cfg.blockDim = dim3(kLpThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, lp_write_kernel<TIn>, a, tiles) != cudaSuccess) return LS_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}

ls_status dispatch_lp_write(const KernelArgs& a, ls_dtype dtype, int32_t n, cudaStream_t stream) {
  return dtype == LS_DTYPE_BF16 ? launch_lp_write<bf16_tag>(a, n, stream) : launch_lp_write<float>(a, n, stream);
}

}  // namespace lsg
