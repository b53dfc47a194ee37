#pragma once
// ls_kernel.cuh -- GB300 (sm_103a) kernel of the token sampler and its
// host-side launch helpers.  Each ls_mode_*.cu instantiates `dispatch` for one
// mode (so the modes compile in parallel); ls_sampler.cu holds the C ABI.
//
// One CTA of 512 threads owns one sampled row.  The row is read from HBM once,
// with 256-bit loads, by a single streaming pass that keeps, per group of 16
// logits, the group maximum in shared memory and, per thread, a running
// maximum and (when the row needs it) the online sum of exp((l - max) / T).
// Everything after that pass touches only candidate groups -- groups whose
// maximum clears a provable lower bound of what can be kept or sampled -- and
// re-reads them from L2 once, into a shared-memory candidate list:
//   * exact top-k cut: an adaptive 11-bit radix select on order-preserving keys
//     (its first level built while collecting);
//   * exact top-p cut: the same select weighted by fixed-point masses (32-bit
//     atomics on (lo, hi) pairs, or per-key counts scaled by the key's weight,
//     deterministic run to run), joint = top-k cut first;
//   * Gumbel-max over the kept set with in-register Philox4x32-10 noise, only
//     for entries within the noise span of the best score of the maximum's ties.
// The log-probs mode runs the same selection and then writes the full [vocab]
// row of log-probs; the fused mode does both (and the raw log-prob of the
// sampled id) from the same pass.
//
// The behaviour follows "core.inference.sampling.base" (Sampling.sample_kernel,
// Sampling.sample_speculative), "core.inference.sampling.flashinfer_sampling"
// (FlashInferSampling: per-step top-p-only / top-k-only / joint dispatch from
// host flags, log_probs_kernel) and the TokenSpeed "backends/triton.py" page
// (TritonSamplingBackend: Gumbel-max sampling from per-request pools).

#include <atomic>
#include <cfloat>
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "ls_device.cuh"
#include "ls_sampler.h"

namespace lsg {

enum MapMode { MAP_IDENTITY = 0, MAP_T2R = 1, MAP_SPEC = 2 };
// MODE_BOTH: ids, and from the same pass the processed log-prob rows and/or
// the selected token's log-prob under the raw logits.
enum Mode { MODE_SAMPLE = 0, MODE_LOGPROBS = 1, MODE_BOTH = 2 };
enum Route { ROUTE_NONE = 0, ROUTE_K = 1, ROUTE_P = 2, ROUTE_KP = 3 };

// Scalars of a deferred log-prob row (the row kernel leaves them for
// lp_write_kernel): kept = v >= lo; value = (v - M) / T - lnS for T > 0, the
// constant -lnS for T == 0 (rows whose kept set is the maximum's ties); M NaN
// marks an error row (NaN throughout).
struct alignas(16) LpRow {
  float M, T, lnS, lo;
};

struct KernelArgs {
  const void* logits;
  int64_t logits_rows, vocab, stride;
  const int32_t* gather;
  const int32_t* t2r;
  int map_mode;
  int32_t spec_decode_rows;  // num_decode * (1 + S)
  int32_t spec_per_req;      // 1 + S
  int32_t spec_num_decode;
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const uint64_t* seed;
  int32_t num_requests;
  uint64_t step;
  const uint64_t* step_ptr;  // when not NULL the step word is read from device memory
  int32_t* out_ids;
  int32_t* out_t2r;
  float* out_lp;   // log-prob rows (MODE_LOGPROBS; MODE_BOTH when not NULL)
  float* out_sel;  // raw log-prob of the sampled id per row (MODE_BOTH, when not NULL)
  int32_t* error_word;
  int32_t cand_cap;   // capacity of the shared-memory candidate list
  int32_t gslot_cap;  // group-maximum slots of one CTA's slice (split sampler)
  int32_t ent_cap;    // capacity of the candidate-entry list (split sampler)
  int32_t pool_cap;   // captured-group slots shared by the warps once their own are full (split sampler)
  LpRow* lp_rows;     // when not NULL the log-prob rows are written by lp_write_kernel from these
};

constexpr int kWarpList = 128;  // candidate groups a warp lists before loading them
constexpr int kTieList = 32;    // ties of the maximum recorded while collecting
// Slack of the top-p candidate bound: the entries below it carry at most
// e^-kTopPSlack of the mass that the cut leaves out.  The bound decides only
// which entries are examined first; a build may override it (a negative slack
// puts the bound above the cut, so every top-p row takes the full re-select).
#ifndef LS_TOPP_SLACK
#define LS_TOPP_SLACK 0.25f
#endif
constexpr float kTopPSlack = LS_TOPP_SLACK;

// Group-maximum slots of a row: worst-case row alignment, rounded up to whole
// 16-byte vectors (the candidate list that follows stays 16-byte aligned).
__host__ __device__ inline int64_t group_slots(int64_t vocab) {
  return ((vocab + 2 * kGroup - 1) / kGroup + 3) & ~(int64_t)3;
}

// Fixed part of the dynamic shared memory; the group maxima follow it.
struct alignas(16) Shared {
  // Histogram: u32 counts, or masses as (lo, hi) u32 pairs updated with
  // carry-propagating 32-bit atomics (shared-memory 64-bit adds are not
  // native and degrade badly under contention).
  unsigned int hist[2 * kBins];
  unsigned long long red_u64[kWarps];
  float red_f[kWarps];
  int red_i[kWarps];
  unsigned long long best;
  unsigned int acc[2];  // a count in acc[0], or a mass as a (lo, hi) pair
  unsigned long long cut_above;
  unsigned long long cut_total, cut_target;  // level total and (joint) target, from thread 0
  unsigned long long cut_mass;
  int cut_bin;
  int min_index;
  int cand_count;
  unsigned long long step;  // the Philox step word of the call
  int tie_count;        // ties of the maximum met while collecting
  int tie_j[kTieList];  // their vocabulary indices (the first kTieList)
  int glist[kWarps * kWarpList];  // candidate group indices, one slice per warp
  float red_m[kWarps];
  float red_s[kWarps];
  float red_s2[kWarps];  // raw (T = 1) mass per warp, for the selected log-prob
  float row_M, row_S, row_S2, row_gamma, row_Lp;  // row scalars from warp 0
};

// Exact 64-bit add into a (lo, hi) pair of u32 counters with two native
// 32-bit atomics: the thread whose addition wraps the low word carries one
// into the high word, so the pair ends at the exact sum in any order.
__device__ __forceinline__ void add_mass(unsigned int* pair, unsigned long long w) {
  const unsigned int lo = (unsigned int)w, hi = (unsigned int)(w >> 32);
  const unsigned int old = atomicAdd(pair, lo);
  const unsigned int carry = (old + lo < old) ? 1u : 0u;
  if (hi + carry) atomicAdd(pair + 1, hi + carry);
}
__device__ __forceinline__ unsigned long long read_mass(const unsigned int* pair) {
  return ((unsigned long long)pair[1] << 32) | pair[0];
}

// round(w * 2^40) for a weight w in [0, 1], from the float's bits with integer
// operations only (64-bit float/integer conversions run on the slow FP64
// pipe).  Weights below 2^-41 give 0.
// Branch-free: a right shift by r >= 25 (weights below 2^-40 and the clamp
// at 63) leaves 0, since mant + 2^(r-1) < 2^r.
__device__ __forceinline__ unsigned long long mass_fixed(float w) {
  const uint32_t b = __float_as_uint(w);
  const int e = (int)((b >> 23) & 0xFFu);
  const unsigned long long mant = (unsigned long long)((b & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 110;  // w * 2^40 = mant * 2^(e - 127 - 23 + 40)
  const int r = min(max(-sh, 0), 63);
  const unsigned long long up = mant << min(max(sh, 0), 63);
  const unsigned long long dn = (mant + ((1ull << r) >> 1)) >> r;
  return e == 0 ? 0ull : sh >= 0 ? up : dn;
}

// ---------------------------------------------------------------------------
// Row view: groups of 16 logits aligned to the group size in bytes, so that
// every interior group is one (bf16) or two (fp32) aligned 256-bit loads.
// Group g covers row entries [16 g - off, 16 g - off + 16); entries outside
// [0, vocab) read as -inf.
// ---------------------------------------------------------------------------
template <typename TIn>
struct RowView;

__device__ __forceinline__ void ld256(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

// The same load under an L2 eviction policy (createpolicy): the log-prob
// modes keep the row in L2 for the write pass (evict_last) and let that pass's
// re-read go first (evict_first); sampling streams evict_first.
__device__ __forceinline__ void ld256_hint(const void* p, uint32_t (&r)[8], uint64_t policy) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p), "l"(policy));
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

template <>
struct RowView<bf16_tag> {
  static constexpr int kBytes = 2;
  const uint16_t* row;
  const unsigned char* base;  // group 0, aligned to 32 bytes
  int off;
  int64_t V;
  int NG;
  __device__ __forceinline__ void init(const void* logits, int64_t src, int64_t stride, int64_t vocab) {
    row = static_cast<const uint16_t*>(logits) + src * stride;
    const uintptr_t a = reinterpret_cast<uintptr_t>(row);
    base = reinterpret_cast<const unsigned char*>(a & ~uintptr_t(31));
    off = (int)((a - reinterpret_cast<uintptr_t>(base)) / 2);
    V = vocab;
    NG = (int)((off + vocab + kGroup - 1) / kGroup);
    g_full_lo = off > 0 ? 1 : 0;
    g_full_hi = (int)((off + vocab) / kGroup) - 1;
  }
  int g_full_lo, g_full_hi;  // groups lying entirely inside the row
  __device__ __forceinline__ int64_t index(int g, int e) const { return (int64_t)g * kGroup - off + e; }
  static constexpr int kWords = 8;
  // Raw words of a group that straddles the row's ends; outside entries read as -inf.
  __device__ __forceinline__ void load_words_partial(int g, uint32_t (&w)[kWords]) const {
    const int64_t j0 = index(g, 0);
#pragma unroll
    for (int q = 0; q < kWords; ++q) {
      const int64_t a = j0 + 2 * q, b = a + 1;
      const uint32_t lo = (a >= 0 && a < V) ? (uint32_t)row[a] : 0xFF80u;
      const uint32_t hi = (b >= 0 && b < V) ? (uint32_t)row[b] : 0xFF80u;
      w[q] = lo | (hi << 16);
    }
  }
  // Maximum of the 16 entries (NaN ignored unless all are NaN).
  __device__ __forceinline__ static float group_max(const uint32_t (&w)[kWords]) {
    const uint32_t a = bmax2(bmax2(w[0], w[1]), bmax2(w[2], w[3]));
    const uint32_t b = bmax2(bmax2(w[4], w[5]), bmax2(w[6], w[7]));
    const uint32_t m = bmax2(a, b);
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  // Bit e set when entry e is >= lo (NaN never).
  __device__ __forceinline__ static uint32_t ge_mask(const uint32_t (&w)[kWords], float lo) {
    uint32_t m = 0u;
#pragma unroll
    for (int q = 0; q < kWords; ++q) {
      m |= (__uint_as_float(w[q] << 16) >= lo ? 1u : 0u) << (2 * q);
      m |= (__uint_as_float(w[q] & 0xFFFF0000u) >= lo ? 1u : 0u) << (2 * q + 1);
    }
    return m;
  }
  // Entry e of the group for an index known at compile time.
  __device__ __forceinline__ static float element_at(const uint32_t (&w)[kWords], int e) {
    return __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
  }
  // Entry e of the group (a select chain, so the words stay in registers).
  __device__ __forceinline__ static float element(const uint32_t (&w)[kWords], int e) {
    uint32_t word = w[0];
#pragma unroll
    for (int q = 1; q < kWords; ++q) word = select_word(word, w[q], (e >> 1) == q);
    return __uint_as_float((e & 1) ? (word & 0xFFFF0000u) : (word << 16));
  }
  // Packed partial sums of 2^(v c - r) over the 16 entries.
  __device__ __forceinline__ static f32x2 exp_sum(const uint32_t (&w)[kWords], f32x2 c2, f32x2 nr2) {
    f32x2 s0 = 0ull, s1 = 0ull;
#pragma unroll
    for (int q = 0; q < kWords; ++q) {
      const f32x2 t = fma2(pack2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xFFFF0000u)), c2, nr2);
      float t0, t1;
      unpack2(t, t0, t1);
      const f32x2 e = pack2(ex2(t0), ex2(t1));
      if (q & 1)
        s1 = add2(s1, e);
      else
        s0 = add2(s0, e);
    }
    return add2(s0, s1);
  }
  __device__ __forceinline__ float at(int64_t j) const { return bf16_bits_to_float(row[j]); }
  __device__ __forceinline__ bool full(int g) const { return g >= g_full_lo && g <= g_full_hi; }
  __device__ __forceinline__ void load_words(int g, uint32_t (&w)[kWords]) const { ld256(base + (size_t)g * 32, w); }
  __device__ __forceinline__ void load_words(int g, uint32_t (&w)[kWords], uint64_t pol) const {
    ld256_hint(base + (size_t)g * 32, w, pol);
  }
  __device__ __forceinline__ static void unpack(const uint32_t (&w)[kWords], float (&v)[kGroup]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[2 * q] = __uint_as_float(w[q] << 16);
      v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ void load(int g, float (&v)[kGroup]) const {
    const int64_t j0 = index(g, 0);
    if (j0 >= 0 && j0 + kGroup <= V) {
      uint32_t r[kWords];
      load_words(g, r);
      unpack(r, v);
    } else {
#pragma unroll
      for (int e = 0; e < kGroup; ++e) {
        const int64_t j = j0 + e;
        v[e] = (j >= 0 && j < V) ? at(j) : kNegInf;
      }
    }
  }
};

template <>
struct RowView<float> {
  static constexpr int kBytes = 4;
  const float* row;
  const unsigned char* base;  // group 0, aligned to 64 bytes
  int off;
  int64_t V;
  int NG;
  __device__ __forceinline__ void init(const void* logits, int64_t src, int64_t stride, int64_t vocab) {
    row = static_cast<const float*>(logits) + src * stride;
    const uintptr_t a = reinterpret_cast<uintptr_t>(row);
    base = reinterpret_cast<const unsigned char*>(a & ~uintptr_t(63));
    off = (int)((a - reinterpret_cast<uintptr_t>(base)) / 4);
    V = vocab;
    NG = (int)((off + vocab + kGroup - 1) / kGroup);
    g_full_lo = off > 0 ? 1 : 0;
    g_full_hi = (int)((off + vocab) / kGroup) - 1;
  }
  int g_full_lo, g_full_hi;  // groups lying entirely inside the row
  __device__ __forceinline__ int64_t index(int g, int e) const { return (int64_t)g * kGroup - off + e; }
  static constexpr int kWords = 16;
  __device__ __forceinline__ void load_words_partial(int g, uint32_t (&w)[kWords]) const {
    const int64_t j0 = index(g, 0);
#pragma unroll
    for (int q = 0; q < kWords; ++q) {
      const int64_t j = j0 + q;
      w[q] = (j >= 0 && j < V) ? __float_as_uint(row[j]) : 0xFF800000u;
    }
  }
  __device__ __forceinline__ static float group_max(const uint32_t (&w)[kWords]) {
    float v[kGroup];
#pragma unroll
    for (int q = 0; q < kGroup; ++q) v[q] = __uint_as_float(w[q]);
    const float a = fmax3(v[0], v[1], v[2]), b = fmax3(v[3], v[4], v[5]), c = fmax3(v[6], v[7], v[8]);
    const float d = fmax3(v[9], v[10], v[11]), e = fmax3(v[12], v[13], v[14]);
    return fmaxf(fmax3(a, b, c), fmax3(d, e, v[15]));
  }
  __device__ __forceinline__ static uint32_t ge_mask(const uint32_t (&w)[kWords], float lo) {
    uint32_t m = 0u;
#pragma unroll
    for (int q = 0; q < kWords; ++q) m |= (__uint_as_float(w[q]) >= lo ? 1u : 0u) << q;
    return m;
  }
  __device__ __forceinline__ static float element_at(const uint32_t (&w)[kWords], int e) {
    return __uint_as_float(w[e]);
  }
  __device__ __forceinline__ static float element(const uint32_t (&w)[kWords], int e) {
    uint32_t word = w[0];
#pragma unroll
    for (int q = 1; q < kWords; ++q) word = select_word(word, w[q], e == q);
    return __uint_as_float(word);
  }
  __device__ __forceinline__ static f32x2 exp_sum(const uint32_t (&w)[kWords], f32x2 c2, f32x2 nr2) {
    f32x2 s0 = 0ull, s1 = 0ull;
#pragma unroll
    for (int q = 0; q < kWords / 2; ++q) {
      const f32x2 t = fma2(pack2(__uint_as_float(w[2 * q]), __uint_as_float(w[2 * q + 1])), c2, nr2);
      float t0, t1;
      unpack2(t, t0, t1);
      const f32x2 e = pack2(ex2(t0), ex2(t1));
      if (q & 1)
        s1 = add2(s1, e);
      else
        s0 = add2(s0, e);
    }
    return add2(s0, s1);
  }
  __device__ __forceinline__ float at(int64_t j) const { return row[j]; }
  __device__ __forceinline__ bool full(int g) const { return g >= g_full_lo && g <= g_full_hi; }
  __device__ __forceinline__ void load_words(int g, uint32_t (&w)[kWords]) const {
    ld256(base + (size_t)g * 64, *reinterpret_cast<uint32_t(*)[8]>(&w[0]));
    ld256(base + (size_t)g * 64 + 32, *reinterpret_cast<uint32_t(*)[8]>(&w[8]));
  }
  __device__ __forceinline__ void load_words(int g, uint32_t (&w)[kWords], uint64_t pol) const {
    ld256_hint(base + (size_t)g * 64, *reinterpret_cast<uint32_t(*)[8]>(&w[0]), pol);
    ld256_hint(base + (size_t)g * 64 + 32, *reinterpret_cast<uint32_t(*)[8]>(&w[8]), pol);
  }
  __device__ __forceinline__ static void unpack(const uint32_t (&w)[kWords], float (&v)[kGroup]) {
#pragma unroll
    for (int q = 0; q < kGroup; ++q) v[q] = __uint_as_float(w[q]);
  }
  __device__ __forceinline__ void load(int g, float (&v)[kGroup]) const {
    const int64_t j0 = index(g, 0);
    if (j0 >= 0 && j0 + kGroup <= V) {
      uint32_t r[kWords];
      load_words(g, r);
      unpack(r, v);
    } else {
#pragma unroll
      for (int e = 0; e < kGroup; ++e) {
        const int64_t j = j0 + e;
        v[e] = (j >= 0 && j < V) ? at(j) : kNegInf;
      }
    }
  }
};

template <typename TIn>
struct KeyOf {
  using type = KeyOps<TIn>;
};

__device__ __forceinline__ float max16(const float (&v)[kGroup]) {
  float a = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
  float b = fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7]));
  float c = fmaxf(fmaxf(v[8], v[9]), fmaxf(v[10], v[11]));
  float d = fmaxf(fmaxf(v[12], v[13]), fmaxf(v[14], v[15]));
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

// Calls f(value, vocabulary index) for each entry >= lo of group g, in
// order: one mask over the group's words, then a single call site for f (an
// unrolled loop would copy f, often a Gumbel scorer with its Philox rounds,
// sixteen times into the caller's code).
template <typename RV, typename F>
__device__ __forceinline__ void each_in_group(const RV& rv, int g, float lo, F&& f) {
  uint32_t w[RV::kWords];
  if (rv.full(g))
    rv.load_words(g, w);
  else
    rv.load_words_partial(g, w);
  uint32_t mm = RV::ge_mask(w, lo);
  // One trip count for the lanes that arrive together: a loop over each
  // lane's own bits diverges, and took about 1.6x as long on flat rows.
  const int trips = __reduce_max_sync(__activemask(), (unsigned)__popc(mm));
#pragma unroll 1
  for (int it = 0; it < trips; ++it) {
    if (mm != 0u) {
      const int e = __ffs(mm) - 1;
      mm &= mm - 1u;
      f(RV::element(w, e), rv.index(g, e));
    }
  }
}

// Visit every row entry whose value is >= lo (NaN never qualifies), looking
// only at groups whose maximum is >= lo.  Candidate groups are re-read from
// global memory (normally still in L2 after the streaming pass).
template <typename TIn, typename F>
__device__ __forceinline__ void visit_candidates(const RowView<TIn>& rv, const float* gmax, float lo, F&& f) {
  for (int g = threadIdx.x; g < rv.NG; g += kThreads)
    if (gmax[g] >= lo) each_in_group(rv, g, lo, f);
}

// The row entries that later phases examine.  After the streaming pass one
// visit of the candidate groups copies every entry >= the row's candidate
// bound into a shared-memory list (value, index); all later phases then read
// that list.  If the list would overflow, phases fall back to re-reading the
// candidate groups from global memory.
// Total mass 2^(v c - R) of a row with NaN entries (read as -inf): a second
// pass over the row, off the common path.  All threads call it.
template <typename TIn>
__device__ float total_mass_nan(const RowView<TIn>& rv, float c, float R, float* red) {
  float nacc = 0.f;
  for (int g = threadIdx.x; g < rv.NG; g += kThreads) {
    float v[kGroup];
    rv.load(g, v);
#pragma unroll
    for (int q = 0; q < kGroup; ++q) {
      const float x = v[q] == v[q] ? v[q] : kNegInf;
      nacc += ex2(fmaf(x, c, -R));
    }
  }
  return block_reduce(nacc, OpAddF(), red);
}

template <typename TIn>
struct Cands {
  const RowView<TIn>* rv;
  const float* gmax;
  const float* lv;    // values
  const int32_t* lj;  // vocabulary indices
  int count;
  bool listed;
  template <typename F>
  __device__ __forceinline__ void each(float lo, F&& f) const {
    if (listed) {
      for (int c = threadIdx.x; c < count; c += kThreads) {
        const float v = lv[c];
        if (v >= lo) f(v, (int64_t)lj[c]);
      }
    } else {
      visit_candidates(*rv, gmax, lo, f);
    }
  }
};

// Gumbel-max over the kept entries with value >= lo, given in sh.best the
// exact score of the best of the maximum's ties (always kept): s_lb, a lower
// bound of the winner's score.  Only entries with z >= s_lb - 16.6356 can
// still win (g <= 16.6356); of those, an entry needs g >= s_lb - z, i.e.
// u >= exp(-exp(z - s_lb)).  That test (taken 1e-3 looser in g) runs on the
// Philox word alone, and only entries passing it compute the two logarithms.
// Leaves the winner's key in sh.best.
// One Philox block yields the noise words of four consecutive vocabulary
// entries; a thread walking consecutive entries reuses it.
struct PhiloxCache {
  uint32_t id = 0xFFFFFFFFu;
  uint4 blk = make_uint4(0u, 0u, 0u, 0u);
  __device__ __forceinline__ uint32_t word(uint64_t seed, uint64_t step, uint32_t row, int64_t j) {
    const uint32_t b = (uint32_t)((uint64_t)j >> 2);
    if (b != id) {
      id = b;
      blk = philox4x32_10(make_uint4(b, row, (uint32_t)step, (uint32_t)(step >> 32)),
                          make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
    }
    const uint32_t ln = (uint32_t)j & 3u;
    return ln == 0 ? blk.x : ln == 1 ? blk.y : ln == 2 ? blk.z : blk.w;
  }
};

// Exact Gumbel score of entry j (value x) raised into *best.
__device__ __forceinline__ void score_entry(unsigned long long* best, float x, float T, uint64_t seed, uint64_t step,
                                         uint32_t row, int64_t j) {
  atomicMax(best, argmax_key(__fdiv_rn(x, T) + gumbel_of_word(noise_word(seed, step, row, j)), j));
}

template <typename TIn>
__device__ void gumbel_argmax(Shared& sh, const Cands<TIn>& cs, float M, float lo, float T, uint64_t seed,
                              uint64_t step, uint32_t row) {
  using RVT = RowView<TIn>;
  const float s_lb = f32_from_key((uint32_t)(sh.best >> 32));
  // z >= s_lb - 16.6356, in logit units (T > 0), lowered by a rounding margin
  float lb = (s_lb - 16.6366f) * T;
  lb -= fabsf(lb) * 1e-5f + 1e-30f;
  const float lo2 = fmaxf(lo, lb);
  PhiloxCache pc;
  auto test_word = [&](float v, int64_t j, uint32_t x) {
    const float z = __fdiv_rn(v, T);
    const float need = s_lb - z - 1e-3f;
    const float thr = ex2(-ex2(-need * kLog2e) * kLog2e) * (1.f - 4e-7f);
    const float u = __uint2float_rn(((x >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
    if (u >= thr) atomicMax(&sh.best, argmax_key(z + gumbel_of_word(x), j));
  };
  auto test = [&](float v, int64_t j) { test_word(v, j, pc.word(seed, step, row, j)); };
  if (cs.listed) {
    // each thread walks a contiguous run of the list (entries of one group are
    // consecutive there), so neighbouring entries share Philox blocks
    const int per = (cs.count + kThreads - 1) / kThreads;
    const int c0 = threadIdx.x * per, c1 = min(cs.count, c0 + per);
#pragma unroll 1
    for (int q = c0; q < c1; ++q) {
      const float v = cs.lv[q];
      if (v >= lo2 && v < M) test(v, (int64_t)cs.lj[q]);
    }
  } else {
    // Candidate groups re-read from global memory (normally L2), the next
    // one in flight while the current one is tested.  An interior group
    // whose first index is a multiple of 4 spans exactly four Philox blocks:
    // they are drawn together (four independent chains), and a group-level
    // threshold taken at the group's largest z rejects most entries with one
    // integer compare of their uniform; survivors take the exact test.
    const RowView<TIn>& rv = *cs.rv;
    const uint2 key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
    auto next = [&](int g) {
      while (g < rv.NG && !(cs.gmax[g] >= lo2)) g += kThreads;
      return g;
    };
    auto load = [&](int g, uint32_t (&w)[RVT::kWords]) {
      if (rv.full(g))
        rv.load_words(g, w);
      else
        rv.load_words_partial(g, w);
    };
    constexpr bool kAhead = RVT::kWords <= 8;  // next group in flight (bf16: registers allow it)
    int g = next(threadIdx.x);
    uint32_t w[RVT::kWords];
    if (kAhead && g < rv.NG) load(g, w);
    while (g < rv.NG) {
      const int gn = next(g + kThreads);
      uint32_t wn[RVT::kWords];
      if (kAhead) {
        if (gn < rv.NG) load(gn, wn);
      } else {
        load(g, w);
      }
      const int64_t j0 = rv.index(g, 0);
      if (rv.full(g) && (j0 & 3) == 0) {
        // every entry of the group has z <= fl(gmax / T): its threshold is at
        // least the group's, so u below the group's threshold rejects it
        const float zg = __fdiv_rn(cs.gmax[g], T);
        const float need_g = s_lb - zg - 1e-3f;
        const float thr_g = ex2(-ex2(-need_g * kLog2e) * kLog2e) * (1.f - 4e-7f);
        // u = (2 (x >> 9) + 1) 2^-24 >= thr_g  implies  2 (x >> 9) + 1 >= floor(thr_g 2^24)
        const uint32_t thr_i = (uint32_t)(thr_g * 16777216.f);
        const uint32_t b0 = (uint32_t)((uint64_t)j0 >> 2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two blocks (eight entries) at a time
          const uint4 p0 = philox4x32_10(make_uint4(b0 + 2 * h, row, (uint32_t)step, (uint32_t)(step >> 32)), key);
          const uint4 p1 = philox4x32_10(make_uint4(b0 + 2 * h + 1, row, (uint32_t)step, (uint32_t)(step >> 32)), key);
#pragma unroll
          for (int e8 = 0; e8 < 8; ++e8) {
            const int e = 8 * h + e8;
            const uint4 bq = e8 < 4 ? p0 : p1;
            const uint32_t x = (e & 3) == 0 ? bq.x : (e & 3) == 1 ? bq.y : (e & 3) == 2 ? bq.z : bq.w;
            const float v = RVT::element_at(w, e);
            if (v >= lo2 && v < M && (((x >> 9) << 1) | 1u) >= thr_i) test_word(v, j0 + e, x);
          }
        }
      } else {
        uint32_t mm = RVT::ge_mask(w, lo2);
#pragma unroll 1
        while (mm) {
          const int e = __ffs(mm) - 1;
          mm &= mm - 1u;
          const float v = RVT::element(w, e);
          if (v < M) test(v, rv.index(g, e));
        }
      }
      g = gn;
      if (kAhead) {
#pragma unroll
        for (int q = 0; q < RVT::kWords; ++q) w[q] = wn[q];
      }
    }
  }
  __syncthreads();
}

// Bin weights of one select level.  A bin holds a count (top-k), the exact
// fixed-point mass of its entries as a (lo, hi) pair (top-p, bins spanning
// several keys) or, when every bin is a single key, a count that is scaled
// here by that key's weight: the same fixed-point mass, since every entry of
// the bin has the same value.
enum BinMode { BIN_COUNT = 0, BIN_MASS = 1, BIN_KEY_COUNT = 2 };

// load() reads a bin's words, weight() turns them into its weight: a level
// issues every load of a thread before the first weight.
template <typename TIn>
struct BinWeight {
  const Shared* sh;
  int mode;
  uint32_t klo;  // key of bin 0 (BIN_KEY_COUNT)
  float c, R;
  __device__ __forceinline__ void load(int b, unsigned int& lo, unsigned int& hi) const {
    const bool pair = mode == BIN_MASS;
    lo = sh->hist[pair ? 2 * b : b];
    hi = pair ? sh->hist[2 * b + 1] : 0u;
  }
  __device__ __forceinline__ unsigned long long weight(int b, unsigned int lo, unsigned int hi) const {
    if (mode == BIN_MASS) return ((unsigned long long)hi << 32) | lo;
    if (mode == BIN_COUNT) return lo;
    return (unsigned long long)lo * mass_fixed(ex2(fmaf(KeyOps<TIn>::value(klo + (uint32_t)b), c, -R)));
  }
};

// Find the highest bin b with above + (weight of bins >= b) >= target.
// Thread t holds bins nb-1-4t .. nb-4-4t; one block scan over the threads.
// With joint_p >= 0 the target becomes joint_p * (total weight of the level)
// (written back to `target`, the same in every thread).
// Writes sh.cut_bin (-1 when the total never reaches the target, possible
// only through rounding of a top-p target), sh.cut_above (weight strictly
// above bin b, including `above`) and sh.cut_mass (weight of bin b); returns
// the level's total weight.  Two block barriers.
template <typename W>
__device__ __forceinline__ unsigned long long find_cut_bin(Shared& sh, int nb, unsigned long long above,
                                                           unsigned long long& target, float joint_p,
                                                           const W& weight) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int top = nb - 1 - t * kBinsPerThread;
  // warps holding no bin only write a zero total and meet the barriers
  const bool has_bins = nb - 1 - warp * 32 * kBinsPerThread >= 0;
  unsigned long long w[kBinsPerThread], local = 0, incl = 0;
  if (has_bins) {
    unsigned int lo[kBinsPerThread], hi[kBinsPerThread];
#pragma unroll
    for (int q = 0; q < kBinsPerThread; ++q) weight.load(max(top - q, 0), lo[q], hi[q]);
#pragma unroll
    for (int q = 0; q < kBinsPerThread; ++q) {
      w[q] = top - q >= 0 ? weight.weight(top - q, lo[q], hi[q]) : 0ull;
      local += w[q];
    }
    incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += u;
    }
  }
  if (t == 0) sh.cut_bin = -1;
  if (lane == 31) sh.red_u64[warp] = incl;
  __syncthreads();
  if (has_bins) {
    unsigned long long base = 0, total = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      const unsigned long long x = sh.red_u64[i];
      base += i < warp ? x : 0ull;
      total += x;
    }
    if (joint_p >= 0.f) target = __float2ull_ru(joint_p * __ull2float_rn(total));
    if (target < 1ull) target = 1ull;
    if (t == 0) {
      sh.cut_total = total;
      sh.cut_target = target;
    }
    unsigned long long cum = above + base + incl - local;
    if (cum < target && cum + local >= target) {
#pragma unroll
      for (int q = 0; q < kBinsPerThread; ++q) {
        if (cum + w[q] >= target) {
          sh.cut_bin = top - q;
          sh.cut_above = cum;
          sh.cut_mass = w[q];
          break;
        }
        cum += w[q];
      }
    }
  }
  __syncthreads();
  target = sh.cut_target;  // the same in every thread (set by warp 0, which always holds bins)
  return sh.cut_total;
}

struct SelResult {
  uint32_t key;                 // kept set: entries with key >= this
  unsigned long long mass_ge;   // weight of the kept entries
  bool short_total;             // the whole range weighs less than the target
};

// Exact threshold select over the row entries with keys in [klo, khi], given
// the weight `above` of the entries with larger keys: returns the largest key
// kappa such that above + (weight of entries with key in [kappa, khi]) >=
// target, where weight is 1 (top-k, target = k) or the fixed-point
// probability mass exp((l - M)/T) * 2^40 (top-p, `mass`).  With joint_p >= 0
// the target is joint_p * (total weight of the range).  Each level splits the
// remaining key range into at most 2048 bins: bf16 keys (16 bits) need at most
// two levels, fp32 keys at most three.  With `built` the first level's
// histogram (same binning) is already in shared memory.  If the total weight
// never reaches the target (possible only through rounding of a top-p target)
// the whole range is kept.
template <typename TIn>
__device__ SelResult radix_select(Shared& sh, const Cands<TIn>& cs, uint32_t klo, uint32_t khi,
                                  unsigned long long target, float joint_p, float R, float c,
                                  unsigned long long above, bool mass, bool built) {
  using K = KeyOps<TIn>;
  unsigned long long mass_at = 0;
  for (;;) {
    const uint32_t width = khi - klo;
    const int bits = width ? 32 - __clz(width) : 0;
    const int shift = bits > kBinBits ? bits - kBinBits : 0;
    const int nb = (int)(width >> shift) + 1;
    const int mode = !mass ? BIN_COUNT : shift == 0 ? BIN_KEY_COUNT : BIN_MASS;
    if (!built) {
      for (int b = threadIdx.x; b < (mode == BIN_MASS ? 2 * nb : nb); b += kThreads) sh.hist[b] = 0u;
      __syncthreads();
      const float lo = K::value(klo), hi = K::value(khi);
      const uint32_t base = klo, top = khi;
      cs.each(lo, [&](float v, int64_t) {
        const uint32_t kk = K::key(v);
        if (v <= hi && kk >= base && kk <= top) {
          const int bin = (int)((kk - base) >> shift);
          if (mode == BIN_MASS)
            add_mass(&sh.hist[2 * bin], mass_fixed(ex2(fmaf(v, c, -R))));
          else
            atomicAdd(&sh.hist[bin], 1u);
        }
      });
      __syncthreads();
    }
    built = false;
    const unsigned long long total =
        find_cut_bin(sh, nb, above, target, joint_p, BinWeight<TIn>{&sh, mode, klo, c, R});
    joint_p = -1.f;
    const int b = sh.cut_bin;
    if (b < 0) return SelResult{klo, above + total, true};  // only reachable on the first level
    above = sh.cut_above;
    mass_at = sh.cut_mass;
    const uint32_t nlo = klo + ((uint32_t)b << shift);
    const unsigned long long nhi = (unsigned long long)nlo + ((1ull << shift) - 1ull);
    khi = nhi < (unsigned long long)khi ? (uint32_t)nhi : khi;
    klo = nlo;
    if (klo >= khi) break;  // a single key left
    __syncthreads();        // the cut fields and the histogram are rewritten by the next level
  }
  return SelResult{klo, above + mass_at, false};
}

// Top-p cut whose first level was binned by value (bin_of_key(k): the bin of
// the entries with key k, non-decreasing in k) rather than by key range: the
// first level's cut bin, then radix_select over exactly that bin's keys (the
// keys k in [klo1, khi1] with bin_of_key(k) == b, found by bisection on the
// monotone bin function).  Same semantics as radix_select over [klo1, khi1].
template <typename TIn, typename BinOfKey>
__device__ SelResult value_binned_select(Shared& sh, const Cands<TIn>& cs, uint32_t klo1, uint32_t khi1,
                                         unsigned long long target, float R, float c, BinOfKey bin_of_key) {
  unsigned long long tg = target;
  const unsigned long long total = find_cut_bin(sh, kBins, 0ull, tg, -1.f, BinWeight<TIn>{&sh, BIN_MASS, klo1, c, R});
  const int b = sh.cut_bin;
  if (b < 0) return SelResult{klo1, total, true};
  const unsigned long long above = sh.cut_above, mass_b = sh.cut_mass;
  // smallest key in [klo1, khi1] whose bin is >= bb (khi1 + 1 if none)
  auto first_key = [&](int bb) {
    uint64_t lo = klo1, hi = (uint64_t)khi1 + 1u;
    while (lo < hi) {
      const uint64_t mid = lo + (hi - lo) / 2u;
      if (bin_of_key((uint32_t)mid) >= bb)
        hi = mid;
      else
        lo = mid + 1u;
    }
    return lo;
  };
  const uint32_t klo = (uint32_t)first_key(b);
  const uint32_t khi = b + 1 < kBins ? (uint32_t)(first_key(b + 1) - 1u) : khi1;
  __syncthreads();  // every thread has read the cut fields before the next level rewrites them
  if (klo >= khi) return SelResult{klo, above + mass_b, false};  // the bin holds one key
  return radix_select<TIn>(sh, cs, klo, khi, target, -1.f, R, c, above, true, false);
}

// Exact cuts over a short candidate list (at most kSmallList entries, all of
// them listed) by direct counting: for each entry x, the number and the
// fixed-point mass of the listed entries strictly above it.  x survives the
// top-k cut iff fewer than k entries lie above it, and a top-p cut with
// target t iff the mass strictly above it is below t -- the kept sets of
// radix_select (the largest key whose upward-closed weight reaches the
// target), without its per-level histograms and scans.  With k_on and p_on
// the top-p target is p times the weight of the top-k set, as in the joint
// level of radix_select.  Four threads share an entry, a quarter of the list
// each.  The histogram area is the scratch.  Returns the final cut; for a
// top-p cut alone whose candidates weigh less than the target, the short
// result radix_select gives (the whole range from klo kept).
constexpr int kSmallList = 128;
static_assert(kThreads == 4 * kSmallList, "four threads per listed entry");

template <typename TIn>
__device__ SelResult small_select(Shared& sh, const Cands<TIn>& cs, uint32_t klo, bool k_on, bool p_on, int32_t k,
                                  float joint_p, unsigned long long target, float R, float c) {
  using K = KeyOps<TIn>;
  unsigned long long* ms = reinterpret_cast<unsigned long long*>(sh.hist);  // [kSmallList] masses
  unsigned int* pc = sh.hist + 2 * kSmallList;                              // [4][kSmallList] counts above
  unsigned long long* pm = ms + 3 * kSmallList;                             // [4][kSmallList] masses above
  unsigned long long* cell = pm + 4 * kSmallList;                           // sum, kept mass, lowest kept key
  static_assert(7 * kSmallList + 3 <= kBins, "scratch inside the histogram");
  const int n = cs.count, t = threadIdx.x, lane = t & 31;
  auto add_u64 = [](unsigned long long a, unsigned long long b) { return a + b; };
  auto sum_into = [&](unsigned long long w, unsigned long long* dst) {
    w = warp_reduce(w, add_u64);
    if (lane == 0 && w) atomicAdd(dst, w);
  };
  if (t < n) ms[t] = mass_fixed(ex2(fmaf(cs.lv[t], c, -R)));
  if (t < 3) cell[t] = t == 2 ? 0xFFFFFFFFull : 0ull;
  __syncthreads();
  const int x = t & (kSmallList - 1), q = t / kSmallList;
  const bool own = q == 0 && x < n;  // the thread that decides entry x
  const float vx = x < n ? cs.lv[x] : 0.f;
  if (x < n) {
    unsigned int cnt = 0u;
    unsigned long long m = 0ull;
    const int y1 = min(n, (q + 1) * (kSmallList / 4));
    for (int y = q * (kSmallList / 4); y < y1; ++y) {
      const bool gt = cs.lv[y] > vx;
      cnt += gt ? 1u : 0u;
      m += gt ? ms[y] : 0ull;
    }
    pc[q * kSmallList + x] = cnt;
    pm[q * kSmallList + x] = m;
  }
  // the candidates' total mass (top-p alone) or the top-k set's (joint)
  __syncthreads();
  unsigned int cgt = 0u;
  unsigned long long mgt = 0ull;
  const unsigned long long mx = own ? ms[x] : 0ull;
  if (own) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      cgt += pc[r * kSmallList + x];
      mgt += pm[r * kSmallList + x];
    }
  }
  bool keep = own && (!k_on || cgt < (unsigned int)k);
  if (!k_on || p_on) {
    sum_into(keep ? mx : 0ull, &cell[0]);
    __syncthreads();
    const unsigned long long w = cell[0];
    if (k_on) {
      target = __float2ull_ru(joint_p * __ull2float_rn(w));
      if (target < 1ull) target = 1ull;
    } else if (w < target) {
      __syncthreads();  // every thread has read the total before the histogram is reused
      return SelResult{klo, w, true};
    }
    keep = keep && mgt < target;
  }
  sum_into(keep ? mx : 0ull, &cell[1]);
  if (keep) atomicMin(reinterpret_cast<unsigned int*>(&cell[2]), K::key(vx));
  __syncthreads();
  const SelResult r{(uint32_t)cell[2], cell[1], false};
  __syncthreads();
  return r;
}

__device__ __forceinline__ void row_error(const KernelArgs& a, int64_t i, int mode, int err) {
  if (threadIdx.x == 0) {
    if (mode != MODE_LOGPROBS) a.out_ids[i] = -1;
    if (mode == MODE_BOTH && a.out_sel) a.out_sel[i] = __uint_as_float(0x7FC00000u);
    if (a.error_word) atomicOr(a.error_word, err);
  }
  if (mode == MODE_LOGPROBS || (mode == MODE_BOTH && a.out_lp)) {
    const float nan = __uint_as_float(0x7FC00000u);
    if (a.lp_rows) {
      if (threadIdx.x == 0) a.lp_rows[i] = LpRow{nan, 0.f, 0.f, 0.f};
      return;
    }
    float* out = a.out_lp + i * a.vocab;
    for (int64_t j = threadIdx.x; j < a.vocab; j += kThreads) out[j] = nan;
  }
}

// 16-byte store that is evicted first (the log-prob rows are written once and
// not read back here).
__device__ __forceinline__ void st_stream4(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// 8- or 16-byte load of four consecutive logits (no L1 allocation, an L2
// eviction policy).
__device__ __forceinline__ void ld_quad(const void* p, uint32_t (&r)[2], uint64_t pol) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
               : "=r"(r[0]), "=r"(r[1])
               : "l"(p), "l"(pol));
}
__device__ __forceinline__ void ld_quad(const void* p, uint32_t (&r)[4], uint64_t pol) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "l"(p), "l"(pol));
}
__device__ __forceinline__ float quad_at(const uint32_t (&r)[2], int e) {
  return __uint_as_float((e & 1) ? (r[e >> 1] & 0xFFFF0000u) : (r[e >> 1] << 16));
}
__device__ __forceinline__ float quad_at(const uint32_t (&r)[4], int e) { return __uint_as_float(r[e]); }

// Whether a row's outputs can go out as 16-byte stores: its groups' first
// entries land on 16-byte boundaries of `out` (the same for every group).
template <typename TIn>
__device__ __forceinline__ bool out_vec(const RowView<TIn>& rv, const float* out) {
  const uintptr_t oa = reinterpret_cast<uintptr_t>(out);
  return (oa & 3u) == 0u && (((oa >> 2) - (uintptr_t)rv.off) & 3u) == 0u;
}

// out[j] = kept(v_j) ? value(v_j) : -inf for the 16 entries of group g (words
// w, loaded already unless the group is ragged), four at a time as 16-byte
// streaming stores when vec, else one by one.
template <typename TIn, typename KeptF, typename ValF>
__device__ __forceinline__ void write_group(const RowView<TIn>& rv, float* out, bool vec, int g,
                                            uint32_t (&w)[RowView<TIn>::kWords], KeptF kept, ValF val) {
  using RVT = RowView<TIn>;
  const bool full = rv.full(g);
  if (!full) rv.load_words_partial(g, w);
  const int64_t j0 = rv.index(g, 0);
#pragma unroll
  for (int h = 0; h < kGroup / 4; ++h) {
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float v = RVT::element_at(w, 4 * h + e);
      o[e] = kept(v) ? val(v) : kNegInf;
    }
    if (vec && full) {
      st_stream4(out + j0 + 4 * h, o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t j = j0 + 4 * h + e;
        if (j >= 0 && j < rv.V) out[j] = o[e];
      }
    }
  }
}

// Write out[j] = kept(v_j) ? value(v_j) : -inf over the whole row, reading
// the row again (normally from L2).  When the row and the output allow it,
// entries go four at a time: a warp's loads and 16-byte streaming stores
// cover consecutive addresses (kWriteQuads quads of a thread in flight
// together); otherwise group by group with the streaming pass's 256-bit loads.
constexpr int kWriteQuads = 8;
template <typename TIn, typename KeptF, typename ValF>
__device__ __forceinline__ void write_row(const RowView<TIn>& rv, float* out, KeptF kept, ValF val) {
  using RVT = RowView<TIn>;
  constexpr int E = RVT::kBytes;
  constexpr int QW = E == 2 ? 2 : 4;
  const uint64_t pol = l2_evict_first_policy();  // the row's last use
  const int64_t V = rv.V;
  if ((reinterpret_cast<uintptr_t>(rv.row) & (4 * E - 1)) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const int64_t nq = V / 4;  // whole quads; the last 1-3 entries one by one
    for (int64_t q0 = threadIdx.x; q0 < nq; q0 += (int64_t)kWriteQuads * kThreads) {
      uint32_t w[kWriteQuads][QW];
#pragma unroll
      for (int u = 0; u < kWriteQuads; ++u) {
        const int64_t q = q0 + (int64_t)u * kThreads;
        if (q < nq) ld_quad(rv.row + 4 * q, w[u], pol);
      }
#pragma unroll
      for (int u = 0; u < kWriteQuads; ++u) {
        const int64_t q = q0 + (int64_t)u * kThreads;
        if (q < nq) {
          float o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = quad_at(w[u], e);
            o[e] = kept(v) ? val(v) : kNegInf;
          }
          st_stream4(out + 4 * q, o[0], o[1], o[2], o[3]);
        }
      }
    }
    for (int64_t j = 4 * nq + threadIdx.x; j < V; j += kThreads) {
      const float v = rv.at(j);
      out[j] = kept(v) ? val(v) : kNegInf;
    }
    return;
  }
  const bool vec = out_vec(rv, out);
  for (int g = threadIdx.x; g < rv.NG; g += kThreads) {
    uint32_t w[RVT::kWords];
    if (rv.full(g)) rv.load_words(g, w, pol);
    write_group(rv, out, vec, g, w, kept, val);
  }
}

// Value of a kept entry of a log-prob row: (v - M) / T - lnS, the division a
// multiplication by RN(1/T) while |(v - M) / T| < 256 (an error below
// 3 2^-24 256 + half an ulp of the result, inside the 1e-4 the log-probs are
// held to), the correctly rounded division beyond.
struct LpValue {
  float M, T, lnS, invT, lim;
  __device__ __forceinline__ float operator()(float v) const {
    const float d = v - M;
    return (fabsf(d) < lim ? d * invT : __fdiv_rn(d, T)) - lnS;
  }
};
__device__ __forceinline__ LpValue lp_value(float M, float T, float lnS) {
  return LpValue{M, T, lnS, __frcp_rn(T), 256.f * T};
}

template <typename TIn, int ROUTE, int MODE>
__global__ void __launch_bounds__(kThreads, 2) sampler_row_kernel(const KernelArgs a) {
  using K = KeyOps<TIn>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  float* gmax = reinterpret_cast<float*>(smem_raw + sizeof(Shared));
  const int tid = threadIdx.x;
  const int64_t ng_cap = group_slots(a.vocab);
  float* cand_v = gmax + ng_cap;
  int32_t* cand_j = reinterpret_cast<int32_t*>(cand_v + a.cand_cap);
  const int64_t i = blockIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's writes are visible

  // ---- row -> (logits row, request) ------------------------------------
  int err = 0;
  int64_t src = i;
  if (a.gather) {
    src = a.gather[i];
    if (src < 0 || src >= a.logits_rows) err |= LS_ROW_ERR_BAD_GATHER;
  }
  int64_t req = i;
  if (a.map_mode == MAP_T2R) {
    req = a.t2r[i];
  } else if (a.map_mode == MAP_SPEC) {
    req = i < a.spec_decode_rows ? i / a.spec_per_req : a.spec_num_decode + (i - a.spec_decode_rows);
  }
  if (a.out_t2r && tid == 0) a.out_t2r[i] = (int32_t)req;
  if (req < 0 || req >= a.num_requests) err |= LS_ROW_ERR_BAD_REQUEST;
  if (err) {
    row_error(a, i, MODE, err);
    return;
  }

  const int64_t V = a.vocab;
  RowView<TIn> rv;
  rv.init(a.logits, src, a.stride, V);

  // ---- streaming pass: group maxima, running max, online mass ----------
  // Weights are 2^(v c - R) with c = log2(e) / T and R = RN(max * c): every
  // mass in the row (total, candidate and kept masses) uses this one formula,
  // so the rounding of R cancels in each ratio the cuts compare.  Each thread
  // keeps its own reference r = RN(m c) for its running maximum m.
  // Two register stages: the loads of the next groups are in flight while
  // the current ones are reduced.  The first two stages are issued before
  // the request's parameters are read.
  using RV = RowView<TIn>;
  constexpr int U = RV::kBytes == 2 ? 2 : 1;  // groups per stage
  constexpr int STEP = U * kThreads;
  // log-prob modes: the row stays in L2 for the write pass (the rows in
  // flight fit there; the outputs are stored evict-first).  Sampling streams
  // evict-first: the row is needed again only by this call's candidate
  // re-reads, and the stream no longer pushes out of L2 what every call
  // reuses (this kernel's code among it: top_p 19.5 -> 19.0 us, speculative
  // 52.3 -> 49.8).
  const uint64_t keep = MODE == MODE_SAMPLE ? l2_evict_first_policy() : l2_evict_last_policy();
  auto issue = [&](int g0, uint32_t (&w)[U][RV::kWords]) {
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (rv.full(g0 + u * kThreads)) rv.load_words(g0 + u * kThreads, w[u], keep);
  };
  uint32_t wa[U][RV::kWords], wb[U][RV::kWords];
  issue(tid, wa);
  issue(tid + STEP, wb);

  const float T = a.temperature[req];
  const int32_t k = a.top_k[req];
  const float p = a.top_p[req];
  const bool greedy = !(T >= 1e-5f);
  const bool k_on = !greedy && (ROUTE & ROUTE_K) && k >= 1 && (int64_t)k < V;
  const bool p_on = !greedy && (ROUTE & ROUTE_P) && p < 0.99999f;
  constexpr bool kSample = MODE != MODE_LOGPROBS;  // an id per row
  const bool want_lp = MODE == MODE_LOGPROBS || (MODE == MODE_BOTH && a.out_lp != nullptr);
  const bool want_raw = MODE == MODE_BOTH && a.out_sel != nullptr;  // raw log-sum-exp of the row
  const bool need_sum = !greedy && !k_on && (p_on || want_lp);
  const float c = greedy ? 0.f : kLog2e / T;

  float m = kNegInf, r = 0.f, r2 = 0.f;
  f32x2 acc = 0ull, acc2 = 0ull;
  const f32x2 c2 = pack2(c, c);
  const f32x2 l2 = pack2(kLog2e, kLog2e);
  auto consume = [&](int g0, uint32_t (&w)[U][RV::kWords]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = g0 + u * kThreads;
      if (g < rv.NG) {
        if (!rv.full(g)) rv.load_words_partial(g, w[u]);
        const float gm = RV::group_max(w[u]);
        gmax[g] = gm;
        if (MODE == MODE_BOTH && want_raw) {
          // raw weights 2^(v log2 e - r2) beside the processed ones
          if (gm > m) {
            const float rn = __fmul_rn(gm, kLog2e);
            const float sc = ex2(r2 - rn);
            acc2 = m > kNegInf ? mul2(acc2, pack2(sc, sc)) : 0ull;
            r2 = rn;
          }
          if (gm > kNegInf) acc2 = add2(acc2, RV::exp_sum(w[u], l2, pack2(-r2, -r2)));
        }
        if (need_sum) {
          if (gm > m) {
            const float rn = __fmul_rn(gm, c);  // rounded: never fused into r - rn
            const float sc = ex2(r - rn);
            acc = m > kNegInf ? mul2(acc, pack2(sc, sc)) : 0ull;
            m = gm;
            r = rn;
          }
          if (gm > kNegInf) acc = add2(acc, RV::exp_sum(w[u], c2, pack2(-r, -r)));
        } else {
          m = fmaxf(m, gm);
        }
      }
    }
  };
  for (int g0 = tid; g0 < rv.NG; g0 += 2 * STEP) {
    consume(g0, wa);
    issue(g0 + 2 * STEP, wa);
    consume(g0 + STEP, wb);
    issue(g0 + 3 * STEP, wb);
  }
  // the next kernel on the stream may be scheduled now (it waits for this grid
  // to complete before it reads memory)
  asm volatile("griddepcontrol.launch_dependents;");
  // ---- one block reduction: row maximum, total mass, top-k bound --------
  const uint64_t seed = kSample ? a.seed[req] : 0ull;  // its latency overlaps the reduction
  // Each warp reduces its maximum, rescales every lane's sum to the warp's
  // reference RN(max * c) and adds; after one barrier every warp combines the
  // 16 warp results the same way (fixed order, so S is deterministic and the
  // same in every warp).  For a top-k row each of the w warps that streamed
  // groups (thread t streamed groups t, t + 512, ...; w = 16 unless the row
  // is short) also extracts the j-th largest of its 32 thread maxima,
  // j = ceil(k / w): those warps then hold >= j w >= k thread maxima (distinct
  // entries) at or above the smallest of those, gamma.
  const int wact = min(kWarps, (rv.NG + 31) / 32);
  {
    uint4* h4 = reinterpret_cast<uint4*>(sh.hist);
    for (int q = tid; q < 2 * kBins / 4; q += kThreads) h4[q] = make_uint4(0u, 0u, 0u, 0u);
  }
  const int lane = tid & 31;
  {
    const float mw = warp_max(m);
    float sw = 0.f;
    if (need_sum && mw > kNegInf) {
      float lo, hi;
      unpack2(acc, lo, hi);
      sw = m > kNegInf ? (lo + hi) * ex2(r - __fmul_rn(mw, c)) : 0.f;
      sw = warp_reduce(sw, OpAddF());
    }
    float sw2 = 0.f;
    if (MODE == MODE_BOTH && want_raw && mw > kNegInf) {
      float lo, hi;
      unpack2(acc2, lo, hi);
      sw2 = m > kNegInf ? (lo + hi) * ex2(r2 - __fmul_rn(mw, kLog2e)) : 0.f;
      sw2 = warp_reduce(sw2, OpAddF());
    }
    float gj = kNegInf;
    if (k_on && (tid >> 5) < wact && k <= 32 * wact) {
      const int jrank = (k + wact - 1) / wact;
      if (jrank <= 8) {  // a few dependent extractions of the warp maximum
        float cur = m;
        for (int t = 0; t < jrank; ++t) {
          gj = warp_max(cur);
          const unsigned holders = __ballot_sync(0xFFFFFFFFu, cur == gj);
          if (lane == __ffs(holders) - 1) cur = kNegInf;
        }
      } else {  // each lane's rank among the 32 (ties by lane), all shuffles independent
        int rank = 0;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
          const float o = __shfl_sync(0xFFFFFFFFu, m, l);
          rank += (o > m || (o == m && l < lane)) ? 1 : 0;
        }
        const unsigned at = __ballot_sync(0xFFFFFFFFu, rank == jrank - 1);
        gj = __shfl_sync(0xFFFFFFFFu, m, __ffs(at) - 1);
      }
    }
    if (lane == 0) {
      sh.red_m[tid >> 5] = mw;
      sh.red_s[tid >> 5] = sw;
      sh.red_s2[tid >> 5] = sw2;
      sh.red_f[tid >> 5] = gj;
    }
  }
  if (tid == 0) {
    sh.best = 0ull;
    sh.acc[0] = 0u;
    sh.acc[1] = 0u;
    sh.min_index = 0x7FFFFFFF;
    sh.cand_count = 0;
    sh.tie_count = 0;
    sh.step = kSample && a.step_ptr ? *a.step_ptr : a.step;  // kept in shared memory, read late
  }
  __syncthreads();
  // warp 0 combines the 16 warp results (fixed order: S is deterministic) and
  // derives the top-p bound's log; the other warps wait at one more barrier
  // instead of repeating that work
  if (tid < 32) {
    const float mq = lane < kWarps ? sh.red_m[lane] : kNegInf;
    const float Mw = warp_max(mq);
    const float gw = warp_min(lane < wact ? sh.red_f[lane] : kPosInf);
    float Sw = 0.f, S2w = 0.f, Lpw = kNegInf;
    if (Mw > kNegInf && Mw < kPosInf) {
      if (need_sum) {
        const float Rw = __fmul_rn(Mw, c);
        const float sq = lane < kWarps && mq > kNegInf ? sh.red_s[lane] * ex2(__fmul_rn(mq, c) - Rw) : 0.f;
        Sw = warp_reduce(sq, OpAddF());
        // entries below Lp = M + T (ln((1 - p) S / V) - slack) carry less than (1 - p) S e^-slack
        if (p_on && !k_on && Sw <= FLT_MAX) Lpw = Mw + T * (logf((1.f - p) * Sw / (float)V) - kTopPSlack);
      }
      if (MODE == MODE_BOTH && want_raw) {
        const float R2w = __fmul_rn(Mw, kLog2e);
        const float sq = lane < kWarps && mq > kNegInf ? sh.red_s2[lane] * ex2(__fmul_rn(mq, kLog2e) - R2w) : 0.f;
        S2w = warp_reduce(sq, OpAddF());
      }
    }
    if (lane == 0) {
      sh.row_M = Mw;
      sh.row_S = Sw;
      sh.row_S2 = S2w;
      sh.row_gamma = gw;
      sh.row_Lp = Lpw;
    }
  }
  __syncthreads();
  const float M = sh.row_M, gamma = sh.row_gamma;
  if (M == kNegInf) {
    row_error(a, i, MODE, LS_ROW_ERR_NO_FINITE);
    return;
  }
  const float R = __fmul_rn(M, c);  // reference exponent of the row (rounded product, never fused)
  float S = sh.row_S;
  float Lp = sh.row_Lp;
  const bool tie_only = greedy || M == kPosInf;  // no temperature-scaled distribution
  // raw mass S2 = sum 2^(v log2 e - R2), R2 = RN(M log2 e) (MODE_BOTH, selected log-prob)
  const float R2 = __fmul_rn(M, kLog2e);
  float S2 = sh.row_S2;
  if (MODE == MODE_BOTH && want_raw && M < kPosInf && !(S2 <= FLT_MAX)) S2 = total_mass_nan(rv, kLog2e, R2, sh.red_f);

  // ---- total mass when a NaN entry poisoned the online sum ---------------
  if (!tie_only && need_sum && !(S <= FLT_MAX)) {
    S = total_mass_nan(rv, c, R, sh.red_f);
    if (p_on && !k_on) Lp = M + T * (logf((1.f - p) * S / (float)V) - kTopPSlack);
  }

  // ---- candidate bound --------------------------------------------------
  // Every entry that a later phase needs is >= lc:
  //  * ties-only rows (greedy, +inf maximum): the maximum itself;
  //  * top-k: gamma (at least k entries are >= gamma);
  //  * top-p alone: the entries below Lp carry less than (1 - p) S e^-slack,
  //    so the cut lies above Lp (if rounding of S, or of Lp for a tiny T and
  //    large logits, ever beat the slack, the cut detects it: see there);
  //  * no filter: an entry with z more than the noise span below max z can
  //    never beat the maximum's perturbed score.
  const float lg = M - kGumbelSpan * T;
  float lc;
  int kind = 0;  // first-level histogram: 0 none, 1 count (top-k), 2 mass (top-p alone)
  if (tie_only) {
    lc = M;
  } else if (k_on) {
    lc = gamma > kNegInf ? gamma : -FLT_MAX;
    kind = 1;
  } else if (p_on) {
    lc = fminf(fmaxf(Lp, -FLT_MAX), M);
    kind = 2;
  } else {
    // Unfiltered rows build no list: sampling reads only the groups above its
    // noise bounds (the maximum's ties, then the pruned Gumbel pass) straight
    // from global memory, and unfiltered log-probs need no candidates at all.
    lc = kPosInf;
  }
  lc = fmaxf(lc, -FLT_MAX);
  const uint32_t key_max = K::key(M);
  const uint32_t klo1 = K::key(lc);
  const uint32_t width1 = key_max - klo1;
  const int bits1 = width1 ? 32 - __clz(width1) : 0;
  const int shift1 = bits1 > kBinBits ? bits1 - kBinBits : 0;
  // first select level, built while collecting (the binning radix_select uses)
  const int mode1 = kind == 1 ? BIN_COUNT : shift1 == 0 ? BIN_KEY_COUNT : BIN_MASS;
  // A top-p cut over a wide key range bins that first level by value, linearly
  // over [lc, M]: key-range bins put a flat bf16 row's thousands of candidates
  // into a few dozen of the 2048 bins, and their mass atomics serialised.
  const float vscale = (float)kBins / (M - lc);
  const bool vbin = kind == 2 && mode1 == BIN_MASS && vscale <= FLT_MAX;
  auto value_bin = [&](float v) {
    const float t = (v - lc) * vscale;
    return t <= 0.f ? 0 : t >= (float)(kBins - 1) ? kBins - 1 : (int)t;
  };
  // sampling rows score the maximum's ties while collecting
  const bool ties_in_take = kSample && !tie_only;

  // ---- collect: candidate groups -> entries >= lc -----------------------
  // Each thread tests the maxima of the groups it streamed; a warp prefix
  // lists the candidate groups (maximum >= lc) in the warp's own slice of the
  // group list, kWarpList at a time.  The warp loads the listed groups (two
  // per lane per round for bf16, one for fp32, all loads in flight at once)
  // and takes their entries >= lc: they are appended to the shared-memory
  // candidate list (one atomic per warp and round), feed the first select
  // level's histogram and, when sampling, the maximum's ties are recorded.
  // No block barrier until every warp is done.
  using RVT = RowView<TIn>;
  int count = 0;
  // Entry >= lc of a loaded group: append it to the list and feed the first
  // select level's histogram.
  // Every lane of the warp calls it; one trip count for the warp (a loop over
  // each lane's own bits diverges, and took about 1.6x as long on flat rows).
  auto take = [&](int g, const uint32_t (&w)[RVT::kWords], uint32_t mm, int at) {
    const int trips = __reduce_max_sync(__activemask(), (unsigned)__popc(mm));
#pragma unroll 1
    for (int it = 0; it < trips; ++it) {
      if (mm == 0u) continue;
      const int e = __ffs(mm) - 1;
      mm &= mm - 1u;
      const float x = RVT::element(w, e);
      if (at < a.cand_cap) {
        cand_v[at] = x;
        cand_j[at] = (int32_t)rv.index(g, e);
      }
      ++at;
      if (kind != 0) {
        const uint32_t kk = K::key(x);
        if (vbin) {
          add_mass(&sh.hist[2 * value_bin(x)], mass_fixed(ex2(fmaf(x, c, -R))));
        } else if (kk >= klo1 && kk <= key_max) {
          const int bin = (int)((kk - klo1) >> shift1);
          if (mode1 == BIN_MASS)
            add_mass(&sh.hist[2 * bin], mass_fixed(ex2(fmaf(x, c, -R))));
          else
            atomicAdd(&sh.hist[bin], 1u);
        }
      }
      if (ties_in_take && x >= M) {
        const int q = atomicAdd(&sh.tie_count, 1);
        if (q < kTieList) sh.tie_j[q] = (int)rv.index(g, e);
      }
    }
  };
  if (lc <= M) {
    int* wl = sh.glist + (tid >> 5) * kWarpList;
    // load the n listed groups of this warp (kPer per lane per round, all
    // loads in flight at once) and take their entries
    constexpr int kPer = RVT::kWords <= 8 ? 2 : 1;
    auto flush = [&](int n) {
      __syncwarp();
      for (int c0 = 0; c0 < n; c0 += 32 * kPer) {
        uint32_t w[kPer][RVT::kWords];
        int gg[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int cu = c0 + 32 * u + lane;
          gg[u] = cu < n ? wl[cu] : -1;
          if (gg[u] >= 0 && rv.full(gg[u])) rv.load_words(gg[u], w[u]);
        }
        uint32_t mm[kPer];
        int cnt = 0;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          mm[u] = 0u;
          if (gg[u] >= 0) {
            if (!rv.full(gg[u])) rv.load_words_partial(gg[u], w[u]);
            mm[u] = RVT::ge_mask(w[u], lc);
            cnt += __popc(mm[u]);
          }
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += t2;
        }
        int base = 0;
        if (lane == 31) base = atomicAdd(&sh.cand_count, incl);
        int at = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          take(gg[u], w[u], mm[u], at);
          at += __popc(mm[u]);
        }
      }
      __syncwarp();
    };
    // Each thread tests the maxima of its own groups (tid + 512 s, the ones
    // it streamed), 32 slots at a time; one warp prefix over the per-thread
    // counts places the candidate groups in the warp's list slice, which is
    // loaded and taken kWarpList groups at a time.
    const int nslots = (rv.NG + kThreads - 1) / kThreads;
    for (int sb = 0; sb < nslots; sb += 32) {
      const int send = min(32, nslots - sb);
      // eight maxima in flight (indices clamped into the row), then the tests
      uint32_t mask = 0u;
      for (int q0 = 0; q0 < send; q0 += 8) {
        float gm[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) gm[u] = gmax[min(tid + (sb + q0 + u) * kThreads, rv.NG - 1)];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int g = tid + (sb + q0 + u) * kThreads;
          mask |= (g < rv.NG && gm[u] >= lc ? 1u : 0u) << (q0 + u);
        }
      }
      const int cnt = __popc(mask);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t2;
      }
      const int wtot = __shfl_sync(0xFFFFFFFFu, incl, 31);
      for (int w0 = 0; w0 < wtot; w0 += kWarpList) {
        uint32_t mm = mask;
        int at = incl - cnt;
        while (mm) {
          const int q = __ffs(mm) - 1;
          mm &= mm - 1u;
          if (at >= w0 && at < w0 + kWarpList) wl[at - w0] = tid + (sb + q) * kThreads;
          ++at;
        }
        flush(min(kWarpList, wtot - w0));
      }
    }
    __syncthreads();
    count = sh.cand_count;
  }
  Cands<TIn> cs{&rv, gmax, cand_v, cand_j, count, lc <= M && count <= a.cand_cap};

  // The maximum's ties: lowest index (greedy), count (log-probs of ties-only
  // rows) or exact Gumbel score (sampling; the best is a lower bound of the
  // winner's score).  Sampling rows that collected candidates recorded their
  // ties there: one thread of the last warps scores each (those warps hold no
  // bin of a small first select level, whose scan leads warp 0; sh.best is
  // next read after the cut's barriers); only more than kTieList ties take a
  // pass over the list.
  const uint64_t step = sh.step;
  // A sampling row whose whole list fits one entry per thread scores every
  // candidate here, the last threads first (the first warps hold the cut's
  // bins): the kept set lies in the list, and an entry that can never win
  // (below the noise bound) may be scored too.  The ties' scores go to
  // sh.best at once, as below; after the cut the best kept score is a warp
  // maximum and one atomic per warp instead of a Gumbel pass.  Not in the
  // fused fp32 kernel, whose long write pass pays for the extra live state in
  // spills (1024 x 262144 fp32: 648 against 638 us a call).
  constexpr bool kPre = kSample && !(MODE == MODE_BOTH && RowView<TIn>::kBytes == 4);
  const bool pre = kPre && !tie_only && cs.listed && count <= kThreads;
  const int pe = kThreads - 1 - tid;  // this thread's entry
  float pv = kNegInf;
  unsigned long long pkey = 0ull;
  if (pre && pe < count) {
    pv = cand_v[pe];
    const int64_t j = cand_j[pe];
    pkey = argmax_key(__fdiv_rn(pv, T) + gumbel_of_word(noise_word(seed, step, (uint32_t)i, j)), j);
    if (pv >= M) atomicMax(&sh.best, pkey);
  }
  const int nties = ties_in_take && lc <= M ? sh.tie_count : -1;
  if (pre) {
    // the ties were scored with the list
  } else if (nties >= 0 && nties <= kTieList) {
    const int q = kThreads - 1 - tid;
    if (q < nties) score_entry(&sh.best, M, T, seed, step, (uint32_t)i, sh.tie_j[q]);
  } else if (tie_only || kSample) {
    cs.each(M, [&](float x, int64_t j) {
      if (MODE != MODE_SAMPLE && tie_only) atomicAdd(&sh.acc[0], 1u);
      if (kSample) {
        if (greedy) {
          atomicMin(&sh.min_index, (int)j);
        } else {
          const float z = M == kPosInf ? 0.f : __fdiv_rn(x, T);
          atomicMax(&sh.best, argmax_key(z + gumbel_of_word(noise_word(seed, step, (uint32_t)i, j)), j));
        }
      }
    });
    __syncthreads();
  }
  // Raw log-prob of the sampled entry: (v - M) - ln sum exp(v - M); the raw
  // masses carry the residual 2^(M log2 e - R2) of R2's rounding.  A +inf
  // maximum shares the probability among its +inf entries.
  auto selected_lp = [&](int32_t id) {
    const float v = rv.at(id);
    if (M == kPosInf) return v == kPosInf ? -logf((float)sh.acc[0]) : kNegInf;
    return (v - M) - (logf(S2) - fmaf(M, kLog2e, -R2) * 0.6931471805599453f);
  };
  if (tie_only) {
    if (kSample && tid == 0) {
      const int32_t id = greedy ? sh.min_index : argmax_index(sh.best);
      a.out_ids[i] = id;
      if (MODE == MODE_BOTH && want_raw) a.out_sel[i] = selected_lp(id);
    }
    if (want_lp) {
      const float lp = -logf((float)sh.acc[0]);
      if (a.lp_rows) {
        if (tid == 0) a.lp_rows[i] = LpRow{M, 0.f, -lp, M};
      } else {
        write_row(rv, a.out_lp + i * V, [&](float v) { return v >= M; }, [&](float) { return lp; });
      }
    }
    return;
  }

  // ---- exact top-k and top-p cuts ---------------------------------------
  uint32_t lo_key = K::key(-FLT_MAX);  // no filter: every finite entry
  unsigned long long kept_mass = 0ull;
  // a short list takes both cuts by direct counting
  const bool small = kind != 0 && cs.listed && count <= kSmallList;
  if (kind != 0) {
    // the first level's histogram was built while collecting
    const unsigned long long target =
        kind == 1 ? (unsigned long long)k : max(1ull, __float2ull_ru(fmaxf(p, 0.f) * S * kMassScale));
    SelResult r1 =
        small  ? small_select<TIn>(sh, cs, klo1, k_on, p_on, k, fmaxf(p, 0.f), target, R, c)
        : vbin ? value_binned_select<TIn>(sh, cs, klo1, key_max, target, R, c,
                                          [&](uint32_t kk) { return value_bin(K::value(kk)); })
               : radix_select<TIn>(sh, cs, klo1, key_max, target, -1.f, R, c, 0ull, kind == 2, true);
    if (kind == 2 && r1.short_total && lc > -FLT_MAX) {
      // The candidates weigh less than the top-p target, so the cut lies
      // below the bound: select again over every finite entry, visiting the
      // groups from global memory (the list holds only entries >= lc).  The
      // maximum's ties are all candidates, so their scores stand.
      cs.listed = false;
      r1 = radix_select<TIn>(sh, cs, K::key(-FLT_MAX), key_max, target, -1.f, R, c, 0ull, true, false);
    }
    lo_key = r1.key;
    kept_mass = r1.mass_ge;
  }
  if (k_on && p_on && !small) {
    const SelResult r2 =
        radix_select<TIn>(sh, cs, lo_key, key_max, 0ull, fmaxf(p, 0.f), R, c, 0ull, true, false);
    lo_key = r2.key;
    kept_mass = r2.mass_ge;
  }
  const float lo_val = K::value(lo_key);

  if (kSample) {
    // ---- Gumbel-max over the kept set ------------------------------------
    if (pre && cs.listed) {
      unsigned long long kk = pv >= lo_val ? pkey : 0ull;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long u = __shfl_xor_sync(0xFFFFFFFFu, kk, o);
        kk = u > kk ? u : kk;
      }
      if (lane == 0 && kk != 0ull) atomicMax(&sh.best, kk);
      __syncthreads();
    } else {
      gumbel_argmax(sh, cs, M, fmaxf(lo_val, lg), T, seed, step, (uint32_t)i);
    }
    if (tid == 0) {
      const int32_t id = argmax_index(sh.best);
      a.out_ids[i] = id;
      if (MODE == MODE_BOTH && want_raw) a.out_sel[i] = selected_lp(id);
    }
  }
  if (want_lp) {
    // ---- log-probs of the processed distribution -------------------------
    float lnS;
    if (p_on) {
      lnS = logf(__ull2float_rn(kept_mass) / kMassScale);
    } else if (k_on) {
      cs.each(lo_val, [&](float v, int64_t) { add_mass(sh.acc, mass_fixed(ex2(fmaf(v, c, -R)))); });
      __syncthreads();
      lnS = logf(__ull2float_rn(read_mass(sh.acc)) / kMassScale);
    } else {
      lnS = logf(S);
    }
    // The masses are 2^(v c - R) = exp((v - M) / T) * 2^(M c - R); remove the
    // exactly computable residual of R's rounding from the normaliser.
    lnS -= fmaf(M, c, -R) * 0.6931471805599453f;
    if (a.lp_rows) {
      if (tid == 0) a.lp_rows[i] = LpRow{M, T, lnS, lo_val};
    } else {
      write_row(rv, a.out_lp + i * V, [&](float v) { return v >= lo_val; }, lp_value(M, T, lnS));
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Shared memory of one CTA: fixed part, group maxima (worst-case row
// alignment), candidate list of `cap` (value, index) pairs.
static size_t smem_bytes(int64_t vocab, int cap) {
  const int64_t ng = group_slots(vocab);
  return sizeof(Shared) + (size_t)ng * sizeof(float) + (size_t)cap * (sizeof(float) + sizeof(int32_t));
}

// Candidate-list capacity: up to 8192 entries while a CTA stays within 96 KB
// of shared memory, never below 256.  Two such CTAs per SM leave at least
// 60 KB of the SM's 256 KB L1/shared array to L1, which the streaming loads
// need for their requests in flight: with 104 KB per CTA a plain 256-row
// bf16 read of this shape was measured a quarter slower.
static int cand_capacity(int64_t vocab) {
  constexpr size_t kPerCta = 96 * 1024;
  const size_t base = smem_bytes(vocab, 0);
  int cap = 8192;
  while (cap > 256 && base + (size_t)cap * 8 > kPerCta) cap -= 256;
  return cap;
}

constexpr int kMaxDevices = 64;

static int max_dyn_smem() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && (v = cache[dev].load(std::memory_order_relaxed)) > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

template <typename TIn, int ROUTE, int MODE>
static ls_status launch_rows(const KernelArgs& a, int32_t n, size_t smem, cudaStream_t stream) {
  auto kern = sampler_row_kernel<TIn, ROUTE, MODE>;
  // The dynamic shared-memory opt-in is set once per device and size class.
  static std::atomic<size_t> opted[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LS_ERR_CUDA;
  if (smem > 48 * 1024 && (dev < 0 || dev >= kMaxDevices || opted[dev].load(std::memory_order_relaxed) < smem)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return LS_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) opted[dev].store(smem, std::memory_order_relaxed);
  }
  // Programmatic dependent launch: the grid may be scheduled while the
  // previous kernel on the stream drains; every CTA waits for that kernel's
  // completion (griddepcontrol.wait) before it reads any memory.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return LS_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}

// The deferred log-prob write (ls_lpwrite.cu): every row's log-probs from
// the LpRow scalars the row kernel left in a.lp_rows, tiled over all SMs.
ls_status dispatch_lp_write(const KernelArgs& a, ls_dtype dtype, int32_t n, cudaStream_t stream);

template <int MODE>
ls_status dispatch(KernelArgs a, ls_dtype dtype, int route, int32_t n, cudaStream_t stream) {
  a.cand_cap = cand_capacity(a.vocab);
  const size_t smem = smem_bytes(a.vocab, a.cand_cap);
  const int lim = max_dyn_smem();
  if (lim <= 0) return LS_ERR_CUDA;
  if (smem > (size_t)lim) return LS_ERR_UNSUPPORTED;
  if (dtype == LS_DTYPE_BF16) {
    switch (route) {
      case ROUTE_NONE: return launch_rows<bf16_tag, ROUTE_NONE, MODE>(a, n, smem, stream);
      case ROUTE_K: return launch_rows<bf16_tag, ROUTE_K, MODE>(a, n, smem, stream);
      case ROUTE_P: return launch_rows<bf16_tag, ROUTE_P, MODE>(a, n, smem, stream);
      default: return launch_rows<bf16_tag, ROUTE_KP, MODE>(a, n, smem, stream);
    }
  }
  switch (route) {
    case ROUTE_NONE: return launch_rows<float, ROUTE_NONE, MODE>(a, n, smem, stream);
    case ROUTE_K: return launch_rows<float, ROUTE_K, MODE>(a, n, smem, stream);
    case ROUTE_P: return launch_rows<float, ROUTE_P, MODE>(a, n, smem, stream);
    default: return launch_rows<float, ROUTE_KP, MODE>(a, n, smem, stream);
  }
}

static bool params_ok(const ls_params* prm, bool need_seed) {
  return prm && prm->temperature && prm->top_k && prm->top_p && (!need_seed || prm->seed) && prm->num_requests >= 1;
}

static bool common_ok(const void* logits, ls_dtype dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride) {
  return logits && (dtype == LS_DTYPE_F32 || dtype == LS_DTYPE_BF16) && vocab >= 1 && row_stride >= vocab &&
         logits_rows >= 1 && vocab <= 0x7FFFFFF0ll;
}

static KernelArgs make_args(const void* logits, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                            const int32_t* gather, const ls_params* prm, uint64_t step, int32_t* error_word) {
  KernelArgs a{};
  a.logits = logits;
  a.logits_rows = logits_rows;
  a.vocab = vocab;
  a.stride = row_stride;
  a.gather = gather;
  a.temperature = prm->temperature;
  a.top_k = prm->top_k;
  a.top_p = prm->top_p;
  a.seed = prm->seed;
  a.num_requests = prm->num_requests;
  a.step = step;
  a.error_word = error_word;
  return a;
}

}  // namespace lsg
