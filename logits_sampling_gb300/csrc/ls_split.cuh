#pragma once
// ls_split.cuh -- the streaming sampler (ids only): one HBM pass per row that
// also collects everything the cuts and the Gumbel-max need, with a row split
// over a thread-block cluster of C CTAs when the batch is small.
//
// Row r is owned by cluster r (C = 1: a single CTA).  CTA q of the cluster
// streams a contiguous slice of the row's 16-logit groups with 256-bit loads
// (two register stages) and, in the same pass:
//   * keeps the slice maximum, the online sum of exp((l - max) / T) (top-p
//     rows) and each group's maximum (2 bytes, rounded up, in shared memory);
//   * top-k and top-p rows: appends to a shared-memory list every entry at or
//     above a running lower bound of the final candidate bound -- for top-p
//     M_run - T (ln(V / (1 - p)) + slack), valid since the total mass relative
//     to the maximum is at least 1; for top-k the smallest over the warps of
//     each warp's j-th largest lane maximum, j = ceil(k / warps), since then
//     at least k entries lie at or above it;
//   * rows without a filter: draws the Philox noise of every entry within the
//     noise span of the best score seen so far and keeps the best (Gumbel-max
//     as a running maximum), so such rows need no later phase.
// After the pass the CTAs all-gather their partial results over distributed
// shared memory (one cluster barrier), every CTA derives the same row scalars,
// and the exact cuts run as radix selects whose per-level histograms are built
// by every CTA from its own list and merged into the leader CTA's.  The
// Gumbel-max over the kept set scores only the kept entries of each list, and
// the leader takes the best key.  A list that overflowed, a row whose
// maximum is +inf or whose mass sum met a NaN re-read the slice from global
// memory (normally L2) instead: the list decides only the speed.
//
// Behaviour as "core.inference.sampling.base" (Sampling.sample_kernel,
// sample_speculative), "core.inference.sampling.flashinfer_sampling"
// (FlashInferSampling: top-k-only / top-p-only / joint dispatch from host
// flags) and the TokenSpeed "backends/triton.py" page (TritonSamplingBackend:
// Gumbel-max sampling; split-row partial results combined per row, there in
// global buffers of per-block maxima, sums and arg-maxima, here in the
// cluster's shared memory).

#include <type_traits>

#include "ls_kernel.cuh"

namespace lsg {

enum RowKind { KIND_GREEDY = 0, KIND_FREE = 1, KIND_TOPK = 2, KIND_TOPP = 3 };

// Threads per CTA, CTAs per SM the register budget is sized for, histogram
// bins per select level and the cap of one CTA's shared-memory budget, per
// cluster size.  Smaller CTAs for larger clusters keep about a wave of
// resident CTAs.
template <int C>
struct SplitCfg;
template <>
struct SplitCfg<1> {
  static constexpr int kB = 512, kMinBlocks = 2, kBinBits = 11;
  static constexpr size_t kBudget = 96 * 1024;
};
template <>
struct SplitCfg<2> {
  static constexpr int kB = 256, kMinBlocks = 2, kBinBits = 10;
  static constexpr size_t kBudget = 112 * 1024;
};
template <>
struct SplitCfg<4> {
  static constexpr int kB = 128, kMinBlocks = 4, kBinBits = 10;
  static constexpr size_t kBudget = 112 * 1024;
};
template <>
struct SplitCfg<8> {
  static constexpr int kB = 128, kMinBlocks = 4, kBinBits = 10;
  static constexpr size_t kBudget = 112 * 1024;
};

constexpr int kMaxCluster = 8;
constexpr int kSplitWarps = 16;  // most warps of a CTA (512 threads)

// One CTA's results of the streaming pass, gathered in every CTA.
struct alignas(16) SplitPart {
  float m;      // slice maximum
  float s;      // mass sum of the slice relative to 2^RN(m c)
  float bound;  // the list holds every entry of the slice at or above this
  int count;    // groups captured by the CTA, or -1 when a warp's segment overflowed
  unsigned long long best;  // best Gumbel score key (rows without a filter)
  int gidx;     // lowest index of the slice maximum (greedy rows)
  int pad;
};

struct alignas(16) SplitShared {
  SplitPart part[kMaxCluster];
  unsigned long long fbest[kMaxCluster];  // per-CTA best key of the final Gumbel-max (leader)
  float fsum[kMaxCluster];                // per-CTA mass sums when a NaN poisoned the online sum
  unsigned long long wbest[kSplitWarps];  // per-warp running best score key (rows without a filter)
  unsigned long long red_u64[kSplitWarps];
  float wrun[kSplitWarps];  // per-warp source of the running list bound
  float wlse[kSplitWarps];  // per-warp running log2-mass (top-p rows)
  float wm[kSplitWarps], ws[kSplitWarps], wb[kSplitWarps];
  unsigned int wj[kSplitWarps];
  int wcnt[kSplitWarps];  // groups each warp captured (more than its segment holds: overflow)
  unsigned long long cut_above, cut_mass, cut_total, cut_target;
  unsigned long long step;
  int cut_bin;
  int ecount;  // candidate entries gathered in the leader's list
  int pool;    // captured groups placed in the shared pool
  // top-p probe rounds: per-CTA two best score keys and their values, the
  // per-warp ones, per-CTA masses above each and in total
  unsigned long long pkey[kMaxCluster][2];
  float pval[kMaxCluster][2];
  unsigned long long pabove[kMaxCluster][2], ptotal[kMaxCluster];
  unsigned long long wkey[kSplitWarps][2];
  float wval[kSplitWarps][2];
  unsigned long long red2_u64[kSplitWarps], red3_u64[kSplitWarps];
  // top-k bound refinement: this CTA's candidate counts per value bin, and
  // every CTA's (all-gathered)
  unsigned int lbin[32];
  unsigned int kbin[kMaxCluster][32];
};

// ---------------------------------------------------------------------------
// Cluster primitives (distributed shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer(uint32_t a, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(rank));
  return d;
}
__device__ __forceinline__ void st_peer(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_peer(uint32_t a, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_peer(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atom_peer_add(uint32_t a, uint32_t v) {
  uint32_t o;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(o) : "r"(a), "r"(v) : "memory");
  return o;
}
__device__ __forceinline__ void red_peer_add(uint32_t a, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Barrier over the row's CTAs: the cluster, or the CTA itself.
template <int C>
__device__ __forceinline__ void row_sync() {
  if (C > 1)
    cluster_sync_all();
  else
    __syncthreads();
}

// Group maximum as the bf16 bit pattern of the smallest bf16 value >= it (the
// maximum itself for bf16 rows); a group of -inf / NaN entries stores -inf.
__device__ __forceinline__ uint16_t gmax_bits(float gm) {
  if (!(gm > kNegInf)) return (uint16_t)0xFF80u;
  const uint32_t b = __float_as_uint(gm);
  if ((b & 0xFFFFu) == 0u || (b & 0x80000000u)) return (uint16_t)(b >> 16);  // exact, or negative: truncation rounds up
  return (uint16_t)((b >> 16) + 1u);
}
__device__ __forceinline__ float gmax_value(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Warp-wide maximum of a 64-bit key (every lane gets it).
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {
  const unsigned int hi = __reduce_max_sync(0xFFFFFFFFu, (unsigned int)(k >> 32));
  const unsigned int lo = __reduce_max_sync(0xFFFFFFFFu, (unsigned int)(k >> 32) == hi ? (unsigned int)k : 0u);
  return ((unsigned long long)hi << 32) | lo;
}

// Gumbel-max scoring of candidate entries by one thread: exact score of every
// entry that can still beat the best the thread holds; an entry whose Philox
// uniform lies below the level it would need (exp(-exp(z - s_best)), taken
// 1e-3 looser in g) is skipped without the logarithms.
struct Scorer {
  float T;
  uint64_t seed, step;
  uint32_t row;
  bool zero_z;  // +inf row: the +inf entries share the probability, z = 0
  unsigned long long best;
  PhiloxCache pc;
  __device__ __forceinline__ void operator()(float v, int64_t j) {
    const float z = zero_z ? 0.f : __fdiv_rn(v, T);
    const uint32_t x = pc.word(seed, step, row, j);
    if (best != 0ull) {
      const float s_lb = f32_from_key((uint32_t)(best >> 32));
      const float need = s_lb - z - 1e-3f;
      const float thr = ex2(-ex2(-need * kLog2e) * kLog2e) * (1.f - 4e-7f);
      const float u = __uint2float_rn(((x >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
      if (!(u >= thr)) return;
    }
    const unsigned long long key = argmax_key(z + gumbel_of_word(x), j);
    if (key > best) best = key;
  }
};

// The two best score keys (k1 > k2, 0 when absent) and their entries'
// values.
struct TopTwo {
  unsigned long long k1, k2;
  float v1, v2;
  __device__ __forceinline__ void add(unsigned long long k, float v) {
    if (k > k1) {
      k2 = k1;
      v2 = v1;
      k1 = k;
      v1 = v;
    } else if (k > k2 && k != k1) {
      k2 = k;
      v2 = v;
    }
  }
  // Merge another pair (keys are unique per entry: an equal key is the same
  // entry).
  __device__ __forceinline__ void merge(const TopTwo& o) {
    add(o.k2, o.v2);
    add(o.k1, o.v1);
  }
  __device__ __forceinline__ void warp_merge() {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      TopTwo o;
      o.k1 = __shfl_xor_sync(0xFFFFFFFFu, k1, off);
      o.k2 = __shfl_xor_sync(0xFFFFFFFFu, k2, off);
      o.v1 = __shfl_xor_sync(0xFFFFFFFFu, v1, off);
      o.v2 = __shfl_xor_sync(0xFFFFFFFFu, v2, off);
      merge(o);
    }
  }
};

// Gumbel-max scoring that keeps the two best entries: an entry takes its
// exact score only if it can still beat the second best (the Scorer's test
// against k2).
struct TwoScorer {
  float T;
  uint64_t seed, step;
  uint32_t row;
  TopTwo t;
  PhiloxCache pc;
  __device__ __forceinline__ void operator()(float v, int64_t j) {
    const float z = __fdiv_rn(v, T);
    const uint32_t x = pc.word(seed, step, row, j);
    if (t.k2 != 0ull) {
      const float s_lb = f32_from_key((uint32_t)(t.k2 >> 32));
      const float need = s_lb - z - 1e-3f;
      const float thr = ex2(-ex2(-need * kLog2e) * kLog2e) * (1.f - 4e-7f);
      const float u = __uint2float_rn(((x >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
      if (!(u >= thr)) return;
    }
    t.add(argmax_key(z + gumbel_of_word(x), j), v);
  }
};

// Smallest value of 2 (x >> 9) + 1, for the noise word x of an entry whose z
// is at most fl(gm / T), that can still beat the best score key `best` (the
// Scorer's test, 1e-3 looser in g): every entry of a group whose maximum is
// gm needs u >= exp(-exp(z - s_best)) >= the group's level, and
// u = (2 (x >> 9) + 1) 2^-24 >= thr implies 2 (x >> 9) + 1 >= floor(thr 2^24).
// 0 (nothing rejected) while no best is held.
__device__ __forceinline__ uint32_t group_word_threshold(unsigned long long best, float gm, float T) {
  if (best == 0ull) return 0u;
  const float need = f32_from_key((uint32_t)(best >> 32)) - __fdiv_rn(gm, T) - 1e-3f;
  const float thr = ex2(-ex2(-need * kLog2e) * kLog2e) * (1.f - 4e-7f);
  return (uint32_t)(thr * 16777216.f);
}

// Per-warp buffer of the entries that passed a noise-word test (value,
// vocabulary index).  Their exact tests run in batches with one entry per
// lane: code that only a few entries reach then runs once per batch, instead
// of once for every entry that some lane passes (a rarely taken branch into
// code that other warps' code had evicted from the instruction caches).
// `n` is the same in every lane; all lanes call push and flush.
struct SurvivorBuffer {
  float* v;
  int32_t* j;
  int cap;  // entries, a multiple of 32
  int n;
  template <typename S>
  __device__ __forceinline__ void flush(S& sc) {
    __syncwarp();
    for (int q = (int)(threadIdx.x & 31); q < n; q += 32) sc(v[q], (int64_t)j[q]);
    __syncwarp();
    n = 0;
  }
  // Appends the entries of `surv` of a group (words w; idx(e): vocabulary
  // index of entry e).
  template <typename RV, typename Idx, typename S>
  __device__ __forceinline__ void push(uint32_t surv, const uint32_t (&w)[RV::kWords], Idx idx, S& sc) {
    const int lane = threadIdx.x & 31;
    const int cnt = __popc(surv);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const int tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (tot == 0) return;
    if (n + tot > cap) flush(sc);
    if (tot > cap) {  // more than a whole buffer at once: exact tests in place
      while (surv) {
        const int e = __ffs(surv) - 1;
        surv &= surv - 1u;
        sc(RV::element(w, e), idx(e));
      }
      return;
    }
    int at = n + incl - cnt;
    while (surv) {
      const int e = __ffs(surv) - 1;
      surv &= surv - 1u;
      v[at] = RV::element(w, e);
      j[at] = (int32_t)idx(e);
      ++at;
    }
    n += tot;
  }
};

// Entries of a group whose noise word clears the level thr_i (bit e for
// entry e; only entries in `mm`).  A group whose first index j0 is a multiple
// of 4 spans exactly four Philox blocks: they are drawn together, four
// independent chains, and the sixteen tests need no branch; other groups
// draw entry by entry.
template <typename RV, typename Idx>
__device__ __forceinline__ uint32_t word_survivors(uint32_t mm, int64_t j0, Idx idx, uint32_t thr_i, uint64_t seed,
                                                   uint64_t step, uint32_t row, PhiloxCache& pc) {
  if (mm == 0u || thr_i == 0u) return mm;
  uint32_t surv = 0u;
  if ((j0 & 3) == 0 && j0 >= 0) {
    const uint32_t b0 = (uint32_t)((uint64_t)j0 >> 2);
    uint4 c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = make_uint4(b0 + q, row, (uint32_t)step, (uint32_t)(step >> 32));
    philox4x32_10_x4(c, make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
#pragma unroll
    for (int e = 0; e < kGroup; ++e) {
      const uint4 bq = c[e >> 2];
      const uint32_t x = (e & 3) == 0 ? bq.x : (e & 3) == 1 ? bq.y : (e & 3) == 2 ? bq.z : bq.w;
      surv |= ((((x >> 9) << 1) | 1u) >= thr_i ? 1u : 0u) << e;
    }
    return surv & mm;
  }
  while (mm) {
    const int e = __ffs(mm) - 1;
    mm &= mm - 1u;
    if ((((pc.word(seed, step, row, idx(e)) >> 9) << 1) | 1u) >= thr_i) surv |= 1u << e;
  }
  return surv;
}

// Smallest float above a finite x (the lower bound of "strictly above x").
__device__ __forceinline__ float next_above(float x) {
  if (x == 0.f) return __uint_as_float(1u);
  const uint32_t b = __float_as_uint(x);
  return __uint_as_float(x > 0.f ? b + 1u : b - 1u);
}

// Entry sources of the post-stream phases, per CTA:
//   SRC_ENTRIES  the compacted list of candidate entries (value, index);
//   SRC_GROUPS   the groups captured during the stream (their raw words and
//                slice-local indices; warp w's k-th group in slot k W + w);
//   SRC_SLICE    the slice re-read from global memory (normally L2);
//   SRC_ROW      the whole row re-read from global memory (one CTA finishing
//                a row alone).
// Except for SRC_ROW, only groups whose maximum reaches `lo` are opened.
enum SrcMode { SRC_ENTRIES = 0, SRC_GROUPS = 1, SRC_SLICE = 2, SRC_ROW = 3 };

template <typename TIn, int B>
struct SplitSource {
  using RV = RowView<TIn>;
  static constexpr int W = B / 32;
  const RV* rv;
  const uint16_t* gmax;
  const uint32_t* cw;
  const int32_t* cl;
  const int* wcnt;  // per-warp captured groups
  int capw;         // own slots per warp (warp w's k-th group in slot k W + w)
  int maxk;         // largest number of own slots any warp filled
  int npool;        // groups in the pool (slots W capw ...)
  const float* ev;
  const int32_t* ej;
  int ecount;
  int gb, nl;  // first group and group count of the slice
  int mode;
  // slot of the q-th captured-group candidate, or -1 when that slot is unused
  __device__ __forceinline__ int slot(int q) const {
    if (q < W * maxk) return q / W < min(wcnt[q % W], capw) ? q : -1;
    return W * capw + (q - W * maxk);
  }
  __device__ __forceinline__ int slots() const { return W * maxk + npool; }
  __device__ __forceinline__ void load_group(int sl, uint32_t (&w)[RV::kWords]) const {
    const uint4* src4 = reinterpret_cast<const uint4*>(cw + (size_t)sl * RV::kWords);
#pragma unroll
    for (int h = 0; h < RV::kWords / 4; ++h) {
      const uint4 x = src4[h];
      w[4 * h] = x.x;
      w[4 * h + 1] = x.y;
      w[4 * h + 2] = x.z;
      w[4 * h + 3] = x.w;
    }
  }
  template <typename F>
  __device__ __forceinline__ void each(float lo, F&& f) const {
    if (mode == SRC_ENTRIES) {
      for (int q = threadIdx.x; q < ecount; q += B) {
        const float v = ev[q];
        if (v >= lo) f(v, (int64_t)ej[q]);
      }
    } else if (mode == SRC_GROUPS) {
      const int nq = slots();
      for (int q = threadIdx.x; q < nq; q += B) {
        const int sl = slot(q);
        if (sl >= 0) {
          const int l = cl[sl];
          if (gmax_value(gmax[l]) >= lo) {
            uint32_t w[RV::kWords];
            load_group(sl, w);
            uint32_t mm = RV::ge_mask(w, lo);
            while (mm) {
              const int e = __ffs(mm) - 1;
              mm &= mm - 1u;
              f(RV::element(w, e), rv->index(gb + l, e));
            }
          }
        }
      }
    } else if (mode == SRC_SLICE) {
      for (int l = threadIdx.x; l < nl; l += B)
        if (gmax_value(gmax[l]) >= lo) each_in_group(*rv, gb + l, lo, f);
    } else {
      for (int g = threadIdx.x; g < rv->NG; g += B) each_in_group(*rv, g, lo, f);
    }
  }
  // As each, but over the entry list a thread walks a contiguous run (the
  // entries of one group are adjacent there, so they share Philox blocks).
  template <typename F>
  __device__ __forceinline__ void each_run(float lo, F&& f) const {
    if (mode == SRC_ENTRIES) {
      const int per = (ecount + B - 1) / B;
      const int c0 = threadIdx.x * per, c1 = min(ecount, c0 + per);
      for (int q = c0; q < c1; ++q) {
        const float v = ev[q];
        if (v >= lo) f(v, (int64_t)ej[q]);
      }
    } else {
      each(lo, f);
    }
  }
};

template <typename TIn>
struct HistWeight {
  const unsigned int* hist;
  int mode;
  uint32_t klo;
  float c, R;
  __device__ __forceinline__ unsigned long long operator()(int b) const {
    if (mode == BIN_MASS) return ((unsigned long long)hist[2 * b + 1] << 32) | hist[2 * b];
    const unsigned int n = hist[b];
    if (mode == BIN_COUNT || n == 0u) return n;
    return (unsigned long long)n * mass_fixed(ex2(fmaf(KeyOps<TIn>::value(klo + (uint32_t)b), c, -R)));
  }
};

// Highest bin b with above + (weight of bins >= b) >= target, over one CTA's
// histogram (as the one-CTA kernel's cut, for B threads and NB bins).
template <int B, int NB, typename Wt>
__device__ __forceinline__ unsigned long long split_find_cut(SplitShared& sh, int nb, unsigned long long above,
                                                             unsigned long long& target, float joint_p,
                                                             const Wt& weight) {
  constexpr int PER = NB / B;
  constexpr int W = B / 32;
  static_assert(NB % B == 0, "bins must split evenly over threads");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int top = nb - 1 - t * PER;
  const bool has_bins = nb - 1 - warp * 32 * PER >= 0;
  unsigned long long w[PER], local = 0, incl = 0;
  if (has_bins) {
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      w[q] = top - q >= 0 ? weight(top - q) : 0ull;
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
    for (int q = 0; q < W; ++q) {
      const unsigned long long x = sh.red_u64[q];
      base += q < warp ? x : 0ull;
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
      for (int q = 0; q < PER; ++q) {
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
  target = sh.cut_target;
  return sh.cut_total;
}

// Exact threshold select over the row entries with keys in [klo, khi] (as the
// one-CTA kernel's radix_select): each level every CTA histograms its own
// entries, the other CTAs add their bins into the leader's histogram, the
// leader finds the cut bin and writes it into every CTA.  The leader's
// histogram is cleared before the cluster barrier that precedes the next
// level's additions (the first level: the barrier of the row-scalar
// exchange).
template <typename TIn, int C, int B, int BITS, typename Src>
__device__ SelResult split_select(SplitShared& sh, unsigned int* hist, const Src& src, uint32_t klo, uint32_t khi,
                                  unsigned long long target, float joint_p, float R, float c, bool mass) {
  using K = KeyOps<TIn>;
  constexpr int NB = 1 << BITS;
  const int tid = threadIdx.x;
  const uint32_t rank = C > 1 ? cluster_rank() : 0u;
  unsigned long long above = 0, mass_at = 0;
  for (;;) {
    const uint32_t width = khi - klo;
    const int bits = width ? 32 - __clz(width) : 0;
    const int shift = bits > BITS ? bits - BITS : 0;
    const int nb = (int)(width >> shift) + 1;
    const int mode = !mass ? BIN_COUNT : shift == 0 ? BIN_KEY_COUNT : BIN_MASS;
    if (C == 1 || rank != 0) {
      for (int b = tid; b < (mode == BIN_MASS ? 2 * nb : nb); b += B) hist[b] = 0u;
      __syncthreads();
    }
    {
      const float lo = K::value(klo), hi = K::value(khi);
      src.each(lo, [&](float v, int64_t) {
        const uint32_t kk = K::key(v);
        if (v <= hi && kk >= klo && kk <= khi) {
          const int bin = (int)((kk - klo) >> shift);
          if (mode == BIN_MASS)
            add_mass(&hist[2 * bin], mass_fixed(ex2(fmaf(v, c, -R))));
          else
            atomicAdd(&hist[bin], 1u);
        }
      });
    }
    __syncthreads();
    if (C > 1) {
      if (rank != 0) {
        const uint32_t base = peer(smem_u32(hist), 0u);
        if (mode == BIN_MASS) {
          for (int b = tid; b < nb; b += B) {
            const unsigned int lo32 = hist[2 * b], hi32 = hist[2 * b + 1];
            if (lo32 | hi32) {
              const unsigned int old = atom_peer_add(base + 8u * (uint32_t)b, lo32);
              const unsigned int carry = (old + lo32 < old) ? 1u : 0u;
              if (hi32 + carry) red_peer_add(base + 8u * (uint32_t)b + 4u, hi32 + carry);
            }
          }
        } else {
          for (int b = tid; b < nb; b += B) {
            const unsigned int n = hist[b];
            if (n) red_peer_add(base + 4u * (uint32_t)b, n);
          }
        }
      }
      cluster_sync_all();
    }
    if (C == 1 || rank == 0) {
      split_find_cut<B, NB>(sh, nb, above, target, joint_p, HistWeight<TIn>{hist, mode, klo, c, R});
      if (C > 1) {
        for (int b = tid; b < 2 * NB; b += B) hist[b] = 0u;
        if (tid >= 1 && tid < C) {
          const uint32_t r = (uint32_t)tid;
          st_peer(peer(smem_u32(&sh.cut_bin), r), (uint32_t)sh.cut_bin);
          st_peer(peer(smem_u32(&sh.cut_above), r), sh.cut_above);
          st_peer(peer(smem_u32(&sh.cut_mass), r), sh.cut_mass);
          st_peer(peer(smem_u32(&sh.cut_total), r), sh.cut_total);
          st_peer(peer(smem_u32(&sh.cut_target), r), sh.cut_target);
        }
      }
    }
    if (C > 1) cluster_sync_all();
    joint_p = -1.f;
    const int b = sh.cut_bin;
    const unsigned long long total = sh.cut_total;
    target = sh.cut_target;
    if (b < 0) return SelResult{klo, above + total, true};  // only reachable on the first level
    above = sh.cut_above;
    mass_at = sh.cut_mass;
    const uint32_t nlo = klo + ((uint32_t)b << shift);
    const unsigned long long nhi = (unsigned long long)nlo + ((1ull << shift) - 1ull);
    khi = nhi < (unsigned long long)khi ? (uint32_t)nhi : khi;
    klo = nlo;
    if (klo >= khi) break;
    if (C == 1) __syncthreads();  // the cut fields and the histogram are rewritten by the next level
  }
  return SelResult{klo, above + mass_at, false};
}

// Sources for one warp: the leader's entry list, or the whole row re-read
// from global memory; lane L visits items L, L + 32, ...
struct WarpEntries {
  const float* ev;
  int E;
  template <typename F>
  __device__ __forceinline__ void each(float lo, F&& f) const {
    for (int q = threadIdx.x & 31; q < E; q += 32) {
      const float v = ev[q];
      if (v >= lo) f(v, q);
    }
  }
};
template <typename TIn>
struct WarpRow {
  const RowView<TIn>* rv;
  template <typename F>
  __device__ __forceinline__ void each(float lo, F&& f) const {
    for (int g = threadIdx.x & 31; g < rv->NG; g += 32) each_in_group(*rv, g, lo, f);
  }
};

// One warp's exact threshold select (the semantics of split_select: the
// largest key kappa with above + weight(keys in [kappa, khi]) >= target, the
// target joint_p times the range's weight when joint_p >= 0): at most 256
// bins per level (8 per lane) in the first 512 words of `hist`, only
// __syncwarp between the steps.  All 32 lanes call it; every lane returns the
// same result.
template <typename TIn, typename Src>
__device__ SelResult warp_select(unsigned int* hist, const Src& src, uint32_t klo, uint32_t khi,
                                 unsigned long long target, float joint_p, float R, float c, bool mass) {
  using K = KeyOps<TIn>;
  constexpr int WBITS = 8, PER = 8;
  const int lane = threadIdx.x & 31;
  unsigned long long above = 0, mass_at = 0;
  for (;;) {
    const uint32_t width = khi - klo;
    const int bits = width ? 32 - __clz(width) : 0;
    const int shift = bits > WBITS ? bits - WBITS : 0;
    const int nb = (int)(width >> shift) + 1;
    const int mode = !mass ? BIN_COUNT : shift == 0 ? BIN_KEY_COUNT : BIN_MASS;
#pragma unroll
    for (int b = lane; b < 512; b += 32) hist[b] = 0u;
    __syncwarp();
    {
      const float lo = K::value(klo), hi = K::value(khi);
      src.each(lo, [&](float v, int64_t) {
        const uint32_t kk = K::key(v);
        if (v <= hi && kk >= klo && kk <= khi) {
          const int bin = (int)((kk - klo) >> shift);
          if (mode == BIN_MASS)
            add_mass(&hist[2 * bin], mass_fixed(ex2(fmaf(v, c, -R))));
          else
            atomicAdd(&hist[bin], 1u);
        }
      });
    }
    __syncwarp();
    const HistWeight<TIn> weight{hist, mode, klo, c, R};
    const int top = nb - 1 - lane * PER;  // lane 0 holds the highest bins
    unsigned long long w[PER], local = 0;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      w[q] = top - q >= 0 ? weight(top - q) : 0ull;
      local += w[q];
    }
    unsigned long long incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += u;
    }
    const unsigned long long total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (joint_p >= 0.f) target = __float2ull_ru(joint_p * __ull2float_rn(total));
    if (target < 1ull) target = 1ull;
    joint_p = -1.f;
    unsigned long long cum = above + incl - local, ab = 0, ms = 0;
    int bin = -1;
    if (cum < target && cum + local >= target) {
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        if (bin < 0 && cum + w[q] >= target) {
          bin = top - q;
          ab = cum;
          ms = w[q];
        }
        cum += w[q];
      }
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, bin >= 0);
    if (!hit) return SelResult{klo, above + total, true};  // only reachable on the first level
    const int from = __ffs(hit) - 1;
    bin = __shfl_sync(0xFFFFFFFFu, bin, from);
    above = __shfl_sync(0xFFFFFFFFu, ab, from);
    mass_at = __shfl_sync(0xFFFFFFFFu, ms, from);
    __syncwarp();  // the histogram is rewritten by the next level
    const uint32_t nlo = klo + ((uint32_t)bin << shift);
    const unsigned long long nhi = (unsigned long long)nlo + ((1ull << shift) - 1ull);
    khi = nhi < (unsigned long long)khi ? (uint32_t)nhi : khi;
    klo = nlo;
    if (klo >= khi) break;
  }
  return SelResult{klo, above + mass_at, false};
}

// Best key of the CTA (every thread gets it).  Uses sh.red_u64; ends with a
// barrier so that the slots may be reused.
template <int B>
__device__ __forceinline__ unsigned long long cta_max_key(SplitShared& sh, unsigned long long k) {
  constexpr int W = B / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long kw = warp_max_key(k);
  if (lane == 0) sh.red_u64[warp] = kw;
  __syncthreads();
  unsigned long long r = 0ull;
#pragma unroll
  for (int q = 0; q < W; ++q) r = sh.red_u64[q] > r ? sh.red_u64[q] : r;
  __syncthreads();
  return r;
}

// Block-wide sums of two 64-bit values (every thread gets both).
template <int B>
__device__ __forceinline__ void cta_sum2(SplitShared& sh, unsigned long long& x, unsigned long long& y) {
  constexpr int W = B / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    y += __shfl_xor_sync(0xFFFFFFFFu, y, o);
  }
  if (lane == 0) {
    sh.red_u64[warp] = x;
    sh.red2_u64[warp] = y;
  }
  __syncthreads();
  x = 0ull;
  y = 0ull;
#pragma unroll
  for (int q = 0; q < W; ++q) {
    x += sh.red_u64[q];
    y += sh.red2_u64[q];
  }
  __syncthreads();
}

// Block-wide sums of three 64-bit values (every thread gets them).
template <int B>
__device__ __forceinline__ void cta_sum3(SplitShared& sh, unsigned long long& x, unsigned long long& y,
                                         unsigned long long& z) {
  constexpr int W = B / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    y += __shfl_xor_sync(0xFFFFFFFFu, y, o);
    z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
  }
  if (lane == 0) {
    sh.red_u64[warp] = x;
    sh.red2_u64[warp] = y;
    sh.red3_u64[warp] = z;
  }
  __syncthreads();
  x = y = z = 0ull;
#pragma unroll
  for (int q = 0; q < W; ++q) {
    x += sh.red_u64[q];
    y += sh.red2_u64[q];
    z += sh.red3_u64[q];
  }
  __syncthreads();
}

// Probe rounds a top-p row takes before it falls back to the select.
constexpr int kProbeRounds = 4;
// Gathered lists up to this length take their cuts in the whole leader CTA by
// direct counting (one entry per thread).
constexpr int kLeadList = 128;
// Captured groups over the row from which a top-p row probes instead of
// gathering its candidates for the select.
constexpr int kProbeGroups = 64;

template <typename TIn, int ROUTE, int C>
__global__ void __launch_bounds__(SplitCfg<C>::kB, SplitCfg<C>::kMinBlocks) split_sampler_kernel(const KernelArgs a) {
  using K = KeyOps<TIn>;
  using RV = RowView<TIn>;
  constexpr int B = SplitCfg<C>::kB;
  constexpr int W = B / 32;
  constexpr int NB = 1 << SplitCfg<C>::kBinBits;
  static_assert(W <= kSplitWarps && C <= kMaxCluster, "shared slots");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SplitShared& sh = *reinterpret_cast<SplitShared*>(smem_raw);
  unsigned int* hist = reinterpret_cast<unsigned int*>(smem_raw + sizeof(SplitShared));
  uint16_t* gmax = reinterpret_cast<uint16_t*>(hist + 2 * NB);
  // captured groups: raw words (16-byte aligned: gslot_cap is a multiple of
  // 8), their slice-local indices, then the compacted entry list
  uint32_t* cw = reinterpret_cast<uint32_t*>(gmax + a.gslot_cap);
  int32_t* cl = reinterpret_cast<int32_t*>(cw + (size_t)a.cand_cap * RV::kWords);
  float* ev = reinterpret_cast<float*>(cl + a.cand_cap);
  int32_t* ej = reinterpret_cast<int32_t*>(ev + a.ent_cap);
  float* es = reinterpret_cast<float*>(ej + a.ent_cap);  // Gumbel scores of the entries
  const int capw = (a.cand_cap - a.pool_cap) / W;  // own capture slots per warp
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the warp's survivor buffer in the entry list (rows without a filter, and
  // top-p probes: neither gathers into that list while it is in use)
  const int capb = (a.ent_cap / W) & ~31;
  SurvivorBuffer sb{ev + warp * capb, ej + warp * capb, capb, 0};
  const uint32_t rank = C > 1 ? cluster_rank() : 0u;
  const int64_t i = (int64_t)(blockIdx.x / C);
  const bool lead = rank == 0u;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's writes are visible

  // ---- row -> (logits row, request): the same in every CTA of the row ----
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
  if (a.out_t2r && lead && tid == 0) a.out_t2r[i] = (int32_t)req;
  if (req < 0 || req >= a.num_requests) err |= LS_ROW_ERR_BAD_REQUEST;
  if (err) {  // every CTA of the row leaves here, before any cluster barrier
    if (lead && tid == 0) {
      a.out_ids[i] = -1;
      if (a.error_word) atomicOr(a.error_word, err);
    }
    return;
  }

  const int64_t V = a.vocab;
  RV rv;
  rv.init(a.logits, src, a.stride, V);
  const int per = (rv.NG + C - 1) / C;
  const int gb = (int)rank * per;                       // first group of this CTA's slice
  const int nl = max(0, min(rv.NG, gb + per) - gb);    // groups of the slice
  constexpr int U = RV::kBytes == 2 ? 2 : 1;           // groups per stage and thread
  constexpr int STEP = U * B;
  const int iters = (nl + 2 * STEP - 1) / (2 * STEP);  // the same for every thread of the CTA
  auto issue = [&](int l0, uint32_t (&w)[U][RV::kWords]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int l = l0 + u * B;
      if (l < nl && rv.full(gb + l)) rv.load_words(gb + l, w[u]);
    }
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
  const int kind = greedy ? KIND_GREEDY : k_on ? KIND_TOPK : p_on ? KIND_TOPP : KIND_FREE;
  const bool need_sum = kind == KIND_TOPP;
  const float c = greedy ? 0.f : kLog2e / T;
  const uint64_t seed = greedy ? 0ull : a.seed[req];
  // top-p: entries below M - T dp carry less than (1 - p) e^-slack of the mass (S >= 1);
  // in log2 units, an entry whose weight 2^(v c) lies dp2 below the row's
  // total log2-mass carries less than (1 - p) e^-slack / V of it
  const float dp = kind == KIND_TOPP ? logf((float)V / (1.f - p)) + kTopPSlack : 0.f;
  const float dp2 = dp * kLog2e;
  // top-k: each warp's j-th largest lane maximum; the warps that hold groups
  // (Wa of them) then have Wa j >= k entries at or above the smallest of those
  const int wact = min(W, (nl + 31) / 32);
  const int jrank = kind == KIND_TOPK && wact > 0 && k <= 32 * wact ? (k + wact - 1) / wact : 0;

  if (lane == 0) {
    sh.wrun[warp] = kNegInf;
    sh.wlse[warp] = kNegInf;
    sh.wbest[warp] = 0ull;
  }
  if (tid == 0) {
    sh.ecount = 0;
    sh.pool = 0;
    sh.step = a.step_ptr ? *a.step_ptr : a.step;
  }
  // the first select level adds into the leader's histogram after the
  // exchange barrier: clear it now
  for (int b = tid; b < 2 * NB; b += B) hist[b] = 0u;

  // ---- streaming pass ---------------------------------------------------
  // One copy of the loop per row kind (the kind is the same for every thread
  // of the CTA): each copy keeps only its own state live in registers.
  float m = kNegInf, r = 0.f;
  f32x2 acc = 0ull;
  int mg = -1;            // greedy: first local group holding the thread maximum
  float bound = kNegInf;  // the thread's current list / noise bound (never decreases)
  unsigned long long best = 0ull;  // rows without a filter: the thread's best score key
  int wcnt = 0;           // groups this warp captured (the same in every lane)
  auto stream = [&](auto kind_c) {
    constexpr int KD = decltype(kind_c)::value;
    const f32x2 c2 = pack2(c, c);
    Scorer sc{T, seed, 0ull, (uint32_t)i, false, 0ull, PhiloxCache{}};
    // heavy stages also refresh the top-p bound from the running mass
    auto stage = [&](int l0, uint32_t (&w)[U][RV::kWords], bool first, bool heavy) {
      float gmv[U];
      // group maxima, running maximum, online mass
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int l = l0 + u * B;
        gmv[u] = kNegInf;
        if (l < nl) {
          const int g = gb + l;
          if (!rv.full(g)) rv.load_words_partial(g, w[u]);
          const float gm = RV::group_max(w[u]);
          gmv[u] = gm;
          gmax[l] = gmax_bits(gm);
          if constexpr (KD == KIND_TOPP) {
            if (gm > m) {
              const float rn = __fmul_rn(gm, c);
              const float sc2 = ex2(r - rn);
              acc = m > kNegInf ? mul2(acc, pack2(sc2, sc2)) : 0ull;
              m = gm;
              r = rn;
            }
            if (gm > kNegInf) acc = add2(acc, RV::exp_sum(w[u], c2, pack2(-r, -r)));
          } else {
            if (gm > m) {
              m = gm;
              if constexpr (KD == KIND_GREEDY) mg = l;
            }
          }
        }
      }
      if constexpr (KD == KIND_GREEDY) return;
      // publish this warp's bound source (values only grow and are valid
      // whenever they are read: no barrier needed)
      if constexpr (KD == KIND_TOPK) {
        if (jrank > 0) {
          float cur = m, gj = kNegInf;
          for (int t = 0; t < jrank; ++t) {
            gj = warp_max(cur);
            const unsigned holders = __ballot_sync(0xFFFFFFFFu, cur == gj);
            if (lane == __ffs(holders) - 1) cur = kNegInf;
          }
          if (lane == 0) sh.wrun[warp] = gj;
        }
      } else {
        const float mw = warp_max(m);
        if (lane == 0) sh.wrun[warp] = mw;
        if constexpr (KD == KIND_FREE) {
          const unsigned long long kw = warp_max_key(sc.best);
          if (lane == 0) sh.wbest[warp] = kw;
        }
        if constexpr (KD == KIND_TOPP) {
          if (heavy && mw > kNegInf) {
            // the warp's log2-mass RN(mw c) + log2(sum): one word, so a
            // reader never pairs a maximum with another time's sum
            float lo, hi;
            unpack2(acc, lo, hi);
            const float sw = warp_reduce(m > kNegInf ? (lo + hi) * ex2(r - __fmul_rn(mw, c)) : 0.f, OpAddF());
            if (lane == 0) sh.wlse[warp] = __fmul_rn(mw, c) + __log2f(sw);
          }
        }
      }
      if (first) {
        __syncthreads();  // every warp has published: the bounds are defined from here on
        sc.step = sh.step;
      }
      // refresh the bound
      {
        float b;
        if constexpr (KD == KIND_TOPK) {
          b = jrank > 0 ? warp_min(lane < wact ? sh.wrun[lane] : kPosInf) : kNegInf;
        } else if constexpr (KD == KIND_TOPP) {
          const float mx = warp_max(lane < W ? sh.wrun[lane] : kNegInf);
          b = mx - T * dp;
          if (heavy) {
            // the warps' masses summed: a lower bound of the row's log2-mass
            const float x = lane < W ? sh.wlse[lane] : kNegInf;
            const float lx = warp_max(x);
            if (lx > kNegInf) {
              const float sx = warp_reduce(x > kNegInf ? ex2(x - lx) : 0.f, OpAddF());
              b = fmaxf(b, (lx + __log2f(sx) - dp2) / c);
            }
          }
          b -= fabsf(b) * 1e-5f + fabsf(mx) * 1e-6f;
        } else {
          // no filter: an entry more than the noise span below the maximum,
          // or more than the largest noise below the best score, cannot win
          const float mx = warp_max(lane < W ? sh.wrun[lane] : kNegInf);
          const unsigned long long kb = warp_max_key(lane < W ? sh.wbest[lane] : 0ull);
          if (kb > sc.best) sc.best = kb;
          b = mx - kGumbelSpan * T;
          if (sc.best) b = fmaxf(b, (f32_from_key((uint32_t)(sc.best >> 32)) - 16.6366f) * T);
          b -= fabsf(b) * 1e-5f + 1e-30f;
        }
        bound = fmaxf(bound, fmaxf(b, -FLT_MAX));  // -inf entries are never needed
      }
      if constexpr (KD == KIND_FREE) {
        if (first) {
          // Warp seed: the exact score of the largest entry among the warp's
          // groups of this stage, so that the thresholds prune from the first
          // group on (without it every lane scores its first entries in full).
          float gv = kNegInf;
          int us = 0;
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (l0 + u * B < nl && gmv[u] > gv) {
              gv = gmv[u];
              us = u;
            }
          const float wv = warp_max(gv);
          const unsigned holders = __ballot_sync(0xFFFFFFFFu, wv > kNegInf && gv == wv);
          if (holders && lane == __ffs(holders) - 1) {
            uint32_t ms = 0u;
            int ls = l0;
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (u == us) {
                ms = RV::ge_mask(w[u], wv);
                ls = l0 + u * B;
              }
            sc(wv, rv.index(gb + ls, __ffs(ms) - 1));
          }
          const unsigned long long kw = warp_max_key(sc.best);
          if (kw > sc.best) sc.best = kw;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int l = l0 + u * B;
        const bool over = l < nl && gmv[u] >= bound;
        if constexpr (KD == KIND_FREE) {
          // Gumbel-max as a running maximum over the entries that can win;
          // a threshold taken at the group's largest z against the thread's
          // best rejects most entries on their Philox word alone.
          // (the survivors of the word test take their exact tests in
          // batches: see SurvivorBuffer)
          const uint32_t mm = over ? RV::ge_mask(w[u], bound) : 0u;
          const uint32_t thr_i = mm ? group_word_threshold(sc.best, gmv[u], T) : 0u;
          auto idx = [&](int e) { return rv.index(gb + l, e); };
          const uint32_t surv = word_survivors<RV>(mm, rv.index(gb + l, 0), idx, thr_i, seed, sc.step, (uint32_t)i, sc.pc);
          sb.push<RV>(surv, w[u], idx, sc);
        } else {
          // capture the groups whose maximum clears the bound into the warp's
          // own slots (k W + warp): a ballot places them, no atomics; once
          // those are full, into the shared pool (one atomic per group)
          const unsigned hits = __ballot_sync(0xFFFFFFFFu, over);
          if (hits) {
            if (over) {
              const int kk = wcnt + __popc(hits & ((1u << lane) - 1u));
              int sl = -1;
              if (kk < capw) {
                sl = kk * W + warp;
              } else {
                const int pq = atomicAdd(&sh.pool, 1);
                if (pq < a.pool_cap) sl = W * capw + pq;
              }
              if (sl >= 0) {
                uint4* dst4 = reinterpret_cast<uint4*>(cw + (size_t)sl * RV::kWords);
#pragma unroll
                for (int h = 0; h < RV::kWords / 4; ++h)
                  dst4[h] = make_uint4(w[u][4 * h], w[u][4 * h + 1], w[u][4 * h + 2], w[u][4 * h + 3]);
                cl[sl] = l;
              }
            }
            wcnt += __popc(hits);
          }
        }
      }
    };
    for (int it = 0; it < iters; ++it) {
      const int l0 = it * 2 * STEP + tid;
      if constexpr (KD == KIND_GREEDY) {
        stage(l0, wa, false, false);
      } else {
        stage(l0, wa, it == 0, true);
      }
      issue(l0 + 2 * STEP, wa);
      stage(l0 + STEP, wb, false, it == 0);
      issue(l0 + 3 * STEP, wb);
    }
    if constexpr (KD == KIND_FREE) sb.flush(sc);
    best = sc.best;
  };
  switch (kind) {
    case KIND_GREEDY: stream(std::integral_constant<int, KIND_GREEDY>{}); break;
    case KIND_FREE: stream(std::integral_constant<int, KIND_FREE>{}); break;
    case KIND_TOPK:
      if constexpr ((ROUTE & ROUTE_K) != 0) stream(std::integral_constant<int, KIND_TOPK>{});
      break;
    default:
      if constexpr ((ROUTE & ROUTE_P) != 0) stream(std::integral_constant<int, KIND_TOPP>{});
      break;
  }
  // the next kernel on the stream may be scheduled now (it waits for this
  // grid to complete before it reads memory)
  asm volatile("griddepcontrol.launch_dependents;");
  __syncthreads();  // the step word and the list count are settled for every kind
  const uint64_t step = sh.step;

  // ---- this CTA's partial results --------------------------------------
  {
    const float mw = warp_max(m);
    float sw = 0.f;
    if (need_sum && mw > kNegInf) {
      float lo, hi;
      unpack2(acc, lo, hi);
      sw = m > kNegInf ? (lo + hi) * ex2(r - __fmul_rn(mw, c)) : 0.f;
      sw = warp_reduce(sw, OpAddF());
    }
    unsigned int jw = 0xFFFFFFFFu;
    if (kind == KIND_GREEDY) {
      unsigned int jt = 0xFFFFFFFFu;
      if (mg >= 0) {
        uint32_t w[RV::kWords];
        const int g = gb + mg;
        if (rv.full(g))
          rv.load_words(g, w);
        else
          rv.load_words_partial(g, w);
#pragma unroll
        for (int e = kGroup - 1; e >= 0; --e)
          if (RV::element_at(w, e) == m) jt = (unsigned int)rv.index(g, e);
      }
      jw = __reduce_min_sync(0xFFFFFFFFu, m == mw ? jt : 0xFFFFFFFFu);
    }
    const float bw = warp_max(bound);
    const unsigned long long kw = kind == KIND_FREE ? warp_max_key(best) : 0ull;
    if (lane == 0) {
      sh.wm[warp] = mw;
      sh.ws[warp] = sw;
      sh.wb[warp] = bw;
      sh.wj[warp] = jw;
      sh.red_u64[warp] = kw;
      sh.wcnt[warp] = wcnt;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const float mq = lane < W ? sh.wm[lane] : kNegInf;
    const float Mc = warp_max(mq);
    float Sc = 0.f;
    if (need_sum && Mc > kNegInf && Mc < kPosInf) {
      const float Rc = __fmul_rn(Mc, c);
      const float sq = lane < W && mq > kNegInf ? sh.ws[lane] * ex2(__fmul_rn(mq, c) - Rc) : 0.f;
      Sc = warp_reduce(sq, OpAddF());
    }
    const int wc = lane < W ? sh.wcnt[lane] : 0;
    SplitPart pt;
    pt.m = Mc;
    pt.s = Sc;
    pt.bound = warp_max(lane < W ? sh.wb[lane] : kNegInf);
    pt.count = sh.pool > a.pool_cap ? -1 : __reduce_add_sync(0xFFFFFFFFu, wc);
    pt.best = kind == KIND_FREE ? warp_max_key(lane < W ? sh.red_u64[lane] : 0ull) : 0ull;
    pt.gidx = kind == KIND_GREEDY
                  ? (int)__reduce_min_sync(0xFFFFFFFFu, lane < W && mq == Mc ? sh.wj[lane] : 0xFFFFFFFFu)
                  : -1;
    pt.pad = 0;
    if (C == 1) {
      if (lane == 0) sh.part[0] = pt;
    } else if (lane < C) {
      // all-gather: this CTA's part into slot `rank` of every CTA of the row
      const uint32_t dst = peer(smem_u32(&sh.part[rank]), (uint32_t)lane);
      const uint32_t* src_w = reinterpret_cast<const uint32_t*>(&pt);
#pragma unroll
      for (int q = 0; q < 8; ++q) st_peer(dst + 4u * q, src_w[q]);
    }
  }
  row_sync<C>();

  // ---- row scalars, identical in every CTA (fixed combination order) -----
  float M = kNegInf;
#pragma unroll
  for (int q = 0; q < C; ++q) M = fmaxf(M, sh.part[q].m);
  if (M == kNegInf) {  // no entry above -inf (no CTA touches another's memory after the exchange)
    if (lead && tid == 0) {
      a.out_ids[i] = -1;
      if (a.error_word) atomicOr(a.error_word, LS_ROW_ERR_NO_FINITE);
    }
    return;
  }
  if (kind == KIND_GREEDY) {  // lowest index of the maximum
    if (lead && tid == 0) {
      unsigned int J = 0xFFFFFFFFu;
#pragma unroll
      for (int q = 0; q < C; ++q)
        if (sh.part[q].m == M) J = min(J, (unsigned int)sh.part[q].gidx);
      a.out_ids[i] = (int32_t)J;
    }
    return;
  }
  int maxk = 0;
#pragma unroll
  for (int q = 0; q < W; ++q) maxk = max(maxk, min(sh.wcnt[q], capw));
  SplitSource<TIn, B> srcs{&rv, gmax, cw, cl, sh.wcnt, capw, maxk, min(sh.pool, a.pool_cap), ev, ej, 0, gb, nl,
                           SRC_SLICE};
  // The last phase of every remaining route: the best key of each CTA goes to
  // the leader, which writes the id.
  auto finish = [&](unsigned long long local) {
    const unsigned long long kc = cta_max_key<B>(sh, local);
    if (C == 1) {
      if (tid == 0) a.out_ids[i] = argmax_index(kc);
      return;
    }
    if (tid == 0) st_peer(peer(smem_u32(&sh.fbest[rank]), 0u), kc);
    cluster_sync_all();
    if (lead && tid == 0) {
      unsigned long long kb = 0ull;
#pragma unroll
      for (int q = 0; q < C; ++q) kb = sh.fbest[q] > kb ? sh.fbest[q] : kb;
      a.out_ids[i] = argmax_index(kb);
    }
  };

  if (M == kPosInf) {  // the +inf entries share the probability: Gumbel-max among them, z = 0
    Scorer s2{T, seed, step, (uint32_t)i, true, 0ull, PhiloxCache{}};
    srcs.each(kPosInf, s2);
    finish(s2.best);
    return;
  }
  if (kind == KIND_FREE) {  // the Gumbel-max ran in the stream
    if (lead && tid == 0) {
      unsigned long long kb = 0ull;
#pragma unroll
      for (int q = 0; q < C; ++q) kb = sh.part[q].best > kb ? sh.part[q].best : kb;
      a.out_ids[i] = argmax_index(kb);
    }
    return;
  }

  // ---- top-k / top-p: exact cuts over the lists -------------------------
  const float R = __fmul_rn(M, c);  // reference exponent of the row's masses (rounded, never fused)
  float S = 0.f;
  bool overflow = false;
  float bmax = kNegInf;
#pragma unroll
  for (int q = 0; q < C; ++q) {
    const SplitPart& pq = sh.part[q];
    if (need_sum && pq.m > kNegInf) S += pq.s * ex2(__fmul_rn(pq.m, c) - R);
    overflow |= pq.count < 0;
    bmax = fmaxf(bmax, pq.bound);
  }
  if (need_sum && !(S <= FLT_MAX)) {
    // a NaN entry poisoned the online sum: sum the slice again with NaN read
    // as -inf (a second read of the slice, off the common path)
    float s1 = 0.f;
    for (int l = tid; l < nl; l += B) {
      float v[kGroup];
      rv.load(gb + l, v);
#pragma unroll
      for (int e = 0; e < kGroup; ++e) {
        const float x = v[e] == v[e] ? v[e] : kNegInf;
        s1 += ex2(fmaf(x, c, -R));
      }
    }
    s1 = warp_reduce(s1, OpAddF());
    if (lane == 0) sh.wm[warp] = s1;
    __syncthreads();
    if (tid < C) {
      float t = 0.f;
#pragma unroll
      for (int q = 0; q < W; ++q) t += sh.wm[q];
      if (C == 1)
        sh.fsum[0] = t;
      else
        st_peer(peer(smem_u32(&sh.fsum[rank]), (uint32_t)tid), __float_as_uint(t));
    }
    row_sync<C>();
    S = 0.f;
#pragma unroll
    for (int q = 0; q < C; ++q) S += sh.fsum[q];
  }
  float lc;
  if (kind == KIND_TOPK) {
    lc = bmax;
  } else {
    const float Lp = M + T * (logf((1.f - p) * S / (float)V) - kTopPSlack);
    lc = fmaxf(Lp, bmax);
  }
  lc = fminf(fmaxf(lc, -FLT_MAX), M);
  const uint32_t key_max = K::key(M);
  const unsigned long long target =
      kind == KIND_TOPK ? (unsigned long long)k : max(1ull, __float2ull_ru(fmaxf(p, 0.f) * S * kMassScale));

  // ---- top-k: a bound from the whole row -----------------------------------
  // Each CTA's bound guarantees k entries in its own slice, so the row's bound
  // (the largest of them) lies well below the row's k-th largest entry.  The
  // candidates counted in 32 value bins over [lc, M], summed over the
  // cluster, raise it to half a bin below the highest bin edge with at least
  // k entries above (half a bin absorbs the rounding of the binning): the
  // gathered list then holds little more than k entries.
  if (kind == KIND_TOPK && !overflow && lc < M) {
    constexpr int NT = 32;
    const float scale = (float)NT / (M - lc);
    if (tid < NT) sh.lbin[tid] = 0u;
    __syncthreads();
    srcs.mode = SRC_GROUPS;
    srcs.each(lc, [&](float v, int64_t) { atomicAdd(&sh.lbin[min(NT - 1, (int)((v - lc) * scale))], 1u); });
    __syncthreads();
    for (int t = tid; t < NT * C; t += B) {
      const int q = t / NT, b = t % NT;
      if (C == 1)
        sh.kbin[0][b] = sh.lbin[b];
      else
        st_peer(peer(smem_u32(&sh.kbin[rank][b]), (uint32_t)q), sh.lbin[b]);
    }
    row_sync<C>();
    unsigned int cum = 0u;
    int bk = 0;
    for (int b = NT - 1; b > 0; --b) {
#pragma unroll
      for (int q = 0; q < C; ++q) cum += sh.kbin[q][b];
      if (cum >= (unsigned int)k) {
        bk = b;
        break;
      }
    }
    if (bk > 0) lc = fmaxf(lc, lc + ((float)bk - 0.5f) / scale);
  }

  // ---- top-p alone over many candidates: probe the best scores ------------
  // The Gumbel-max over the kept set is the best-scoring candidate whose
  // value clears the cut, and an entry clears it iff the mass of the entries
  // strictly above it is below the target (the kept set is the smallest
  // upward-closed set whose mass reaches the target).  Each round scores the
  // candidates >= lo in every CTA, takes the row's best over the cluster and
  // tests it with one sum of masses: no histogram and no gathered list.  An
  // entry that fails lies below the cut, so the next round raises lo above
  // it (the candidates >= lo then still weigh at least the target).  After
  // kProbeRounds rounds, or when the candidates weigh less than the target,
  // the row falls through to the select.
  {
    int ncap = 0;
#pragma unroll
    for (int q = 0; q < C; ++q) ncap += max(sh.part[q].count, 0);
    if (kind == KIND_TOPP && (overflow || ncap >= kProbeGroups)) {
      srcs.mode = overflow ? SRC_SLICE : SRC_GROUPS;
      // Scoring of this CTA's candidates >= lo (captured groups, or the slice
      // re-read): a warp seed (the exact score of the largest entry among the
      // lanes' first groups), then per group the threshold against the lane's
      // best, so most entries are rejected on their Philox word alone.
      auto score_pass = [&](float lo, TwoScorer& ts) {
        const bool grp = srcs.mode == SRC_GROUPS;
        const int nq = grp ? srcs.slots() : nl;
        for (int q0 = 0; q0 < nq; q0 += B) {  // rounds: the same count in every thread
          const int q = q0 + tid;
          int l = -1;
          uint32_t w[RV::kWords];
          if (q < nq) {
            if (grp) {
              const int sl = srcs.slot(q);
              if (sl >= 0 && gmax_value(gmax[cl[sl]]) >= lo) {
                l = cl[sl];
                srcs.load_group(sl, w);
              }
            } else if (gmax_value(gmax[q]) >= lo) {
              l = q;
              if (rv.full(gb + l))
                rv.load_words(gb + l, w);
              else
                rv.load_words_partial(gb + l, w);
            }
          }
          uint32_t mm = l >= 0 ? RV::ge_mask(w, lo) : 0u;
          const float gm = mm ? RV::group_max(w) : kNegInf;
          if (q0 == 0) {
            // warp seed: exact scores of the largest entries of the two lanes
            // with the largest group maxima, merged into every lane
            const float wv1 = warp_max(gm);
            const unsigned h1 = __ballot_sync(0xFFFFFFFFu, wv1 > kNegInf && gm == wv1);
            const int l1 = h1 ? __ffs(h1) - 1 : -1;
            const float gm2 = lane == l1 ? kNegInf : gm;
            const float wv2 = warp_max(gm2);
            const unsigned h2 = __ballot_sync(0xFFFFFFFFu, wv2 > kNegInf && gm2 == wv2);
            const int l2 = h2 ? __ffs(h2) - 1 : -1;
            if (lane == l1 || lane == l2) ts(gm, rv.index(gb + l, __ffs(RV::ge_mask(w, gm)) - 1));
            ts.t.warp_merge();
          }
          // the entries whose word clears the group's level against the
          // second best; their exact tests run in batches (SurvivorBuffer)
          const uint32_t thr_i = mm ? group_word_threshold(ts.t.k2, gm, T) : 0u;
          auto idx = [&](int e) { return rv.index(gb + l, e); };
          const uint32_t surv = word_survivors<RV>(mm, rv.index(gb + l, 0), idx, thr_i, seed, step, (uint32_t)i, ts.pc);
          sb.push<RV>(surv, w, idx, ts);
        }
        sb.flush(ts);
      };
      float lo = lc;
      for (int round = 0; round < kProbeRounds; ++round) {
        TwoScorer ts{T, seed, step, (uint32_t)i, TopTwo{0ull, 0ull, 0.f, 0.f}, PhiloxCache{}};
        score_pass(lo, ts);
        // the CTA's two best, then the row's (all-gathered over the cluster)
        ts.t.warp_merge();
        if (lane == 0) {
          sh.wkey[warp][0] = ts.t.k1;
          sh.wkey[warp][1] = ts.t.k2;
          sh.wval[warp][0] = ts.t.v1;
          sh.wval[warp][1] = ts.t.v2;
        }
        __syncthreads();
        TopTwo ct{0ull, 0ull, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < W; ++q) ct.merge(TopTwo{sh.wkey[q][0], sh.wkey[q][1], sh.wval[q][0], sh.wval[q][1]});
        if (tid < C) {
          if (C == 1) {
            sh.pkey[0][0] = ct.k1;
            sh.pkey[0][1] = ct.k2;
            sh.pval[0][0] = ct.v1;
            sh.pval[0][1] = ct.v2;
          } else {
            const uint32_t q = (uint32_t)tid;
            st_peer(peer(smem_u32(&sh.pkey[rank][0]), q), ct.k1);
            st_peer(peer(smem_u32(&sh.pkey[rank][1]), q), ct.k2);
            st_peer(peer(smem_u32(&sh.pval[rank][0]), q), __float_as_uint(ct.v1));
            st_peer(peer(smem_u32(&sh.pval[rank][1]), q), __float_as_uint(ct.v2));
          }
        }
        row_sync<C>();
        TopTwo rt{0ull, 0ull, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < C; ++q) rt.merge(TopTwo{sh.pkey[q][0], sh.pkey[q][1], sh.pval[q][0], sh.pval[q][1]});
        // masses strictly above each of the two, and of every candidate
        unsigned long long above1 = 0ull, above2 = 0ull, total = 0ull;
        srcs.each(lo, [&](float v, int64_t) {
          const unsigned long long w = mass_fixed(ex2(fmaf(v, c, -R)));
          total += w;
          above1 += v > rt.v1 ? w : 0ull;
          above2 += v > rt.v2 ? w : 0ull;
        });
        cta_sum3<B>(sh, above1, above2, total);
        if (tid < C) {
          if (C == 1) {
            sh.pabove[0][0] = above1;
            sh.pabove[0][1] = above2;
            sh.ptotal[0] = total;
          } else {
            const uint32_t q = (uint32_t)tid;
            st_peer(peer(smem_u32(&sh.pabove[rank][0]), q), above1);
            st_peer(peer(smem_u32(&sh.pabove[rank][1]), q), above2);
            st_peer(peer(smem_u32(&sh.ptotal[rank]), q), total);
          }
        }
        row_sync<C>();
        unsigned long long A1 = 0ull, A2 = 0ull, Tt = 0ull;
#pragma unroll
        for (int q = 0; q < C; ++q) {
          A1 += sh.pabove[q][0];
          A2 += sh.pabove[q][1];
          Tt += sh.ptotal[q];
        }
        if (Tt < target || rt.k1 == 0ull) break;  // the cut lies below lc: the select re-selects
        // the best is kept: it wins; else the second best, if kept, wins
        // (every entry scoring above it is the best)
        const unsigned long long win = A1 < target ? rt.k1 : rt.k2 != 0ull && A2 < target ? rt.k2 : 0ull;
        if (win != 0ull) {
          if (lead && tid == 0) a.out_ids[i] = argmax_index(win);
          return;  // no CTA reads another's shared memory after the last barrier
        }
        // both lie below the cut
        lo = next_above(rt.k2 != 0ull ? fmaxf(rt.v1, rt.v2) : rt.v1);
      }
      srcs.mode = overflow ? SRC_SLICE : SRC_GROUPS;
    }
  }

  // ---- common case: gather the candidates at the leader -------------------
  // Every CTA's captured groups hold all of its slice's entries >= lc (unless
  // its pool overflowed).  Each CTA appends those entries, with their Gumbel
  // scores, to the leader's entry list (one atomic per warp and round, on the
  // leader's counter); after one barrier the other CTAs are done and the
  // leader finds the cuts over its list and takes the best kept score.
  if (!overflow) {
    srcs.mode = SRC_GROUPS;
    const uint32_t cnt_a = C > 1 ? peer(smem_u32(&sh.ecount), 0u) : smem_u32(&sh.ecount);
    const uint32_t ev_a = C > 1 ? peer(smem_u32(ev), 0u) : smem_u32(ev);
    const uint32_t ej_a = C > 1 ? peer(smem_u32(ej), 0u) : smem_u32(ej);
    const uint32_t es_a = C > 1 ? peer(smem_u32(es), 0u) : smem_u32(es);
    const int nq = srcs.slots();
    PhiloxCache pc;
    for (int q0 = 0; q0 < nq; q0 += B) {  // rounds: the same count in every thread
      const int q = q0 + tid;
      uint32_t w[RV::kWords];
      uint32_t mm = 0u;
      int l = 0;
      const int sl = q < nq ? srcs.slot(q) : -1;
      if (sl >= 0) {
        l = cl[sl];
        if (gmax_value(gmax[l]) >= lc) {
          srcs.load_group(sl, w);
          mm = RV::ge_mask(w, lc);
        }
      }
      const int cnt = __popc(mm);
      if (__any_sync(0xFFFFFFFFu, cnt != 0)) {
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += t2;
        }
        int base = 0;
        if (lane == 31) base = (int)(C > 1 ? atom_peer_add(cnt_a, (uint32_t)incl) : atomicAdd(&sh.ecount, incl));
        int at = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
        while (mm) {
          const int e = __ffs(mm) - 1;
          mm &= mm - 1u;
          if (at < a.ent_cap) {
            const float v = RV::element(w, e);
            const int64_t j = rv.index(gb + l, e);
            const float sc = __fdiv_rn(v, T) + gumbel_of_word(pc.word(seed, step, (uint32_t)i, j));
            if (C > 1) {
              st_peer(ev_a + 4u * (uint32_t)at, __float_as_uint(v));
              st_peer(ej_a + 4u * (uint32_t)at, (uint32_t)j);
              st_peer(es_a + 4u * (uint32_t)at, __float_as_uint(sc));
            } else {
              ev[at] = v;
              ej[at] = (int32_t)j;
              es[at] = sc;
            }
          }
          ++at;
        }
      }
    }
    row_sync<C>();
    const int E = C > 1 && !lead ? (int)ld_peer(cnt_a) : sh.ecount;  // final after the barrier
    // the leader stays resident until every CTA has read its count (no CTA
    // may read the shared memory of one that has exited)
    if (C > 1) cluster_sync_all();
    if (E <= a.ent_cap) {
      if (!lead) return;  // nothing touches this CTA's shared memory any more
      // A short list: the leader CTA takes the cuts by direct counting (one
      // entry per thread: the count and the fixed-point mass of the entries
      // strictly above it; kept by top-k iff fewer than k lie above, by a
      // top-p target t iff the mass above is below t, the target of the joint
      // route p times the top-k set's mass), then the best stored score among
      // the kept entries.  A top-p cut whose candidates weigh less than the
      // target goes on to the warp's re-select below.
      if (E <= kLeadList) {
        unsigned long long* ms = reinterpret_cast<unsigned long long*>(hist);
        const bool own = tid < E;
        const float vx = own ? ev[tid] : 0.f;
        const unsigned long long mx = own ? mass_fixed(ex2(fmaf(vx, c, -R))) : 0ull;
        if (own) ms[tid] = mx;
        __syncthreads();
        unsigned int cgt = 0u;
        unsigned long long mgt = 0ull;
        if (own)
          for (int y = 0; y < E; ++y) {
            const bool gt = ev[y] > vx;
            cgt += gt ? 1u : 0u;
            mgt += gt ? ms[y] : 0ull;
          }
        bool keep = own && (kind != KIND_TOPK || cgt < (unsigned int)k);
        bool decided = true;
        if (kind == KIND_TOPP || p_on) {
          unsigned long long w = keep ? mx : 0ull, unused = 0ull;
          cta_sum2<B>(sh, w, unused);
          unsigned long long tg = target;
          if (kind == KIND_TOPK) {
            tg = __float2ull_ru(fmaxf(p, 0.f) * __ull2float_rn(w));
            if (tg < 1ull) tg = 1ull;
          } else if (w < target) {
            decided = false;
          }
          keep = keep && mgt < tg;
        }
        if (decided) {
          const unsigned long long kb = cta_max_key<B>(sh, keep ? argmax_key(es[tid], ej[tid]) : 0ull);
          if (tid == 0) a.out_ids[i] = argmax_index(kb);
          return;
        }
      }
      // The leader's warp 0 finishes the row alone: the cuts over the entry
      // list (warp-level selects), then the best stored score at or above the
      // cut.  The other warps are done.
      if (warp != 0) return;
      const WarpEntries wl{ev, E};
      SelResult q1 = warp_select<TIn>(hist, wl, K::key(lc), key_max, target, -1.f, R, c, kind == KIND_TOPP);
      if (!(kind == KIND_TOPP && q1.short_total && lc > -FLT_MAX)) {
        uint32_t lk = q1.key;
        if (kind == KIND_TOPK && p_on) lk = warp_select<TIn>(hist, wl, lk, key_max, 0ull, fmaxf(p, 0.f), R, c, true).key;
        const float tau = K::value(lk);
        unsigned long long kb = 0ull;
        for (int q = lane; q < E; q += 32)
          if (ev[q] >= tau) {
            const unsigned long long kq = argmax_key(es[q], ej[q]);
            kb = kq > kb ? kq : kb;
          }
        kb = warp_max_key(kb);
        if (lane == 0) a.out_ids[i] = argmax_index(kb);
        return;
      }
      // The candidates weigh less than the target (the cut lies below the
      // bound): the warp selects again over every finite entry of the whole
      // row, re-read from global memory, and draws the Gumbel-max over the
      // kept entries (off the common path).
      const WarpRow<TIn> wr{&rv};
      const SelResult q2 = warp_select<TIn>(hist, wr, K::key(-FLT_MAX), key_max, target, -1.f, R, c, true);
      Scorer s4{T, seed, step, (uint32_t)i, false, 0ull, PhiloxCache{}};
      wr.each(K::value(q2.key), s4);
      const unsigned long long kb = warp_max_key(s4.best);
      if (lane == 0) a.out_ids[i] = argmax_index(kb);
      return;
    }
    // the entry list overflowed: every CTA takes the general path below
  }

  SelResult r1 = split_select<TIn, C, B, SplitCfg<C>::kBinBits>(sh, hist, srcs, K::key(lc), key_max, target, -1.f, R, c, kind == KIND_TOPP);
  if (kind == KIND_TOPP && r1.short_total && lc > -FLT_MAX) {
    // the candidates weigh less than the target: the cut lies below the
    // bound, select again over every finite entry of the slices
    srcs.mode = SRC_SLICE;
    r1 = split_select<TIn, C, B, SplitCfg<C>::kBinBits>(sh, hist, srcs, K::key(-FLT_MAX), key_max, target, -1.f, R, c, true);
  }
  uint32_t lo_key = r1.key;
  if (kind == KIND_TOPK && p_on) {
    const SelResult r2 = split_select<TIn, C, B, SplitCfg<C>::kBinBits>(sh, hist, srcs, lo_key, key_max, 0ull, fmaxf(p, 0.f), R, c, true);
    lo_key = r2.key;
  }
  // ---- Gumbel-max over the kept set ---------------------------------------
  Scorer s3{T, seed, step, (uint32_t)i, false, 0ull, PhiloxCache{}};
  srcs.each_run(K::value(lo_key), s3);
  finish(s3.best);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Group-maximum slots of one CTA's slice (a multiple of 8: the list that
// follows stays 16-byte aligned).
inline int split_gslots(int64_t vocab, int C) {
  const int64_t ng = group_slots(vocab);
  return (int)(((ng + C - 1) / C + 7) & ~(int64_t)7);
}

// Bytes of one captured group (its words and its slice-local index) and of
// one candidate entry of the leader's list (value, index, Gumbel score).
inline size_t split_group_bytes(ls_dtype dtype) { return (dtype == LS_DTYPE_BF16 ? 32u : 64u) + 4u; }
constexpr size_t kSplitEntryBytes = 12;

template <int C>
inline size_t split_smem_bytes(int64_t vocab, ls_dtype dtype, int cap, int ecap) {
  constexpr int NB = 1 << SplitCfg<C>::kBinBits;
  return sizeof(SplitShared) + (size_t)NB * 8u + (size_t)split_gslots(vocab, C) * 2u +
         (size_t)cap * split_group_bytes(dtype) + (size_t)ecap * kSplitEntryBytes;
}

// Shared-memory budget of one CTA: what lets all n C CTAs of the grid (or
// as many as the registers allow) be resident at once (228 KB per SM, 1 KB of
// it reserved per CTA), never more than the cluster size's cap (one CTA per
// row: 96 KB, leaving the SM's L1 room for the streaming loads in flight).
template <int C>
inline size_t split_budget(int32_t n, int sms) {
  const int64_t ctas = (int64_t)n * C;
  int64_t per_sm = sms > 0 ? (ctas + sms - 1) / sms : 1;
  if (per_sm > SplitCfg<C>::kMinBlocks) per_sm = SplitCfg<C>::kMinBlocks;  // more run in waves anyway
  if (per_sm < 1) per_sm = 1;
  size_t b = (size_t)(228 * 1024) / (size_t)per_sm;
  b = b > 1024 ? b - 1024 : 0;
  return b < SplitCfg<C>::kBudget ? b : SplitCfg<C>::kBudget;
}

// Capacities within the budget: captured-group slots take up to 70% of what
// the fixed part leaves (never more than the slice holds; a multiple of the
// warps for an equal segment per warp, plus a shared pool of about a quarter,
// or of the whole slice when that fits), the leader's entry list -- the
// candidates of the whole row are gathered there -- takes the rest (at least
// 256 entries).
template <int C>
inline void split_capacity(int64_t vocab, ls_dtype dtype, size_t budget, int& cap, int& pool, int& ecap) {
  constexpr int B = SplitCfg<C>::kB;
  constexpr int W = B / 32;
  const int64_t slice = split_gslots(vocab, C);
  const size_t base = split_smem_bytes<C>(vocab, dtype, 0, 0);
  const size_t room = budget > base ? budget - base : 0;
  int64_t g = (int64_t)(room * 7 / 10 / split_group_bytes(dtype));
  g = g < slice ? g : slice;
  // a warp captures at most 32 lanes x ceil(slice / B) groups
  const int64_t most = 32 * ((slice + B - 1) / B);
  int64_t own = (g * 3 / 4) / W;
  own = own < most ? own : most;
  own = own > 4 ? own : 4;
  int64_t pl = g - own * W;
  pl = pl > 32 ? pl : 32;
  // a group is captured at most once: a pool as large as the slice never
  // overflows, whichever warps capture -- take it when it fits
  if ((own * W + slice) * (int64_t)split_group_bytes(dtype) <= (int64_t)(room * 7 / 10)) pl = slice;
  cap = (int)(own * W + pl);
  pool = (int)pl;
  const size_t used = (size_t)cap * split_group_bytes(dtype);
  int64_t e = room > used ? (int64_t)((room - used) / kSplitEntryBytes) : 0;
  e = e > 256 ? e : 256;
  ecap = (int)(e & ~(int64_t)3);
}

inline int split_sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && (v = cache[dev].load(std::memory_order_relaxed)) > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

template <typename TIn, int ROUTE, int C>
static ls_status launch_split(const KernelArgs& a, int32_t n, size_t smem, cudaStream_t stream) {
  auto kern = split_sampler_kernel<TIn, ROUTE, C>;
  static std::atomic<size_t> opted[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LS_ERR_CUDA;
  if (smem > 48 * 1024 && (dev < 0 || dev >= kMaxDevices || opted[dev].load(std::memory_order_relaxed) < smem)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return LS_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) opted[dev].store(smem, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n * (unsigned)C);
  cfg.blockDim = dim3(SplitCfg<C>::kB);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return LS_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}

template <int C>
ls_status dispatch_split(KernelArgs a, ls_dtype dtype, int route, int32_t n, cudaStream_t stream) {
  if ((int64_t)n * C > 0x7FFFFFFFll) return LS_ERR_UNSUPPORTED;  // grid size
  a.gslot_cap = split_gslots(a.vocab, C);
  split_capacity<C>(a.vocab, dtype, split_budget<C>(n, split_sm_count()), a.cand_cap, a.pool_cap, a.ent_cap);
  const size_t smem = split_smem_bytes<C>(a.vocab, dtype, a.cand_cap, a.ent_cap);
  const int lim = max_dyn_smem();
  if (lim <= 0) return LS_ERR_CUDA;
  if (smem > (size_t)lim) return LS_ERR_UNSUPPORTED;
  if (dtype == LS_DTYPE_BF16) {
    switch (route) {
      case ROUTE_NONE: return launch_split<bf16_tag, ROUTE_NONE, C>(a, n, smem, stream);
      case ROUTE_K: return launch_split<bf16_tag, ROUTE_K, C>(a, n, smem, stream);
      case ROUTE_P: return launch_split<bf16_tag, ROUTE_P, C>(a, n, smem, stream);
      default: return launch_split<bf16_tag, ROUTE_KP, C>(a, n, smem, stream);
    }
  }
  switch (route) {
    case ROUTE_NONE: return launch_split<float, ROUTE_NONE, C>(a, n, smem, stream);
    case ROUTE_K: return launch_split<float, ROUTE_K, C>(a, n, smem, stream);
    case ROUTE_P: return launch_split<float, ROUTE_P, C>(a, n, smem, stream);
    default: return launch_split<float, ROUTE_KP, C>(a, n, smem, stream);
  }
}

}  // namespace lsg
