// ls_device.cuh -- device building blocks of the GB300 token sampler.
//
// Keys, Philox4x32-10, Gumbel noise, block-wide reductions and scans.  Nothing
// here is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lsg {

constexpr int kThreads = 512;            // threads per CTA (one CTA per sampled row)
constexpr int kWarps = kThreads / 32;
constexpr int kGroup = 16;               // logits per group: one 32-byte sector of bf16, two of fp32
constexpr int kBinBits = 11;
constexpr int kBins = 1 << kBinBits;     // bins per radix-select level
constexpr int kBinsPerThread = kBins / kThreads;
static_assert(kBins % kThreads == 0, "bins must split evenly over threads");

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();
constexpr float kLog2e = 1.4426950408889634f;
// Fixed-point scale of probability masses (weights are <= 1 relative to the row max).
constexpr float kMassScale = 1099511627776.0f;  // 2^40
// Span of the Gumbel noise for u in [2^-24, 1 - 2^-24]: g in [-2.81161, 16.63553].
// An entry whose z is more than this (plus a rounding margin) below the row maximum
// can never win the Gumbel-max.
constexpr float kGumbelSpan = 19.4572f;

// ---------------------------------------------------------------------------
// Order-preserving keys: key(a) < key(b) <=> a < b for non-NaN floats, with -0
// and +0 mapped to the same key (they compare equal as floats).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f32_key(float v) {
  uint32_t b = __float_as_uint(v);
  if ((b << 1) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float f32_from_key(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

// Keys used by the radix select.  bf16 values have only 16 significant bits, so
// their keys are the top 16 bits of the fp32 key (two select levels at most);
// fp32 values use the full 32-bit key (three levels at most).
template <typename TIn>
struct KeyOps;

template <>
struct KeyOps<float> {
  static constexpr int kBits = 32;
  __device__ __forceinline__ static uint32_t key(float v) { return f32_key(v); }
  __device__ __forceinline__ static float value(uint32_t k) { return f32_from_key(k); }
};

struct bf16_tag {};
template <>
struct KeyOps<bf16_tag> {
  static constexpr int kBits = 16;
  // For a float that is not a bf16 value this rounds the key down, i.e. towards
  // the next bf16 value in key order; every bf16 value >= v keeps key >= key(v).
  __device__ __forceinline__ static uint32_t key(float v) { return f32_key(v) >> 16; }
  __device__ __forceinline__ static float value(uint32_t k) {
    uint32_t full = (k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu);
    return f32_from_key(full);
  }
};

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 products by the published
// multipliers, cross-xored with the other counter words and the round key; the
// key advances by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// Four Philox4x32-10 blocks at once (counters c[0..3], one key): the same
// rounds as philox4x32_10, four independent chains per round, the ten rounds
// kept a loop (a short body: it serves code that runs about once per warp).
__device__ __forceinline__ void philox4x32_10_x4(uint4 (&c)[4], uint2 k) {
#pragma unroll 1
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo0 = 0xD2511F53u * c[q].x, hi0 = __umulhi(0xD2511F53u, c[q].x);
      const uint32_t lo1 = 0xCD9E8D57u * c[q].z, hi1 = __umulhi(0xCD9E8D57u, c[q].z);
      c[q] = make_uint4(hi1 ^ c[q].y ^ k.x, lo1, hi0 ^ c[q].w ^ k.y, lo0);
    }
  }
}

// Noise word of vocabulary entry j for (seed, step, row): lane j%4 of
// Philox(counter = (j/4, row, lo32 step, hi32 step), key = (lo32 seed, hi32 seed)).
__device__ __forceinline__ uint32_t noise_word(uint64_t seed, uint64_t step, uint32_t row, int64_t j) {
  const uint4 blk = philox4x32_10(make_uint4((uint32_t)((uint64_t)j >> 2), row, (uint32_t)step,
                                             (uint32_t)(step >> 32)),
                                  make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  const uint32_t lane = (uint32_t)j & 3u;
  return lane == 0 ? blk.x : lane == 1 ? blk.y : lane == 2 ? blk.z : blk.w;
}

// g = -ln(-ln u), u = (2*(x>>9)+1) * 2^-24 (exact in fp32, never 0 or 1).
__device__ __forceinline__ float gumbel_of_word(uint32_t x) {
  const float u = __uint2float_rn(((x >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
  return -logf(-logf(u));
}

// Argmax key: larger score first, lower index first on an exact tie.
__device__ __forceinline__ unsigned long long argmax_key(float s, int64_t j) {
  return ((unsigned long long)f32_key(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)j);
}
__device__ __forceinline__ int32_t argmax_index(unsigned long long key) {
  return (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

// ---------------------------------------------------------------------------
// Packed arithmetic (sm_100+): two fp32 lanes in a 64-bit register, bf16x2
// max, 3-input fp32 max, and the hardware base-2 exponential.
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(f32x2 r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Lane-wise max of two bf16 pairs; a NaN lane yields the other operand.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Max of three floats; NaN inputs are ignored like fmaxf.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// take ? cand : cur, opaque to the compiler so that a chain of these over a
// register array is not turned back into (local-memory) indexing.
__device__ __forceinline__ uint32_t select_word(uint32_t cur, uint32_t cand, bool take) {
  uint32_t r;
  asm("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %3, 0;\n\tselp.b32 %0, %1, %2, p;\n\t}"
      : "=r"(r)
      : "r"(cand), "r"(cur), "r"((uint32_t)take));
  return r;
}

// 2^x with results below 2^-126 flushed to zero (they are far below the
// resolution of any sum here).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Block-wide reductions (all threads must call; result returned to all).
// `red` must hold kWarps elements of the reduced type (8-byte aligned).
// ---------------------------------------------------------------------------
template <typename T, typename Op>
__device__ __forceinline__ T warp_reduce(T v, Op op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, Op op, T* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_reduce(v, op);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  T r = red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) r = op(r, red[i]);
  return r;
}

// Warp-wide max / min of a float in one instruction (NaN inputs ignored).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float warp_min(float v) {
  float r;
  asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

struct OpAddF {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

}  // namespace lsg
