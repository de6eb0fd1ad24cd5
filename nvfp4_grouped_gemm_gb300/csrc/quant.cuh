// The activation quantiser Q (device side), shared by the kernels that quantise x and h.
//
// Q (the pages never quantise activations; the block-scaled FP4 x FP4 tensor-core product
// needs it): s = the smallest integer with amax_row <= 6*448*2^s; block scale = the UE4M3
// value nearest to amax_16 / (6*2^s) (ties to the even encoding); code = the E2M1 value
// nearest to v / (scale*2^s), saturating at 6, ties to even, sign bit iff v < 0.  Every
// decision is an exact float32 comparison of |v|*2^-s against midpoint*scale products.
#pragma once

#include <cstdint>

#include "moe_internal.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// number formats (written from the format definitions)
// ---------------------------------------------------------------------------

// Value of UE4M3 encoding b (0 <= b <= 0x7E).
__device__ __forceinline__ float ue4m3_val(int b) {
  const int e = b >> 3, m = b & 7;
  if (e == 0) return (float)m * (1.0f / 512.0f);                    // m/8 * 2^-6
  return __uint_as_float((uint32_t)(e + 120) << 23 | (uint32_t)m << 20);   // (1+m/8)*2^(e-7)
}

// Decision threshold between UE4M3 encodings j and j+1, times 6: 3 * (v(j) + v(j+1)).
__device__ __forceinline__ float ue4m3_thr6(int j) { return 3.0f * (ue4m3_val(j) + ue4m3_val(j + 1)); }

// Threshold j "passed" by key: above it, or on it when the upper neighbour is the even code.
__device__ __forceinline__ bool ue4m3_passed(float key, int j) {
  const float t = ue4m3_thr6(j);
  return key > t || (key == t && ((j + 1) & 1) == 0);
}

// Nearest UE4M3 encoding to key/6 (key = block amax * 2^-s <= 2688), ties to even: the
// number of thresholds passed.  A first guess from the float bits of key/6 is corrected
// by exact comparisons with the neighbouring thresholds.
__device__ __forceinline__ int ue4m3_code_of(float key) {
  const float r = key * (1.0f / 6.0f);
  int cand;
  if (r < 0.015625f) {
    cand = (int)(r * 512.0f);                        // subnormal encodings m/8 * 2^-6
  } else {
    const uint32_t b = __float_as_uint(r);
    const int e = (int)((b >> 23) & 0xff) - 127;       // -6 .. 8
    cand = ((e + 7) << 3) | (int)((b >> 20) & 7);
  }
  cand = min(max(cand, 0), 126);
  while (cand < 126 && ue4m3_passed(key, cand)) ++cand;
  while (cand > 0 && !ue4m3_passed(key, cand - 1)) --cand;
  return cand;
}

// key[i] * 2^-s in place: one multiply by the exact power of two m = 2^-s when that is a
// float (the same correctly rounded value as ldexpf), else ldexpf.  The choice is made once
// for the whole array, so the common case is a plain multiply per element (a per-element
// select could let the compiler evaluate the long ldexpf path for every element).
template <int N>
__device__ __forceinline__ void scale_down_n(float (&key)[N], int s, bool fast, float m) {
  if (fast) {
#pragma unroll
    for (int i = 0; i < N; ++i) key[i] *= m;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) key[i] = ldexpf(key[i], -s);
  }
}

// Row exponent: smallest s with amax <= 2688 * 2^s (2688 = 0.65625 * 2^12).
__device__ __forceinline__ int row_exp_of(float amax) {
  if (!(amax > 0.0f)) return 0;
  int ea;
  const float m = frexpf(amax, &ea);
  return ea - 12 + (m > 0.65625f ? 1 : 0);
}

// Quantise 16 values (already |v| * 2^-s in `key`, signs in `neg`) with block code sbc.
// The E2M1 magnitude code of key / scale is the number of midpoints passed between the
// values 0 .5 1 1.5 2 3 4 6 (midpoints .25 .75 1.25 1.75 2.5 3.5 5).  The seven decision
// thresholds midpoint * scale are exact f32 products, formed once per block; a key passes
// an even-indexed threshold when above it and an odd-indexed one when at or above it, so
// a tie goes to the even code.
__device__ __forceinline__ uint64_t quant_block(const float (&key)[16], uint32_t negmask, int sbc) {
  if (sbc == 0) return 0ull;
  const float sbv = ue4m3_val(sbc);
  const float t0 = 0.25f * sbv, t1 = 0.75f * sbv, t2 = 1.25f * sbv, t3 = 1.75f * sbv;
  const float t4 = 2.5f * sbv, t5 = 3.5f * sbv, t6 = 5.0f * sbv;
  // thresholds are increasing, so the count is found by a three-step search
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float v = key[i];
    const bool b2 = v >= t3;
    const bool b1 = v >= (b2 ? t5 : t1);
    const bool b0 = v > (b2 ? (b1 ? t6 : t4) : (b1 ? t2 : t0));
    const uint32_t c = (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u) | (((negmask >> i) & 1u) << 3);
    if (i < 8) lo |= c << (4 * i); else hi |= c << (4 * (i - 8));
  }
  const uint64_t out = (uint64_t)lo | ((uint64_t)hi << 32);
  return out;
}

}  // namespace
}  // namespace moe
