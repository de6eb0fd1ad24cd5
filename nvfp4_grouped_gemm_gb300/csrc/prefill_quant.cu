// Activation quantisers (the quantiser Q itself is in quant.cuh) and the prefill combine:
//
//   quant_x_kernel      Q(x): each token's bf16 row to NVFP4 with a power-of-two row scale
//                       (one CTA per token), written to every CSR row of the token's pairs
//   quant_h_kernel      Q(h) per CSR row
//   combine_f16_kernel  y[t] = sum_j w[t,j] * z16[pos_j] * 2^(e_j + c_F), ascending j
//   slice_x_kernel, slice_h_kernel   the decode tensor-core form's four residual slices
//                       of each x row (per pair or per token, written to the pairs' rows)
//                       and h row
#include <cmath>

#include "moe_internal.cuh"
#include "quant.cuh"

namespace moe {

namespace {

// ---------------------------------------------------------------------------
// Q(x): one CTA per token, one thread per 16-value block (H <= 16 * blockDim.x), the
// result copied to each of the token's CSR rows
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_x_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                      int k, const int32_t* __restrict__ pair_pos,
                                                      uint8_t* __restrict__ qc,
                                                      uint8_t* __restrict__ qs,
                                                      int32_t* __restrict__ qe) {
  __shared__ float red[8];
  __shared__ int s_pos[kMaxK];
  const int t = blockIdx.x, b = threadIdx.x;
  const int lane = b & 31, warp = b >> 5;
  const int nblk = H / 16;
  const bool has = b < nblk;
  uint32_t w[8];
  {
    const uint4* p = reinterpret_cast<const uint4*>(x + (size_t)t * H + b * 16);
    const uint4 v0 = has ? __ldg(p) : make_uint4(0, 0, 0, 0);
    const uint4 v1 = has ? __ldg(p + 1) : make_uint4(0, 0, 0, 0);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
    amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xffff0000u)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = 0.0f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const int s = row_exp_of(amax);
  const bool fast = s >= -127 && s <= 149;
  const float m = fast ? pow2f(-s) : 0.0f;
  float key[16];
  uint32_t neg = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
    key[2 * i] = fabsf(lo);
    key[2 * i + 1] = fabsf(hi);
    neg |= (lo < 0.0f ? 1u : 0u) << (2 * i);
    neg |= (hi < 0.0f ? 1u : 0u) << (2 * i + 1);
  }
  scale_down_n(key, s, fast, m);
  float bmax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, key[i]);
  const int sbc = ue4m3_code_of(bmax);
  const uint64_t codes = quant_block(key, neg, sbc);
  // the codes depend on x alone and are formed while the CSR kernel runs; where they go
  // (the token's CSR rows) waits for it
  pdl_wait();
  pdl_trigger();
  if (b < k) s_pos[b] = pair_pos[(size_t)t * k + b];
  __syncthreads();
  if (!has) return;
  for (int j = 0; j < k; ++j) {
    const int pj = s_pos[j];
    if (pj < 0) continue;                          // invalid expert id: the pair has no row
    *reinterpret_cast<uint64_t*>(qc + (size_t)pj * (H / 2) + b * 8) = codes;
    qs[(size_t)pj * nblk + b] = (uint8_t)sbc;
    if (b == 0) qe[pj] = s;
  }
}

// ---------------------------------------------------------------------------
// Q(h): one warp per CSR row, the row's blocks in registers as for Q(x)
// ---------------------------------------------------------------------------
// LPR lanes per row (32 / LPR rows per warp), lane l of a row taking its blocks l, l + LPR,
// ...: LPR is chosen so that the row's F/16 blocks fill every lane in every pass
// (F = 640: 8 lanes x 5 blocks), since the per-block work is ALU-bound.  Two passes over
// the row: the largest magnitude (reduced over the row's lanes), then each block read again
// (from L1) and quantised, so that no lane holds more than one block.
template <int LPR>
__global__ void __launch_bounds__(256) quant_h_kernel(const float* __restrict__ h, int P, int F,
                                                      int sf_pitch,
                                                      const int32_t* __restrict__ offsets, int E,
                                                      uint8_t* __restrict__ qc,
                                                      uint8_t* __restrict__ qs,
                                                      int32_t* __restrict__ qe) {
  static_assert(LPR >= 4 && LPR <= 32 && (LPR & (LPR - 1)) == 0, "lanes per row");
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;
  const int r = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * (32 / LPR) + lane / LPR;
  const bool valid = r < P && r < offsets[E];
  const float* row = h + (size_t)r * F;
  const int nblk = F / 16;
  float amax = 0.0f;
  if (valid)
    for (int b = sub; b < nblk; b += LPR) {
      const float4* p = reinterpret_cast<const float4*>(row + b * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = __ldg(p + q);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
    }
  // the row's lanes are LPR consecutive lanes starting at a multiple of LPR
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (!valid) return;
  const int s = row_exp_of(amax);
  const bool fast = s >= -127 && s <= 149;
  const float m = fast ? pow2f(-s) : 0.0f;
  if (sub == 0) qe[r] = s;
  for (int b = sub; b < nblk; b += LPR) {
    const float4* p = reinterpret_cast<const float4*>(row + b * 16);
    float key[16];
    uint32_t neg = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v4 = __ldcs(p + q);
      const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        key[4 * q + e] = fabsf(vv[e]);
        neg |= (vv[e] < 0.0f ? 1u : 0u) << (4 * q + e);
      }
    }
    scale_down_n(key, s, fast, m);
    float bmax = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) bmax = fmaxf(bmax, key[e]);
    const int sbc = ue4m3_code_of(bmax);
    *reinterpret_cast<uint64_t*>(qc + (size_t)r * (F / 2) + b * 8) = quant_block(key, neg, sbc);
    qs[(size_t)r * sf_pitch + b] = (uint8_t)sbc;
  }
}

// ---------------------------------------------------------------------------
// Activation slices for the decode form of the tensor-core path: a row v is written as
// NS rows q_0..q_{NS-1}, each the quantiser Q of what the earlier ones left over
// (q_i = Q(v - q_0 - ... - q_{i-1}), exact f32 residuals), so that sum_i q_i approximates v
// to about 6^-NS of each block's largest magnitude.  The GEMM multiplies every slice and
// sums the NS accumulator rows of a pair in its epilogue.  One thread per 16-value block.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float e2m1_mag(uint32_t m) {      // magnitude code 0..7
  return m < 2 ? 0.5f * (float)m : __uint_as_float(((m >> 1) + 126u) << 23 | (m & 1u) << 22);
}

// Row max of |v| over the CTA (one value per thread in `x`); `red` holds one slot per warp.
__device__ __forceinline__ float cta_max(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  float m = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  return m;
}

// One slice of part of a block: the EPT residual values r of this thread (elements
// EPT*q .. EPT*q + EPT-1 of a 16-value block whose other parts sit in the neighbouring lanes).
// Row exponent from row_amax, block scale from the block's max key (shared by the block's
// lanes), E2M1 codes as in quant_block; r becomes the remainder.  Returns the EPT codes as
// 4*EPT bits.
template <int EPT>
__device__ __forceinline__ uint32_t slice_part(float (&r)[EPT], float row_amax, int& s_out,
                                               int& sbc_out) {
  const int s = row_exp_of(row_amax);
  const bool fast = s >= -127 && s <= 149;
  const float m = fast ? pow2f(-s) : 0.0f;
  float key[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) key[i] = fabsf(r[i]);
  scale_down_n(key, s, fast, m);
  float bmax = 0.0f;
#pragma unroll
  for (int i = 0; i < EPT; ++i) bmax = fmaxf(bmax, key[i]);
#pragma unroll
  for (int o = 1; o < 16 / EPT; o <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
  const int sbc = ue4m3_code_of(bmax);
  uint32_t codes = 0;
  if (sbc != 0) {
    const float sbv = ue4m3_val(sbc);
    const float t0 = 0.25f * sbv, t1 = 0.75f * sbv, t2 = 1.25f * sbv, t3 = 1.75f * sbv;
    const float t4 = 2.5f * sbv, t5 = 3.5f * sbv, t6 = 5.0f * sbv;
    // each code's value times 2^s, removed from the residual: the values are formed first,
    // then scaled by one exact power-of-two multiply (ldexpf only when 2^s is not a float)
    float qv[EPT];
    uint32_t negs = 0;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const float v = key[i];
      // the same three-step threshold search as quant_block (ties to the even code)
      const bool b2 = v >= t3;
      const bool b1 = v >= (b2 ? t5 : t1);
      const bool b0 = v > (b2 ? (b1 ? t6 : t4) : (b1 ? t2 : t0));
      const uint32_t mag = (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u);
      const bool neg = r[i] < 0.0f;
      negs |= (neg ? 1u : 0u) << i;
      codes |= (mag | (neg ? 8u : 0u)) << (4 * i);
      qv[i] = e2m1_mag(mag) * sbv;                        // exact: <= 6 significant bits
    }
    scale_down_n(qv, -s, s >= -126 && s <= 127, s >= -126 && s <= 127 ? pow2f(s) : 0.0f);
#pragma unroll
    for (int i = 0; i < EPT; ++i) r[i] = ((negs >> i) & 1u) ? r[i] + qv[i] : r[i] - qv[i];
  }
  s_out = s;
  sbc_out = sbc;
  return codes;
}

// Elements per thread in the slice kernels: a 16-value block is shared by two lanes.
constexpr int kSliceEPT = 8;

// x: 16/EPT threads per 16-value block (thread (16/EPT)*b + q holds elements 16b + EPT*q
// ..).  PER_PAIR: one CTA per pair p = t*k + j, which forms the slices of its token's row
// and writes them to its own pair's NS rows (pair_pos * NS + i); the k CTAs of a token
// repeat the work, spreading it over k times more SMs when there are few tokens.
// Otherwise one CTA per token, writing to all k of its pairs' rows.  The slices depend only
// on x, so they are formed before the wait; only the stores wait for the CSR.
template <int NS, bool PER_PAIR>
__global__ void __launch_bounds__(1024) slice_x_kernel(const uint16_t* __restrict__ x, int H, int k,
                                                       const int32_t* __restrict__ pair_pos,
                                                       uint8_t* __restrict__ qc,
                                                       uint8_t* __restrict__ qs,
                                                       int32_t* __restrict__ qe) {
  constexpr int EPT = kSliceEPT, TPB = 16 / EPT;
  __shared__ float red[NS][32];
  __shared__ int s_pos[kMaxK];
  const int t = PER_PAIR ? blockIdx.x / k : blockIdx.x, tid = threadIdx.x;
  const int b = tid / TPB, q = tid % TPB;
  const int nblk = H / 16;
  const bool has = b < nblk;
  float r[EPT];
  {
    const uint4 w = has ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + 16 * b + EPT * q))
                        : make_uint4(0, 0, 0, 0);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r[2 * i] = __uint_as_float(ww[i] << 16);
      r[2 * i + 1] = __uint_as_float(ww[i] & 0xffff0000u);
    }
  }
  uint32_t codes[NS];
  int sbc[NS], sx[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) a = fmaxf(a, fabsf(r[e]));
    codes[i] = slice_part<EPT>(r, cta_max(a, red[i]), sx[i], sbc[i]);
  }
  pdl_wait();                                       // pair_pos is complete
  pdl_trigger();
  const int npairs = PER_PAIR ? 1 : k;
  // the positions of this CTA's pairs, read once (all loads in flight together)
  if (tid < npairs) s_pos[tid] = pair_pos[PER_PAIR ? (size_t)blockIdx.x : (size_t)t * k + tid];
  __syncthreads();
  if (!has) return;
  for (int j = 0; j < npairs; ++j) {
    const int pos = s_pos[j];
    if (pos < 0) continue;                          // invalid expert id: the pair has no rows
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const size_t row = (size_t)pos * NS + i;
      *reinterpret_cast<uint32_t*>(qc + row * (H / 2) + 8 * b + (EPT / 2) * q) = codes[i];
      if (q == 0) qs[row * nblk + b] = (uint8_t)sbc[i];
      if (tid == 0) qe[row] = sx[i];
    }
  }
}

// h: one CTA per CSR row (f32 h, rows in CSR order), rows r * NS + i.
template <int NS>
__global__ void __launch_bounds__(1024) slice_h_kernel(const float* __restrict__ h, int F,
                                                       int sf_pitch,
                                                       const int32_t* __restrict__ offsets, int E,
                                                       uint8_t* __restrict__ qc,
                                                       uint8_t* __restrict__ qs,
                                                       int32_t* __restrict__ qe) {
  constexpr int EPT = kSliceEPT, TPB = 16 / EPT;
  __shared__ float red[NS][32];
  pdl_wait();
  pdl_trigger();
  const int row0 = blockIdx.x, tid = threadIdx.x;
  if (row0 >= offsets[E]) return;                  // uniform over the CTA
  const int b = tid / TPB, q = tid % TPB;
  const int nblk = F / 16;
  const bool has = b < nblk;
  float r[EPT];
  {
    const float4* p = reinterpret_cast<const float4*>(h + (size_t)row0 * F + 16 * b + EPT * q);
#pragma unroll
    for (int i = 0; i < EPT / 4; ++i) {
      const float4 v = has ? __ldcs(p + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
    }
  }
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) a = fmaxf(a, fabsf(r[e]));
    int s, sbc;
    const uint32_t c = slice_part<EPT>(r, cta_max(a, red[i]), s, sbc);
    if (has) {
      const size_t row = (size_t)row0 * NS + i;
      *reinterpret_cast<uint32_t*>(qc + row * (F / 2) + 8 * b + (EPT / 2) * q) = c;
      if (q == 0) qs[row * sf_pitch + b] = (uint8_t)sbc;
      if (tid == 0) qe[row] = s;
    }
  }
}

// combine for the prefill path: y[t, :] = sum_j w[t, j] * f32(z16[pos_j, :]) * 2^(e_j + cF)
// The token's k positions and scaled weights are read once into shared memory; the
// partial rows are then loaded eight pairs at a time and summed in ascending j.
// Columns [c0, c0 + HS) of y from a partial slice [P][HS].
__global__ void __launch_bounds__(256)
combine_f16_kernel(const float* __restrict__ w, const int32_t* __restrict__ pair_pos,
                   const __half* __restrict__ partial, const int32_t* __restrict__ hexp,
                   int shift, int H, int c0, int HS, int k, float* __restrict__ y) {
  __shared__ int s_pos[kMaxK];
  __shared__ float s_w[kMaxK];
  const int t = blockIdx.y;
  if (threadIdx.x < k) {
    const int pos = pair_pos[(size_t)t * k + threadIdx.x];
    s_pos[threadIdx.x] = pos;
    s_w[threadIdx.x] = pos >= 0 ? ldexpf(w[(size_t)t * k + threadIdx.x], hexp[pos] + shift) : 0.0f;
  }
  __syncthreads();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) * 8;   // column within the slice
  if (r >= HS) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < k; j0 += 8) {
    uint4 z[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q;
      const int pos = j < k ? s_pos[j] : -1;
      z[q] = pos >= 0 ? __ldcs(reinterpret_cast<const uint4*>(partial + (size_t)pos * HS + r))
                      : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q;
      if (j >= k || s_pos[j] < 0) continue;
      const float wj = s_w[j];
      const uint32_t zz[4] = {z[q].x, z[q].y, z[q].z, z[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&zz[e]));
        acc[2 * e] = fmaf(wj, f.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(wj, f.y, acc[2 * e + 1]);
      }
    }
  }
  float4* out = reinterpret_cast<float4*>(y + (size_t)t * H + c0 + r);
  __stcs(out, make_float4(acc[0], acc[1], acc[2], acc[3]));
  __stcs(out + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
}

}  // namespace

cudaError_t launch_quant_x(const uint16_t* x_bf16, int T, int H, int k, const int32_t* pair_pos,
                           uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s) {
  const int threads = (H / 16 + 31) / 32 * 32;     // one thread per 16-value block
  if (threads > 256) return cudaErrorInvalidValue;
  return launch_pdl(quant_x_kernel, dim3(T), dim3(threads), 0, s, x_bf16, T, H, k, pair_pos, qc,
                    qs, qe);
}

cudaError_t launch_slice_x(const uint16_t* x_bf16, int T, int H, int k, const int32_t* pair_pos,
                           uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s) {
  const int threads = (H / kSliceEPT + 31) / 32 * 32;
  if (threads > 1024) return cudaErrorInvalidValue;
  // one CTA per pair while that keeps at most ~4 CTAs per SM: few tokens alone would leave
  // most SMs idle (the k-fold repeated work is cheaper than the idle SMs up to there)
  if ((long long)T * k <= 4LL * num_sms())
    return launch_pdl(slice_x_kernel<kDecodeSlices, true>, dim3(T * k), dim3(threads), 0, s,
                      x_bf16, H, k, pair_pos, qc, qs, qe);
  return launch_pdl(slice_x_kernel<kDecodeSlices, false>, dim3(T), dim3(threads), 0, s, x_bf16,
                    H, k, pair_pos, qc, qs, qe);
}

cudaError_t launch_slice_h(const float* h, int P, int F, int sf_pitch, const int32_t* offsets,
                           int E, uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s) {
  const int threads = (F / kSliceEPT + 31) / 32 * 32;
  if (threads > 1024) return cudaErrorInvalidValue;
  return launch_pdl(slice_h_kernel<kDecodeSlices>, dim3(P), dim3(threads), 0, s, h, F, sf_pitch,
                    offsets, E, qc, qs, qe);
}
cudaError_t launch_quant_h(const float* h, int P, int F, int sf_pitch, const int32_t* offsets,
                           int E, uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s) {
  // lanes per row: the fewest idle lane-passes (lanes x passes - blocks), ties to more lanes
  const int nblk = F / 16;
  int lpr = 32, waste = 32 * ((nblk + 31) / 32) - nblk;
  for (int c = 16; c >= 4; c /= 2) {
    const int w = c * ((nblk + c - 1) / c) - nblk;
    if (w < waste) { lpr = c; waste = w; }
  }
  const int rows_per_cta = 8 * (32 / lpr);
  auto kq = lpr == 4 ? quant_h_kernel<4> : lpr == 8 ? quant_h_kernel<8>
          : lpr == 16 ? quant_h_kernel<16> : quant_h_kernel<32>;
  kq<<<(P + rows_per_cta - 1) / rows_per_cta, 256, 0, s>>>(h, P, F, sf_pitch, offsets, E, qc, qs,
                                                           qe);
  return cudaGetLastError();
}// Exponent c_F with F * 2688^2 * 2^-c_F < 2^15: the fixed shift of the f16 partials.
int down_shift_for(int F) {
  const double bound = (double)F * 2688.0 * 2688.0;
  int c = 0;
  while (std::ldexp(bound, -c) >= 32768.0) ++c;
  return c;
}

cudaError_t launch_prefill_combine(const float* w, int T, int H, int F, int k, int c0, int HS,
                                   const moe_ws_layout& L, char* ws, float* y, cudaStream_t s) {
  dim3 grid((HS / 8 + 255) / 256, T);
  combine_f16_kernel<<<grid, 256, 0, s>>>(w, reinterpret_cast<const int32_t*>(ws + L.pair_pos),
                                          reinterpret_cast<const __half*>(ws + L.partial),
                                          reinterpret_cast<const int32_t*>(ws + L.qh_exp),
                                          down_shift_for(F), H, c0, HS, k, y);
  return cudaGetLastError();
}

}  // namespace moe
