// Decode path: few pairs per expert, memory-bound on the NVFP4 weight bytes.
//
// Every active expert's rows are streamed from HBM exactly once per call with 128-bit
// non-allocating loads (the union-of-experts gather: the grid is indexed by active
// expert, not by pair), dequantised in registers (E2M1 -> f16 via cvt, times the UE4M3
// scale, exact in f16), and multiplied on the tensor cores (mma.sync m16n8k16, f32
// accumulate) against the expert's activation rows, which are staged once per CTA in
// shared memory as f16 with a per-row power-of-two prescale (exact for bf16 inputs in
// f16's normal range: the row's largest magnitude lands in [2^14, 2^15)) and reused by
// every weight row of the CTA.
//
// Lane layout of one m16n8k16 step: lane = 4g + c holds 16 contiguous code bytes (32
// elements) of weight rows g and g+8 per 128-element k-block; MMA step s consumes bytes
// 2s, 2s+1, i.e. elements 32c + 4s .. 32c + 4s + 3, and the activation fragment is read
// from the same four elements.  The tensor core sums over k in any order, so this
// permutation of k (identical for both operands) leaves the product unchanged.
#include "moe_internal.cuh"

namespace moe {

namespace {

// Byte offset of 16-byte chunk `lc` of a staged f16 row: XOR-swizzled so that the
// quarter-warp reading chunks 4c+u of rows g, g+1 touches eight distinct bank groups.
__device__ __forceinline__ int swz_chunk(int lc) { return (lc ^ (((lc >> 3) & 1) << 1)) * 16; }

// Dequantise one MMA step's A fragment for a pair of rows (g, g+8): bytes 2s, 2s+1.
template <int S>
__device__ __forceinline__ void a_frag(const uint4& r0, const uint4& r1, uint32_t sc0,
                                       uint32_t sc1, uint32_t (&a)[4]) {
  const uint32_t w0 = (S / 2 == 0) ? r0.x : (S / 2 == 1) ? r0.y : (S / 2 == 2) ? r0.z : r0.w;
  const uint32_t w1 = (S / 2 == 0) ? r1.x : (S / 2 == 1) ? r1.y : (S / 2 == 2) ? r1.z : r1.w;
  const int sh = (S & 1) * 16;
  a[0] = hmul2_u32(e2m1x2_to_f16x2(w0 >> sh), sc0);
  a[1] = hmul2_u32(e2m1x2_to_f16x2(w1 >> sh), sc1);
  a[2] = hmul2_u32(e2m1x2_to_f16x2(w0 >> (sh + 8)), sc0);
  a[3] = hmul2_u32(e2m1x2_to_f16x2(w1 >> (sh + 8)), sc1);
}

// Same for 8-byte (64-element k-block) lanes: bytes 2s, 2s+1 of a uint2.
template <int S>
__device__ __forceinline__ void a_frag64(const uint2& r0, const uint2& r1, uint32_t sc0,
                                         uint32_t sc1, uint32_t (&a)[4]) {
  const uint32_t w0 = (S / 2 == 0) ? r0.x : r0.y;
  const uint32_t w1 = (S / 2 == 0) ? r1.x : r1.y;
  const int sh = (S & 1) * 16;
  a[0] = hmul2_u32(e2m1x2_to_f16x2(w0 >> sh), sc0);
  a[1] = hmul2_u32(e2m1x2_to_f16x2(w1 >> sh), sc1);
  a[2] = hmul2_u32(e2m1x2_to_f16x2(w0 >> (sh + 8)), sc0);
  a[3] = hmul2_u32(e2m1x2_to_f16x2(w1 >> (sh + 8)), sc1);
}

// ---------------------------------------------------------------------------
// gate/up + SiLU
// ---------------------------------------------------------------------------
// CTA = KS x RB warps: RB row blocks (16 gate rows + the matching 16 up rows each), the
// H reduction split over KS warps and summed in shared memory in a fixed order.
// grid = (ceil(F / (16 RB)), max_active).  Tokens of the expert are processed 8*NT at a time.
struct GateUpArgs {
  const uint16_t* x;      // bf16 [T][H]
  const uint8_t* codes;
  const uint8_t* scales;
  int H, F, k;
  const int32_t* offsets;
  const int32_t* pair_ids;
  const int32_t* active;
  const int32_t* n_active;
  float* h;
};

template <int KS, int RB, int NT>
__global__ void __launch_bounds__(32 * KS * RB)
decode_gate_up_kernel(const GateUpArgs args) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int a_idx = blockIdx.y;
  if (a_idx >= *args.n_active) return;
  const int H = args.H, F = args.F;
  const int e = args.active[a_idx];
  const int off = args.offsets[e];
  const int m = args.offsets[e + 1] - off;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int kw = warp % KS, rbw = warp / KS;
  const int i0 = (blockIdx.x * RB + rbw) * 16;     // first gate row of this warp
  const bool rows_ok = i0 < F;

  const int row_bytes = H / 2, srow_bytes = H / 16;
  const size_t rows2F = (size_t)2 * F;
  const uint8_t* cb = args.codes + (size_t)e * rows2F * row_bytes;
  const uint8_t* sb = args.scales + (size_t)e * rows2F * srow_bytes;
  const int ig = rows_ok ? i0 + g : 0;
  const uint8_t* pg0 = cb + (size_t)ig * row_bytes + 16 * c;
  const uint8_t* pg1 = pg0 + (size_t)8 * row_bytes;
  const uint8_t* pu0 = pg0 + (size_t)F * row_bytes;
  const uint8_t* pu1 = pu0 + (size_t)8 * row_bytes;
  const uint8_t* sg0 = sb + (size_t)ig * srow_bytes + 2 * c;
  const uint8_t* sg1 = sg0 + (size_t)8 * srow_bytes;
  const uint8_t* su0 = sg0 + (size_t)F * srow_bytes;
  const uint8_t* su1 = su0 + (size_t)8 * srow_bytes;

  const int nkb = H / 128;
  const int kb_beg = kw * nkb / KS, kb_end = (kw + 1) * nkb / KS;

  const int xrow_bytes = H * 2 + 16;
  unsigned char* xs = smem;                                        // [8NT][xrow_bytes]
  int* slot_exp = reinterpret_cast<int*>(smem + 8 * NT * xrow_bytes);   // [8NT]
  uint32_t* slot_amax = reinterpret_cast<uint32_t*>(slot_exp + 8 * NT);  // [8NT]
  int* slot_tok = reinterpret_cast<int*>(slot_amax + 8 * NT);             // [8NT]
  float* red = reinterpret_cast<float*>(smem + 8 * NT * xrow_bytes + 24 * NT * sizeof(int));

  for (int tok0 = 0; tok0 < m; tok0 += 8 * NT) {
    // prefetch the first k-block of weights before staging the activations
    uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0, c2 = c0, c3 = c0;
    uint32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    if (rows_ok && kb_beg < kb_end) {
      c0 = ldg_stream(pg0 + kb_beg * 64); c1 = ldg_stream(pg1 + kb_beg * 64);
      c2 = ldg_stream(pu0 + kb_beg * 64); c3 = ldg_stream(pu1 + kb_beg * 64);
      s0 = *reinterpret_cast<const uint16_t*>(sg0 + kb_beg * 8);
      s1 = *reinterpret_cast<const uint16_t*>(sg1 + kb_beg * 8);
      s2 = *reinterpret_cast<const uint16_t*>(su0 + kb_beg * 8);
      s3 = *reinterpret_cast<const uint16_t*>(su1 + kb_beg * 8);
    }
    __syncthreads();   // previous pass done with xs
    // stage the pass's activation rows (only the live ones): raw bf16 first, with each
    // row's amax; dead slots keep stale data, which only reaches discarded output columns
    const int live = min(8 * NT, m - tok0);
    if (threadIdx.x < 8 * NT) {
      slot_amax[threadIdx.x] = 0u;
      slot_tok[threadIdx.x] =
          threadIdx.x < live ? args.pair_ids[off + tok0 + threadIdx.x] / args.k : 0;
    }
    __syncthreads();
    const int nchunk = H / 8;
    for (int idx = threadIdx.x; idx < live * nchunk; idx += blockDim.x) {
      const int slot = idx / nchunk, ch = idx - slot * nchunk;
      const uint4 v =
          *reinterpret_cast<const uint4*>(args.x + (size_t)slot_tok[slot] * H + ch * 8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t am = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        am = max(am, (w[i] << 16) & 0x7fffffffu);
        am = max(am, w[i] & 0x7fff0000u);
      }
      if (am) atomicMax(&slot_amax[slot], am);         // |x| as ordered integer bits
      *reinterpret_cast<uint4*>(xs + slot * xrow_bytes + swz_chunk(ch)) = v;
    }
    __syncthreads();
    if (threadIdx.x < 8 * NT)
      slot_exp[threadIdx.x] = f16_prescale_exp(__uint_as_float(slot_amax[threadIdx.x]));
    __syncthreads();
    // convert in place to f16 times 2^-exp (same thread, same chunk as above)
    for (int idx = threadIdx.x; idx < live * nchunk; idx += blockDim.x) {
      const int slot = idx / nchunk, ch = idx - slot * nchunk;
      uint4* q = reinterpret_cast<uint4*>(xs + slot * xrow_bytes + swz_chunk(ch));
      const uint4 v = *q;
      const int ex = slot_exp[slot];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 hv = __floats2half2_rn(ldexpf(__uint_as_float(w[i] << 16), -ex),
                                             ldexpf(__uint_as_float(w[i] & 0xffff0000u), -ex));
        o[i] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *q = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();

    float accg[NT][4], accu[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) accg[nt][q] = accu[nt][q] = 0.0f;

    if (rows_ok) {
      for (int kb = kb_beg; kb < kb_end; ++kb) {
        uint4 n0 = c0, n1 = c1, n2 = c2, n3 = c3;
        uint32_t t0 = s0, t1 = s1, t2 = s2, t3 = s3;
        if (kb + 1 < kb_end) {
          n0 = ldg_stream(pg0 + (kb + 1) * 64); n1 = ldg_stream(pg1 + (kb + 1) * 64);
          n2 = ldg_stream(pu0 + (kb + 1) * 64); n3 = ldg_stream(pu1 + (kb + 1) * 64);
          t0 = *reinterpret_cast<const uint16_t*>(sg0 + (kb + 1) * 8);
          t1 = *reinterpret_cast<const uint16_t*>(sg1 + (kb + 1) * 8);
          t2 = *reinterpret_cast<const uint16_t*>(su0 + (kb + 1) * 8);
          t3 = *reinterpret_cast<const uint16_t*>(su1 + (kb + 1) * 8);
        }
        const uint32_t f0 = e4m3x2_to_f16x2(s0), f1 = e4m3x2_to_f16x2(s1);
        const uint32_t f2 = e4m3x2_to_f16x2(s2), f3 = e4m3x2_to_f16x2(s3);
        // activation fragments for this k-block: 4 chunks of 16 B per n-tile
        uint4 xb[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            xb[nt][u] = *reinterpret_cast<const uint4*>(
                xs + (nt * 8 + g) * xrow_bytes + swz_chunk(kb * 16 + 4 * c + u));
#define MOE_GU_STEP(S)                                                                     \
  {                                                                                        \
    uint32_t ag[4], au[4];                                                                 \
    const uint32_t scg0 = (S < 4) ? bcast_lo(f0) : bcast_hi(f0);                           \
    const uint32_t scg1 = (S < 4) ? bcast_lo(f1) : bcast_hi(f1);                           \
    const uint32_t scu0 = (S < 4) ? bcast_lo(f2) : bcast_hi(f2);                           \
    const uint32_t scu1 = (S < 4) ? bcast_lo(f3) : bcast_hi(f3);                           \
    a_frag<S>(c0, c1, scg0, scg1, ag);                                                     \
    a_frag<S>(c2, c3, scu0, scu1, au);                                                     \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                    \
      const uint32_t b0 = (S & 1) ? xb[nt][S / 2].z : xb[nt][S / 2].x;                     \
      const uint32_t b1 = (S & 1) ? xb[nt][S / 2].w : xb[nt][S / 2].y;                     \
      mma_f16_16816(accg[nt], ag[0], ag[1], ag[2], ag[3], b0, b1);                         \
      mma_f16_16816(accu[nt], au[0], au[1], au[2], au[3], b0, b1);                         \
    }                                                                                      \
  }
        MOE_GU_STEP(0) MOE_GU_STEP(1) MOE_GU_STEP(2) MOE_GU_STEP(3)
        MOE_GU_STEP(4) MOE_GU_STEP(5) MOE_GU_STEP(6) MOE_GU_STEP(7)
#undef MOE_GU_STEP
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        s0 = t0; s1 = t1; s2 = t2; s3 = t3;
      }
    }

    // fixed-order reduction over the KS warps sharing a row block
    if (KS > 1) {
      float* mine = red + (((size_t)(kw * RB + rbw) * NT) * 32 + lane) * 8;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mine[nt * 256 + q] = accg[nt][q];
          mine[nt * 256 + 4 + q] = accu[nt][q];
        }
      __syncthreads();
      if (kw == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) { accg[nt][q] = 0.0f; accu[nt][q] = 0.0f; }
        for (int w = 0; w < KS; ++w) {
          const float* src = red + (((size_t)(w * RB + rbw) * NT) * 32 + lane) * 8;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              accg[nt][q] += src[nt * 256 + q];
              accu[nt][q] += src[nt * 256 + 4 + q];
            }
        }
      }
    }
    if (kw == 0 && rows_ok) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int n = nt * 8 + 2 * c + (q & 1);
          const int i = i0 + g + 8 * (q >> 1);
          if (tok0 + n < m) {
            const int ex = slot_exp[n];
            const float gv = ldexpf(accg[nt][q], ex), uv = ldexpf(accu[nt][q], ex);
            args.h[(size_t)(off + tok0 + n) * F + i] = silu_f(gv) * uv;
          }
        }
    }
  }
}

// ---------------------------------------------------------------------------
// down projection: z_p = W_down[e] h_p, rows of the per-pair partials in CSR order
// ---------------------------------------------------------------------------
struct DownArgs {
  const float* h;
  const uint8_t* codes;
  const uint8_t* scales;
  int H, F;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  float* partial;
};

// CTA = WARPS warps of 16 output rows each; grid = (ceil(H / (16 WARPS)), max_active).
// KB = 128 (uint4 lanes) when F % 128 == 0, else 64 (uint2 lanes).
template <int WARPS, int NT, int KB>
__global__ void __launch_bounds__(32 * WARPS)
decode_down_kernel(const DownArgs args) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int a_idx = blockIdx.y;
  if (a_idx >= *args.n_active) return;
  const int H = args.H, F = args.F;
  const int e = args.active[a_idx];
  const int off = args.offsets[e];
  const int m = args.offsets[e + 1] - off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int r0 = (blockIdx.x * WARPS + warp) * 16;
  const bool rows_ok = r0 < H;
  const int row_bytes = F / 2, srow_bytes = F / 16;
  constexpr int LB = KB / 8;                       // code bytes per lane per k-block
  const uint8_t* cb = args.codes + (size_t)e * H * row_bytes;
  const uint8_t* sb = args.scales + (size_t)e * H * srow_bytes;
  const int rg = rows_ok ? r0 + g : 0;
  const uint8_t* p0 = cb + (size_t)rg * row_bytes + LB * c;
  const uint8_t* p1 = p0 + (size_t)8 * row_bytes;
  const uint8_t* q0 = sb + (size_t)rg * srow_bytes + (KB / 64) * c;
  const uint8_t* q1 = q0 + (size_t)8 * srow_bytes;
  const int nkb = F / KB;

  const int hrow_bytes = F * 2 + 16;
  unsigned char* hs = smem;                                          // [8NT][hrow_bytes]
  int* slot_exp = reinterpret_cast<int*>(smem + 8 * NT * hrow_bytes);

  for (int tok0 = 0; tok0 < m; tok0 += 8 * NT) {
    __syncthreads();
    // stage h rows as f16 with a per-row power-of-two prescale (one warp per row)
    const int nlive = min(8 * NT, m - tok0);
    for (int slot = warp; slot < nlive; slot += WARPS) {
      const bool live = true;
      const float* hr = args.h + (size_t)(off + tok0 + slot) * F;
      float amax = 0.0f;
      if (live)
        for (int i = lane * 4; i < F; i += 128) {
          float4 v = *reinterpret_cast<const float4*>(hr + i);
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int ex = f16_prescale_exp(amax);
      if (lane == 0) slot_exp[slot] = ex;
      for (int ch = lane; ch < F / 8; ch += 32) {
        uint4 o = make_uint4(0, 0, 0, 0);
        if (live) {
          float4 v0 = *reinterpret_cast<const float4*>(hr + ch * 8);
          float4 v1 = *reinterpret_cast<const float4*>(hr + ch * 8 + 4);
          __half2 h0 = __floats2half2_rn(ldexpf(v0.x, -ex), ldexpf(v0.y, -ex));
          __half2 h1 = __floats2half2_rn(ldexpf(v0.z, -ex), ldexpf(v0.w, -ex));
          __half2 h2 = __floats2half2_rn(ldexpf(v1.x, -ex), ldexpf(v1.y, -ex));
          __half2 h3 = __floats2half2_rn(ldexpf(v1.z, -ex), ldexpf(v1.w, -ex));
          o = make_uint4(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                         *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3));
        }
        *reinterpret_cast<uint4*>(hs + slot * hrow_bytes + swz_chunk(ch)) = o;
      }
    }
    __syncthreads();
    if (!rows_ok) continue;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[nt][q] = 0.0f;

    if (KB == 128) {
      uint4 a0 = ldg_stream(p0), a1 = ldg_stream(p1);
      uint32_t w0 = *reinterpret_cast<const uint16_t*>(q0);
      uint32_t w1 = *reinterpret_cast<const uint16_t*>(q1);
      for (int kb = 0; kb < nkb; ++kb) {
        uint4 b0n = a0, b1n = a1;
        uint32_t w0n = w0, w1n = w1;
        if (kb + 1 < nkb) {
          b0n = ldg_stream(p0 + (kb + 1) * (KB / 2));
          b1n = ldg_stream(p1 + (kb + 1) * (KB / 2));
          w0n = *reinterpret_cast<const uint16_t*>(q0 + (kb + 1) * (KB / 16));
          w1n = *reinterpret_cast<const uint16_t*>(q1 + (kb + 1) * (KB / 16));
        }
        const uint32_t f0 = e4m3x2_to_f16x2(w0), f1 = e4m3x2_to_f16x2(w1);
        uint4 xb[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            xb[nt][u] = *reinterpret_cast<const uint4*>(
                hs + (nt * 8 + g) * hrow_bytes + swz_chunk(kb * 16 + 4 * c + u));
#define MOE_DN_STEP(S)                                                                     \
  {                                                                                        \
    uint32_t af[4];                                                                        \
    const uint32_t sc0 = (S < 4) ? bcast_lo(f0) : bcast_hi(f0);                            \
    const uint32_t sc1 = (S < 4) ? bcast_lo(f1) : bcast_hi(f1);                            \
    a_frag<S>(a0, a1, sc0, sc1, af);                                                       \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                    \
      const uint32_t bb0 = (S & 1) ? xb[nt][S / 2].z : xb[nt][S / 2].x;                    \
      const uint32_t bb1 = (S & 1) ? xb[nt][S / 2].w : xb[nt][S / 2].y;                    \
      mma_f16_16816(acc[nt], af[0], af[1], af[2], af[3], bb0, bb1);                        \
    }                                                                                      \
  }
        MOE_DN_STEP(0) MOE_DN_STEP(1) MOE_DN_STEP(2) MOE_DN_STEP(3)
        MOE_DN_STEP(4) MOE_DN_STEP(5) MOE_DN_STEP(6) MOE_DN_STEP(7)
#undef MOE_DN_STEP
        a0 = b0n; a1 = b1n; w0 = w0n; w1 = w1n;
      }
    } else {
      for (int kb = 0; kb < nkb; ++kb) {
        const uint2 a0 = ldg_stream64(p0 + kb * (KB / 2));
        const uint2 a1 = ldg_stream64(p1 + kb * (KB / 2));
        const uint32_t w0 = q0[kb * (KB / 16)], w1 = q1[kb * (KB / 16)];
        const uint32_t f0 = bcast_lo(e4m3x2_to_f16x2(w0)), f1 = bcast_lo(e4m3x2_to_f16x2(w1));
        uint4 xb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int u = 0; u < 2; ++u)
            xb[nt][u] = *reinterpret_cast<const uint4*>(
                hs + (nt * 8 + g) * hrow_bytes + swz_chunk(kb * 8 + 2 * c + u));
#define MOE_DN64_STEP(S)                                                                   \
  {                                                                                        \
    uint32_t af[4];                                                                        \
    a_frag64<S>(a0, a1, f0, f1, af);                                                       \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                    \
      const uint32_t bb0 = (S & 1) ? xb[nt][S / 2].z : xb[nt][S / 2].x;                    \
      const uint32_t bb1 = (S & 1) ? xb[nt][S / 2].w : xb[nt][S / 2].y;                    \
      mma_f16_16816(acc[nt], af[0], af[1], af[2], af[3], bb0, bb1);                        \
    }                                                                                      \
  }
        MOE_DN64_STEP(0) MOE_DN64_STEP(1) MOE_DN64_STEP(2) MOE_DN64_STEP(3)
#undef MOE_DN64_STEP
      }
    }

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = nt * 8 + 2 * c + (q & 1);
        const int r = r0 + g + 8 * (q >> 1);
        if (tok0 + n < m)
          args.partial[(size_t)(off + tok0 + n) * H + r] = ldexpf(acc[nt][q], slot_exp[n]);
      }
  }
}

// ---------------------------------------------------------------------------
// combine: y[t, :] = sum_j w[t, j] * z[pair_pos[t*k + j], :] in ascending j
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ w, const int32_t* __restrict__ pair_pos,
               const float* __restrict__ partial, int H, int k, float* __restrict__ y) {
  const int t = blockIdx.y;
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (r >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int pos = pair_pos[(size_t)t * k + j];
    if (pos < 0) continue;
    const float wj = w[(size_t)t * k + j];
    const float4 z = *reinterpret_cast<const float4*>(partial + (size_t)pos * H + r);
    acc.x = fmaf(wj, z.x, acc.x);
    acc.y = fmaf(wj, z.y, acc.y);
    acc.z = fmaf(wj, z.z, acc.z);
    acc.w = fmaf(wj, z.w, acc.w);
  }
  *reinterpret_cast<float4*>(y + (size_t)t * H + r) = acc;
}

template <int KS, int RB, int NT>
cudaError_t run_gate_up(const GateUpArgs& a, int F, int max_active, cudaStream_t s) {
  const int H = a.H;
  const size_t smem = (size_t)8 * NT * (H * 2 + 16) + 24 * NT * sizeof(int) +
                      (KS > 1 ? (size_t)KS * RB * NT * 32 * 8 * sizeof(float) : 0);
  auto kern = decode_gate_up_kernel<KS, RB, NT>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem);
  if (st != cudaSuccess) return st;
  dim3 grid((F + 16 * RB - 1) / (16 * RB), max_active);
  kern<<<grid, 32 * KS * RB, smem, s>>>(a);
  return cudaGetLastError();
}

template <int WARPS, int NT, int KB>
cudaError_t run_down(const DownArgs& a, int max_active, cudaStream_t s) {
  const size_t smem = (size_t)8 * NT * (a.F * 2 + 16) + 8 * NT * sizeof(int);
  auto kern = decode_down_kernel<WARPS, NT, KB>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem);
  if (st != cudaSuccess) return st;
  dim3 grid((a.H + 16 * WARPS - 1) / (16 * WARPS), max_active);
  kern<<<grid, 32 * WARPS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                  const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                  char* ws, cudaStream_t s) {
  GateUpArgs a{x_bf16, b.codes, b.scales, H, F, k, csr.expert_offsets, csr.pair_ids,
               csr.active_experts, csr.n_active, reinterpret_cast<float*>(ws + L.h)};
  const int P = T * k;
  const int max_active = P < b.E ? P : b.E;
  if (P <= 160) return run_gate_up<8, 1, 1>(a, F, max_active, s);
  return run_gate_up<2, 4, 2>(a, F, max_active, s);
}

cudaError_t launch_decode_down(const moe_nvfp4_bank& b, moe_csr csr, int T, int H, int F, int k,
                               const moe_ws_layout& L, char* ws, cudaStream_t s) {
  DownArgs a{reinterpret_cast<const float*>(ws + L.h), b.codes, b.scales, H, F,
             csr.expert_offsets, csr.active_experts, csr.n_active,
             reinterpret_cast<float*>(ws + L.partial)};
  const int P = T * k;
  const int max_active = P < b.E ? P : b.E;
  if (F % 128 == 0) {
    if (P <= 160) return run_down<4, 1, 128>(a, max_active, s);
    return run_down<8, 2, 128>(a, max_active, s);
  }
  return run_down<4, 1, 64>(a, max_active, s);
}

cudaError_t launch_combine(const float* w, int T, int H, int k, const moe_ws_layout& L, char* ws,
                           float* y, cudaStream_t s) {
  dim3 grid((H / 4 + 255) / 256, T);
  combine_kernel<<<grid, 256, 0, s>>>(w, reinterpret_cast<const int32_t*>(ws + L.pair_pos),
                                      reinterpret_cast<const float*>(ws + L.partial), H, k, y);
  return cudaGetLastError();
}

}  // namespace moe
