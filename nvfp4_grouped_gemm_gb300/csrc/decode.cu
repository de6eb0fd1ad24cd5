// Decode path: few pairs per expert, memory-bound on the NVFP4 weight bytes.
//
// Work is indexed by active expert, not by pair, so every active expert's rows are
// streamed from HBM exactly once per call (the union-of-experts gather).  Kernels:
//
//   x_gather_kernel   CSR row r <- token x row as f16 times 2^-e (e from the row's amax,
//                     so the largest magnitude lands in [2^14, 2^15): exact for bf16
//                     values in f16's normal range); also zeroes the call's counters
//   gate_up_kernel    warp unit = (active expert, 8 gate rows + the matching 8 up rows);
//                     one m16n8k16 MMA carries gate rows in M rows 0..7 and up rows in
//                     8..15, so each lane holds a gate and an up value of the same (row,
//                     pair) and writes h = silu(g)*u itself.  The unit's codes go from
//                     HBM straight into MMA fragments (128-bit loads, 4 k-blocks ahead).
//                     The last unit of an expert to finish converts that expert's h
//                     rows to f16 times 2^-e (as for x).
//   down_kernel       warp unit = (active expert, 32 output rows) over the whole F, the
//                     same register-direct loop; per-pair partials z (f32).  The last of
//                     the units that cover a (token, 64-row chunk) combines that chunk:
//                     y[t, rows] = sum_j w[t,j] z[pos(t,j), rows] in ascending j.
//
// Units are taken from a per-call counter (the first unit of each warp is fixed, so its
// loads can be issued before the kernel waits for its predecessor).  Arrival counters are
// integers; every sum is taken in a fixed order, so results do not depend on scheduling.
//
// FP4 codes are dequantised in registers (cvt.rn.f16x2.e2m1x2, times the UE4M3 scale via
// cvt.rn.f16x2.e4m3x2: every product has <= 6 significant bits, exact in f16) and fed
// to mma.sync.m16n8k16 (f32 accumulate).  Lane 4g+c of an MMA step s uses elements
// 32c + 4s .. 32c + 4s + 3 of a 128-element k-block for both operands; the tensor core
// sums over k in any order, so this shared permutation leaves the product unchanged.
#include "moe_internal.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Same for 64-element k-blocks: bytes 2S, 2S+1 of the lane's 8-byte piece.
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

// Counter region of the decode workspace: [0] gate/up unit queue, [1] down unit queue,
// [2, 2 + A) per-active-expert gate/up arrivals, then [T][H/64] combine arrivals.
constexpr int kCtrGu = 0, kCtrDn = 1, kCtrExpert = 2;

// Next unit of this warp: the first is fixed (warp id), later ones come from the queue.
__device__ __forceinline__ int next_unit(int32_t* queue, int n_warps) {
  int u = 0;
  if ((threadIdx.x & 31) == 0) u = n_warps + atomicAdd(queue, 1);
  return __shfl_sync(0xffffffffu, u, 0);
}

// ---------------------------------------------------------------------------
// gather + f16 prescale of the activation rows of every CSR row (decode stage a3)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) x_gather_kernel(const uint16_t* __restrict__ x, int H, int k,
                                                       const int32_t* __restrict__ pair_ids,
                                                       const int32_t* __restrict__ offsets, int E,
                                                       __half* __restrict__ xg,
                                                       int32_t* __restrict__ xe,
                                                       int32_t* __restrict__ ctr, int n_ctr) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_ctr; i += blockDim.x) ctr[i] = 0;
  const int pos = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pos >= offsets[E]) return;
  const uint16_t* row = x + (size_t)(pair_ids[pos] / k) * H;
  // the whole row in registers (H <= 4096: at most 16 pieces of 8 values per lane)
  uint4 v[16];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int c = (lane + 32 * i) * 8;
    v[i] = c < H ? *reinterpret_cast<const uint4*>(row + c) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xffff0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = f16_prescale_exp(amax);
  if (lane == 0) xe[pos] = e;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int c = (lane + 32 * i) * 8;
    if (c >= H) break;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 hv = __floats2half2_rn(ldexpf(__uint_as_float(w[q] << 16), -e),
                                           ldexpf(__uint_as_float(w[q] & 0xffff0000u), -e));
      o[q] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(xg + (size_t)pos * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}


// ---------------------------------------------------------------------------
// gate/up + SiLU
// ---------------------------------------------------------------------------
struct GateUpArgs {
  const __half* xg;        // [P][H] gathered f16 activations
  const int32_t* xe;       // [P]
  const uint8_t* codes;
  const uint8_t* scales;
  int H, F;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  float* h;                // [P][F]
  __half* hg;              // [P][F] h times 2^-he
  int32_t* he;             // [P]
  int32_t* ctr;
};

constexpr int kPf = 4;     // k-blocks of codes in flight per warp

// h row `pos` (f32, written by other warps: read through L2) to f16 times 2^-e.
__device__ void h_to_f16(const float* __restrict__ h, int F, int pos, __half* __restrict__ hg,
                         int32_t* __restrict__ he) {
  const int lane = threadIdx.x & 31;
  const float* row = h + (size_t)pos * F;
  float amax = 0.0f;
  for (int c = lane * 4; c < F; c += 128) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(row + c));
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = f16_prescale_exp(amax);
  if (lane == 0) he[pos] = e;
  for (int c = lane * 4; c < F; c += 128) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(row + c));
    const __half2 h0 = __floats2half2_rn(ldexpf(a.x, -e), ldexpf(a.y, -e));
    const __half2 h1 = __floats2half2_rn(ldexpf(a.z, -e), ldexpf(a.w, -e));
    *reinterpret_cast<uint2*>(hg + (size_t)pos * F + c) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
  }
}

__global__ void __launch_bounds__(256) gate_up_kernel(const GateUpArgs args) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int H = args.H, F = args.F;
  const int row_bytes = H / 2, srow = H / 16;
  const int nkb = H / 128;
  const int nrb = F / 8;                       // units per expert
  const int n_warps = gridDim.x * (blockDim.x >> 5);
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int n_units = *args.n_active * nrb;    // the CSR is complete (two kernels back)
  const size_t rows2F = (size_t)2 * F;

  uint4 wg[kPf], wu[kPf];
  uint32_t sg[kPf], su[kPf];
  const uint8_t* pg = nullptr;                 // this lane's 16-byte column of the gate row
  const uint8_t* pu = nullptr;
  const uint8_t* qg = nullptr;                 // its two scale bytes
  const uint8_t* qu = nullptr;
  auto set_unit = [&](int u) {
    const int e = args.active[u / nrb];
    const size_t rg = (size_t)e * rows2F + (u % nrb) * 8 + g;
    pg = args.codes + rg * row_bytes + 16 * c;
    pu = pg + (size_t)F * row_bytes;
    qg = args.scales + rg * srow + 2 * c;
    qu = qg + (size_t)F * srow;
  };
  auto load_kb = [&](int kb, int d) {
    wg[d] = ldg_stream(pg + kb * 64);
    wu[d] = ldg_stream(pu + kb * 64);
    sg[d] = __ldg(reinterpret_cast<const uint16_t*>(qg + kb * 8));
    su[d] = __ldg(reinterpret_cast<const uint16_t*>(qu + kb * 8));
  };

  int u = gw;
  // the first unit's codes are independent of the previous kernel: issue them first
  if (u < n_units) {
    set_unit(u);
#pragma unroll
    for (int d = 0; d < kPf; ++d)
      if (d < nkb) load_kb(d, d);
  }
  pdl_wait();                                  // gathered activations and counters are ready
  pdl_trigger();

  while (u < n_units) {
    const int un = next_unit(args.ctr + kCtrGu, n_warps);
    const int a = u / nrb;
    const int e = args.active[a];
    const int i0 = (u % nrb) * 8;
    const int off = args.offsets[e];
    const int m = args.offsets[e + 1] - off;
    for (int tok0 = 0; tok0 < m; tok0 += 8) {
      const int live = min(8, m - tok0);
      if (tok0 > 0) {                           // codes again for the next 8 pairs
#pragma unroll
        for (int d = 0; d < kPf; ++d)
          if (d < nkb) load_kb(d, d);
      }
      const __half* xrow = args.xg + (size_t)(off + tok0 + (g < live ? g : 0)) * H + 32 * c;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      uint4 xb[4], xn[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        xb[q] = g < live ? __ldg(reinterpret_cast<const uint4*>(xrow + 8 * q)) : make_uint4(0, 0, 0, 0);
      for (int kb0 = 0; kb0 < nkb; kb0 += kPf) {
#pragma unroll
        for (int d = 0; d < kPf; ++d) {
          const int kb = kb0 + d;
          if (kb < nkb) {
            // next k-block's activation fragments
#pragma unroll
            for (int q = 0; q < 4; ++q)
              xn[q] = (g < live && kb + 1 < nkb)
                          ? __ldg(reinterpret_cast<const uint4*>(xrow + (kb + 1) * 128 + 8 * q))
                          : make_uint4(0, 0, 0, 0);
            const uint32_t fg = e4m3x2_to_f16x2(sg[d]), fu = e4m3x2_to_f16x2(su[d]);
            const uint32_t s_g[2] = {bcast_lo(fg), bcast_hi(fg)};
            const uint32_t s_u[2] = {bcast_lo(fu), bcast_hi(fu)};
            const uint32_t WG[4] = {wg[d].x, wg[d].y, wg[d].z, wg[d].w};
            const uint32_t WU[4] = {wu[d].x, wu[d].y, wu[d].z, wu[d].w};
            if (kb + kPf < nkb) load_kb(kb + kPf, d);
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              uint32_t gq[4], uq[4];
              e2m1x8_to_f16x2x4(WG[wi], gq[0], gq[1], gq[2], gq[3]);
              e2m1x8_to_f16x2x4(WU[wi], uq[0], uq[1], uq[2], uq[3]);
              const int sb = wi >> 1;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
                mma_f16_16816(acc, hmul2_u32(gq[2 * hh], s_g[sb]), hmul2_u32(uq[2 * hh], s_u[sb]),
                              hmul2_u32(gq[2 * hh + 1], s_g[sb]), hmul2_u32(uq[2 * hh + 1], s_u[sb]),
                              hh ? xb[wi].z : xb[wi].x, hh ? xb[wi].w : xb[wi].y);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) xb[q] = xn[q];
          }
        }
      }
      // acc[0..1]: gate row i0+g, pairs 2c, 2c+1; acc[2..3]: up row i0+g, same pairs
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int n = 2 * c + q;
        if (n < live) {
          const int pos = off + tok0 + n;
          const int ex = args.xe[pos];
          args.h[(size_t)pos * F + i0 + g] = silu_f(ldexpf(acc[q], ex)) * ldexpf(acc[2 + q], ex);
        }
      }
    }
    // the expert's last unit converts its h rows for the down projection
    __threadfence();
    int last = 0;
    if (lane == 0) last = atomicAdd(args.ctr + kCtrExpert + a, 1) == nrb - 1;
    if (__shfl_sync(0xffffffffu, last, 0)) {
      __threadfence();
      for (int pos = off; pos < off + m; ++pos) h_to_f16(args.h, F, pos, args.hg, args.he);
    }
    u = un;
    if (u < n_units) {
      set_unit(u);
#pragma unroll
      for (int d = 0; d < kPf; ++d)
        if (d < nkb) load_kb(d, d);
    }
  }
}

// ---------------------------------------------------------------------------
// down + combine
// ---------------------------------------------------------------------------
struct DownArgs {
  const __half* hg;
  const int32_t* he;
  const uint8_t* codes;
  const uint8_t* scales;
  int H, F, k, T;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  const int32_t* pair_ids;
  const int32_t* pair_pos;
  const float* w;          // [T][k]
  float* partial;          // [P][H]
  float* y;                // [T][H]
  int32_t* ctr;
  int cc_off;              // first combine counter
};

constexpr int kDnRows = 32;           // output rows per down unit
constexpr int kPfDn = 2;              // k-blocks of codes in flight per down warp (4 rows each)
constexpr int kChunk = 64;            // rows per combine chunk

// Number of valid pairs of token t.
__device__ __forceinline__ int valid_pairs(const int32_t* pair_pos, int t, int k) {
  int v = 0;
  for (int j = 0; j < k; ++j) v += pair_pos[(size_t)t * k + j] >= 0;
  return v;
}

// y[t, r0 .. r0 + 64) = sum_j w[t, j] z[pos_j, same rows], ascending j (partials of
// other warps: read through L2).
__device__ void combine_chunk(const DownArgs& args, int t, int r0) {
  const int lane = threadIdx.x & 31;
  const int r = r0 + 2 * lane;
  float2 acc = make_float2(0.f, 0.f);
  for (int j = 0; j < args.k; ++j) {
    const int pos = args.pair_pos[(size_t)t * args.k + j];
    if (pos < 0) continue;
    const float wj = args.w[(size_t)t * args.k + j];
    const float2 z = __ldcg(reinterpret_cast<const float2*>(args.partial + (size_t)pos * args.H + r));
    acc.x = fmaf(wj, z.x, acc.x);
    acc.y = fmaf(wj, z.y, acc.y);
  }
  *reinterpret_cast<float2*>(args.y + (size_t)t * args.H + r) = acc;
}

template <int KB>
__global__ void __launch_bounds__(256, 2) down_kernel(const DownArgs args) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int H = args.H, F = args.F;
  const int row_bytes = F / 2, srow = F / 16;
  const int nkb = F / KB;
  const int nrb = H / kDnRows;                 // units per expert
  const int n_warps = gridDim.x * (blockDim.x >> 5);
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int n_units = *args.n_active * nrb;
  constexpr int LB = KB / 8;                   // code bytes per lane per k-block and row
  using WT = typename std::conditional<KB == 128, uint4, uint2>::type;

  // 4 rows per lane: r0 + g + 8i, i = 0..3
  WT wr[kPfDn][4];
  uint32_t sr[kPfDn][4];
  const uint8_t* pr = nullptr;
  const uint8_t* qr = nullptr;
  auto set_unit = [&](int u) {
    const int e = args.active[u / nrb];
    const size_t r = (size_t)e * H + (u % nrb) * kDnRows + g;
    pr = args.codes + r * row_bytes + LB * c;
    qr = args.scales + r * srow + (KB == 128 ? 2 * c : c);
  };
  auto load_kb = [&](int kb, int d) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (KB == 128) {
        wr[d][i] = ldg_stream(pr + (size_t)(8 * i) * row_bytes + kb * 64);
        sr[d][i] = __ldg(reinterpret_cast<const uint16_t*>(qr + (size_t)(8 * i) * srow + kb * 8));
      } else {
        wr[d][i] = ldg_stream64(pr + (size_t)(8 * i) * row_bytes + kb * 32);
        sr[d][i] = __ldg(qr + (size_t)(8 * i) * srow + kb * 4);
      }
    }
  };

  int u = gw;
  if (u < n_units) {
    set_unit(u);
#pragma unroll
    for (int d = 0; d < kPfDn; ++d)
      if (d < nkb) load_kb(d, d);
  }
  pdl_wait();                                  // h in f16 is complete
  pdl_trigger();

  // tokens without a valid pair get y = 0 (no unit covers them)
  for (int t = gw; t < args.T; t += n_warps)
    if (valid_pairs(args.pair_pos, t, args.k) == 0)
      for (int r = lane * 4; r < H; r += 128)
        *reinterpret_cast<float4*>(args.y + (size_t)t * H + r) = make_float4(0.f, 0.f, 0.f, 0.f);

  while (u < n_units) {
    const int un = next_unit(args.ctr + kCtrDn, n_warps);
    const int e = args.active[u / nrb];
    const int r0 = (u % nrb) * kDnRows;
    const int off = args.offsets[e];
    const int m = args.offsets[e + 1] - off;
    for (int tok0 = 0; tok0 < m; tok0 += 8) {
      const int live = min(8, m - tok0);
      if (tok0 > 0) {
#pragma unroll
        for (int d = 0; d < kPfDn; ++d)
          if (d < nkb) load_kb(d, d);
      }
      const __half* hrow = args.hg + (size_t)(off + tok0 + (g < live ? g : 0)) * F;
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      for (int kb0 = 0; kb0 < nkb; kb0 += kPfDn) {
#pragma unroll
        for (int d = 0; d < kPfDn; ++d) {
          const int kb = kb0 + d;
          if (kb < nkb) {
            if constexpr (KB == 128) {
              uint4 xb[4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                xb[q] = g < live ? __ldg(reinterpret_cast<const uint4*>(hrow + kb * 128 + 32 * c + 8 * q))
                                 : make_uint4(0, 0, 0, 0);
              uint32_t s[4][2];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t f = e4m3x2_to_f16x2(sr[d][i]);
                s[i][0] = bcast_lo(f);
                s[i][1] = bcast_hi(f);
              }
              const uint4 W[4] = {wr[d][0], wr[d][1], wr[d][2], wr[d][3]};
              if (kb + kPfDn < nkb) load_kb(kb + kPfDn, d);
#pragma unroll
              for (int wi = 0; wi < 4; ++wi) {
                const uint32_t w0 = wi == 0 ? W[0].x : wi == 1 ? W[0].y : wi == 2 ? W[0].z : W[0].w;
                const uint32_t w1 = wi == 0 ? W[1].x : wi == 1 ? W[1].y : wi == 2 ? W[1].z : W[1].w;
                const uint32_t w2 = wi == 0 ? W[2].x : wi == 1 ? W[2].y : wi == 2 ? W[2].z : W[2].w;
                const uint32_t w3 = wi == 0 ? W[3].x : wi == 1 ? W[3].y : wi == 2 ? W[3].z : W[3].w;
                uint32_t p0[4], p1[4], p2[4], p3[4];
                e2m1x8_to_f16x2x4(w0, p0[0], p0[1], p0[2], p0[3]);
                e2m1x8_to_f16x2x4(w1, p1[0], p1[1], p1[2], p1[3]);
                e2m1x8_to_f16x2x4(w2, p2[0], p2[1], p2[2], p2[3]);
                e2m1x8_to_f16x2x4(w3, p3[0], p3[1], p3[2], p3[3]);
                const int sb = wi >> 1;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const uint32_t b0 = hh ? xb[wi].z : xb[wi].x, b1 = hh ? xb[wi].w : xb[wi].y;
                  mma_f16_16816(acc[0], hmul2_u32(p0[2 * hh], s[0][sb]), hmul2_u32(p1[2 * hh], s[1][sb]),
                                hmul2_u32(p0[2 * hh + 1], s[0][sb]), hmul2_u32(p1[2 * hh + 1], s[1][sb]),
                                b0, b1);
                  mma_f16_16816(acc[1], hmul2_u32(p2[2 * hh], s[2][sb]), hmul2_u32(p3[2 * hh], s[3][sb]),
                                hmul2_u32(p2[2 * hh + 1], s[2][sb]), hmul2_u32(p3[2 * hh + 1], s[3][sb]),
                                b0, b1);
                }
              }
            } else {
              uint4 xb[2];
#pragma unroll
              for (int q = 0; q < 2; ++q)
                xb[q] = g < live ? __ldg(reinterpret_cast<const uint4*>(hrow + kb * 64 + 16 * c + 8 * q))
                                 : make_uint4(0, 0, 0, 0);
              uint32_t s[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) s[i] = bcast_lo(e4m3x2_to_f16x2(sr[d][i]));
              const uint2 W[4] = {wr[d][0], wr[d][1], wr[d][2], wr[d][3]};
              if (kb + kPfDn < nkb) load_kb(kb + kPfDn, d);
#define MOE_DN64_STEP(S)                                                                      \
  {                                                                                           \
    uint32_t af[4], bf[4];                                                                    \
    a_frag64<S>(W[0], W[1], s[0], s[1], af);                                                  \
    a_frag64<S>(W[2], W[3], s[2], s[3], bf);                                                  \
    const uint32_t b0 = (S & 1) ? xb[S / 2].z : xb[S / 2].x;                                  \
    const uint32_t b1 = (S & 1) ? xb[S / 2].w : xb[S / 2].y;                                  \
    mma_f16_16816(acc[0], af[0], af[1], af[2], af[3], b0, b1);                                \
    mma_f16_16816(acc[1], bf[0], bf[1], bf[2], bf[3], b0, b1);                                \
  }
              MOE_DN64_STEP(0) MOE_DN64_STEP(1) MOE_DN64_STEP(2) MOE_DN64_STEP(3)
#undef MOE_DN64_STEP
            }
          }
        }
      }
      // acc[h][q]: row r0 + 16h + g + 8(q>>1), pair 2c + (q&1)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int n = 2 * c + (q & 1);
          if (n < live) {
            const int pos = off + tok0 + n;
            args.partial[(size_t)pos * H + r0 + 16 * hh + g + 8 * (q >> 1)] =
                ldexpf(acc[hh][q], args.he[pos]);
          }
        }
    }
    // arrivals on the (token, 64-row chunk) of every pair of the unit; the last combines
    __threadfence();
    const int chunk = r0 / kChunk;
    for (int p0 = 0; p0 < m; p0 += 32) {
      int t = -1, last = 0;
      if (p0 + lane < m) {
        t = args.pair_ids[off + p0 + lane] / args.k;
        const int need = (kChunk / kDnRows) * valid_pairs(args.pair_pos, t, args.k);
        last = atomicAdd(args.ctr + args.cc_off + t * (H / kChunk) + chunk, 1) == need - 1;
      }
      unsigned todo = __ballot_sync(0xffffffffu, last);
      if (todo) __threadfence();
      while (todo) {
        const int src = __ffs(todo) - 1;
        todo &= todo - 1;
        combine_chunk(args, __shfl_sync(0xffffffffu, t, src), chunk * kChunk);
      }
    }
    u = un;
    if (u < n_units) {
      set_unit(u);
#pragma unroll
      for (int d = 0; d < kPfDn; ++d)
        if (d < nkb) load_kb(d, d);
    }
  }
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <typename K>
int resident_blocks(K kern, int threads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

int E_active_bound(int P, int E) { return P < E ? P : E; }

}  // namespace

cudaError_t launch_decode_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                  const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                  char* ws, cudaStream_t s) {
  const int P = T * k;
  __half* xg = reinterpret_cast<__half*>(ws + L.xg);
  int32_t* xe = reinterpret_cast<int32_t*>(ws + L.xe);
  int32_t* ctr = reinterpret_cast<int32_t*>(ws + L.counters);
  const int n_ctr = decode_counter_count(T, H, E_active_bound(P, b.E));
  cudaError_t st = launch_pdl(x_gather_kernel, dim3((P + 7) / 8), dim3(256), 0, s, x_bf16, H, k,
                              (const int32_t*)csr.pair_ids, (const int32_t*)csr.expert_offsets,
                              b.E, xg, xe, ctr, n_ctr);
  if (st != cudaSuccess) return st;
  GateUpArgs a{xg, xe, b.codes, b.scales, H, F, csr.expert_offsets, csr.active_experts,
               csr.n_active, reinterpret_cast<float*>(ws + L.h),
               reinterpret_cast<__half*>(ws + L.hg), reinterpret_cast<int32_t*>(ws + L.he), ctr};
  const long long max_units = (long long)E_active_bound(P, b.E) * (F / 8);
  long long grid = (long long)resident_blocks(gate_up_kernel, 256) * sm_count();
  if (grid > (max_units + 7) / 8) grid = (max_units + 7) / 8;
  if (grid < 1) grid = 1;
  return launch_pdl(gate_up_kernel, dim3((unsigned)grid), dim3(256), 0, s, a);
}

cudaError_t launch_decode_down(const moe_nvfp4_bank& b, moe_csr csr, const float* w, int T, int H,
                               int F, int k, const moe_ws_layout& L, char* ws, float* y,
                               cudaStream_t s) {
  const int P = T * k;
  const int A = E_active_bound(P, b.E);
  DownArgs a{reinterpret_cast<const __half*>(ws + L.hg), reinterpret_cast<const int32_t*>(ws + L.he),
             b.codes, b.scales, H, F, k, T, csr.expert_offsets, csr.active_experts, csr.n_active,
             csr.pair_ids, reinterpret_cast<const int32_t*>(ws + L.pair_pos), w,
             reinterpret_cast<float*>(ws + L.partial), y, reinterpret_cast<int32_t*>(ws + L.counters),
             kCtrExpert + A};
  const long long max_units = (long long)A * (H / kDnRows);
  auto kern = (F % 128 == 0) ? down_kernel<128> : down_kernel<64>;
  long long grid = (long long)resident_blocks(kern, 256) * sm_count();
  if (grid > (max_units + 7) / 8) grid = (max_units + 7) / 8;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(256), 0, s, a);
}

int decode_counter_count(int T, int H, int A) { return kCtrExpert + A + T * (H / kChunk); }

}  // namespace moe
