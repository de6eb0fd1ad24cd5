// The work units of the TMA-fed decode kernels, shared by the per-call kernels (decode.cu)
// and the one-kernel decode layer (decode_layer.cu).
//
// A CTA runs kTmaProd producer warps and kTmaWarps consumer warps.  Each consumer warp owns
// a ring of 2^slog stage slots in shared memory (slot0 .. slot0 + 2^slog - 1), each with a
// `full` and an `empty` mbarrier; the consumer's q-th stage sits in slot slot0 + q mod
// 2^slog and completes phase (q >> slog) & 1 of that slot's barriers.  Producer warp p
// fills the rings of consumers p*PER .. p*PER+PER-1 in turn, in the order each consumes
// them, so a unit's stages never depend on another consumer.
//
//   gate/up unit = (active expert, 8 gate rows + the matching 8 up rows) over the whole H,
//                  one stage per K-chunk (nh of them) and per group of 8 pairs: two 4-D
//                  TMA boxes, codes {128 B, 8 rows, gate/up, nb K-boxes} (SWIZZLE_128B) and
//                  scales {16 B, 8 rows, gate/up, nb}; one m16n8k16 MMA carries the gate
//                  rows in M rows 0..7 and the up rows in 8..15, so each lane holds a gate
//                  and an up value of the same (row, pair) and writes h = silu(g) * u.
//   down unit    = (active expert, 16 output rows) over the whole F, one stage per group
//                  of 8 pairs: two contiguous bulk copies (16 x F/2 code bytes, then
//                  16 x F/16 scale bytes).
//
// FP4 codes are dequantised in registers (cvt.rn.f16x2.e2m1x2, times the UE4M3 scale via
// cvt.rn.f16x2.e4m3x2: every product has <= 6 significant bits, exact in f16) and fed to
// mma.sync.m16n8k16 (f32 accumulate).  Lane 4g+c of an MMA step s uses elements
// 32c + 4s .. 32c + 4s + 3 of a 128-element k-block for both operands; the tensor core
// sums over k in any order, so this shared permutation leaves the product unchanged.
#pragma once

#include "moe_internal.cuh"
#include "tma_sync.cuh"

namespace moe {
namespace {

constexpr int kTmaWarps = 16;                 // consumer warps
constexpr int kTmaSlots = 2;                  // stages per consumer warp (per-call kernels)
constexpr int kTmaProd = 4;                   // producer warps, each feeding kTmaWarps/kTmaProd

// A consumer warp's ring of stage slots.
struct Ring {
  int slot0, slog;
  __device__ __forceinline__ int slot(int q) const { return slot0 + (q & ((1 << slog) - 1)); }
  __device__ __forceinline__ uint32_t parity(int q) const { return (uint32_t)((q >> slog) & 1); }
};

// After an abort: wait (bounded) until every stage issued into the ring (q of them) has
// landed, so that no copy is still writing shared memory when the CTA exits.
__device__ __forceinline__ void ring_drain(uint64_t* full, const Ring& r, int q) {
  const int n = 1 << r.slog;
  for (int s = 0; s < n; ++s) {
    if (q <= s) continue;
    const int last = s + (((q - 1 - s) >> r.slog) << r.slog);   // last stage issued in slot s
    const uint64_t t0 = global_ns();
    while (!mbar_try(&full[r.slot0 + s], r.parity(last)) && global_ns() - t0 < 100000000ull) {
    }
  }
}

// ---------------------------------------------------------------------------
// activation rows: bf16 x and f32 h rows to f16 times a power of two
// ---------------------------------------------------------------------------
// A bf16 row of H <= 256*NP values, read by one warp (8 values per lane and piece), as f16
// times 2^-e (e from the row's amax, so the largest magnitude lands in [2^14, 2^15): exact
// for bf16 values in f16's normal range).  Returns e.
template <int NP>
__device__ __forceinline__ int x_row_f16(const uint16_t* row, bool has, int H, int lane,
                                         uint4 (&v)[NP]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int c = (lane + 32 * i) * 8;
    v[i] = has && c < H ? *reinterpret_cast<const uint4*>(row + c) : make_uint4(0, 0, 0, 0);
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
  // times 2^-e as two power-of-two factors (each a normal float for every e of a bf16 row)
  const float s1 = pow2f(-e / 2), s2 = pow2f(-e - (-e / 2));
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 hv = __floats2half2_rn((__uint_as_float(w[q] << 16) * s1) * s2,
                                           (__uint_as_float(w[q] & 0xffff0000u) * s1) * s2);
      w[q] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    v[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return e;
}
template <int NP>
__device__ __forceinline__ void x_row_store(const uint4 (&v)[NP], int H, int lane, __half* dst) {
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int c = (lane + 32 * i) * 8;
    if (c >= H) break;
    *reinterpret_cast<uint4*>(dst + c) = v[i];
  }
}

// The same conversion of a bf16 row of H values (H % 256 == 0) in two passes over the row
// (the largest magnitude, then the converted values straight to dst), so that no register
// holds more than one 16-byte piece; the second pass reads the row from L1.  Returns e.
__device__ __forceinline__ int x_row_f16_store(const uint16_t* row, int H, int lane, __half* dst) {
  float amax = 0.0f;
  for (int c = lane * 8; c < H; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xffff0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = f16_prescale_exp(amax);
  const float s1 = pow2f(-e / 2), s2 = pow2f(-e - (-e / 2));
  for (int c = lane * 8; c < H; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + c);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 hv = __floats2half2_rn((__uint_as_float(w[q] << 16) * s1) * s2,
                                           (__uint_as_float(w[q] & 0xffff0000u) * s1) * s2);
      w[q] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return e;
}

// An f32 row of F <= 128*NR values, one warp: f16 times 2^-e into dst, e into *e_out.  The
// row stays in registers, so it is read once.
template <int NR>
__device__ __forceinline__ void h_row_f16(const float* row, int F, int lane, __half* dst,
                                          int32_t* e_out) {
  float4 v[NR];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int c = 4 * lane + 128 * i;
    v[i] = c < F ? *reinterpret_cast<const float4*>(row + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = f16_prescale_exp(amax);
  if (lane == 0) *e_out = e;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int c = 4 * lane + 128 * i;
    if (c >= F) break;
    const __half2 h0 = __floats2half2_rn(ldexpf(v[i].x, -e), ldexpf(v[i].y, -e));
    const __half2 h1 = __floats2half2_rn(ldexpf(v[i].z, -e), ldexpf(v[i].w, -e));
    *reinterpret_cast<uint2*>(dst + c) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
  }
}

// combine: columns r..r+3 of y[t] = sum_j w[t, j] * z[pos(t, j)] in ascending j, with the
// token's k positions and weights in s_pos / s_w (a position < 0: the pair has no row).
// The partial rows are loaded eight pairs at a time.
__device__ __forceinline__ float4 combine4(const float* __restrict__ partial, const int* s_pos,
                                           const float* s_w, int k, int H, int r) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += 8) {
    float4 z[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q;
      const int pos = j < k ? s_pos[j] : -1;
      z[q] = pos >= 0 ? __ldcs(reinterpret_cast<const float4*>(partial + (size_t)pos * H + r))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q;
      if (j >= k || s_pos[j] < 0) continue;
      const float wj = s_w[j];
      acc.x = fmaf(wj, z[q].x, acc.x);
      acc.y = fmaf(wj, z[q].y, acc.y);
      acc.z = fmaf(wj, z[q].z, acc.z);
      acc.w = fmaf(wj, z[q].w, acc.w);
    }
  }
  return acc;
}

// A 16-byte piece of an activation row.  RO: the row was written by an earlier kernel, so
// it is read-only for this one and may take the non-coherent path; otherwise (written
// earlier in the same kernel, before a grid-wide barrier) a plain coherent load.
template <bool RO>
__device__ __forceinline__ uint4 ld_act(const __half* p) {
  if (RO) return __ldg(reinterpret_cast<const uint4*>(p));
  return *reinterpret_cast<const uint4*>(p);
}

// ---------------------------------------------------------------------------
// gate/up units
// ---------------------------------------------------------------------------
struct GuTmaArgs {
  const __half* xg;           // f16 activation rows times 2^-xe: row pos of the CSR, or (with
  const int32_t* xe;          // row_tok) row row_tok[pos], one per token
  int H, F, nh, nb;                           // K-chunks per unit, 128-byte boxes per chunk
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  float* h;
  uint32_t* err;
  const float* alpha = nullptr;   // [E] per-expert second-level weight scale, or none
  const int32_t* row_tok = nullptr;   // [P] token of each CSR row (xg / xe rows per token)
};

__host__ __device__ constexpr int gu_stage_bytes(int nb) {
  return ((2 * nb * 1024 + 2 * 8 * nb * 16) + 1023) / 1024 * 1024;
}
// byte offsets inside a stage: codes land as [K-box][gate, up][row][128 B] (the 128-byte
// swizzle puts chunk c of row r at c ^ r, so the quarter-warp reads of rows g..g+7 hit
// distinct banks), scales as [K-box][gate, up][row][16 B]
__device__ __forceinline__ uint32_t gu_code_off(int kbox, int mat, int row, int chunk16) {
  return kbox * 2048 + mat * 1024 + row * 128 + ((chunk16 ^ row) << 4);
}
__device__ __forceinline__ uint32_t gu_scale_off(int nb, int kbox, int mat, int row) {
  return 2 * nb * 1024 + kbox * 256 + mat * 128 + row * 16;
}

// Producer cursor over one consumer's gate/up units: unit, pair group, K-chunk, stages issued.
struct GuCursor {
  int u, pass, chunk, q;
};

// Issue the stage at the cursor into the consumer's ring and advance the cursor (the next
// unit of this consumer is u + u_step).  False if the wait for the slot gave up.
__device__ __forceinline__ bool gu_issue(const GuTmaArgs& a, const CUtensorMap* tmap_c,
                                         const CUtensorMap* tmap_s, GuCursor& cur, int u_step,
                                         unsigned char* smem, int stage_bytes, uint64_t* full,
                                         uint64_t* empty, const Ring& ring,
                                         volatile int* abort_flag) {
  const int nb = a.nb, nrb = a.F / 8;
  const int slot = ring.slot(cur.q);
  if (!mbar_wait(&empty[slot], ring.parity(cur.q) ^ 1, abort_flag, a.err)) return false;
  const int e = a.active[cur.u / nrb];
  unsigned char* sb = smem + slot * stage_bytes;
  mbar_expect_tx(&full[slot], (uint32_t)(2 * nb * 1024 + 2 * 8 * nb * 16));
  // coordinates {byte in K-box, row of the matrix, 2e (gate) .. 2e+1 (up), K-box}
  tma_load_4d(sb, tmap_c, 0, (cur.u % nrb) * 8, 2 * e, cur.chunk * nb, &full[slot]);
  tma_load_4d(sb + 2 * nb * 1024, tmap_s, 0, (cur.u % nrb) * 8, 2 * e, cur.chunk * nb, &full[slot]);
  ++cur.q;
  if (++cur.chunk == a.nh) {
    cur.chunk = 0;
    const int m = a.offsets[e + 1] - a.offsets[e];
    if (++cur.pass * 8 >= m) { cur.pass = 0; cur.u += u_step; }
  }
  return true;
}

// Consume gate/up unit u (all its pair groups and K-chunks) and write its h values (f32,
// CSR order).  q counts the stages this warp consumed.  False if a wait gave up.
// TOK: activation rows per token (args.row_tok), else per CSR row.
template <int NB, bool ALPHA, bool RO = true, bool TOK = false>
__device__ __forceinline__ bool gu_consume_unit(const GuTmaArgs& args, int u, unsigned char* smem,
                                                int stage_bytes, uint64_t* full, uint64_t* empty,
                                                const Ring& ring, int& q, volatile int* abort_flag) {
  constexpr int nb = NB;                                   // 128-byte K-boxes per stage
  const int lane = threadIdx.x & 31;
  const int H = args.H, F = args.F, nh = args.nh;
  const int nrb = F / 8;                                   // units per expert
  const int g = lane >> 2, c = lane & 3;
  const int e = args.active[u / nrb];
  const int i0 = (u % nrb) * 8;
  const int off = args.offsets[e];
  const int m = args.offsets[e + 1] - off;
  for (int tok0 = 0; tok0 < m; tok0 += 8) {
    const int live = min(8, m - tok0);
    const int xr = off + tok0 + (g < live ? g : 0);
    const __half* xrow = args.xg + (size_t)(TOK ? args.row_tok[xr] : xr) * H + 32 * c;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    uint4 xb[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
      xb[qq] = g < live ? ld_act<RO>(xrow + 8 * qq) : make_uint4(0, 0, 0, 0);
    for (int hc = 0; hc < nh; ++hc, ++q) {
      const int slot = ring.slot(q);
      if (!mbar_wait_warp(&full[slot], ring.parity(q), abort_flag, args.err)) return false;
      const uint32_t sb = smem_u32(smem + slot * stage_bytes);
#pragma unroll
      for (int kl = 0; kl < 2 * nb; ++kl) {             // 128-element k-blocks of the chunk
        const int kbg = hc * 2 * nb + kl;               // k-block within the row
        uint4 xn[4];
        const bool nxt = g < live && kbg + 1 < H / 128;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq)
          xn[qq] = nxt ? ld_act<RO>(xrow + (kbg + 1) * 128 + 8 * qq) : make_uint4(0, 0, 0, 0);
        const int chunk = ((kl & 1) << 2) + c;           // 16-byte chunk within the K-box row
        const int kbox = kl >> 1;
        uint4 WGv, WUv;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(WGv.x), "=r"(WGv.y), "=r"(WGv.z), "=r"(WGv.w) : "r"(sb + gu_code_off(kbox, 0, g, chunk)));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(WUv.x), "=r"(WUv.y), "=r"(WUv.z), "=r"(WUv.w) : "r"(sb + gu_code_off(kbox, 1, g, chunk)));
        // the K-box's 16 scale bytes per row: 8 for each of its two 128-element k-blocks
        unsigned short s16g, s16u;
        const uint32_t so = ((kl & 1) << 3) + 2 * c;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(s16g) : "r"(sb + gu_scale_off(nb, kbox, 0, g) + so));
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(s16u) : "r"(sb + gu_scale_off(nb, kbox, 1, g) + so));
        const uint32_t fg = e4m3x2_to_f16x2(s16g), fu = e4m3x2_to_f16x2(s16u);
        const uint32_t s_g[2] = {bcast_lo(fg), bcast_hi(fg)};
        const uint32_t s_u[2] = {bcast_lo(fu), bcast_hi(fu)};
        const uint32_t WG[4] = {WGv.x, WGv.y, WGv.z, WGv.w};
        const uint32_t WU[4] = {WUv.x, WUv.y, WUv.z, WUv.w};
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          uint32_t gq[4], uq[4];
          e2m1x8_to_f16x2x4(WG[wi], gq[0], gq[1], gq[2], gq[3]);
          e2m1x8_to_f16x2x4(WU[wi], uq[0], uq[1], uq[2], uq[3]);
          const int sbk = wi >> 1;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            mma_f16_16816(acc, hmul2_u32(gq[2 * hh], s_g[sbk]), hmul2_u32(uq[2 * hh], s_u[sbk]),
                          hmul2_u32(gq[2 * hh + 1], s_g[sbk]), hmul2_u32(uq[2 * hh + 1], s_u[sbk]),
                          hh ? xb[wi].z : xb[wi].x, hh ? xb[wi].w : xb[wi].y);
        }
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) xb[qq] = xn[qq];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    // acc[0..1]: gate row i0+g, pairs 2c, 2c+1; acc[2..3]: up row i0+g, same pairs
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const int n = 2 * c + qq;
      if (n < live) {
        const int pos = off + tok0 + n;
        const int ex = args.xe[TOK ? args.row_tok[pos] : pos];
        const float al = ALPHA ? __ldg(args.alpha + e) : 1.0f;
        args.h[(size_t)pos * F + i0 + g] =
            silu_f(al * ldexpf(acc[qq], ex)) * (al * ldexpf(acc[2 + qq], ex));
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// down units
// ---------------------------------------------------------------------------
// With F/2 bytes per row the quarter-warp reads of rows g, g+1 at 64 kb + 16 c fall in
// different bank halves whenever F/2 is an odd multiple of 64 bytes.
struct DnTmaArgs {
  const __half* hg;
  const int32_t* he;
  const uint8_t* codes;
  const uint8_t* scales;
  int H, F;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  float* partial;
  uint32_t* err;
  const float* alpha = nullptr;   // [E] per-expert second-level weight scale, or none
};

__host__ __device__ constexpr int dn_stage_bytes(int F) {
  return ((16 * (F / 2) + 16 * (F / 16)) + 1023) / 1024 * 1024;
}

struct DnCursor {
  int u, pass, q;
};

// Issue the stage at the cursor (the unit's 16 rows: codes, then scales) and advance.
__device__ __forceinline__ bool dn_issue(const DnTmaArgs& a, DnCursor& cur, int u_step,
                                         unsigned char* smem, int stage_bytes, uint64_t* full,
                                         uint64_t* empty, const Ring& ring,
                                         volatile int* abort_flag) {
  const int H = a.H, nrb = H / 16;
  const int row_bytes = a.F / 2, srow = a.F / 16;
  const uint32_t codes_bytes = 16 * row_bytes, scale_bytes = 16 * srow;
  const int slot = ring.slot(cur.q);
  if (!mbar_wait(&empty[slot], ring.parity(cur.q) ^ 1, abort_flag, a.err)) return false;
  const int e = a.active[cur.u / nrb];
  const size_t r0 = (size_t)e * H + (cur.u % nrb) * 16;
  unsigned char* sb = smem + slot * stage_bytes;
  mbar_expect_tx(&full[slot], codes_bytes + scale_bytes);
  bulk_load(sb, a.codes + r0 * row_bytes, codes_bytes, &full[slot]);
  bulk_load(sb + codes_bytes, a.scales + r0 * srow, scale_bytes, &full[slot]);
  ++cur.q;
  const int m = a.offsets[e + 1] - a.offsets[e];
  if (++cur.pass * 8 >= m) { cur.pass = 0; cur.u += u_step; }
  return true;
}

// Consume down unit u and write its rows of the per-pair partials (f32, CSR order).
template <bool RO = true>
__device__ __forceinline__ bool dn_consume_unit(const DnTmaArgs& args, int u, unsigned char* smem,
                                                int stage_bytes, uint64_t* full, uint64_t* empty,
                                                const Ring& ring, int& q, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int H = args.H, F = args.F;
  const int row_bytes = F / 2, srow = F / 16;
  const uint32_t codes_bytes = 16 * row_bytes;
  const int nrb = H / 16;
  const int g = lane >> 2, c = lane & 3;
  const int nkb = F / 128;
  const int e = args.active[u / nrb];
  const int r0 = (u % nrb) * 16;
  const int off = args.offsets[e];
  const int m = args.offsets[e + 1] - off;
  for (int tok0 = 0; tok0 < m; tok0 += 8, ++q) {
    const int live = min(8, m - tok0);
    const __half* hrow = args.hg + (size_t)(off + tok0 + (g < live ? g : 0)) * F + 32 * c;
    const int slot = ring.slot(q);
    if (!mbar_wait_warp(&full[slot], ring.parity(q), abort_flag, args.err)) return false;
    const uint32_t sb = smem_u32(smem + slot * stage_bytes);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    uint4 xb[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
      xb[qq] = g < live ? ld_act<RO>(hrow + 8 * qq) : make_uint4(0, 0, 0, 0);
    for (int kb = 0; kb < nkb; ++kb) {
      uint4 xn[4];
      const bool nxt = g < live && kb + 1 < nkb;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        xn[qq] = nxt ? ld_act<RO>(hrow + (kb + 1) * 128 + 8 * qq) : make_uint4(0, 0, 0, 0);
      uint4 A0, A1;
      const uint32_t a0 = sb + g * row_bytes + kb * 64 + 16 * c;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(A0.x), "=r"(A0.y), "=r"(A0.z), "=r"(A0.w) : "r"(a0));
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(A1.x), "=r"(A1.y), "=r"(A1.z), "=r"(A1.w) : "r"(a0 + 8 * row_bytes));
      unsigned short s0, s1;
      const uint32_t sa = sb + codes_bytes + g * srow + kb * 8 + 2 * c;
      asm volatile("ld.shared.u16 %0, [%1];" : "=h"(s0) : "r"(sa));
      asm volatile("ld.shared.u16 %0, [%1];" : "=h"(s1) : "r"(sa + 8 * srow));
      const uint32_t f0 = e4m3x2_to_f16x2(s0), f1 = e4m3x2_to_f16x2(s1);
      const uint32_t sc0[2] = {bcast_lo(f0), bcast_hi(f0)};
      const uint32_t sc1[2] = {bcast_lo(f1), bcast_hi(f1)};
      const uint32_t W0[4] = {A0.x, A0.y, A0.z, A0.w}, W1[4] = {A1.x, A1.y, A1.z, A1.w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        uint32_t p0[4], p1[4];
        e2m1x8_to_f16x2x4(W0[wi], p0[0], p0[1], p0[2], p0[3]);
        e2m1x8_to_f16x2x4(W1[wi], p1[0], p1[1], p1[2], p1[3]);
        const int sbk = wi >> 1;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          mma_f16_16816(acc, hmul2_u32(p0[2 * hh], sc0[sbk]), hmul2_u32(p1[2 * hh], sc1[sbk]),
                        hmul2_u32(p0[2 * hh + 1], sc0[sbk]), hmul2_u32(p1[2 * hh + 1], sc1[sbk]),
                        hh ? xb[wi].z : xb[wi].x, hh ? xb[wi].w : xb[wi].y);
      }
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) xb[qq] = xn[qq];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    // acc[q]: row r0 + g + 8(q>>1), pair 2c + (q&1)
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int n = 2 * c + (qq & 1);
      if (n < live) {
        const int pos = off + tok0 + n;
        args.partial[(size_t)pos * H + r0 + g + 8 * (qq >> 1)] =
            (args.alpha ? __ldg(args.alpha + e) : 1.0f) * ldexpf(acc[qq], args.he[pos]);
      }
    }
  }
  return true;
}

}  // namespace
}  // namespace moe
