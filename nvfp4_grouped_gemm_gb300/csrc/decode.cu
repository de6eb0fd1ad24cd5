// Decode path below the tensor-core switch (fewer than moe_decode_tensor_core_min_pairs()
// pairs; from there on sliced.cu): few pairs per expert, memory-bound on the NVFP4 weight
// bytes.
//
// The grid is indexed by active expert, not by pair, so every active expert's rows are
// streamed from HBM exactly once per call (the union-of-experts gather).  Kernels:
//
//   x_gather_kernel   token t's x row as f16 times 2^-e (e from the row's amax, so the
//                     largest magnitude lands in [2^14, 2^15): exact for bf16 values in
//                     f16's normal range), one warp per token, converted and stored before
//                     the wait for the CSR; after it, each of the token's CSR rows gets
//                     the token's index (row_tok), through which the gate/up units read x
//   gate_up_kernel    CTA = (active expert, 16 gate rows + the matching 16 up rows); the
//                     CTA's weight bytes land in shared memory with 16-byte cp.async
//                     issued by every thread up front, the activation fragments come
//                     straight from the gathered f16 rows, 8 warps split the H
//                     reduction (summed in a fixed order), one warp writes h = silu(g)*u
//   h_prep_kernel     CSR row r of h (f32) -> f16 times 2^-e, as for x
//   down_kernel       CTA = (active expert, 128 output rows), weights and the expert's h
//                     rows in shared memory, warp w owns 16 rows over the whole F
//   gate_up_tma_kernel, down_tma_kernel   from 8 units per SM on: one CTA per SM, four
//                     producer warps feed a TMA / bulk-copy ring, sixteen consumer warps
//                     each multiply whole units (8 gate + 8 up rows, or 16 down rows)
//   combine_kernel    y[t] = sum_j w[t,j] z[pos(t,j)] in ascending j, no atomics (also the
//                     combine of the sliced form)
//
// FP4 codes are dequantised in registers (cvt.rn.f16x2.e2m1x2, times the UE4M3 scale via
// cvt.rn.f16x2.e4m3x2: every product has <= 6 significant bits, exact in f16) and fed
// to mma.sync.m16n8k16 (f32 accumulate).  Lane 4g+c of an MMA step s uses elements
// 32c + 4s .. 32c + 4s + 3 of a 128-element k-block for both operands; the tensor core
// sums over k in any order, so this shared permutation leaves the product unchanged.
//
// Kernels after the CSR are launched with programmatic dependent launch: each issues
// the loads that depend only on the CSR (two or more kernels back, complete before its
// predecessor passed its own griddepcontrol.wait) and then waits for its predecessor.
#include "decode_units.cuh"

namespace moe {

namespace {


__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src) : "memory");
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

// Byte offset of 16-byte chunk `q` of row `r` in a shared code tile: with `swz` (rows a
// multiple of 128 bytes) odd rows swap the two 64-byte halves of each 128-byte window, so
// the quarter-warp reading the same chunk of rows g, g+1 hits distinct banks.
__device__ __forceinline__ int wchunk(int r, int q, int row_bytes, bool swz) {
  return r * row_bytes + ((swz ? (q ^ ((r & 1) << 2)) : q) << 4);
}

// Byte offset of 16-byte chunk `lc` of a staged f16 activation row: XOR-swizzled so the
// quarter-warp reading chunks 4c+u of rows g, g+1 touches eight distinct bank groups.
__device__ __forceinline__ int swz_chunk(int lc) { return (lc ^ (((lc >> 3) & 1) << 1)) * 16; }

// ---------------------------------------------------------------------------
// gather + f16 prescale of the activation rows of every CSR row (decode stage a3)
// ---------------------------------------------------------------------------
// One warp per pair p = t*k + j.  The token's row depends only on x, so it is read and
// converted before the wait; after it, the row goes to the pair's CSR row pair_pos[p].
template <int NP>
__global__ void __launch_bounds__(256) x_gather_kernel(const uint16_t* __restrict__ x, int H, int k,
                                                       int T, const int32_t* __restrict__ pair_pos,
                                                       __half* __restrict__ xg,
                                                       int32_t* __restrict__ xe,
                                                       int32_t* __restrict__ row_tok) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const bool has = t < T;
  // the whole row in registers (H <= 256 * NP: NP pieces of 8 values per lane); the row and
  // its exponent depend on x alone, so they are stored before the wait
  uint4 v[NP];
  const int e = x_row_f16<NP>(x + (size_t)(has ? t : 0) * H, has, H, lane, v);
  if (has) {
    if (lane == 0) xe[t] = e;
    x_row_store<NP>(v, H, lane, xg + (size_t)t * H);
  }
  pdl_wait();                                  // pair_pos is complete
  pdl_trigger();
  if (!has || lane >= k) return;
  const int pos = pair_pos[(size_t)t * k + lane];
  if (pos >= 0) row_tok[pos] = t;              // invalid expert id: the pair has no row
}

// Same for h (f32 rows already in CSR order), F <= 128*NR: the row stays in registers, so
// h is read once.
template <int NR>
__global__ void __launch_bounds__(256) h_prep_kernel(const float* __restrict__ h, int F,
                                                     const int32_t* __restrict__ offsets, int E,
                                                     __half* __restrict__ hg,
                                                     int32_t* __restrict__ he) {
  pdl_wait();
  pdl_trigger();
  const int pos = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (pos >= offsets[E]) return;
  h_row_f16<NR>(h + (size_t)pos * F, F, threadIdx.x & 31, hg + (size_t)pos * F, he + pos);
}

// ---------------------------------------------------------------------------
// gate/up + SiLU
// ---------------------------------------------------------------------------
struct GateUpArgs {
  const __half* xg;        // [T][H] f16 activation rows, one per token
  const int32_t* xe;       // [T]
  const uint8_t* codes;
  const uint8_t* scales;
  int H, F;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  float* h;
  const float* alpha = nullptr;   // [E] per-expert second-level weight scale, or none
  const int32_t* row_tok = nullptr;   // [P] token of each CSR row
};

// Persistent: CTA c owns a contiguous range of work units u = (active expert, 16-row
// block), ordered by expert.  Each unit's weight rows (16 gate + 16 up) land in one of two
// shared buffers with 16-byte cp.async issued by every thread; the next unit's copy is in
// flight while the current one is multiplied.  KMAX = ceil(H / 128 / 8): k-blocks per
// warp, whose activation fragments stay in registers while the expert does not change.
template <int KMAX>
__global__ void __launch_bounds__(256, 2) gate_up_kernel(const GateUpArgs args) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = args.H, F = args.F;
  const int row_bytes = H / 2, srow = H / 16;
  const int nrb = F / 16;
  const int wbytes = (32 * row_bytes + 32 * srow + 127) & ~127;
  float* red = reinterpret_cast<float*>(smem + 2 * wbytes);      // [8 warps][32][8]
  const int n_units = *args.n_active * nrb;                        // CSR is complete
  const int u_beg = (int)((long long)blockIdx.x * n_units / gridDim.x);
  const int u_end = (int)((long long)(blockIdx.x + 1) * n_units / gridDim.x);
  const size_t rows2F = (size_t)2 * F;
  const int cpr = row_bytes / 16, spr = srow / 16;

  // thread t copies row t/8 (rows 0..15 gate, 16..31 up), chunks t%8, t%8 + 8, ...
  // (H % 256 == 0, so a code row has a multiple of 8 chunks); no divisions in the loop
  const int my_r = threadIdx.x >> 3, my_q = threadIdx.x & 7;
  auto issue = [&](int u, int buf) {
    const int e = args.active[u / nrb];
    const int i0 = (u % nrb) * 16;
    unsigned char* wc = smem + buf * wbytes;
    unsigned char* ws = wc + 32 * row_bytes;
    const size_t wrow = (size_t)e * rows2F + (my_r < 16 ? i0 + my_r : F + i0 + my_r - 16);
    const uint8_t* src = args.codes + wrow * row_bytes;
    unsigned char* dst = wc + my_r * row_bytes;
    const int swz = (my_r & 1) << 2;
    for (int q = my_q; q < cpr; q += 8) cp_async16(dst + ((q ^ swz) << 4), src + q * 16);
    const uint8_t* ssrc = args.scales + wrow * srow;
    for (int q = my_q; q < spr; q += 8) cp_async16(ws + my_r * srow + q * 16, ssrc + q * 16);
  };

  if (u_beg < u_end) issue(u_beg, 0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  pdl_wait();                                   // the gathered activations are complete

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int nkb = H / 128;
  const int kb_beg = warp * nkb / 8, kb_end = (warp + 1) * nkb / 8;
  uint4 xb[KMAX][4];
  int cur_e = -1, cur_t0 = -1;

  for (int u = u_beg, i = 0; u < u_end; ++u, ++i) {
    if (u + 1 < u_end) issue(u + 1, (i + 1) & 1);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    const unsigned char* wc = smem + (i & 1) * wbytes;
    const unsigned char* ws = wc + 32 * row_bytes;
    const int e = args.active[u / nrb];
    const int i0 = (u % nrb) * 16;
    const int off = args.offsets[e];
    const int m = args.offsets[e + 1] - off;
    for (int tok0 = 0; tok0 < m; tok0 += 8) {
      const int live = min(8, m - tok0);
      if (e != cur_e || tok0 != cur_t0) {
        const int xr = g < live ? args.row_tok[off + tok0 + g] : 0;
        const __half* xrow = args.xg + (size_t)xr * H + 32 * c;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kb = kb_beg + j;
            xb[j][q] = (g < live && kb < kb_end)
                           ? __ldg(reinterpret_cast<const uint4*>(xrow + kb * 128 + 8 * q))
                           : make_uint4(0, 0, 0, 0);
          }
        cur_e = e;
        cur_t0 = tok0;
      }
      float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        const int kb = kb_beg + j;
        if (kb < kb_end) {
          const uint4 c0 = *reinterpret_cast<const uint4*>(wc + wchunk(g, kb * 4 + c, row_bytes, true));
          const uint4 c1 = *reinterpret_cast<const uint4*>(wc + wchunk(g + 8, kb * 4 + c, row_bytes, true));
          const uint4 c2 = *reinterpret_cast<const uint4*>(wc + wchunk(g + 16, kb * 4 + c, row_bytes, true));
          const uint4 c3 = *reinterpret_cast<const uint4*>(wc + wchunk(g + 24, kb * 4 + c, row_bytes, true));
          const unsigned char* sp = ws + g * srow + kb * 8 + 2 * c;
          const uint32_t f0 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sp));
          const uint32_t f1 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sp + 8 * srow));
          const uint32_t f2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sp + 16 * srow));
          const uint32_t f3 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sp + 24 * srow));
          // words 0,1 of a row use the scale of block 2c, words 2,3 that of block 2c+1
          const uint32_t s0[2] = {bcast_lo(f0), bcast_hi(f0)}, s1[2] = {bcast_lo(f1), bcast_hi(f1)};
          const uint32_t s2[2] = {bcast_lo(f2), bcast_hi(f2)}, s3[2] = {bcast_lo(f3), bcast_hi(f3)};
          const uint32_t W0[4] = {c0.x, c0.y, c0.z, c0.w}, W1[4] = {c1.x, c1.y, c1.z, c1.w};
          const uint32_t W2[4] = {c2.x, c2.y, c2.z, c2.w}, W3[4] = {c3.x, c3.y, c3.z, c3.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            // one word per row = two MMA steps (2wi, 2wi+1); each byte converted once
            uint32_t g0[4], g1[4], u0[4], u1[4];
            e2m1x8_to_f16x2x4(W0[wi], g0[0], g0[1], g0[2], g0[3]);
            e2m1x8_to_f16x2x4(W1[wi], g1[0], g1[1], g1[2], g1[3]);
            e2m1x8_to_f16x2x4(W2[wi], u0[0], u0[1], u0[2], u0[3]);
            e2m1x8_to_f16x2x4(W3[wi], u1[0], u1[1], u1[2], u1[3]);
            const int sb = wi >> 1;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t b0 = h ? xb[j][wi].z : xb[j][wi].x;
              const uint32_t b1 = h ? xb[j][wi].w : xb[j][wi].y;
              mma_f16_16816(accg, hmul2_u32(g0[2 * h], s0[sb]), hmul2_u32(g1[2 * h], s1[sb]),
                            hmul2_u32(g0[2 * h + 1], s0[sb]), hmul2_u32(g1[2 * h + 1], s1[sb]), b0, b1);
              mma_f16_16816(accu, hmul2_u32(u0[2 * h], s2[sb]), hmul2_u32(u1[2 * h], s3[sb]),
                            hmul2_u32(u0[2 * h + 1], s2[sb]), hmul2_u32(u1[2 * h + 1], s3[sb]), b0, b1);
            }
          }
        }
      }
      // fixed-order sum over the 8 warps' k ranges
      float* mine = red + (warp * 32 + lane) * 8;
#pragma unroll
      for (int q = 0; q < 4; ++q) { mine[q] = accg[q]; mine[4 + q] = accu[q]; }
      __syncthreads();
      if (warp == 0) {
        float sg[4] = {0.f, 0.f, 0.f, 0.f}, su[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < 8; ++w) {
          const float* src = red + (w * 32 + lane) * 8;
#pragma unroll
          for (int q = 0; q < 4; ++q) { sg[q] += src[q]; su[q] += src[4 + q]; }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int n = 2 * c + (q & 1);
          const int ii = i0 + g + 8 * (q >> 1);
          if (n < live) {
            const int ex = args.xe[args.row_tok[off + tok0 + n]];
            const float al = args.alpha ? __ldg(args.alpha + e) : 1.0f;
            args.h[(size_t)(off + tok0 + n) * F + ii] =
                silu_f(al * ldexpf(sg[q], ex)) * (al * ldexpf(su[q], ex));
          }
        }
      }
      __syncthreads();
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------------------
// down projection: z_p = W_down[e] h_p, rows of the per-pair partials in CSR order
// ---------------------------------------------------------------------------
struct DownArgs {
  const __half* hg;        // [P][F]
  const int32_t* he;       // [P]
  const uint8_t* codes;
  const uint8_t* scales;
  int H, F;
  const int32_t* offsets;
  const int32_t* active;
  const int32_t* n_active;
  float* partial;
  const float* alpha = nullptr;   // [E] per-expert second-level weight scale, or none
};

// Persistent like the gate/up kernel: unit = (active expert, 128 output rows), two weight
// buffers, the expert's h rows staged once while the expert does not change.
// KB = 128 (16-byte lane pieces) when F % 128 == 0, else 64 (8-byte pieces).
template <int KB>
__global__ void __launch_bounds__(256, 2) down_kernel(const DownArgs args) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = args.H, F = args.F;
  const int nrb = H / 128;
  const int row_bytes = F / 2, srow = F / 16;
  const bool swz = (row_bytes % 128) == 0;
  const int wbytes = (128 * row_bytes + 128 * srow + 127) & ~127;
  const int hrow_bytes = F * 2 + 16;
  unsigned char* hs = smem + 2 * wbytes;                            // [8][hrow_bytes]
  const int n_units = *args.n_active * nrb;
  const int u_beg = (int)((long long)blockIdx.x * n_units / gridDim.x);
  const int u_end = (int)((long long)(blockIdx.x + 1) * n_units / gridDim.x);
  const int cpr = row_bytes / 16;

  // thread t copies row t/2, chunks t%2, t%2 + 2, ... of the unit's 128 rows
  const int my_r = threadIdx.x >> 1, my_q = threadIdx.x & 1;
  auto issue = [&](int u, int buf) {
    const int e = args.active[u / nrb];
    const int r0 = (u % nrb) * 128;
    unsigned char* wc = smem + buf * wbytes;
    unsigned char* ws = wc + 128 * row_bytes;
    const unsigned char* src = args.codes + ((size_t)e * H + r0 + my_r) * row_bytes;
    unsigned char* dst = wc + my_r * row_bytes;
    const int sw = swz ? (my_r & 1) << 2 : 0;
    for (int q = my_q; q < cpr; q += 2) cp_async16(dst + ((q ^ sw) << 4), src + q * 16);
    const unsigned char* ssrc = args.scales + ((size_t)e * H + r0) * srow;
    for (int idx = threadIdx.x; idx < 128 * srow / 16; idx += 256)
      cp_async16(ws + idx * 16, ssrc + idx * 16);
  };

  if (u_beg < u_end) issue(u_beg, 0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  pdl_wait();                                   // h in f16 is complete

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int nkb = F / KB;
  constexpr int LB = KB / 8;          // code bytes per lane per k-block
  int cur_e = -1, cur_t0 = -1;

  for (int u = u_beg, i = 0; u < u_end; ++u, ++i) {
    const int e = args.active[u / nrb];
    const int r0 = (u % nrb) * 128;
    const int off = args.offsets[e];
    const int m = args.offsets[e + 1] - off;
    const unsigned char* wc = smem + (i & 1) * wbytes;
    const unsigned char* ws = wc + 128 * row_bytes;
    for (int tok0 = 0; tok0 < m; tok0 += 8) {
      const int live = min(8, m - tok0);
      // stage the expert's h rows (copy group committed before the next unit's weights)
      if (e != cur_e || tok0 != cur_t0) {
        for (int idx = threadIdx.x; idx < live * (F / 8); idx += 256) {
          const int slot = idx / (F / 8), ch = idx - slot * (F / 8);
          cp_async16(hs + slot * hrow_bytes + swz_chunk(ch),
                     args.hg + (size_t)(off + tok0 + slot) * F + ch * 8);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        cur_e = e;
        cur_t0 = tok0;
      }
      if (tok0 == 0) {
        // prefetch the next unit, then wait for everything but that prefetch
        if (u + 1 < u_end) issue(u + 1, (i + 1) & 1);
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      __syncthreads();
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const int rw = warp * 16 + g;
      for (int kb = 0; kb < nkb; ++kb) {
        if (KB == 128) {
          const uint4 a0 = *reinterpret_cast<const uint4*>(wc + wchunk(rw, kb * 4 + c, row_bytes, swz));
          const uint4 a1 = *reinterpret_cast<const uint4*>(wc + wchunk(rw + 8, kb * 4 + c, row_bytes, swz));
          const unsigned char* sp = ws + rw * srow + kb * 8 + 2 * c;
          const uint32_t f0 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sp));
          const uint32_t f1 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sp + 8 * srow));
          uint4 xb[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            xb[q] = *reinterpret_cast<const uint4*>(hs + g * hrow_bytes + swz_chunk(kb * 16 + 4 * c + q));
          const uint32_t s0[2] = {bcast_lo(f0), bcast_hi(f0)}, s1[2] = {bcast_lo(f1), bcast_hi(f1)};
          const uint32_t W0[4] = {a0.x, a0.y, a0.z, a0.w}, W1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            uint32_t p0[4], p1[4];
            e2m1x8_to_f16x2x4(W0[wi], p0[0], p0[1], p0[2], p0[3]);
            e2m1x8_to_f16x2x4(W1[wi], p1[0], p1[1], p1[2], p1[3]);
            const int sb = wi >> 1;
#pragma unroll
            for (int h = 0; h < 2; ++h)
              mma_f16_16816(acc, hmul2_u32(p0[2 * h], s0[sb]), hmul2_u32(p1[2 * h], s1[sb]),
                            hmul2_u32(p0[2 * h + 1], s0[sb]), hmul2_u32(p1[2 * h + 1], s1[sb]),
                            h ? xb[wi].z : xb[wi].x, h ? xb[wi].w : xb[wi].y);
          }
        } else {
          const unsigned char* rp = wc + rw * row_bytes + LB * c + kb * 32;
          const uint2 a0 = *reinterpret_cast<const uint2*>(rp);
          const uint2 a1 = *reinterpret_cast<const uint2*>(rp + 8 * row_bytes);
          const unsigned char* sp = ws + rw * srow + kb * 4 + c;
          const uint32_t f0 = bcast_lo(e4m3x2_to_f16x2(sp[0]));
          const uint32_t f1 = bcast_lo(e4m3x2_to_f16x2(sp[8 * srow]));
          uint4 xb[2];
#pragma unroll
          for (int q = 0; q < 2; ++q)
            xb[q] = *reinterpret_cast<const uint4*>(hs + g * hrow_bytes + swz_chunk(kb * 8 + 2 * c + q));
#define MOE_DN64_STEP(S)                                                                   \
  {                                                                                        \
    uint32_t af[4];                                                                        \
    a_frag64<S>(a0, a1, f0, f1, af);                                                       \
    mma_f16_16816(acc, af[0], af[1], af[2], af[3], (S & 1) ? xb[S / 2].z : xb[S / 2].x,     \
                  (S & 1) ? xb[S / 2].w : xb[S / 2].y);                                    \
  }
          MOE_DN64_STEP(0) MOE_DN64_STEP(1) MOE_DN64_STEP(2) MOE_DN64_STEP(3)
#undef MOE_DN64_STEP
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = 2 * c + (q & 1);
        const int r = r0 + rw + 8 * (q >> 1);
        if (n < live)
          args.partial[(size_t)(off + tok0 + n) * H + r] =
              (args.alpha ? __ldg(args.alpha + e) : 1.0f) * ldexpf(acc[q], args.he[off + tok0 + n]);
      }
      __syncthreads();
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------------------
// combine: y[t, :] = sum_j w[t, j] * z[pair_pos[t*k + j], :] in ascending j
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ w, const int32_t* __restrict__ pair_pos,
               const float* __restrict__ partial, int H, int k, float* __restrict__ y) {
  __shared__ int s_pos[kMaxK];
  __shared__ float s_w[kMaxK];
  // positions and weights come from the CSR and the router, complete two or more kernels
  // back; only the partial rows need the wait
  const int t = blockIdx.y;
  if (threadIdx.x < k) {
    s_pos[threadIdx.x] = pair_pos[(size_t)t * k + threadIdx.x];
    s_w[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  pdl_wait();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (r >= H) return;
  *reinterpret_cast<float4*>(y + (size_t)t * H + r) = combine4(partial, s_pos, s_w, k, H, r);
}

// ---------------------------------------------------------------------------
// gate/up + SiLU and down, TMA-fed warp units (decode_units.cuh)
// ---------------------------------------------------------------------------
// One CTA per SM: kTmaProd producer warps stream the units' stages with TMA into the rings
// of the kTmaWarps consumer warps (kTmaSlots stages each), and each consumer multiplies
// whole units alone (no CTA barrier, no cross-warp sum).  The CTA takes a contiguous range
// of the units (expert-major); its consumer w takes units w, w + kTmaWarps, ...

// ALPHA: the bank has per-expert second-level scales (a separate instance, so the common
// case keeps every register for the K loop).
template <int NB, bool ALPHA>
__global__ void __launch_bounds__(32 * (kTmaProd + kTmaWarps), 1)
gate_up_tma_kernel(const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_s,
                   const GuTmaArgs args) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = gu_stage_bytes(NB);
  constexpr int NSLOT = kTmaWarps * kTmaSlots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSLOT * stage_bytes);
  uint64_t* empty = full + NSLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NSLOT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrb = args.F / 8;                              // units per expert

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // the producers read only the CSR (complete two kernels back) and the weights, so they
  // start streaming before the gathered activations are ready; the consumers wait
  const int n_units = *args.n_active * nrb;
  const int u_beg = (int)((long long)blockIdx.x * n_units / gridDim.x);
  const int u_end = (int)((long long)(blockIdx.x + 1) * n_units / gridDim.x);

  constexpr int PER = kTmaWarps / kTmaProd;               // consumer warps per producer
  if (warp < kTmaProd) {
    // ---------------- TMA producers: warp p feeds consumers p*PER .. p*PER+PER-1 ----------------
    pdl_trigger();
    if (lane == 0) {
      const int w0 = warp * PER;
      GuCursor cur[PER];
      for (int i = 0; i < PER; ++i) cur[i] = GuCursor{u_beg + w0 + i, 0, 0, 0};
      bool more = true, ok = true;
      while (more && ok) {
        more = false;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          if (!ok) break;
          if (cur[i].u >= u_end) continue;
          more = true;
          ok = gu_issue(args, &tmap_c, &tmap_s, cur[i], kTmaWarps, smem, stage_bytes, full, empty,
                        Ring{(w0 + i) * kTmaSlots, 1}, abort_flag);
        }
      }
      // drain, bounded: every issued stage has landed before the CTA exits
      if (!ok)
        for (int i = 0; i < PER; ++i) ring_drain(full, Ring{(w0 + i) * kTmaSlots, 1}, cur[i].q);
    }
  } else {
    // ---------------- consumer warp ----------------
    pdl_wait();                                            // gathered activations are ready
    pdl_trigger();
    const int cw = warp - kTmaProd;
    const Ring ring{cw * kTmaSlots, 1};
    int q = 0;                                             // stages consumed
    for (int u = u_beg + cw; u < u_end && !*abort_flag; u += kTmaWarps)
      if (!gu_consume_unit<NB, ALPHA, true, true>(args, u, smem, stage_bytes, full, empty, ring, q, abort_flag))
        break;
  }
  __syncthreads();
}

// The down projection in the same organisation: a unit = (active expert, 16 output rows)
// over the whole F, one stage per group of 8 pairs.
__global__ void __launch_bounds__(32 * (kTmaProd + kTmaWarps), 1)
down_tma_kernel(const DnTmaArgs args) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = dn_stage_bytes(args.F);
  constexpr int NSLOT = kTmaWarps * kTmaSlots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSLOT * stage_bytes);
  uint64_t* empty = full + NSLOT;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NSLOT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrb = args.H / 16;                             // units per expert

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int n_units = *args.n_active * nrb;              // the CSR is complete
  const int u_beg = (int)((long long)blockIdx.x * n_units / gridDim.x);
  const int u_end = (int)((long long)(blockIdx.x + 1) * n_units / gridDim.x);
  constexpr int PER = kTmaWarps / kTmaProd;

  if (warp < kTmaProd) {
    // ---------------- producers: warp p feeds consumers p*PER .. p*PER+PER-1 ----------------
    // the weights do not depend on the previous kernel, so the copies start before its end
    if (lane == 0) {
      const int w0 = warp * PER;
      DnCursor cur[PER];
      for (int i = 0; i < PER; ++i) cur[i] = DnCursor{u_beg + w0 + i, 0, 0};
      bool more = true, ok = true;
      while (more && ok) {
        more = false;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          if (!ok) break;
          if (cur[i].u >= u_end) continue;
          more = true;
          ok = dn_issue(args, cur[i], kTmaWarps, smem, stage_bytes, full, empty,
                        Ring{(w0 + i) * kTmaSlots, 1}, abort_flag);
        }
      }
      if (!ok)
        for (int i = 0; i < PER; ++i) ring_drain(full, Ring{(w0 + i) * kTmaSlots, 1}, cur[i].q);
    }
    pdl_wait();
    pdl_trigger();
  } else {
    // ---------------- consumer warp ----------------
    pdl_wait();                                            // h in f16 is complete
    pdl_trigger();
    const int cw = warp - kTmaProd;
    const Ring ring{cw * kTmaSlots, 1};
    int q = 0;
    for (int u = u_beg + cw; u < u_end && !*abort_flag; u += kTmaWarps)
      if (!dn_consume_unit(args, u, smem, stage_bytes, full, empty, ring, q, abort_flag)) break;
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_decode_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                  const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                  char* ws, cudaStream_t s) {
  const int kmax = (H / 128 + 7) / 8;
  if (kmax > 4) return cudaErrorInvalidValue;
  const int P = T * k;
  __half* xg = reinterpret_cast<__half*>(ws + L.xg);
  int32_t* xe = reinterpret_cast<int32_t*>(ws + L.xe);
  int32_t* row_tok = reinterpret_cast<int32_t*>(ws + L.row_tok);
  const int np = H / 256;                         // 16-byte pieces per lane
  auto xk = np <= 4 ? x_gather_kernel<4> : np <= 8 ? x_gather_kernel<8>
          : np <= 12 ? x_gather_kernel<12> : x_gather_kernel<16>;
  cudaError_t st = launch_pdl(xk, dim3((T + 7) / 8), dim3(256), 0, s, x_bf16, H, k,
                              T, (const int32_t*)(ws + L.pair_pos), xg, xe, row_tok);
  if (st != cudaSuccess) return st;
  {
    // TMA-fed warp units: K-chunks of at most 2 boxes of 128 bytes per row
    const int n256 = H / 256;
    int nh = 1;
    while (n256 % nh != 0 || n256 / nh > 2) ++nh;
    const int nb = n256 / nh;
    // stages, 1 KiB of alignment slack, the barriers (16 B per slot) and the abort flag
    const size_t smem = (size_t)kTmaWarps * kTmaSlots * gu_stage_bytes(nb) + 1024 +
                        (size_t)kTmaWarps * kTmaSlots * 16 + 16;
    // the banks as [K-box][E*2 matrices][F rows][bytes of the K-box] (row pitch H/2 or H/16)
    CUtensorMap mc, ms;
    const uint64_t cdims[4] = {128, (uint64_t)F, 2 * (uint64_t)b.E, (uint64_t)n256};
    const uint64_t cstr[3] = {(uint64_t)H / 2, (uint64_t)F * (H / 2), 128};
    const uint32_t cbox[4] = {128, 8, 2, (uint32_t)nb};
    const uint64_t sdims[4] = {16, (uint64_t)F, 2 * (uint64_t)b.E, (uint64_t)n256};
    const uint64_t sstr[3] = {(uint64_t)H / 16, (uint64_t)F * (H / 16), 16};
    const uint32_t sbox[4] = {16, 8, 2, (uint32_t)nb};
    // with fewer than ~8 units per SM the warps cannot keep enough bytes in flight and the
    // CTA kernel below was faster (one token: 40 against 42 us per layer when first
    // measured; level since, 32.9 against 33.0 us)
    const long long units_bound = (long long)(P < b.E ? P : b.E) * (F / 8);
    if (units_bound >= 8LL * num_sms() && smem <= 232448 &&
        make_map4(&mc, b.codes, cdims, cstr, cbox, true) &&
        make_map4(&ms, b.scales, sdims, sstr, sbox, false)) {
      GuTmaArgs ta{xg, xe, H, F, nh, nb, csr.expert_offsets, csr.active_experts, csr.n_active,
                   reinterpret_cast<float*>(ws + L.h), reinterpret_cast<uint32_t*>(ws + L.error_word)};
      ta.alpha = b.alpha;
      ta.row_tok = row_tok;
      auto gk = b.alpha ? (nb == 1 ? gate_up_tma_kernel<1, true> : gate_up_tma_kernel<2, true>)
                        : (nb == 1 ? gate_up_tma_kernel<1, false> : gate_up_tma_kernel<2, false>);
      st = cudaFuncSetAttribute(gk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
      if (st != cudaSuccess) return st;
      const long long units = (long long)(P < b.E ? P : b.E) * (F / 8);
      // every SM streams, even when there are fewer units than consumer warps
      long long grid = num_sms();
      if (grid > units) grid = units;
      if (grid < 1) grid = 1;
      return launch_pdl(gk, dim3((unsigned)grid), dim3(32 * (kTmaProd + kTmaWarps)),
                        smem, s, mc, ms, ta);
    }
  }
  GateUpArgs a{xg, xe, b.codes, b.scales, H, F, csr.expert_offsets, csr.active_experts,
               csr.n_active, reinterpret_cast<float*>(ws + L.h)};
  a.alpha = b.alpha;
  a.row_tok = row_tok;
  const long long max_units = (long long)(P < b.E ? P : b.E) * (F / 16);
  const size_t wbytes = (32 * (size_t)(H / 2) + 32 * (size_t)(H / 16) + 127) & ~size_t(127);
  const size_t smem = 2 * wbytes + 8 * 32 * 8 * sizeof(float);
  auto kern = kmax <= 1 ? gate_up_kernel<1> : kmax == 2 ? gate_up_kernel<2>
                                             : kmax == 3 ? gate_up_kernel<3> : gate_up_kernel<4>;
  st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (st != cudaSuccess) return st;
  long long grid = 2LL * num_sms();
  if (grid > max_units) grid = max_units;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(256), smem, s, a);
}

cudaError_t launch_decode_down(const moe_nvfp4_bank& b, moe_csr csr, int T, int H, int F, int k,
                               const moe_ws_layout& L, char* ws, cudaStream_t s) {
  const int P = T * k;
  __half* hg = reinterpret_cast<__half*>(ws + L.hg);
  int32_t* he = reinterpret_cast<int32_t*>(ws + L.he);
  const int nr = (F + 127) / 128;                 // float4 per lane
  if (nr > 16) return cudaErrorInvalidValue;      // F <= 1408 on this path
  auto hk = nr <= 2 ? h_prep_kernel<2> : nr <= 5 ? h_prep_kernel<5> : nr <= 8 ? h_prep_kernel<8>
                                                                    : h_prep_kernel<16>;
  cudaError_t st = launch_pdl(hk, dim3((P + 7) / 8), dim3(256), 0, s, (const float*)(ws + L.h), F,
                              (const int32_t*)csr.expert_offsets, b.E, hg, he);
  if (st != cudaSuccess) return st;
  {
    // bulk-copy-fed warp units when there are enough of them and the rows fit the loop
    const size_t smem = (size_t)kTmaWarps * kTmaSlots * dn_stage_bytes(F) + 1024 +
                        (size_t)kTmaWarps * kTmaSlots * 16 + 16;
    const long long units = (long long)(P < b.E ? P : b.E) * (H / 16);
    if (F % 128 == 0 && units >= 8LL * num_sms() && smem <= 232448 &&
        (reinterpret_cast<uintptr_t>(b.codes) & 15) == 0 && (reinterpret_cast<uintptr_t>(b.scales) & 15) == 0) {
      DnTmaArgs ta{hg, he, b.codes, b.scales, H, F, csr.expert_offsets, csr.active_experts,
                   csr.n_active, reinterpret_cast<float*>(ws + L.partial),
                   reinterpret_cast<uint32_t*>(ws + L.error_word)};
      ta.alpha = b.alpha;
      st = cudaFuncSetAttribute(down_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (st != cudaSuccess) return st;
      long long grid = num_sms();
      if (grid > units) grid = units;
      return launch_pdl(down_tma_kernel, dim3((unsigned)grid), dim3(32 * (kTmaProd + kTmaWarps)),
                        smem, s, ta);
    }
  }
  DownArgs a{hg, he, b.codes, b.scales, H, F, csr.expert_offsets, csr.active_experts,
             csr.n_active, reinterpret_cast<float*>(ws + L.partial)};
  a.alpha = b.alpha;
  const long long max_units = (long long)(P < b.E ? P : b.E) * (H / 128);
  const size_t wbytes = (128 * (size_t)(F / 2) + 128 * (size_t)(F / 16) + 127) & ~size_t(127);
  const size_t smem = 2 * wbytes + 8 * (size_t)(F * 2 + 16);
  long long grid = 2LL * num_sms();
  if (grid > max_units) grid = max_units;
  auto kern = (F % 128 == 0) ? down_kernel<128> : down_kernel<64>;
  st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (st != cudaSuccess) return st;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(256), smem, s, a);
}

cudaError_t launch_combine(const float* w, int T, int H, int k, const moe_ws_layout& L, char* ws,
                           float* y, cudaStream_t s) {
  return launch_pdl(combine_kernel, dim3((H / 4 + 255) / 256, T), dim3(256), 0, s, w,
                    (const int32_t*)(ws + L.pair_pos), (const float*)(ws + L.partial), H, k, y);
}

}  // namespace moe
