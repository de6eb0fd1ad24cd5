// Prefill path: hundreds of pairs per expert, a dense grouped contraction on the
// block-scaled FP4 tensor cores (tcgen05.mma kind::mxf4nvf4, UE4M3 scale per 16), over the
// 128-row M-tiles (expert, first CSR row, rows) the CSR call lists.
//
//   gemm_kernel     persistent, warp-specialised grouped GEMM over (M-tile, N-tile) work:
//                   TMA (SWIZZLE_128B) feeds FP4 code tiles and row-major images of the
//                   UE4M3 scale factors, four warps write the scale factors into TMEM
//                   with tcgen05.st (with a prepacked bank, the weights' arrive as atoms
//                   that one thread copies in with tcgen05.cp), one thread issues
//                   tcgen05.mma, eight warps drain TMEM with tcgen05.ld and apply the
//                   epilogue (SiLU(g)*u -> h, or z -> f16 partials)
//   down_resident_kernel  the down GEMM with each M-tile's Q(h) held in shared memory
//                   while only the weights stream (F <= 768)
// Q(x), Q(h) and the combine live in prefill_quant.cu.
//
// Every wait on an mbarrier is bounded by a 2 s %globaltimer budget; on expiry the CTA
// sets MOE_DEVERR_TIMEOUT in the workspace error word, drains and frees its TMEM.
#include <cmath>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tma_sync.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace {

// (mbarrier and TMA wrappers: tma_sync.cuh; tcgen05 wrappers: tcgen05.cuh)

// ---------------------------------------------------------------------------
// grouped block-scaled GEMM
// ---------------------------------------------------------------------------
// GATE_UP: A = Q(x) rows [P][H]; the B tile interleaves BN/2 gate rows with the matching
//          up rows of the expert (gate row i, up row i as tile rows 2i, 2i+1: a 3-D tensor
//          map {bytes, gate/up, row}), so one N=BN MMA yields g_i and u_i in accumulator
//          columns 2i and 2i+1; out = h f32 [P][F] (BN/2 columns per tile).
// DOWN:    A = Q(h) rows [P][F], B = BN down rows; out = z * 2^-(row exponent + cF) as f16
//          [P][H] (the combine restores the scale; the bound |acc| <= F * 2688^2 keeps the
//          value below 2^15).
struct GemmArgs {
  const int32_t* a_exp;         // [P]
  const int32_t* tiles;         // n_mtiles, then int4 list
  void* out;                    // f32 [P][F] or f16 [P][H]
  uint32_t* err;
  int P, K, rows_per_expert, n_tiles_n, out_cols, F, down_shift;
  int b_sf_group;               // DOWN: g rows of the weight-scale plane per tensor-map row
  int n_base;                   // first N-tile of this launch (output columns are relative to it)
  const float* alpha = nullptr; // [E] per-expert second-level weight scale, or none
  // Works are taken in groups of `n_group` N-tiles: all M-tiles of group 0, then of group 1,
  // ...; within a group M-tiles in list order, N fastest (n_group = n_tiles_n: one group).
  int n_group = 0;
  // PACKED kernels: the weights' scale factors as 512-byte tensor-memory atoms, one per
  // (expert, 128-row tile, k-step of 64), b_tiles tiles per expert and kst k-steps per row
  const uint8_t* b_atoms = nullptr;
  int b_tiles = 0, kst = 0;
};

// M-tile index and N-tile index of work w (see GemmArgs::n_group).
__device__ __forceinline__ void work_mn(int w, int n_mtiles, int ng, int& m, int& n) {
  const int per = n_mtiles * ng;
  const int g = w / per;
  const int r = w - g * per;
  m = r / ng;
  n = g * ng + (r - m * ng);
}

// Scale factors reach shared memory through TMA, as row-major staging images beside the
// code tiles: A rows [128][16 B] (the stage's 4 k-steps x 4 scales), B rows [BN][16 B]
// (GATE_UP), or for DOWN g sub-row images [128/g][32 B] whose 16-byte windows start at
// byte (s*K/16 + 16*ks) mod 16 (the weight-scale rows are K/16 bytes, not a multiple of
// 16, so g consecutive rows form one tensor-map row).  Four warps, one per TMEM lane
// quarter, rearrange the staging images and store them into the stage's scale-factor
// columns with tcgen05.st: lane r of every quarter holds, in columns 4j..4j+3, the k-step
// j scales of rows r, r+32, r+64, r+96.  No thread waits on global memory, and the MMA
// thread issues nothing but MMAs.
template <int BN, bool GATE_UP>
struct Cfg {
  static constexpr int BM = 128;
  static constexpr int KB = 128;                    // bytes of K per stage (256 elements)
  static constexpr int G = (BN + 127) / 128;        // 128-row scale-factor atoms per B tile
  static constexpr int STAGES = GATE_UP ? 6 : 5;
  static constexpr int OUT_N = GATE_UP ? BN / 2 : BN;   // output columns per tile
  static constexpr int A_BYTES = BM * KB;
  static constexpr int B_BYTES = BN * KB;
  static constexpr int SA_STG = BM * 16;            // A scale staging
  static constexpr int SB_STG = GATE_UP ? BN * 16 : BN * 32;   // B scale staging (DOWN: 32-B windows)
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SA_STG + SB_STG;
  static constexpr int ACC_COLS = 2 * BN;           // two accumulator buffers
  static constexpr int SF_COLS = 16 + 16 * G;       // one stage's scale factors in TMEM
  // one scale-factor buffer per smem stage: a buffer is rewritten only after the stage's
  // empty barrier (committed behind the MMAs that read it) has completed
  static constexpr int TMEM_COLS_USED = ACC_COLS + STAGES * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_COLS_USED <= 256 ? 256 : 512;
  static constexpr int EPI_WARPS = 8;               // two per TMEM lane quarter
  static constexpr int THREADS = 32 * (6 + EPI_WARPS);   // TMA, MMA, 4 transposers, epilogue
  // DOWN: per epilogue warp a 4 KB staging image of its 32 x 64 f16 block of partials,
  // written to global memory by one TMA store (128-byte swizzle, 1024-byte aligned)
  static constexpr int OUT_STG = GATE_UP ? 0 : 8 * 4096;
  static constexpr int SMEM = STAGES * STAGE_BYTES + OUT_STG + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(TMEM_COLS_USED <= 512, "TMEM budget");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// PACKED: the weights' scale factors come as prepacked atoms (GemmArgs::b_atoms), one
// contiguous copy per stage beside the A staging; one thread of the first transposer warp
// moves them into TMEM with tcgen05.cp and commits the copies to the stage's full barrier,
// so the MMA thread still issues nothing but MMAs; the transposer warps handle only A's.
template <int BN, bool GATE_UP, bool PACKED>
__global__ void __launch_bounds__(448, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
            const __grid_constant__ CUtensorMap tmap_out, const GemmArgs args) {
  using C = Cfg<BN, GATE_UP>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full[s]: the stage's code tiles landed and its scale factors are in TMEM (TMA bytes +
  // one arrive per transposer warp); stg_full[s]: the scale staging images landed.
  unsigned char* out_stg = smem + C::STAGES * C::STAGE_BYTES;   // DOWN: [8 warps][4 KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stg + C::OUT_STG);
  uint64_t* stg_full = full + C::STAGES;
  uint64_t* empty = stg_full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;           // [2]
  uint64_t* acc_empty = acc_full + 2;               // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // stage layout: A codes | B codes | A scale staging | B scale staging
  constexpr int OFF_SA = C::A_BYTES + C::B_BYTES;
  constexpr int OFF_SB = OFF_SA + C::SA_STG;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_mtiles = args.tiles[0];
  const int4* tlist = reinterpret_cast<const int4*>(args.tiles + 4);
  const int n_work = n_mtiles * args.n_tiles_n;
  const int k_stages = (args.K / 2 + C::KB - 1) / C::KB;
  const int sfrow = args.K / 16;                    // scale bytes per row

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // TMA expect_tx + 4 transposer warps (+ PACKED: the commit of the atom copies)
      mbar_init(&full[s], PACKED ? 1 + 4 + 1 : 1 + 4);
      mbar_init(&stg_full[s], 1);                    // TMA expect_tx
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::EPI_WARPS);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_holder)), "n"(C::TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t acc_col = tmem;                              // accumulators at column 0
  const uint32_t sf_col0 = tmem + C::ACC_COLS;                 // per-stage scale-factor buffers

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      constexpr uint32_t tx_codes = C::A_BYTES + C::B_BYTES;
      const int g = args.b_sf_group;
      const uint32_t tx_stg =
          C::SA_STG + (PACKED ? 0u : GATE_UP ? C::SB_STG : (uint32_t)(g == 1 ? BN * 16 : BN * 32));
      const uint64_t wpol = l2_evict_first_policy();
      const int sub_rows = BN / g, sub_w = g == 1 ? 16 : 32;
      int it = 0;
      // work descriptors are fetched two works ahead (a DOWN work is only a few stages)
      const int ng = args.n_group;
      auto mtile_of = [&](int w) { int m, n; work_mn(w, n_mtiles, ng, m, n); return tlist[m]; };
      const int w1 = blockIdx.x + gridDim.x;
      int4 tile = blockIdx.x < n_work ? mtile_of(blockIdx.x) : make_int4(0, 0, 0, 0);
      int4 next = w1 < n_work ? mtile_of(w1) : tile;
      for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x) {
        const int w2 = w + 2 * gridDim.x;
        const int4 next2 = w2 < n_work ? mtile_of(w2) : next;
        int wm, wn;
        work_mn(w, n_mtiles, ng, wm, wn);
        const int n0 = wn * C::OUT_N;
        const int brow = tile.z * args.rows_per_expert + args.n_base * C::OUT_N + n0;
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait(&empty[st], ((it / C::STAGES) & 1) ^ 1, abort_flag, args.err)) break;
          unsigned char* sb = smem + st * C::STAGE_BYTES;
          const int nk = PACKED ? min(4, args.kst - 4 * ks) : 0;   // atoms of the stage
          mbar_expect_tx(&stg_full[st], tx_stg + 512u * nk);
          mbar_expect_tx(&full[st], tx_codes);
          // scale staging first: the transposers can start while the code tiles stream in
          tma_load_2d(sb + OFF_SA, &tmap_sfa, ks * 16, tile.x, &stg_full[st]);
          if (PACKED) {
            const int t = args.n_base + wn;                 // the weight tile of this work
            bulk_load(sb + OFF_SB,
                      args.b_atoms + ((size_t)(tile.z * args.b_tiles + t) * args.kst + 4 * ks) * 512,
                      512u * nk, &stg_full[st]);
          } else if (GATE_UP) {
            tma_load_3d_hint(sb + OFF_SB, &tmap_sfb, ks * 16, 0, brow, &stg_full[st], wpol);
          } else {
            for (int s2 = 0; s2 < g; ++s2) {
              const int x = ((s2 * sfrow + 16 * ks) >> 4) << 4;
              tma_load_2d(sb + OFF_SB + s2 * sub_rows * sub_w, &tmap_sfb, x, brow / g,
                          &stg_full[st]);
            }
          }
          tma_load_2d(sb, &tmap_a, ks * C::KB, tile.x, &full[st]);
          if (GATE_UP)
            tma_load_3d_hint(sb + C::A_BYTES, &tmap_b, ks * C::KB, 0, brow, &full[st], wpol);
          else
            tma_load_2d_hint(sb + C::A_BYTES, &tmap_b, ks * C::KB, brow, &full[st], wpol);
        }
        tile = next;
        next = next2;
      }
      // drain: wait (bounded) until every issued stage has landed
      if (*abort_flag) {
        for (int s = 0; s < C::STAGES; ++s) {
          if (it <= s) continue;
          const int last = s + ((it - 1 - s) / C::STAGES) * C::STAGES;   // last issue on s
          const uint64_t t0 = global_ns();
          // full also needs the transposers, which may have stopped: its wait is bounded
          while ((!mbar_try(&stg_full[s], (last / C::STAGES) & 1) ||
                  !mbar_try(&full[s], (last / C::STAGES) & 1)) &&
                 global_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = mxf4_idesc(128, BN);
      const uint32_t s0 = smem_u32(smem);
      // descriptors of stage 0; stage st adds st * STAGE_BYTES to the start address field
      const uint64_t a_desc0 = smem_desc(s0, 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(s0 + C::A_BYTES, 16, 1024, 2);
      int it = 0, tcount = 0;
      for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x, ++tcount) {
        const int ab = tcount & 1;
        if (!mbar_wait(&acc_empty[ab], ((tcount >> 1) & 1) ^ 1, abort_flag, args.err)) break;
        tc_fence_after();
        const uint32_t acc = acc_col + ab * BN;
        bool ok = true;
        int st = it % C::STAGES;
        uint32_t par = (it / C::STAGES) & 1;
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          // code tiles (TMA) and scale factors in TMEM (transposers) of the stage
          if (!mbar_wait(&full[st], par, abort_flag, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t so = (uint64_t)((st * C::STAGE_BYTES) >> 4);
          const uint32_t sfc = sf_col0 + st * C::SF_COLS;
          // k-steps past K (the zero-filled tail of the last stage) are skipped
          const int nk = min(4, (sfrow - 16 * ks) >> 2);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < nk)
              tc_mma(acc, a_desc0 + so + ((32 * j) >> 4), b_desc0 + so + ((32 * j) >> 4), idesc,
                     sfc + 4 * j, sfc + 16 + 4 * C::G * j, (ks | j) != 0);
          tc_commit(&empty[st]);
          if (++st == C::STAGES) { st = 0; par ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&acc_full[ab]);
      }
    }
  } else if (warp < 6) {
    // ---------------- scale-factor transposers (128 threads, one TMEM lane quarter each) ---
    // Lane r of warp w writes TMEM lane 32*(w%4) + r: for k-step j, columns 4j + x hold the
    // scale word of row r + 32x.  Scale bytes past the row's K/16 (the zero-filled tail of
    // the last stage) are written as 0.  PACKED: A's only.
    static_assert(C::G == 1, "one 128-row scale group per operand");
    const int n_it = ((n_work - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) * k_stages;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int g = args.b_sf_group;
    const int sub_rows = BN / g, sub_w = g == 1 ? 16 : 32;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % C::STAGES;
      const int ks = it % k_stages;
      if (!mbar_wait_warp(&stg_full[st], (it / C::STAGES) & 1, abort_flag, args.err)) break;
      tc_fence_after();
      const uint32_t sb = smem_u32(smem + st * C::STAGE_BYTES);
      const int nvalid = min(4, (sfrow - 16 * ks) >> 2);   // u32 words of this stage in a row
      if (PACKED && warp == 2 && lane == 0) {
        // the weight atoms into the stage's B columns, completing on full[st]
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nvalid) tc_cp_sf(sf_col0 + st * C::SF_COLS + 16 + 4 * j, sb + OFF_SB + 512 * j);
        tc_commit(&full[st]);
      }
      uint32_t va[16], vb[16];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int row = lane + 32 * x;
        const uint4 a4 = lds128(sb + OFF_SA + 16 * row);
        const uint32_t a[4] = {a4.x, a4.y, a4.z, a4.w};
        uint32_t b[4] = {0u, 0u, 0u, 0u};
        if (PACKED) {
        } else if (GATE_UP) {
          const uint4 b4 = lds128(sb + OFF_SB + 16 * row);
          b[0] = b4.x; b[1] = b4.y; b[2] = b4.z; b[3] = b4.w;
        } else {
          const int bs = row % g, bi = row / g;
          const int byte0 = bs * sfrow + 16 * ks;
          const uint32_t src = sb + OFF_SB + bs * sub_rows * sub_w + bi * sub_w + (byte0 & 15);
#pragma unroll
          for (int j = 0; j < 4; ++j) b[j] = j < nvalid ? lds32(src + 4 * j) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          va[4 * j + x] = j < nvalid ? a[j] : 0u;
          vb[4 * j + x] = b[j];
        }
      }
      const uint32_t sfc = sf_col0 + st * C::SF_COLS + lane_base;
      tc_st16(sfc, va);
      if (!PACKED) tc_st16(sfc + 16, vb);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
    }
  } else {
    // ---------------- epilogue (warps 6..13: lane quarter warp % 4, column half) ----------
    static_assert(C::THREADS == 448 && C::EPI_WARPS == 8, "epilogue warp map");
    const int quarter = warp & 3;
    const int half = (warp - 6) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    int tcount = 0;
    for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x, ++tcount) {
      const int ab = tcount & 1;
      int wm, wn;
      work_mn(w, n_mtiles, args.n_group, wm, wn);
      const int4 tile = tlist[wm];
      const int n0 = wn * C::OUT_N;
      const bool valid = row < tile.y;
      const int pos = tile.x + row;
      const int sx = GATE_UP ? (valid ? args.a_exp[pos] : 0) : -args.down_shift;
      // x * 2^sx is one exact-power-of-two multiply when 2^sx is a float, else ldexpf
      const bool fast = sx >= -149 && sx <= 127;
      const float m = fast ? pow2f(sx) : 0.0f;
      const float al = args.alpha ? __ldg(args.alpha + tile.z) : 1.0f;
      if (!mbar_wait_warp(&acc_full[ab], (tcount >> 1) & 1, abort_flag, args.err)) break;
      tc_fence_after();
      const uint32_t acc = acc_col + ab * BN + lane_base;
      if (GATE_UP) {
        // this warp: accumulator columns [64*half, +64) = (g_i, u_i) of h columns
        // [32*half, +32)
        float* orow = reinterpret_cast<float*>(args.out) + (size_t)(valid ? pos : 0) * args.out_cols + n0;
        static_assert(BN / 64 == 2, "one 32-column chunk of h per epilogue warp");
        float gu[2][32];
        tc_ld32x2(acc + half * 64, acc + half * 64 + 32, gu[0], gu[1]);
        // the values are in registers: hand the accumulator buffer back to the MMA thread
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float* v = gu[(i + q) >> 4] + 2 * ((i + q) & 15);
              const float gg = al * (fast ? v[0] * m : ldexpf(v[0], sx));
              const float uu = al * (fast ? v[1] * m : ldexpf(v[1], sx));
              o[q] = silu_f(gg) * uu;
            }
            *reinterpret_cast<float4*>(orow + half * 32 + i) = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      } else {
        // this warp: accumulator columns [64*half, +64) -> f16 partials
        __half* orow = reinterpret_cast<__half*>(args.out) + (size_t)(valid ? pos : 0) * args.out_cols + n0;
        static_assert(BN / 32 == 4, "two 32-column chunks per epilogue warp");
        float v[2][32];
        tc_ld32x2(acc + half * 64, acc + half * 64 + 32, v[0], v[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
        uint4 pk[8];                                   // the row's 64 values as f16, 8 x 16 B
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint32_t q4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float a0 = al * (fast ? v[c][i + 2 * q] * m : ldexpf(v[c][i + 2 * q], sx));
              const float a1 = al * (fast ? v[c][i + 2 * q + 1] * m : ldexpf(v[c][i + 2 * q + 1], sx));
              const __half2 h2 = __floats2half2_rn(a0, a1);
              q4[q] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            pk[c * 4 + i / 8] = make_uint4(q4[0], q4[1], q4[2], q4[3]);
          }
        // A warp whose 32 rows are all valid stores them through shared memory with one TMA
        // store, which keeps these 4 KB off the load/store path the transposer warps need; the
        // rows of a ragged last M-tile that end inside this warp's quarter are stored directly
        // (a 32-row box would reach into the next expert's rows).
        if (tile.y - quarter * 32 >= 32) {
          unsigned char* stg = out_stg + (warp - 6) * 4096;
          const uint32_t sa = smem_u32(stg);
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t adr = sa + lane * 128 + ((c ^ (lane & 7)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(adr), "r"(pk[c].x),
                         "r"(pk[c].y), "r"(pk[c].z), "r"(pk[c].w) : "memory");
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            const int x = (n0 + half * 64) * 2;                     // bytes
            const int y = tile.x + quarter * 32;
            asm volatile(
                "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                ::"l"(&tmap_out), "r"(x), "r"(y), "r"(sa) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        } else if (valid) {
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(orow + half * 64 + c * 8) = pk[c];
        }
      }
    }
    // every TMA store of the partials has finished reading shared memory
    if (!GATE_UP && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(C::TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// down GEMM with the activation tile resident (K = F <= 256 * KS)
// ---------------------------------------------------------------------------
// Work comes in chunks: one M-tile (128 CSR rows of Q(h)) x up to kChunkN consecutive
// N-tiles of 128 down rows.  The chunk's A tile (KS k-stages of 128 B codes per row, with
// their scale staging) is loaded once and its scale factors go to TMEM once; only the
// weights then stream, through a ring of B stages (codes + scale staging, 20 KiB), so
// more weight bytes are in flight per SM than with A re-read every stage.  A, its scale
// staging and its TMEM scale factors are double-buffered: chunk i uses buffer i % 2, and
// the producer loads chunk i+1's A right after chunk i's first N-tile of weights, a whole
// chunk before the MMAs need it (an A tile takes about 2 us to land even from L2 while the
// weights stream).  The epilogue stages its partials in 2 KiB per warp (two 32-column TMA
// stores, 64-byte swizzle), which leaves room for five B stages.  Warp roles and outputs
// are those of gemm_kernel<128, false>; with prepacked weight atoms (PACKED) the B stages
// need no transposer work: one thread copies each stage's atoms into TMEM with
// tcgen05.cp and commits the copies to the stage's full barrier.
constexpr int kChunkN = 4;
constexpr int kResidentKS = 3;                      // k-stages of A held (F <= 768)

struct DCfg {
  static constexpr int KS = kResidentKS;
  static constexpr int BN = 128;
  static constexpr int KB = 128;                    // bytes of K per k-stage (256 elements)
  static constexpr int A_CODES = 128 * KB;          // per k-stage
  static constexpr int A_SA = 128 * 16;             // per k-stage: scale staging [128][16 B]
  static constexpr int A_BUF = KS * A_CODES;        // one A buffer's codes
  static constexpr int SA_BUF = KS * A_SA;          // one A buffer's scale staging
  static constexpr int A_BYTES = 2 * (A_BUF + SA_BUF);
  static constexpr int B_CODES = BN * KB;
  static constexpr int B_SB = BN * 32;              // 32-byte windows of g-grouped scale rows
  static constexpr int STAGE_BYTES = B_CODES + B_SB;
  static constexpr int OUT_STG = 8 * 2048;          // per epilogue warp: 32 rows x 32 f16
  static constexpr int STAGES = (232448 - 1024 - 512 - OUT_STG - A_BYTES) / STAGE_BYTES;
  static constexpr int ACC_COLS = 2 * BN;
  static constexpr int SFA_COLS = KS * 16;          // 4 columns per k-step, per buffer
  static constexpr int SFB_COLS = 16;               // per stage
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 32 * (6 + EPI_WARPS);
  static constexpr int SMEM = A_BYTES + STAGES * STAGE_BYTES + OUT_STG + 512 + 1024;
  static_assert(STAGES >= 5, "B ring depth");
  static_assert(ACC_COLS + 2 * SFA_COLS + STAGES * SFB_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(A_BUF % 1024 == 0 && (2 * A_BUF + 2 * SA_BUF) % 1024 == 0 &&
                STAGE_BYTES % 1024 == 0, "alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// chunk c -> M-tile and its N-tile range [n_lo, n_hi)
__device__ __forceinline__ void chunk_range(int c, int nr, int n_tiles_n, int& m, int& n_lo,
                                            int& n_hi) {
  m = c / nr;
  n_lo = (c - m * nr) * kChunkN;
  n_hi = min(n_tiles_n, n_lo + kChunkN);
}

template <bool PACKED>
__global__ void __launch_bounds__(448, 1)
down_resident_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_sfa,
                     const __grid_constant__ CUtensorMap tmap_sfb,
                     const __grid_constant__ CUtensorMap tmap_out, const GemmArgs args) {
  using C = DCfg;
  constexpr int BN = C::BN, KS = C::KS;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // layout: A codes [2][KS][16 KiB] | A scale staging [2][KS][2 KiB] | B ring | epilogue staging
  unsigned char* a_codes = smem;
  unsigned char* a_sa = smem + 2 * C::A_BUF;
  unsigned char* bring = smem + C::A_BYTES;
  unsigned char* out_stg = bring + C::STAGES * C::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stg + C::OUT_STG);   // B codes + B SF in TMEM
  uint64_t* stg_full = full + C::STAGES;            // B scale staging landed
  uint64_t* empty = stg_full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;           // [2]
  uint64_t* acc_empty = acc_full + 2;               // [2]
  uint64_t* a_full = acc_empty + 2;                 // [2] A codes of buffer b landed
  uint64_t* a_stg = a_full + 2;                     // [2] A scale staging of buffer b landed
  uint64_t* a_sf = a_stg + 2;                       // [2] A scale factors of buffer b in TMEM
  uint64_t* a_empty = a_sf + 2;                     // [2] the MMAs reading buffer b are done
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(a_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  static_assert((3 * C::STAGES + 12) * 8 + 8 <= 512, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_mtiles = args.tiles[0];
  const int4* tlist = reinterpret_cast<const int4*>(args.tiles + 4);
  const int nr = (args.n_tiles_n + kChunkN - 1) / kChunkN;
  const int n_chunk = n_mtiles * nr;
  const int k_stages = (args.K / 2 + C::KB - 1) / C::KB;   // <= KS (checked by the host)
  const int sfrow = args.K / 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // the stage's codes (TMA bytes) and its weight scale factors in TMEM: PACKED, the
      // commit of the atom copies; otherwise one arrive per transposer warp
      mbar_init(&full[s], PACKED ? 1 + 1 : 1 + 4);
      mbar_init(&stg_full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::EPI_WARPS);
      mbar_init(&a_full[b], 1);                      // TMA expect_tx
      mbar_init(&a_stg[b], 1);                       // TMA expect_tx
      mbar_init(&a_sf[b], 4);                        // 4 transposer warps
      mbar_init(&a_empty[b], 1);                     // MMA commit
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_holder)), "n"(C::TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t acc_col = tmem;
  const uint32_t sfa_col0 = tmem + C::ACC_COLS;                // A scale factors, 2 buffers
  const uint32_t sfb_col0 = sfa_col0 + 2 * C::SFA_COLS;        // per-stage B scale factors

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int g = args.b_sf_group;
      const int sub_rows = BN / g, sub_w = g == 1 ? 16 : 32;
      const uint32_t tx_sb = (uint32_t)(g == 1 ? BN * 16 : BN * 32);
      const uint64_t wpol = l2_evict_first_policy();
      int it = 0, ca = 0;                          // B stage sequence, chunk sequence
      int a_cnt = 0;                               // A tiles issued
      bool ok = true;
      // A of the chunk with sequence number q (chunk blockIdx.x + q * gridDim.x) into buffer
      // q % 2, once the MMAs of chunk q - 2 (its last reader) are done
      auto load_a = [&](int q) -> bool {
        const int c = blockIdx.x + q * gridDim.x;
        if (c >= n_chunk) return true;
        int m, n_lo, n_hi;
        chunk_range(c, nr, args.n_tiles_n, m, n_lo, n_hi);
        const int4 tile = tlist[m];
        const int b = q & 1;
        if (!mbar_wait(&a_empty[b], ((q >> 1) & 1) ^ 1, abort_flag, args.err)) return false;
        mbar_expect_tx(&a_stg[b], (uint32_t)(k_stages * C::A_SA));
        for (int ks = 0; ks < k_stages; ++ks)
          tma_load_2d(a_sa + b * C::SA_BUF + ks * C::A_SA, &tmap_sfa, ks * 16, tile.x, &a_stg[b]);
        mbar_expect_tx(&a_full[b], (uint32_t)(k_stages * C::A_CODES));
        for (int ks = 0; ks < k_stages; ++ks)
          tma_load_2d(a_codes + b * C::A_BUF + ks * C::A_CODES, &tmap_a, ks * C::KB, tile.x,
                      &a_full[b]);
        ++a_cnt;
        return true;
      };
      ok = load_a(0);
      for (int c = blockIdx.x; c < n_chunk && ok && !*abort_flag; c += gridDim.x, ++ca) {
        int m, n_lo, n_hi;
        chunk_range(c, nr, args.n_tiles_n, m, n_lo, n_hi);
        const int4 tile = tlist[m];
        for (int n = n_lo; n < n_hi && ok; ++n) {
          const int brow = tile.z * args.rows_per_expert + n * BN;
          for (int ks = 0; ks < k_stages; ++ks, ++it) {
            const int st = it % C::STAGES;
            if (!mbar_wait(&empty[st], ((it / C::STAGES) & 1) ^ 1, abort_flag, args.err)) {
              ok = false;
              break;
            }
            unsigned char* sb = bring + st * C::STAGE_BYTES;
            if (PACKED) {
              // the stage's k-steps of atoms: one contiguous copy, on the staging barrier
              const int nk = min(4, args.kst - 4 * ks);
              mbar_expect_tx(&stg_full[st], (uint32_t)(512 * nk));
              mbar_expect_tx(&full[st], (uint32_t)C::B_CODES);
              bulk_load(sb + C::B_CODES,
                        args.b_atoms + ((size_t)(tile.z * args.b_tiles + n) * args.kst + 4 * ks) * 512,
                        512u * nk, &stg_full[st]);
            } else {
              mbar_expect_tx(&stg_full[st], tx_sb);
              mbar_expect_tx(&full[st], C::B_CODES);
              for (int s2 = 0; s2 < g; ++s2) {
                const int x = ((s2 * sfrow + 16 * ks) >> 4) << 4;
                tma_load_2d(sb + C::B_CODES + s2 * sub_rows * sub_w, &tmap_sfb, x, brow / g,
                            &stg_full[st]);
              }
            }
            tma_load_2d_hint(sb, &tmap_b, ks * C::KB, brow, &full[st], wpol);
          }
          // the next chunk's A, after this chunk's first N-tile of weights
          if (n == n_lo && ok) ok = load_a(ca + 1);
        }
      }
      // drain: wait (bounded) until every issued copy has landed
      if (!ok || *abort_flag) {
        const uint64_t t0 = global_ns();
        for (int s = 0; s < C::STAGES; ++s) {
          if (it <= s) continue;
          const int last = s + ((it - 1 - s) / C::STAGES) * C::STAGES;
          while ((!mbar_try(&stg_full[s], (last / C::STAGES) & 1) ||
                  !mbar_try(&full[s], (last / C::STAGES) & 1)) &&
                 global_ns() - t0 < 100000000ull) {
          }
        }
        for (int q = a_cnt - 2; q < a_cnt; ++q) {
          if (q < 0) continue;
          const uint32_t par = (q >> 1) & 1;
          while ((!mbar_try(&a_stg[q & 1], par) || !mbar_try(&a_full[q & 1], par)) &&
                 global_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = mxf4_idesc(128, BN);
      const uint64_t a_desc0 = smem_desc(smem_u32(a_codes), 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(smem_u32(bring), 16, 1024, 2);
      int it = 0, tcount = 0, ca = 0;
      bool ok = true;
      for (int c = blockIdx.x; c < n_chunk && ok && !*abort_flag; c += gridDim.x, ++ca) {
        int m, n_lo, n_hi;
        chunk_range(c, nr, args.n_tiles_n, m, n_lo, n_hi);
        const int b = ca & 1;
        const uint32_t par = (ca >> 1) & 1;
        // the chunk's A codes landed and its scale factors are in TMEM (buffer b)
        if (!mbar_wait(&a_sf[b], par, abort_flag, args.err) ||
            !mbar_wait(&a_full[b], par, abort_flag, args.err))
          break;
        tc_fence_after();
        const uint32_t sfa_col = sfa_col0 + b * C::SFA_COLS;
        const uint64_t a_base = a_desc0 + (uint64_t)((b * C::A_BUF) >> 4);
        for (int n = n_lo; n < n_hi && ok; ++n, ++tcount) {
          const int ab = tcount & 1;
          if (!mbar_wait(&acc_empty[ab], ((tcount >> 1) & 1) ^ 1, abort_flag, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acc = acc_col + ab * BN;
          for (int ks = 0; ks < k_stages; ++ks, ++it) {
            const int st = it % C::STAGES;
            if (!mbar_wait(&full[st], (it / C::STAGES) & 1, abort_flag, args.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ao = (uint64_t)((ks * C::A_CODES) >> 4);
            const uint64_t bo = (uint64_t)((st * C::STAGE_BYTES) >> 4);
            const uint32_t sfb = sfb_col0 + st * C::SFB_COLS;
            const int nk = min(4, (sfrow - 16 * ks) >> 2);   // k-steps past K are skipped
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j < nk)
                tc_mma(acc, a_base + ao + ((32 * j) >> 4), b_desc0 + bo + ((32 * j) >> 4), idesc,
                       sfa_col + 16 * ks + 4 * j, sfb + 4 * j, (ks | j) != 0);
            tc_commit(&empty[st]);
          }
          if (!ok) break;
          tc_commit(&acc_full[ab]);
        }
        // buffer b (codes, staging, TMEM scale factors) may be refilled once these are done
        tc_commit(&a_empty[b]);
      }
    }
  } else if (warp < 6) {
    // ---------------- scale-factor transposers (128 threads, one TMEM lane quarter each) ---
    // The weight scale factors of every B stage, as in gemm_kernel; and the A scale factors
    // of each chunk once, into TMEM buffer q % 2 (lane r of every quarter holds, in columns
    // 16 ks + 4 j + x, the k-step (ks, j) scales of row r + 32 x), in the producer's order:
    // chunk 0's first, chunk q+1's after chunk q's first N-tile of weights.  A chunk's
    // staging lands only after the MMAs that read that buffer before are done.
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int g = args.b_sf_group;
    const int sub_rows = BN / g, sub_w = g == 1 ? 16 : 32;
    auto write_sfa = [&](int q) -> bool {
      const int c = blockIdx.x + q * gridDim.x;
      if (c >= n_chunk) return true;
      const int b = q & 1;
      if (!mbar_wait_warp(&a_stg[b], (q >> 1) & 1, abort_flag, args.err)) return false;
      tc_fence_after();
      for (int ks = 0; ks < KS; ++ks) {
        const int nvalid = ks < k_stages ? min(4, (sfrow - 16 * ks) >> 2) : 0;
        uint32_t va[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint4 a4 = ks < k_stages
                               ? lds128(smem_u32(a_sa + b * C::SA_BUF + ks * C::A_SA) + 16 * (lane + 32 * x))
                               : make_uint4(0, 0, 0, 0);
          const uint32_t a[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) va[4 * j + x] = j < nvalid ? a[j] : 0u;
        }
        tc_st16(sfa_col0 + b * C::SFA_COLS + 16 * ks + lane_base, va);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_sf[b]);
      return true;
    };
    bool ok = write_sfa(0);
    int it = 0, ca = 0;
    // PACKED: one thread of warp 2 copies each stage's weight atoms into TMEM (tcgen05.cp,
    // committed to the stage's full barrier); warps 3-5 arrive on no stage barrier, so they
    // wait on none (a parity wait more than one phase behind would not return) and only
    // write each chunk's A scale factors, in chunk order
    if (PACKED && warp != 2)
      for (int q = 1; ok && blockIdx.x + q * gridDim.x < n_chunk; ++q) ok = write_sfa(q);
    for (int c = blockIdx.x; c < n_chunk && ok && (!PACKED || warp == 2); c += gridDim.x, ++ca) {
      int m, n_lo, n_hi;
      chunk_range(c, nr, args.n_tiles_n, m, n_lo, n_hi);
      for (int n = n_lo; n < n_hi && ok; ++n) {
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait_warp(&stg_full[st], (it / C::STAGES) & 1, abort_flag, args.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = smem_u32(bring + st * C::STAGE_BYTES + C::B_CODES);
          const int nvalid = min(4, (sfrow - 16 * ks) >> 2);
          if (PACKED) {
            if (lane == 0) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (j < nvalid) tc_cp_sf(sfb_col0 + st * C::SFB_COLS + 4 * j, sb + 512 * j);
              tc_commit(&full[st]);
            }
            __syncwarp();
            continue;
          }
          uint32_t vb[16];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int row = lane + 32 * x;
            const int bs = row % g, bi = row / g;
            const int byte0 = bs * sfrow + 16 * ks;
            const uint32_t src = sb + bs * sub_rows * sub_w + bi * sub_w + (byte0 & 15);
#pragma unroll
            for (int j = 0; j < 4; ++j) vb[4 * j + x] = j < nvalid ? lds32(src + 4 * j) : 0u;
          }
          tc_st16(sfb_col0 + st * C::SFB_COLS + lane_base, vb);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[st]);
        }
        if (n == n_lo && ok) ok = write_sfa(ca + 1);
      }
    }
  } else {
    // ---------------- epilogue (warps 6..13: lane quarter warp % 4, column half) ----------
    const int quarter = warp & 3;
    const int half = (warp - 6) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int sx = -args.down_shift;
    const bool fast = sx >= -149 && sx <= 127;
    const float mul = fast ? pow2f(sx) : 0.0f;
    int tcount = 0;
    bool ok = true;
    for (int c = blockIdx.x; c < n_chunk && ok; c += gridDim.x) {
      int m, n_lo, n_hi;
      chunk_range(c, nr, args.n_tiles_n, m, n_lo, n_hi);
      const int4 tile = tlist[m];
      const bool valid = row < tile.y;
      const int pos = tile.x + row;
      const float al = args.alpha ? __ldg(args.alpha + tile.z) : 1.0f;
      for (int n = n_lo; n < n_hi; ++n, ++tcount) {
        const int ab = tcount & 1;
        const int n0 = n * BN;
        if (!mbar_wait_warp(&acc_full[ab], (tcount >> 1) & 1, abort_flag, args.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = acc_col + ab * BN + lane_base;
        __half* orow = reinterpret_cast<__half*>(args.out) + (size_t)(valid ? pos : 0) * args.out_cols + n0;
        float v[2][32];
        tc_ld32x2(acc + half * 64, acc + half * 64 + 32, v[0], v[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ab]);
        uint4 pk[8];                                   // the row's 64 values as f16, 8 x 16 B
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint32_t q4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float a0 = al * (fast ? v[cc][i + 2 * q] * mul : ldexpf(v[cc][i + 2 * q], sx));
              const float a1 = al * (fast ? v[cc][i + 2 * q + 1] * mul : ldexpf(v[cc][i + 2 * q + 1], sx));
              const __half2 h2 = __floats2half2_rn(a0, a1);
              q4[q] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            pk[cc * 4 + i / 8] = make_uint4(q4[0], q4[1], q4[2], q4[3]);
          }
        // full 32-row quarters through shared memory, 32 columns at a time (one TMA store
        // each; 64-byte swizzle: 16-byte chunk c of row r at r*64 + 16*(c ^ ((r >> 1) & 3)),
        // conflict-free); the rows of a ragged last M-tile that end inside this quarter
        // directly (a box would reach the next expert's rows)
        if (tile.y - quarter * 32 >= 32) {
          const uint32_t sa = smem_u32(out_stg + (warp - 6) * 2048);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const uint4 v4 = pk[hh * 4 + cc];
              const uint32_t adr = sa + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4);
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(adr), "r"(v4.x),
                           "r"(v4.y), "r"(v4.z), "r"(v4.w) : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              const int x = (n0 + half * 64 + hh * 32) * 2;
              const int y = tile.x + quarter * 32;
              asm volatile(
                  "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                  ::"l"(&tmap_out), "r"(x), "r"(y), "r"(sa) : "memory");
              asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
          }
        } else if (valid) {
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4*>(orow + half * 64 + cc * 8) = pk[cc];
        }
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(C::TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
template <int BN, bool GATE_UP>
cudaError_t run_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa,
                     const CUtensorMap& msb, const CUtensorMap& mo, const GemmArgs& a, int max_tiles,
                     cudaStream_t s) {
  using C = Cfg<BN, GATE_UP>;
  auto kern = a.b_atoms ? gemm_kernel<BN, GATE_UP, true> : gemm_kernel<BN, GATE_UP, false>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (st != cudaSuccess) return st;
  int grid = max_tiles * a.n_tiles_n;
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  kern<<<grid, C::THREADS, C::SMEM, s>>>(ma, mb, msa, msb, mo, a);
  return cudaGetLastError();
}

cudaError_t run_down_resident(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa,
                              const CUtensorMap& msb, const CUtensorMap& mo, const GemmArgs& a,
                              int max_tiles, cudaStream_t s) {
  using C = DCfg;
  auto kern = a.b_atoms ? down_resident_kernel<true> : down_resident_kernel<false>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (st != cudaSuccess) return st;
  int grid = max_tiles * ((a.n_tiles_n + kChunkN - 1) / kChunkN);
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  kern<<<grid, C::THREADS, C::SMEM, s>>>(ma, mb, msa, msb, mo, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                   const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                   char* ws, cudaStream_t s, bool* unsupported) {
  *unsupported = false;
  if (H % 256 != 0 || F % 64 != 0) { *unsupported = true; return cudaSuccess; }
  const int P = T * k;
  // the 128-row M-tile list was written by the CSR call
  int32_t* tiles = reinterpret_cast<int32_t*>(ws + L.tiles);
  uint8_t* qc = reinterpret_cast<uint8_t*>(ws + L.qx_codes);
  uint8_t* qs = reinterpret_cast<uint8_t*>(ws + L.qx_scales);
  int32_t* qe = reinterpret_cast<int32_t*>(ws + L.qx_exp);
  cudaError_t st = launch_quant_x(x_bf16, T, H, k,
                                  reinterpret_cast<const int32_t*>(ws + L.pair_pos), qc, qs, qe, s);
  if (st != cudaSuccess) return st;
  CUtensorMap ma, mb, msa, msb;
  constexpr int BN = 128;                           // 64 gate rows interleaved with 64 up rows
  // weights: [K bytes][gate, up][row], so the box {128 B, 2, 64} lands gate row i and up row i
  // as shared-memory rows 2i and 2i+1 (and the scale box {16 B, 2, 64} their staging rows);
  // the row extent stops F rows short of the bank so the up coordinate (row + F) stays inside
  const uint64_t wrows = (uint64_t)b.E * 2 * F - F;
  const uint64_t cdims[3] = {(uint64_t)H / 2, 2, wrows};
  const uint64_t cstr[2] = {(uint64_t)F * (H / 2), (uint64_t)H / 2};
  const uint32_t cbox[3] = {128, 2, BN / 2};
  const uint64_t sdims[3] = {(uint64_t)H / 16, 2, wrows};
  const uint64_t sstr[2] = {(uint64_t)F * (H / 16), (uint64_t)H / 16};
  const uint32_t sbox[3] = {16, 2, BN / 2};
  if (!make_map(&ma, qc, H / 2, H / 2, P, 128, 128, true) ||
      !make_map3(&mb, b.codes, cdims, cstr, cbox, true) ||
      !make_map(&msa, qs, H / 16, H / 16, P, 16, 128, false) ||
      !make_map3(&msb, b.scales, sdims, sstr, sbox, false))
    return cudaErrorInvalidValue;
  GemmArgs a{qe, tiles, ws + L.h, reinterpret_cast<uint32_t*>(ws + L.error_word),
             P, H, 2 * F, F / (BN / 2), F, F, 0, 1, 0};
  a.alpha = b.alpha;
  if (b.sf_atoms) {
    a.b_atoms = b.sf_atoms;
    a.b_tiles = F / 64;
    a.kst = H / 64;
  }
  a.n_group = a.n_tiles_n;                          // one group: M-tiles in order, N fastest
  const int max_tiles = P / 128 + (P < b.E ? P : b.E) + 1;
  return run_gemm<BN, true>(ma, mb, msa, msb, ma /* unused */, a, max_tiles, s);
}

cudaError_t launch_prefill_down(const moe_nvfp4_bank& b, moe_csr csr, const float* w, int T, int H,
                                int F, int k, const moe_ws_layout& L, char* ws, float* y,
                                cudaStream_t s, bool* unsupported) {
  *unsupported = false;
  if (H % 256 != 0 || F % 64 != 0) { *unsupported = true; return cudaSuccess; }
  const int P = T * k;
  uint8_t* qc = reinterpret_cast<uint8_t*>(ws + L.qh_codes);
  uint8_t* qs = reinterpret_cast<uint8_t*>(ws + L.qh_scales);
  int32_t* qe = reinterpret_cast<int32_t*>(ws + L.qh_exp);
  const int sfh = qh_scale_pitch(F);
  if ((F / 16 + 31) / 32 > 8) { *unsupported = true; return cudaSuccess; }
  cudaError_t st = launch_quant_h(reinterpret_cast<const float*>(ws + L.h), P, F, sfh,
                                  csr.expert_offsets, b.E, qc, qs, qe, s);
  if (st != cudaSuccess) return st;
  constexpr int BN = 128;
  // the weight-scale rows are F/16 bytes; g of them make a row pitch that is a multiple of 16
  const int sfrow = F / 16;
  int g = 1;
  if (sfrow % 16 != 0)
    for (g = 2; (g * sfrow) % 16 != 0 || g * sfrow < 32; g *= 2) {
    }
  const uint64_t wrows = (uint64_t)b.E * H;
  CUtensorMap ma, mb, msa, msb;
  if (!make_map(&ma, qc, F / 2, F / 2, P, 128, 128, true) ||
      !make_map(&mb, b.codes, F / 2, F / 2, wrows, 128, BN, true) ||
      !make_map(&msa, qs, sfh, sfh, P, 16, 128, false) ||
      !make_map(&msb, b.scales, (uint64_t)g * sfrow, (uint64_t)g * sfrow, wrows / g,
                g == 1 ? 16 : 32, BN / g, false))
    return cudaErrorInvalidValue;
  const int shift = down_shift_for(F);
  const int max_tiles = P / 128 + (P < b.E ? P : b.E) + 1;
  GemmArgs a{qe, reinterpret_cast<const int32_t*>(ws + L.tiles), ws + L.partial,
             reinterpret_cast<uint32_t*>(ws + L.error_word), P, F, H, H / BN, H, F, shift, g, 0};
  a.alpha = b.alpha;
  if (b.sf_atoms) {
    a.b_atoms = b.sf_atoms;
    a.b_tiles = H / 128;
    a.kst = F / 64;
  }
  a.n_group = a.n_tiles_n;                          // one group: M-tiles in order, N fastest
  // the f16 partials [P][H]: box {64 columns, 32 rows}, 128-byte swizzle
  CUtensorMap mo;
  if (!make_map(&mo, ws + L.partial, (uint64_t)H * 2, (uint64_t)H * 2, P, 128, 32, true))
    return cudaErrorInvalidValue;
  // K = F of up to kResidentKS k-stages (F <= 768): the Q(h) tile stays resident and only
  // the weights stream; beyond that the general kernel re-reads both operands per stage
  if ((F / 2 + 127) / 128 <= kResidentKS) {
    // its epilogue stores 32 columns per box: {64 bytes, 32 rows}, 64-byte swizzle
    CUtensorMap mo32;
    if (!make_map(&mo32, ws + L.partial, (uint64_t)H * 2, (uint64_t)H * 2, P, 64, 32,
                  CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    st = run_down_resident(ma, mb, msa, msb, mo32, a, max_tiles, s);
  } else
    st = run_gemm<BN, false>(ma, mb, msa, msb, mo, a, max_tiles, s);
  if (st != cudaSuccess) return st;
  return launch_prefill_combine(w, T, H, F, k, 0, H, L, ws, y, s);
}

}  // namespace moe
