// Decode path: the grouped FP4 GEMMs with the operands the other way round.
//
// A decode layer has a few pairs per expert, so the weights are the big operand.  Each pair's
// activation row v (bf16 x, or f32 h) is written as kDecodeSlices NVFP4 rows (slices,
// prefill_quant.cu): slice i quantises what slices 0..i-1 left over, so their sum is v to
// about 6^-4 of each 16-block's largest magnitude.  The block-scaled tensor core then
// multiplies
//
//   A = 128 weight rows of one expert (M = 128, K-major, SWIZZLE_128B)
//   B = up to 32 slice rows of that expert = 8 pairs x 4 slices (N = 32)
//
// so the weights stream through TMA into shared memory and the tensor core with no
// conversion work in the SMs, and the accumulator row of weight row r holds, in its 32
// columns, the products with every slice: the epilogue sums each pair's 4 columns (each
// scaled by its slice's power of two) in one thread.
//
//   gate/up: the A tile interleaves gate row i and up row i (a 3-D tensor map {128 bytes,
//            gate/up, row}), so they land in TMEM lanes 2i and 2i+1 and one shuffle pairs
//            them for h = silu(g) * u (f32, CSR order).
//   down:    A = 128 down rows; each lane writes its output column of the pair's f32
//            partial row.
//
// Warp roles as in the prefill GEMM: warp 0 issues TMA (codes and scale staging images),
// warp 1's one thread issues tcgen05.mma (kind::mxf4nvf4, scale_vec::4X), warps 2-5 move
// the scale factors into TMEM with tcgen05.st, warps 6-9 (one per TMEM lane quarter) drain
// the double-buffered accumulator.  With a prepacked bank (PACKED) the weights' scale
// factors arrive as atoms, one contiguous copy per stage beside the slice staging; one
// thread of warp 2 moves them into TMEM with tcgen05.cp and commits the copies to the
// stage's full barrier; warps 2-5 then transpose only the slices'.  Every mbarrier wait is bounded by a 2 s %globaltimer
// budget; on expiry the CTA sets MOE_DEVERR_TIMEOUT, drains its copies and frees its TMEM.
#include <cmath>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tma_sync.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr int kSliceTile = kSliceTileRows;         // B rows per tile: 8 pairs x 4 slices

// A stage carries KSUB x 128 bytes of K per row as 128-byte-wide sub-tiles, so the MMA
// thread's per-stage costs (barrier wait, commit) are paid once per 4*KSUB MMAs: two
// sub-tiles for gate/up (K = H), three for down, whose F/2-byte rows (320 at F = 640) then
// fit one stage per work.
template <bool GATE_UP>
struct SCfg {
  static constexpr int NB = kSliceTile;           // MMA N
  static constexpr int KB = 128;                  // bytes of K per sub-tile (256 elements)
  static constexpr int KSUB = GATE_UP ? 2 : 3;    // sub-tiles per stage
  static constexpr int KSTEPS = 4 * KSUB;         // k-steps of 64 per stage
  static constexpr int A_SUB = 128 * KB;          // weight rows
  static constexpr int B_SUB = NB * KB;           // slice rows
  static constexpr int A_BYTES = KSUB * A_SUB;
  static constexpr int B_BYTES = KSUB * B_SUB;
  // weight-scale staging: gate/up [128][32 B] (the stage's window of each row); down: the
  // whole F/16-byte scale rows of the 128 rows (g consecutive rows form one tensor-map row
  // whose pitch is a multiple of 16), 128 * F/16 <= 11264 bytes for F <= 1408
  static constexpr int SA_STG = GATE_UP ? 128 * 16 * KSUB : 11264;
  static constexpr int SB_STG = NB * 16 * KSUB;   // slice-scale staging [NB][16*KSUB B]
  static constexpr int STAGE_BYTES = (A_BYTES + B_BYTES + SA_STG + SB_STG + 1023) / 1024 * 1024;
  static constexpr int STAGES = GATE_UP ? 5 : 3;
  static constexpr int ACC_COLS = 2 * NB;          // two accumulator buffers
  static constexpr int SF_COLS = 8 * KSTEPS;       // per stage: 4 columns per k-step for A and for B
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 4;
  static constexpr int THREADS = 32 * (6 + EPI_WARPS);
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(NB == 32, "one 32-column TMEM load per epilogue warp");
};

struct SlicedArgs {
  const int32_t* b_exp;        // [P * 4] slice exponents
  const int32_t* tiles;        // n_tiles, then int4 {row0, rows, expert, 0}
  float* out;                  // h f32 [P][F] (gate/up) or partial f32 [P][H] (down)
  uint32_t* err;
  int K;                       // reduction length (H or F)
  int rows_per_expert;         // weight rows per expert (2F or H)
  int n_tiles_n;               // weight row tiles per expert (F/64 or H/128)
  int out_cols;                // F or H
  int F;                       // gate/up: row offset of the up rows; down: unused
  int a_sf_group;              // down: g weight-scale rows per tensor-map row
  int sb_w;                    // bytes per slice-scale staging row: min(16*KSUB, scale pitch)
  const float* alpha = nullptr;   // [E] per-expert second-level weight scale, or none
  // PACKED: the weights' 512-byte scale-factor atoms, one per (expert, 128-row tile, k-step
  // of 64); n_tiles_n tiles per expert, kst k-steps per row
  const uint8_t* a_atoms = nullptr;
  int kst = 0;
};


__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&a)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) a[i] = __uint_as_float(r[i]);
}

template <bool GATE_UP, bool PACKED>
__global__ void __launch_bounds__(SCfg<GATE_UP>::THREADS, 1)
sliced_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_sfa,
                   const __grid_constant__ CUtensorMap tmap_sfb, const SlicedArgs args) {
  using C = SCfg<GATE_UP>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full[s]: code tiles landed and the stage's scale factors are in TMEM (TMA bytes + one
  // arrive per transposer warp); stg_full[s]: the scale staging images landed.
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* stg_full = full + C::STAGES;
  uint64_t* empty = stg_full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;           // [2]
  uint64_t* acc_empty = acc_full + 2;               // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // stage layout: A codes (weights) | B codes (slices) | A scale staging | B scale staging
  constexpr int OFF_B = C::A_BYTES;
  constexpr int OFF_SA = C::A_BYTES + C::B_BYTES;
  constexpr int OFF_SB = OFF_SA + C::SA_STG;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The tile list comes from the CSR call, complete before this grid started (the kernel
  // before this one waited for it before letting this grid launch); the slices (and their
  // exponents) come from the kernel just before, which the producer and the epilogue wait
  // for where they first read them.
  const int n_tiles = args.tiles[0];
  const int4* tlist = reinterpret_cast<const int4*>(args.tiles + 4);
  const int n_work = n_tiles * args.n_tiles_n;
  const int k_stages = (args.K / 2 + C::KSUB * C::KB - 1) / (C::KSUB * C::KB);
  const int sfrow = args.K / 16;                    // scale bytes per row
  constexpr int WROWS = GATE_UP ? 64 : 128;         // weight rows of one matrix per work

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // TMA expect_tx + 4 transposer warps (+ PACKED: the commit of the atom copies)
      mbar_init(&full[s], PACKED ? 1 + 4 + 1 : 1 + 4);
      mbar_init(&stg_full[s], 1);
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
  // the next kernel may launch now: it waits for this grid before reading what it writes
  pdl_trigger();
  const uint32_t tmem = *tmem_holder;
  const uint32_t acc_col = tmem;
  const uint32_t sf_col0 = tmem + C::ACC_COLS;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      constexpr uint32_t tx_codes = C::A_BYTES + C::B_BYTES;
      const int g = GATE_UP ? 1 : args.a_sf_group;
      const uint32_t tx_stg = (PACKED ? 0u : (uint32_t)(GATE_UP ? C::SA_STG : 128 * sfrow)) +
                              (uint32_t)(C::NB * args.sb_w);
      const uint64_t wpol = l2_evict_first_policy();
      // The slice half of a stage (B codes and B scale staging) reads what the previous
      // kernel writes; the weight half depends only on the tile list.  The weight halves of
      // the first STAGES stages are issued before waiting for the previous kernel, so the
      // weight stream starts while the slices are still being formed.
      auto issue_b = [&](int st, int ks, int row0, int nsub) {
        unsigned char* sb = smem + st * C::STAGE_BYTES;
        tma_load_2d(sb + OFF_SB, &tmap_sfb, ks * 16 * C::KSUB, row0, &stg_full[st]);
#pragma unroll
        for (int q = 0; q < C::KSUB; ++q)
          if (q < nsub)
            tma_load_2d(sb + OFF_B + q * C::B_SUB, &tmap_b, (ks * C::KSUB + q) * C::KB, row0,
                        &full[st]);
      };
      int pend_st[C::STAGES], pend_ks[C::STAGES], pend_row[C::STAGES], pend_nsub[C::STAGES];
      int npend = 0;
      bool waited = false;
      auto flush_pending = [&]() {
        pdl_wait();
        for (int i = 0; i < npend; ++i) issue_b(pend_st[i], pend_ks[i], pend_row[i], pend_nsub[i]);
        npend = 0;
        waited = true;
      };
      int it = 0;
      // work descriptors are fetched two works ahead
      const int w1 = blockIdx.x + gridDim.x;
      int4 tile = blockIdx.x < n_work ? tlist[blockIdx.x / args.n_tiles_n] : make_int4(0, 0, 0, 0);
      int4 next = w1 < n_work ? tlist[w1 / args.n_tiles_n] : tile;
      for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x) {
        const int w2 = w + 2 * gridDim.x;
        const int4 next2 = w2 < n_work ? tlist[w2 / args.n_tiles_n] : next;
        const int wrow = tile.z * args.rows_per_expert + (w % args.n_tiles_n) * WROWS;
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait(&empty[st], ((it / C::STAGES) & 1) ^ 1, abort_flag, args.err)) break;
          unsigned char* sb = smem + st * C::STAGE_BYTES;
          // sub-tiles that start past the row are not fetched (their k-steps are skipped)
          const int nsub = min(C::KSUB, (args.K / 2 - ks * C::KSUB * C::KB + C::KB - 1) / C::KB);
          const int nk = PACKED ? min(C::KSTEPS, args.kst - C::KSTEPS * ks) : 0;   // atoms
          mbar_expect_tx(&stg_full[st], tx_stg + 512u * nk);
          mbar_expect_tx(&full[st], tx_codes / C::KSUB * nsub);
          // scale staging first: the transposers can start while the code tiles stream in
          if (PACKED) {
            const int t = w % args.n_tiles_n;
            bulk_load(sb + OFF_SA,
                      args.a_atoms + ((size_t)(tile.z * args.n_tiles_n + t) * args.kst + C::KSTEPS * ks) * 512,
                      512u * nk, &stg_full[st]);
          } else if (GATE_UP) {
            tma_load_3d_hint(sb + OFF_SA, &tmap_sfa, ks * 16 * C::KSUB, 0, wrow, &stg_full[st], wpol);
          } else {
            tma_load_2d_hint(sb + OFF_SA, &tmap_sfa, 0, wrow / g, &stg_full[st], wpol);
          }
#pragma unroll
          for (int q = 0; q < C::KSUB; ++q) {
            if (q >= nsub) break;
            const int x = (ks * C::KSUB + q) * C::KB;
            if (GATE_UP)
              tma_load_3d_hint(sb + q * C::A_SUB, &tmap_a, x, 0, wrow, &full[st], wpol);
            else
              tma_load_2d_hint(sb + q * C::A_SUB, &tmap_a, x, wrow, &full[st], wpol);
          }
          if (waited) {
            issue_b(st, ks, tile.x, nsub);
          } else {
            pend_st[npend] = st; pend_ks[npend] = ks; pend_row[npend] = tile.x; pend_nsub[npend] = nsub;
            if (++npend == C::STAGES) flush_pending();
          }
        }
        tile = next;
        next = next2;
      }
      // every issued stage gets its slice half (also when the loop ended early)
      if (!waited) flush_pending();
      // drain: wait (bounded) until every issued stage has landed
      if (*abort_flag) {
        for (int s = 0; s < C::STAGES; ++s) {
          if (it <= s) continue;
          const int last = s + ((it - 1 - s) / C::STAGES) * C::STAGES;
          const uint64_t t0 = global_ns();
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
      constexpr uint32_t idesc = mxf4_idesc(128, C::NB);
      const uint32_t s0 = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(s0, 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(s0 + OFF_B, 16, 1024, 2);
      int it = 0, tcount = 0;
      for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x, ++tcount) {
        const int ab = tcount & 1;
        if (!mbar_wait(&acc_empty[ab], ((tcount >> 1) & 1) ^ 1, abort_flag, args.err)) break;
        tc_fence_after();
        const uint32_t acc = acc_col + ab * C::NB;
        bool ok = true;
        int st = it % C::STAGES;
        uint32_t par = (it / C::STAGES) & 1;
        for (int ks = 0; ks < k_stages; ++ks, ++it) {
          if (!mbar_wait(&full[st], par, abort_flag, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t so = (uint64_t)((st * C::STAGE_BYTES) >> 4);
          const uint32_t sfc = sf_col0 + st * C::SF_COLS;
          // k-steps past K (the zero-filled tail of the last stage) are skipped
          const int nk = min(C::KSTEPS, (sfrow - 16 * C::KSUB * ks) >> 2);
#pragma unroll
          for (int j = 0; j < C::KSTEPS; ++j)
            if (j < nk) {
              const uint32_t ao = (uint32_t)(((j >> 2) * C::A_SUB + 32 * (j & 3)) >> 4);
              const uint32_t bo = (uint32_t)(((j >> 2) * C::B_SUB + 32 * (j & 3)) >> 4);
              tc_mma(acc, a_desc0 + so + ao, b_desc0 + so + bo, idesc, sfc + 4 * j,
                     sfc + 4 * C::KSTEPS + 4 * j, (ks | j) != 0);
            }
          tc_commit(&empty[st]);
          if (++st == C::STAGES) { st = 0; par ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&acc_full[ab]);
      }
    }
  } else if (warp < 6) {
    // ---------------- scale-factor transposers (one TMEM lane quarter each) ----------------
    // Lane r of warp w writes TMEM lane 32*(w%4) + r.  A (weights, 128 rows): for k-step j,
    // columns 4j + x hold the scale word of row r + 32x.  B (32 slice rows), from column
    // 4*KSTEPS on: column 4j holds row r's word, 4j+1..4j+3 are zero.  Words past the row's
    // K/16 bytes are zero.  PACKED: B's only.
    const int n_it = ((n_work - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) * k_stages;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int g = GATE_UP ? 1 : args.a_sf_group;
    constexpr int KW = C::KSTEPS;                            // scale words per row and stage
    for (int it = 0; it < n_it; ++it) {
      const int st = it % C::STAGES;
      const int ks = it % k_stages;
      if (!mbar_wait_warp(&stg_full[st], (it / C::STAGES) & 1, abort_flag, args.err)) break;
      tc_fence_after();
      const uint32_t sb = smem_u32(smem + st * C::STAGE_BYTES);
      const int nvalid = min(KW, (sfrow - 4 * KW * ks) >> 2);
      if (PACKED && warp == 2 && lane == 0) {
        // the weight atoms into the stage's A columns, completing on full[st]
#pragma unroll
        for (int j = 0; j < KW; ++j)
          if (j < nvalid) tc_cp_sf(sf_col0 + st * C::SF_COLS + 4 * j, sb + OFF_SA + 512 * j);
        tc_commit(&full[st]);
      }
      uint32_t va[4 * KW], vb[4 * KW];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        if (PACKED) break;
        const int row = lane + 32 * x;
        uint32_t a[KW];
        if (GATE_UP) {
#pragma unroll
          for (int q = 0; q < KW / 4; ++q) {
            const uint4 a4 = lds128(sb + OFF_SA + 4 * KW * row + 16 * q);
            a[4 * q] = a4.x; a[4 * q + 1] = a4.y; a[4 * q + 2] = a4.z; a[4 * q + 3] = a4.w;
          }
        } else {
          // staged rows: map row r/g holds rows g*(r/g) .. +g-1, sfrow bytes each
          const uint32_t src = sb + OFF_SA + (row / g) * (g * sfrow) + (row % g) * sfrow + 4 * KW * ks;
#pragma unroll
          for (int j = 0; j < KW; ++j) a[j] = j < nvalid ? lds32(src + 4 * j) : 0u;
        }
#pragma unroll
        for (int j = 0; j < KW; ++j) va[4 * j + x] = j < nvalid ? a[j] : 0u;
      }
#pragma unroll
      for (int q = 0; q < KW / 4; ++q) {
        // staging rows are sb_w bytes; words past them are past the row's K (nvalid)
        const uint4 b4 = 16 * q < args.sb_w ? lds128(sb + OFF_SB + args.sb_w * lane + 16 * q)
                                            : make_uint4(0, 0, 0, 0);
        const uint32_t b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * q + jj;
          vb[4 * j] = j < nvalid ? b[jj] : 0u;
          vb[4 * j + 1] = 0u;
          vb[4 * j + 2] = 0u;
          vb[4 * j + 3] = 0u;
        }
      }
      const uint32_t sfc = sf_col0 + st * C::SF_COLS + lane_base;
#pragma unroll
      for (int q = 0; q < KW / 4; ++q) {
        if (!PACKED) tc_st16(sfc + 16 * q, *reinterpret_cast<const uint32_t(*)[16]>(va + 16 * q));
        tc_st16(sfc + 4 * KW + 16 * q, *reinterpret_cast<const uint32_t(*)[16]>(vb + 16 * q));
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
    }
  } else {
    // ---------------- epilogue (warps 6..9, one TMEM lane quarter each) ----------------
    pdl_wait();                                              // the slice exponents are complete
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                     // weight row of the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    int tcount = 0;
    for (int w = blockIdx.x; w < n_work && !*abort_flag; w += gridDim.x, ++tcount) {
      const int ab = tcount & 1;
      const int4 tile = tlist[w / args.n_tiles_n];
      const int nt = w % args.n_tiles_n;
      // lane c holds the exponent of slice row c of the tile (column c of the accumulator)
      const int ex = lane < tile.y ? args.b_exp[tile.x + lane] : 0;
      if (!mbar_wait_warp(&acc_full[ab], (tcount >> 1) & 1, abort_flag, args.err)) break;
      tc_fence_after();
      float v[32];
      tc_ld32(acc_col + ab * C::NB + lane_base, v);
      // pair p of the tile: columns 4p .. 4p+3, summed in slice order
      float z[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        float a = 0.0f;
#pragma unroll
        for (int s = 0; s < 4; ++s) a += ldexpf(v[4 * p + s], __shfl_sync(0xffffffffu, ex, 4 * p + s));
        z[p] = a;
      }
      if (args.alpha) {
        const float al = __ldg(args.alpha + tile.z);
#pragma unroll
        for (int p = 0; p < 8; ++p) z[p] *= al;
      }
      const int np = tile.y >> 2;                           // pairs in the tile
      const int pos0 = tile.x >> 2;                         // CSR row of the tile's first pair
      if (GATE_UP) {
        // lanes 2i (gate row i) and 2i+1 (up row i) of the quarter
        float up[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) up[p] = __shfl_xor_sync(0xffffffffu, z[p], 1);
        if ((lane & 1) == 0) {
          float* o = args.out + nt * 64 + (row >> 1);
#pragma unroll
          for (int p = 0; p < 8; ++p)
            if (p < np) o[(size_t)(pos0 + p) * args.out_cols] = silu_f(z[p]) * up[p];
        }
      } else {
        float* o = args.out + nt * 128 + row;
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < np) o[(size_t)(pos0 + p) * args.out_cols] = z[p];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
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

template <bool GATE_UP>
cudaError_t run_sliced(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa,
                       const CUtensorMap& msb, const SlicedArgs& a, int max_tiles, cudaStream_t s) {
  using C = SCfg<GATE_UP>;
  auto kern = a.a_atoms ? sliced_gemm_kernel<GATE_UP, true> : sliced_gemm_kernel<GATE_UP, false>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (st != cudaSuccess) return st;
  int grid = max_tiles * a.n_tiles_n;
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3(grid), dim3(C::THREADS), (size_t)C::SMEM, s, ma, mb, msa, msb, a);
}

}  // namespace

cudaError_t launch_sliced_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                  const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                  char* ws, cudaStream_t s) {
  constexpr int NS = kDecodeSlices;
  static_assert(NS == 4, "four slices per pair: eight pairs per 32-row tile");
  const int P = T * k;
  uint8_t* qc = reinterpret_cast<uint8_t*>(ws + L.qx_codes);
  uint8_t* qs = reinterpret_cast<uint8_t*>(ws + L.qx_scales);
  int32_t* qe = reinterpret_cast<int32_t*>(ws + L.qx_exp);
  // the slices of x depend only on x: they are formed while the CSR kernel still runs, and
  // only their stores wait for it
  cudaError_t st = launch_slice_x(x_bf16, T, H, k, reinterpret_cast<const int32_t*>(ws + L.pair_pos),
                                  qc, qs, qe, s);
  if (st != cudaSuccess) return st;
  // the 32-row tile list over the slice rows was written by the CSR call
  int32_t* tiles = reinterpret_cast<int32_t*>(ws + L.slice_tiles);
  // weights: [K bytes][gate, up][row], so the box {128 B, 2, 64} lands gate row i and up row i
  // as shared-memory rows 2i and 2i+1; the row extent stops F rows short of the bank so the
  // up coordinate (row + F) stays inside it
  const uint64_t rows = (uint64_t)P * NS;
  const uint64_t wrows = (uint64_t)b.E * 2 * F - F;
  const uint64_t cdims[3] = {(uint64_t)H / 2, 2, wrows};
  const uint64_t cstr[2] = {(uint64_t)F * (H / 2), (uint64_t)H / 2};
  const uint32_t cbox[3] = {128, 2, 64};
  const int sbw = 16 * SCfg<true>::KSUB < H / 16 ? 16 * SCfg<true>::KSUB : H / 16;
  const uint64_t sdims[3] = {(uint64_t)H / 16, 2, wrows};
  const uint64_t sstr[2] = {(uint64_t)F * (H / 16), (uint64_t)H / 16};
  const uint32_t sbox[3] = {32, 2, 64};
  CUtensorMap ma, mb, msa, msb;
  if (!make_map3(&ma, b.codes, cdims, cstr, cbox, true) ||
      !make_map(&mb, qc, H / 2, H / 2, rows, 128, kSliceTile, true) ||
      !make_map3(&msa, b.scales, sdims, sstr, sbox, false) ||
      !make_map(&msb, qs, H / 16, H / 16, rows, sbw, kSliceTile, false))
    return cudaErrorInvalidValue;
  SlicedArgs a{qe, tiles, reinterpret_cast<float*>(ws + L.h),
               reinterpret_cast<uint32_t*>(ws + L.error_word), H, 2 * F, F / 64, F, F, 1, sbw};
  a.alpha = b.alpha;
  if (b.sf_atoms) {
    a.a_atoms = b.sf_atoms;
    a.kst = H / 64;
  }
  const int max_tiles = (int)(rows / kSliceTile) + (P < b.E ? P : b.E) + 1;
  return run_sliced<true>(ma, mb, msa, msb, a, max_tiles, s);
}

cudaError_t launch_sliced_down(const moe_nvfp4_bank& b, moe_csr csr, int T, int H, int F, int k,
                               const moe_ws_layout& L, char* ws, cudaStream_t s) {
  constexpr int NS = kDecodeSlices;
  const int P = T * k;
  uint8_t* qc = reinterpret_cast<uint8_t*>(ws + L.qh_codes);
  uint8_t* qs = reinterpret_cast<uint8_t*>(ws + L.qh_scales);
  int32_t* qe = reinterpret_cast<int32_t*>(ws + L.qh_exp);
  const int sfh = qh_scale_pitch(F);
  cudaError_t st = launch_slice_h(reinterpret_cast<const float*>(ws + L.h), P, F, sfh,
                                  csr.expert_offsets, b.E, qc, qs, qe, s);
  if (st != cudaSuccess) return st;
  // the weight-scale rows are F/16 bytes; g of them make a row pitch that is a multiple of 16
  const int sfrow = F / 16;
  int g = 1;
  if (sfrow % 16 != 0)
    for (g = 2; (g * sfrow) % 16 != 0 || g * sfrow < 32; g *= 2) {
    }
  if (128 % g != 0 || g * sfrow > 256 || 128 * sfrow > 11264) return cudaErrorInvalidValue;
  const uint64_t rows = (uint64_t)P * NS;
  const uint64_t wrows = (uint64_t)b.E * H;
  const int sbw = 16 * SCfg<false>::KSUB < sfh ? 16 * SCfg<false>::KSUB : sfh;
  CUtensorMap ma, mb, msa, msb;
  if (!make_map(&ma, b.codes, F / 2, F / 2, wrows, 128, 128, true) ||
      !make_map(&mb, qc, F / 2, F / 2, rows, 128, kSliceTile, true) ||
      !make_map(&msa, b.scales, (uint64_t)g * sfrow, (uint64_t)g * sfrow, wrows / g,
                g * sfrow, 128 / g, false) ||
      !make_map(&msb, qs, sfh, sfh, rows, sbw, kSliceTile, false))
    return cudaErrorInvalidValue;
  SlicedArgs a{qe, reinterpret_cast<const int32_t*>(ws + L.slice_tiles),
               reinterpret_cast<float*>(ws + L.partial),
               reinterpret_cast<uint32_t*>(ws + L.error_word), F, H, H / 128, H, F, g, sbw};
  a.alpha = b.alpha;
  if (b.sf_atoms) {
    a.a_atoms = b.sf_atoms;
    a.kst = F / 64;
  }
  const int max_tiles = (int)(rows / kSliceTile) + (P < b.E ? P : b.E) + 1;
  return run_sliced<false>(ma, mb, msa, msb, a, max_tiles, s);
}

}  // namespace moe
