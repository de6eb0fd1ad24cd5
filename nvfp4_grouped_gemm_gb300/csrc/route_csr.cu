// Top-k routing and the expert-first CSR.
//
// route_merge_kernel: one CTA per token, one expert per thread.  Each (logit, id) pair
// becomes a 64-bit key whose unsigned order is the routing order (logit descending, then
// id ascending; -0 and +0 share a key, as the float32 comparison makes them equal).  Every
// warp sorts its 32 keys with a shuffle bitonic sort; the sorted lists are then merged
// pairwise through shared memory (the best 32 of two descending lists a, b are
// max(a[i], b[31-i]), a bitonic sequence that five shuffle steps sort), so warp 0 ends with
// the best 32 keys in order and k <= 32 of them are the picks.
//
// build_csr_kernel: one CTA.  The P pairs are cut into 32 contiguous slices, one per warp.
// Pass A counts each slice's pairs per expert in shared memory, pass B turns the
// [slice][expert] counts into starting positions (expert offset + pairs of the same
// expert in earlier slices), pass C walks each slice in ascending p and places pairs with
// a warp-level match so that equal experts keep ascending p.  Placement never depends on
// the order atomics happen to arrive in, so the output is bit-exact.
//
// For many pairs the same three passes run over the whole grid: csr_count_kernel counts
// each 2048-pair chunk's pairs per expert, csr_scan_kernel turns the [chunk][expert]
// counts into each chunk's first row per expert (plus the offsets and the active list),
// csr_place_kernel places each chunk's pairs as above within the chunk.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {


__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
  return a < b ? a : b;
}

// Sort a bitonic sequence held one key per lane into descending lane order.
__device__ __forceinline__ unsigned long long bitonic_merge_desc(unsigned long long key, int lane) {
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, stride);
    key = (lane & stride) == 0 ? umax64(key, o) : umin64(key, o);
  }
  return key;
}

// Descending sort of one key per lane.  Before the last size, blocks alternate between
// descending ((lane & size) == 0) and ascending, so each pair of blocks is bitonic.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long key, int lane) {
#pragma unroll
  for (int size = 2; size < 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      key = keep_max ? umax64(key, o) : umin64(key, o);
    }
  }
  return bitonic_merge_desc(key, lane);
}

// blockDim.x = 32 * ceil(E / 32) threads (E <= 1024); thread e holds expert e.
__global__ void __launch_bounds__(1024)
route_merge_kernel(const float* __restrict__ logits, int T, int E, int k,
                   int32_t* __restrict__ ids, float* __restrict__ w) {
  __shared__ unsigned long long lists[2][32][32];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int e = threadIdx.x;
  unsigned long long key = e < E ? route_key(__ldg(logits + (size_t)t * E + e), e) : 0ull;
  key = warp_sort_desc(key, lane);
  // merge tree: at stride s the warps w = 0 mod 2s take in warp w + s's list
  int buf = 0;
  for (int s = 1; s < nw; s <<= 1) {
    lists[buf][warp][lane] = key;
    __syncthreads();
    if ((warp & (2 * s - 1)) == 0 && warp + s < nw)
      key = bitonic_merge_desc(umax64(key, lists[buf][warp + s][31 - lane]), lane);
    buf ^= 1;
  }
  if (warp == 0) {
    const float first_v = key_logit(__shfl_sync(0xffffffffu, key, 0));
    const float ex = (lane < k) ? expf(key_logit(key) - first_v) : 0.0f;
    // sum in ascending j so every lane sees the same value
    float denom = 0.0f;
    for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
      ids[(size_t)t * k + lane] = key_id(key);
      w[(size_t)t * k + lane] = ex / denom;
    }
  }
}

constexpr int kCsrThreads = 1024;
constexpr int kCsrWarps = kCsrThreads / 32;

// Exclusive scan of four ints per thread across the block at once (one set of barriers
// for all four); scratch: kCsrWarps int4.
__device__ __forceinline__ int4 block_exclusive_scan4(int4 v, int4* scratch, int4* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int4 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, x.x, o), b = __shfl_up_sync(0xffffffffu, x.y, o);
    const int c = __shfl_up_sync(0xffffffffu, x.z, o), d = __shfl_up_sync(0xffffffffu, x.w, o);
    if (lane >= o) { x.x += a; x.y += b; x.z += c; x.w += d; }
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int4 q = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, q.x, o), b = __shfl_up_sync(0xffffffffu, q.y, o);
      const int c = __shfl_up_sync(0xffffffffu, q.z, o), d = __shfl_up_sync(0xffffffffu, q.w, o);
      if (lane >= o) { q.x += a; q.y += b; q.z += c; q.w += d; }
    }
    scratch[lane] = q;   // inclusive
  }
  __syncthreads();
  const int4 base = warp ? scratch[warp - 1] : make_int4(0, 0, 0, 0);
  *total = scratch[kCsrWarps - 1];
  __syncthreads();
  return make_int4(base.x + x.x - v.x, base.y + x.y - v.y, base.z + x.z - v.z, base.w + x.w - v.w);
}

// The cut of an expert's m operand rows (starting at row first) into tiles of tile_rows,
// entries base, base + 1, ... of the list.
__device__ __forceinline__ void write_tiles(int32_t* tiles, int base, int m, int first,
                                            int tile_rows, int e) {
  int4* list = reinterpret_cast<int4*>(tiles + 4);
  for (int i = 0; (i * tile_rows) < m; ++i) {
    const int r = m - i * tile_rows;
    list[base + i] = make_int4(first + i * tile_rows, r < tile_rows ? r : tile_rows, e, 0);
  }
}

// From each expert's pair count (thread e < E holds expert e's; every thread of the CTA
// calls it): the offsets, the active list and count, and both tile lists (the prefill
// GEMMs' 128-row M-tiles, the sliced decode GEMMs' 32-row tiles over kDecodeSlices rows per
// pair, each when the caller passed its region), from one block-wide scan of the four
// per-expert quantities.  Returns the expert's offset.
__device__ __forceinline__ int write_csr_lists(int E, int cnt, int32_t* __restrict__ offsets,
                                               int32_t* __restrict__ active,
                                               int32_t* __restrict__ n_active, int32_t* tiles,
                                               int32_t* slice_tiles, int4* scratch) {
  const int e = threadIdx.x;
  const int c = e < E ? cnt : 0;
  const int m0 = tiles ? c : 0, m1 = slice_tiles ? c * kDecodeSlices : 0;
  const int4 v = make_int4(c, c > 0 ? 1 : 0, (m0 + kTileRows - 1) / kTileRows,
                           (m1 + kSliceTileRows - 1) / kSliceTileRows);
  int4 tot;
  const int4 base = block_exclusive_scan4(v, scratch, &tot);
  if (e < E) {
    offsets[e] = base.x;
    if (c > 0) active[base.y] = e;
    if (tiles) write_tiles(tiles, base.z, m0, base.x, kTileRows, e);
    if (slice_tiles) write_tiles(slice_tiles, base.w, m1, base.x * kDecodeSlices, kSliceTileRows, e);
  }
  if (e == 0) {
    offsets[E] = tot.x;
    *n_active = tot.y;
    if (tiles) tiles[0] = tot.z;
    if (slice_tiles) slice_tiles[0] = tot.w;
  }
  return base.x;
}

__global__ void __launch_bounds__(kCsrThreads, 1)
build_csr_kernel(const int32_t* __restrict__ ids_g, int P, int E, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ pair_ids, int32_t* __restrict__ active,
                 int32_t* __restrict__ n_active, int32_t* __restrict__ pair_pos,
                 uint32_t* __restrict__ err, int ids_in_smem, int32_t* tiles,
                 int32_t* slice_tiles) {
  extern __shared__ int smem[];
  int* hist = smem;                           // [kCsrWarps][E]
  int4* scratch = reinterpret_cast<int4*>(smem + kCsrWarps * E);   // [kCsrWarps]
  int* ids_s = smem + kCsrWarps * E + 4 * kCsrWarps;                // [P] when ids_in_smem
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kCsrWarps * E; i += kCsrThreads) hist[i] = 0;
  pdl_wait();                                 // the expert ids are complete
  pdl_trigger();
  // one coalesced pass over the ids; every later pass reads shared memory
  if (ids_in_smem)
    for (int p = tid; p < P; p += kCsrThreads) ids_s[p] = __ldg(ids_g + p);
  __syncthreads();
  const int32_t* ids = ids_in_smem ? ids_s : ids_g;

  const int slice = (P + kCsrWarps - 1) / kCsrWarps;
  const int p_beg = min(P, warp * slice), p_end = min(P, p_beg + slice);
  int* my = hist + warp * E;
  bool bad = false;
  // pass A: per-slice counts
  for (int p = p_beg + lane; p < p_end; p += 32) {
    int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&my[e], 1);
    else { bad = true; pair_pos[p] = -1; }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, (uint32_t)MOE_DEVERR_EXPERT_ID);
  __syncthreads();

  // pass B: per expert, slice prefix and the expert's total; then the offsets scan
  int cnt = 0;
  if (tid < E) {
    for (int w = 0; w < kCsrWarps; ++w) {
      int c = hist[w * E + tid];
      hist[w * E + tid] = cnt;
      cnt += c;
    }
  }
  const int off = write_csr_lists(E, cnt, offsets, active, n_active, tiles, slice_tiles, scratch);
  if (tid < E)
    for (int w = 0; w < kCsrWarps; ++w) hist[w * E + tid] += off;
  __syncthreads();

  // pass C: stable placement within each slice
  for (int base = p_beg; base < p_end; base += 32) {
    const int p = base + lane;
    const bool in = p < p_end;
    int e = in ? ids[p] : -1;
    const bool valid = in && e >= 0 && e < E;
    if (!valid) e = -1 - lane;                           // unique key: matches nobody
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    int start = valid ? my[e] : 0;
    __syncwarp();
    if (valid) {
      const int pos = start + __popc(lower);
      pair_ids[pos] = p;
      pair_pos[p] = pos;
      if (lower == 0) my[e] = start + __popc(peers);     // lowest lane of the group advances
    }
    __syncwarp();
  }
}


// ---------------------------------------------------------------------------
// grid-wide CSR for many pairs
// ---------------------------------------------------------------------------
constexpr int kChunkPairs = 2048;
constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;
static_assert(kChunkPairs % kChunkThreads == 0 && kChunkPairs % (32 * kChunkWarps) == 0,
              "whole register batches of ids per thread and per warp slice");

__global__ void __launch_bounds__(kChunkThreads)
csr_count_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ cnt,
                 int32_t* __restrict__ pair_pos, uint32_t* __restrict__ err) {
  extern __shared__ int hist[];                // [E]
  for (int i = threadIdx.x; i < E; i += kChunkThreads) hist[i] = 0;
  pdl_wait();                                  // the expert ids are complete
  pdl_trigger();
  __syncthreads();
  const int p0 = blockIdx.x * kChunkPairs, p1 = min(P, p0 + kChunkPairs);
  bool bad = false;
  // the thread's ids loaded together, then counted
  constexpr int kPerThread = kChunkPairs / kChunkThreads;
  int ev[kPerThread];
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int p = p0 + (int)threadIdx.x + i * kChunkThreads;
    ev[i] = p < p1 ? __ldg(ids + p) : 0;
  }
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int p = p0 + (int)threadIdx.x + i * kChunkThreads;
    if (p >= p1) continue;
    const int e = ev[i];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else { bad = true; pair_pos[p] = -1; }
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(err, (uint32_t)MOE_DEVERR_EXPERT_ID);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += kChunkThreads) cnt[(size_t)blockIdx.x * E + i] = hist[i];
}

// One CTA of kCsrThreads: thread e turns expert e's per-chunk counts into chunk starts.
__global__ void __launch_bounds__(kCsrThreads, 1)
csr_scan_kernel(int32_t* __restrict__ cnt, int n_chunks, int E, int32_t* __restrict__ offsets,
                int32_t* __restrict__ active, int32_t* __restrict__ n_active, int32_t* tiles,
                int32_t* slice_tiles) {
  __shared__ int4 scratch[kCsrWarps];
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x;
  // Up to kScanRegChunks chunks the expert's counts are loaded together into registers (the
  // loads are independent, one round trip instead of one per chunk) and written once, as
  // chunk starts, after the offsets are known; beyond that the counts are rewritten in two
  // passes over memory.
  constexpr int kScanRegChunks = 32;
  int c[kScanRegChunks];
  const bool in_regs = n_chunks <= kScanRegChunks;
  int tot = 0;
  if (e < E) {
    if (in_regs) {
#pragma unroll
      for (int b = 0; b < kScanRegChunks; ++b) c[b] = b < n_chunks ? cnt[(size_t)b * E + e] : 0;
#pragma unroll
      for (int b = 0; b < kScanRegChunks; ++b) {
        const int v = c[b];
        c[b] = tot;
        tot += v;
      }
    } else {
      for (int b = 0; b < n_chunks; ++b) {
        const int v = cnt[(size_t)b * E + e];
        cnt[(size_t)b * E + e] = tot;
        tot += v;
      }
    }
  }
  const int off = write_csr_lists(E, tot, offsets, active, n_active, tiles, slice_tiles, scratch);
  if (e < E) {
    if (in_regs) {
#pragma unroll
      for (int b = 0; b < kScanRegChunks; ++b)
        if (b < n_chunks) cnt[(size_t)b * E + e] = c[b] + off;
    } else {
      for (int b = 0; b < n_chunks; ++b) cnt[(size_t)b * E + e] += off;
    }
  }
}

__global__ void __launch_bounds__(kChunkThreads)
csr_place_kernel(const int32_t* __restrict__ ids, int P, int E, const int32_t* __restrict__ cnt,
                 int32_t* __restrict__ pair_ids, int32_t* __restrict__ pair_pos) {
  extern __shared__ int wh[];                  // [kChunkWarps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kChunkWarps * E; i += kChunkThreads) wh[i] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kChunkPairs, p1 = min(P, p0 + kChunkPairs);
  const int slice = (p1 - p0 + kChunkWarps - 1) / kChunkWarps;
  const int s0 = min(p1, p0 + warp * slice), s1 = min(p1, s0 + slice);
  int* my = wh + warp * E;
  // the next kernel may launch now (it waits for this grid before it reads what it writes)
  pdl_trigger();
  // The ids were complete before the count kernel passed its wait (two kernels back), so
  // the warp's slice is loaded (into registers, once) and counted before the wait for the
  // chunk starts.
  constexpr int kPerLane = kChunkPairs / kChunkWarps / 32;
  int ev[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int p = s0 + lane + 32 * i;
    ev[i] = p < s1 ? __ldg(ids + p) : -1;
  }
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int e = ev[i];
    if (s0 + lane + 32 * i < s1 && e >= 0 && e < E) atomicAdd(&my[e], 1);
  }
  pdl_wait();                                  // the chunk starts are complete
  __syncthreads();
  for (int e = tid; e < E; e += kChunkThreads) {
    int run = cnt[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < kChunkWarps; ++w) {
      const int c = wh[w * E + e];
      wh[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int p = s0 + lane + 32 * i;
    const bool in = p < s1;
    int e = ev[i];
    const bool valid = in && e >= 0 && e < E;
    if (!valid) e = -1 - lane;                 // unique key: matches nobody
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    const int start = valid ? my[e] : 0;
    __syncwarp();
    if (valid) {
      const int pos = start + __popc(lower);
      pair_ids[pos] = p;
      pair_pos[p] = pos;
      if (lower == 0) my[e] = start + __popc(peers);
    }
    __syncwarp();
  }
}

// Few pairs (P <= kCsrSmallPairs): one histogram and one scan; pair p's place among the
// pairs of its expert is the number of earlier pairs with the same expert, counted by one
// warp that walks the pairs in groups of 32.
constexpr int kCsrSmallPairs = 256;

__global__ void __launch_bounds__(kCsrThreads, 1)
csr_small_kernel(const int32_t* __restrict__ ids_g, int P, int E, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ pair_ids, int32_t* __restrict__ active,
                 int32_t* __restrict__ n_active, int32_t* __restrict__ pair_pos,
                 uint32_t* __restrict__ err, int32_t* tiles, int32_t* slice_tiles) {
  __shared__ int hist[kMaxE];
  __shared__ int ids_s[kCsrSmallPairs];
  __shared__ int4 scratch[kCsrWarps];
  const int tid = threadIdx.x;
  if (tid < E) hist[tid] = 0;
  pdl_wait();                                 // the expert ids are complete
  pdl_trigger();
  int e = -1;
  bool valid = false;
  if (tid < P) {
    e = __ldg(ids_g + tid);
    valid = e >= 0 && e < E;
    ids_s[tid] = valid ? e : -1;
    if (!valid) {
      pair_pos[tid] = -1;
      atomicOr(err, (uint32_t)MOE_DEVERR_EXPERT_ID);
    }
  }
  __syncthreads();
  if (valid) atomicAdd(&hist[e], 1);
  __syncthreads();
  const int cnt = tid < E ? hist[tid] : 0;
  const int off = write_csr_lists(E, cnt, offsets, active, n_active, tiles, slice_tiles, scratch);
  if (tid < E) hist[tid] = off;
  __syncthreads();
  // one warp places the pairs 32 at a time in ascending p: equal experts in a group are
  // matched and ranked by lane, hist[e] (the expert's next row) advances by the group
  if (tid < 32) {
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + tid;
      const int ep = p < P ? ids_s[p] : -1;
      const bool v = ep >= 0;
      const unsigned peers = __match_any_sync(0xffffffffu, v ? ep : -1 - tid);
      const unsigned lower = peers & ((1u << tid) - 1u);
      const int start = v ? hist[ep] : 0;
      __syncwarp();
      if (v) {
        const int pos = start + __popc(lower);
        pair_ids[pos] = p;
        pair_pos[p] = pos;
        if (lower == 0) hist[ep] = start + __popc(peers);
      }
      __syncwarp();
    }
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t s) {
  const int nw = (E + 31) / 32;
  return launch_pdl(route_merge_kernel, dim3(T), dim3(32 * nw), 0, s, logits, T, E, k, ids, w);
}

size_t csr_scratch_bytes(int P, int E) {
  if (P < kCsrGridMinPairs) return 0;
  return (size_t)((P + kChunkPairs - 1) / kChunkPairs) * E * sizeof(int32_t);
}

cudaError_t launch_build_csr(const int32_t* ids, int P, int k, int E, moe_csr csr,
                             int32_t* pair_pos, uint32_t* err, int32_t* scratch, int32_t* tiles,
                             int32_t* slice_tiles, cudaStream_t s) {
  (void)k;
  if (P <= kCsrSmallPairs)
    return launch_pdl(csr_small_kernel, dim3(1), dim3(kCsrThreads), 0, s, ids, P, E,
                      csr.expert_offsets, csr.pair_ids, csr.active_experts, csr.n_active, pair_pos,
                      err, tiles, slice_tiles);
  if (P >= kCsrGridMinPairs && scratch) {
    const int nb = (P + kChunkPairs - 1) / kChunkPairs;
    cudaError_t st = launch_pdl(csr_count_kernel, dim3(nb), dim3(kChunkThreads),
                                (size_t)E * sizeof(int), s, ids, P, E, scratch, pair_pos, err);
    if (st != cudaSuccess) return st;
    st = launch_pdl(csr_scan_kernel, dim3(1), dim3(kCsrThreads), 0, s, scratch, nb, E,
                    csr.expert_offsets, csr.active_experts, csr.n_active, tiles, slice_tiles);
    if (st != cudaSuccess) return st;
    const size_t smem = (size_t)kChunkWarps * E * sizeof(int);
    st = cudaFuncSetAttribute(csr_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (st != cudaSuccess) return st;
    return launch_pdl(csr_place_kernel, dim3(nb), dim3(kChunkThreads), smem, s, ids, P, E,
                      (const int32_t*)scratch, csr.pair_ids, pair_pos);
  }
  size_t smem = (size_t)(kCsrWarps * E + 4 * kCsrWarps) * sizeof(int);
  const int ids_in_smem = smem + (size_t)P * sizeof(int) <= 200 * 1024 ? 1 : 0;
  if (ids_in_smem) smem += (size_t)P * sizeof(int);
  cudaError_t st = cudaFuncSetAttribute(build_csr_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (st != cudaSuccess) return st;
  return launch_pdl(build_csr_kernel, dim3(1), dim3(kCsrThreads), smem, s, ids, P, E,
                    csr.expert_offsets, csr.pair_ids, csr.active_experts, csr.n_active, pair_pos,
                    err, ids_in_smem, tiles, slice_tiles);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of moe_build_expert_csr
// ---------------------------------------------------------------------------
// Its scratch (the per-pair CSR positions and the device error word, which the regular
// entry point keeps in the caller's workspace) lives in this file-scope device array.
// Every GPU that loads the library holds it until the process exits.
constexpr int kStaticMaxPairs = 65536;
static __device__ __align__(256) int32_t g_csr_scratch[kStaticMaxPairs + 64];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_csr_scratch on the current device, looked up once per device.
// In host code the array's name is only a host-side handle, never a device address.
cudaError_t scratch_for_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    st = cudaGetSymbolAddress(&p, g_csr_scratch);
    if (st != cudaSuccess) return st;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}
}  // namespace

}  // namespace moe

extern "C" moe_status moe_build_expert_csr_static(const int32_t* topk_ids, int32_t T, int32_t k,
                                                  int32_t E, moe_csr csr, void* stream) {
  using namespace moe;
  if (!topk_ids) return MOE_ERR_INVALID_ARG;
  if (T <= 0 || k <= 0 || E <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (!csr.expert_offsets || !csr.pair_ids || !csr.active_experts || !csr.n_active)
    return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k > kStaticMaxPairs) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // every pair's position is rewritten by the kernel; the error word is only OR-ed into
  // and never read back by this entry point, so nothing needs clearing between calls
  cudaError_t st = launch_build_csr(topk_ids, T * k, k, E, csr, scratch,
                                    reinterpret_cast<uint32_t*>(scratch + kStaticMaxPairs),
                                    nullptr, nullptr, nullptr, static_cast<cudaStream_t>(stream));
  return st == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
