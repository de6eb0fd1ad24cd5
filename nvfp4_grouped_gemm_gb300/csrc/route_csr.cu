// Top-k routing and the expert-first CSR.
//
// route_topk_kernel: one warp per token.  Round r selects the largest (logit, -id) pair
// among those ordered strictly after the pair selected in round r-1, so no element is
// ever removed or overwritten and ties resolve to the lower id exactly as the float32
// comparison dictates.
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

__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kNone = 0x7fffffff;   // id of an empty candidate

// a beats b: a is a candidate and either b is empty or a comes first in (logit desc, id asc)
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
  return ai != kNone && (bi == kNone || before(av, ai, bv, bi));
}

// One warp (one CTA) per token; lane l holds experts l, l+32, ... (PL per lane, padded).
// Every untaken expert is ordered after the last pick, so each lane keeps the best of its
// untaken experts; a round is a warp butterfly over those, after which only the winning
// lane marks its slot taken and rescans its own PL slots.
template <int PL>
__global__ void __launch_bounds__(32)
route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                  int32_t* __restrict__ ids, float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
  float v[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : 0.0f;
  }
  uint32_t taken = 0;
  auto local_best = [&](float& bv, int& bi) {
    float cv[PL];
    int ci[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      cv[i] = v[i];
      ci[i] = (e < E && !((taken >> i) & 1u)) ? e : kNone;
    }
#pragma unroll
    for (int s = PL / 2; s >= 1; s >>= 1)
#pragma unroll
      for (int i = 0; i < s; ++i)
        if (beats(cv[i + s], ci[i + s], cv[i], ci[i])) { cv[i] = cv[i + s]; ci[i] = ci[i + s]; }
    bv = cv[0];
    bi = ci[0];
  };
  float lbv;
  int lbi;
  local_best(lbv, lbi);
  float first_v = 0.0f;
  float my_val = 0.0f;   // lane j < k keeps the j-th selected logit
  int my_id = 0;
  for (int r = 0; r < k; ++r) {
    float bv = lbv;
    int bi = lbi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (beats(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (r == 0) first_v = bv;
    if (lane == r) { my_val = bv; my_id = bi; }
    if (bi != kNone && lane == (bi & 31)) {
      taken |= 1u << (bi >> 5);
      local_best(lbv, lbi);
    }
  }
  const float ex = (lane < k) ? expf(my_val - first_v) : 0.0f;
  // sum in ascending j so every lane sees the same value
  float denom = 0.0f;
  for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = ex / denom;
  }
}

// One CTA per token for wider routers: a bitonic sort in shared memory of the N (a power
// of two >= E) keys (logit, id) in the same order (logit descending, then id ascending;
// padding keys of -inf with ids past E sort last); the first k keys are the picks and the
// weights are formed exactly as in route_topk_kernel.
template <int N>
__global__ void __launch_bounds__(N / 2)
route_sort_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                  float* __restrict__ w) {
  __shared__ float sv[N];
  __shared__ int si[N];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const float* row = logits + (size_t)t * E;
  for (int i = tid; i < N; i += N / 2) {
    sv[i] = i < E ? __ldg(row + i) : -INFINITY;
    si[i] = i;
  }
  __syncthreads();
  for (int size = 2; size <= N; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int i = 2 * stride * (tid / stride) + (tid & (stride - 1));
      const int j = i + stride;
      const bool up = (i & size) == 0;          // this block ends ordered best-first
      const float vi = sv[i], vj = sv[j];
      const int ii = si[i], ij = si[j];
      if (before(vj, ij, vi, ii) == up) {
        sv[i] = vj; sv[j] = vi;
        si[i] = ij; si[j] = ii;
      }
      __syncthreads();
    }
  }
  if (tid < 32) {
    const int lane = tid;
    const float first_v = sv[0];
    const float my_val = lane < k ? sv[lane] : 0.0f;
    const float ex = (lane < k) ? expf(my_val - first_v) : 0.0f;
    // sum in ascending j so every lane sees the same value
    float denom = 0.0f;
    for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
      ids[(size_t)t * k + lane] = si[lane];
      w[(size_t)t * k + lane] = ex / denom;
    }
  }
}

constexpr int kCsrThreads = 1024;
constexpr int kCsrWarps = kCsrThreads / 32;

__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  // scratch: kCsrWarps ints
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[lane] = s;   // inclusive
  }
  __syncthreads();
  int base = warp ? scratch[warp - 1] : 0;
  *total = scratch[kCsrWarps - 1];
  __syncthreads();
  return base + x - v;
}

__global__ void __launch_bounds__(kCsrThreads, 1)
build_csr_kernel(const int32_t* __restrict__ ids_g, int P, int E, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ pair_ids, int32_t* __restrict__ active,
                 int32_t* __restrict__ n_active, int32_t* __restrict__ pair_pos,
                 uint32_t* __restrict__ err, int ids_in_smem) {
  extern __shared__ int smem[];
  int* hist = smem;                           // [kCsrWarps][E]
  int* scratch = smem + kCsrWarps * E;        // [kCsrWarps]
  int* ids_s = scratch + kCsrWarps;           // [P] when ids_in_smem
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
  int total;
  int off = block_exclusive_scan(tid < E ? cnt : 0, scratch, &total);
  int act_total;
  int act_pos = block_exclusive_scan((tid < E && cnt > 0) ? 1 : 0, scratch, &act_total);
  if (tid < E) {
    offsets[tid] = off;
    if (cnt > 0) active[act_pos] = tid;
    for (int w = 0; w < kCsrWarps; ++w) hist[w * E + tid] += off;
  }
  if (tid == 0) {
    offsets[E] = total;
    *n_active = act_total;
  }
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
  for (int p = p0 + (int)threadIdx.x; p < p1; p += kChunkThreads) {
    const int e = __ldg(ids + p);
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
                int32_t* __restrict__ active, int32_t* __restrict__ n_active) {
  __shared__ int scratch[kCsrWarps];
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x;
  int tot = 0;
  if (e < E)
    for (int b = 0; b < n_chunks; ++b) {
      const int c = cnt[(size_t)b * E + e];
      cnt[(size_t)b * E + e] = tot;
      tot += c;
    }
  int total, act_total;
  const int off = block_exclusive_scan(e < E ? tot : 0, scratch, &total);
  const int act = block_exclusive_scan((e < E && tot > 0) ? 1 : 0, scratch, &act_total);
  if (e < E) {
    offsets[e] = off;
    if (tot > 0) active[act] = e;
    for (int b = 0; b < n_chunks; ++b) cnt[(size_t)b * E + e] += off;
  }
  if (e == 0) {
    offsets[E] = total;
    *n_active = act_total;
  }
}

__global__ void __launch_bounds__(kChunkThreads)
csr_place_kernel(const int32_t* __restrict__ ids, int P, int E, const int32_t* __restrict__ cnt,
                 int32_t* __restrict__ pair_ids, int32_t* __restrict__ pair_pos) {
  extern __shared__ int wh[];                  // [kChunkWarps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kChunkWarps * E; i += kChunkThreads) wh[i] = 0;
  pdl_wait();                                  // the chunk starts are complete
  pdl_trigger();
  __syncthreads();
  const int p0 = blockIdx.x * kChunkPairs, p1 = min(P, p0 + kChunkPairs);
  const int slice = (p1 - p0 + kChunkWarps - 1) / kChunkWarps;
  const int s0 = min(p1, p0 + warp * slice), s1 = min(p1, s0 + slice);
  int* my = wh + warp * E;
  for (int p = s0 + lane; p < s1; p += 32) {
    const int e = __ldg(ids + p);
    if (e >= 0 && e < E) atomicAdd(&my[e], 1);
  }
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
  for (int base = s0; base < s1; base += 32) {
    const int p = base + lane;
    const bool in = p < s1;
    int e = in ? __ldg(ids + p) : -1;
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
// pairs of its expert is the number of earlier pairs with the same expert.
constexpr int kCsrSmallPairs = 256;

__global__ void __launch_bounds__(kCsrThreads, 1)
csr_small_kernel(const int32_t* __restrict__ ids_g, int P, int E, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ pair_ids, int32_t* __restrict__ active,
                 int32_t* __restrict__ n_active, int32_t* __restrict__ pair_pos,
                 uint32_t* __restrict__ err) {
  __shared__ int hist[kMaxE];
  __shared__ int ids_s[kCsrSmallPairs];
  __shared__ int scratch[kCsrWarps];
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
  int total, act_total;
  const int off = block_exclusive_scan(cnt, scratch, &total);
  const int act = block_exclusive_scan((tid < E && cnt > 0) ? 1 : 0, scratch, &act_total);
  if (tid < E) {
    offsets[tid] = off;
    hist[tid] = off;
    if (cnt > 0) active[act] = tid;
  }
  if (tid == 0) {
    offsets[E] = total;
    *n_active = act_total;
  }
  __syncthreads();
  if (valid) {
    int rank = 0;
    for (int q = 0; q < tid; ++q) rank += ids_s[q] == e;
    const int pos = hist[e] + rank;
    pair_ids[pos] = tid;
    pair_pos[tid] = pos;
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t s) {
  const dim3 grid(T), block(32);
  const int pl = (E + 31) / 32;
  // wider routers: sort per token (the warp version runs k dependent rounds of shuffles)
  if (E > 64) {
    if (E <= 128) return launch_pdl(route_sort_kernel<128>, grid, dim3(64), 0, s, logits, T, E, k, ids, w);
    if (E <= 256) return launch_pdl(route_sort_kernel<256>, grid, dim3(128), 0, s, logits, T, E, k, ids, w);
    if (E <= 512) return launch_pdl(route_sort_kernel<512>, grid, dim3(256), 0, s, logits, T, E, k, ids, w);
    return launch_pdl(route_sort_kernel<1024>, grid, dim3(512), 0, s, logits, T, E, k, ids, w);
  }
  if (pl <= 1) return launch_pdl(route_topk_kernel<1>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (pl <= 2) return launch_pdl(route_topk_kernel<2>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (pl <= 4) return launch_pdl(route_topk_kernel<4>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (pl <= 8) return launch_pdl(route_topk_kernel<8>, grid, block, 0, s, logits, T, E, k, ids, w);
  if (pl <= 16) return launch_pdl(route_topk_kernel<16>, grid, block, 0, s, logits, T, E, k, ids, w);
  return launch_pdl(route_topk_kernel<32>, grid, block, 0, s, logits, T, E, k, ids, w);
}

size_t csr_scratch_bytes(int P, int E) {
  if (P < kCsrGridMinPairs) return 0;
  return (size_t)((P + kChunkPairs - 1) / kChunkPairs) * E * sizeof(int32_t);
}

cudaError_t launch_build_csr(const int32_t* ids, int P, int k, int E, moe_csr csr,
                             int32_t* pair_pos, uint32_t* err, int32_t* scratch, cudaStream_t s) {
  (void)k;
  if (P <= kCsrSmallPairs)
    return launch_pdl(csr_small_kernel, dim3(1), dim3(kCsrThreads), 0, s, ids, P, E,
                      csr.expert_offsets, csr.pair_ids, csr.active_experts, csr.n_active, pair_pos, err);
  if (P >= kCsrGridMinPairs && scratch) {
    const int nb = (P + kChunkPairs - 1) / kChunkPairs;
    cudaError_t st = launch_pdl(csr_count_kernel, dim3(nb), dim3(kChunkThreads),
                                (size_t)E * sizeof(int), s, ids, P, E, scratch, pair_pos, err);
    if (st != cudaSuccess) return st;
    st = launch_pdl(csr_scan_kernel, dim3(1), dim3(kCsrThreads), 0, s, scratch, nb, E,
                    csr.expert_offsets, csr.active_experts, csr.n_active);
    if (st != cudaSuccess) return st;
    const size_t smem = (size_t)kChunkWarps * E * sizeof(int);
    st = cudaFuncSetAttribute(csr_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (st != cudaSuccess) return st;
    return launch_pdl(csr_place_kernel, dim3(nb), dim3(kChunkThreads), smem, s, ids, P, E,
                      (const int32_t*)scratch, csr.pair_ids, pair_pos);
  }
  size_t smem = (size_t)(kCsrWarps * E + kCsrWarps) * sizeof(int);
  const int ids_in_smem = smem + (size_t)P * sizeof(int) <= 200 * 1024 ? 1 : 0;
  if (ids_in_smem) smem += (size_t)P * sizeof(int);
  cudaError_t st = cudaFuncSetAttribute(build_csr_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (st != cudaSuccess) return st;
  return launch_pdl(build_csr_kernel, dim3(1), dim3(kCsrThreads), smem, s, ids, P, E,
                    csr.expert_offsets, csr.pair_ids, csr.active_experts, csr.n_active, pair_pos,
                    err, ids_in_smem);
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
                                    nullptr, static_cast<cudaStream_t>(stream));
  return st == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
