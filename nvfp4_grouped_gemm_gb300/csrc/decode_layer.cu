// The decode layer as one kernel: top-k routing, the expert-first CSR, gate/up + SiLU, down
// and the routing-weighted combine in one cooperative grid (one CTA per SM), for decode
// batches below the tensor-core switch (fewer than moe_decode_tensor_core_min_pairs()
// pairs) with at most kLayerMaxT tokens and F <= 640.
//
// The per-call path runs seven kernels; at a few tokens its time is the chain of their
// latencies (launch, first loads, the drain of each grid), not the HBM bytes.  Here:
//   - every CTA routes all T tokens itself (a warp per token, each lane's keys in
//     registers) and builds the CSR in shared memory, so nothing grid-wide comes before
//     the weight stream; meanwhile one warp per token somewhere in the grid converts that
//     token's x row to f16 (the gate/up units read activation rows per token);
//   - the TMA producers then stream every consumer ring's gate/up stages and, right after
//     them, its down stages (the units of decode_units.cuh), so the down weights are in
//     flight while gate/up finishes;
//   - the consumer warps run  gate/up -> h rows to f16 -> down -> combine,  after a count
//     of the converted x rows and between three grid-wide barriers (h ready, f16 h
//     ready, partials ready): the only points where CTAs wait on one another, each wait
//     bounded by the 2 s budget of the other waits.  The counters only grow, against a
//     per-call epoch in the workspace, so a call needs no reset before it.
// A producer issues all gate/up stages of its consumers before any down stage, so it only
// ever waits for a ring whose consumer still has stages of the current phase to take: a
// ring full of down stages whose consumer waits at a barrier cannot hold up the gate/up
// stages another consumer needs to reach that barrier.
//
// Every step's arithmetic is that of the per-call kernels: the routing kernel's keys and
// weights, and the TMA-fed decode kernels' f16 prescales, units (each unit's K order) and
// combine (ascending j).  The picks and weights are therefore bit-identical to the routing
// call's, and y to the per-call path's wherever that path runs its TMA-fed kernels (from 8
// units per SM); below that it runs CTA kernels that sum K in another order.
#include "decode_units.cuh"

namespace moe {

namespace {

constexpr int kLayerThreads = 32 * (kTmaProd + kTmaWarps);
constexpr int kLayerSlots = kTmaWarps * kTmaSlots;     // stage slots of the CTA
constexpr int kLayerMaxT = 32;                         // tokens routed by every CTA
constexpr int kLayerMaxP = 256;                        // pairs (below the tensor-core switch)
constexpr int kLayerMaxF = 640;                        // a down stage fits one slot
// sync words (u64): the call epoch, three barrier counters, the x-rows counter, the abort word
constexpr int kLayerSyncWords = 6;

struct LayerArgs {
  const float* logits;   // [T][E] f32, or null: ids / w are inputs
  int32_t* ids;          // [T*k] picks (written when routing)
  float* w;              // [T*k] routing weights (written when routing)
  const uint16_t* x;     // bf16 [T][H]
  float* y;              // f32 [T][H]
  __half* xg;            // f16 [T][H] x rows (one per token), times 2^-xe
  int32_t* xe;
  __half* hg;            // f16 [P][F] h rows times 2^-he
  int32_t* he;
  int T, E, k;
  int slot_bytes;        // stride of the stage slots
  int n_cons, slog;      // consumer warps that take units, log2 of their ring length
  GuTmaArgs gu;          // xg / xe / h / err; the CSR pointers are set per CTA
  DnTmaArgs dn;          // hg / he / partial / banks; the CSR pointers are set per CTA
  unsigned long long* sync;   // [kLayerSyncWords], zero before the first call
};

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// the consumer warps of the CTA (named barrier 1)
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kTmaWarps) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu(unsigned long long* p) {
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}

// Wait (bounded) until *cnt reaches target; on the 2 s budget, or when another CTA has
// given up (the abort word), flag MOE_DEVERR_TIMEOUT, poison the sync words and stop.
__device__ __forceinline__ void wait_count(const unsigned long long* cnt, unsigned long long target,
                                           unsigned long long* abort_word,
                                           volatile int* abort_flag, uint32_t* err) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1; ld_acquire_gpu(cnt) < target; ++it) {
    if ((it & 63) == 0 && (ld_acquire_gpu(abort_word) != 0ull || global_ns() - t0 > kWaitBudgetNs)) {
      *abort_flag = 1;
      atomicOr(err, (uint32_t)MOE_DEVERR_TIMEOUT);
      atomicExch(abort_word, 1ull);
      return;
    }
  }
}

// Grid-wide barrier of the consumer warps.  The counters only grow: every call adds
// gridDim.x to each, so call e (the epoch every CTA read at its start) waits for
// (e + 1) * gridDim.x.  After the CTA's consumers meet, its first consumer thread arrives
// with a release reduction (publishing what the CTA wrote) and polls with acquire loads.
// A CTA that stopped early still arrives.
__device__ __forceinline__ void grid_barrier(unsigned long long* cnt, unsigned long long epoch,
                                             unsigned long long* abort_word,
                                             volatile int* abort_flag, uint32_t* err) {
  consumers_sync();
  if (threadIdx.x == 32 * kTmaProd) {
    red_release_gpu(cnt);
    wait_count(cnt, (epoch + 1) * gridDim.x, abort_word, abort_flag, err);
  }
  consumers_sync();
}

template <int NB, bool ALPHA>
__global__ void __launch_bounds__(kLayerThreads, 1)
decode_layer_kernel(const __grid_constant__ CUtensorMap tmap_c,
                    const __grid_constant__ CUtensorMap tmap_s, const LayerArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int SB = a.slot_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kLayerSlots * SB);
  uint64_t* empty = full + kLayerSlots;
  int* s_misc = reinterpret_cast<int*>(empty + kLayerSlots);   // abort flag, n_active
  volatile int* abort_flag = s_misc;
  int* s_ids = s_misc + 4;                                     // [P] picks
  float* s_w = reinterpret_cast<float*>(s_ids + kLayerMaxP);   // [P] routing weights
  int* s_pos = reinterpret_cast<int*>(s_w + kLayerMaxP);       // [P] CSR position, -1 if none
  int* s_rowtok = s_pos + kLayerMaxP;                          // [P] token of each CSR row
  int* s_off = s_rowtok + kLayerMaxP;                          // [E+1] expert offsets
  int* s_active = s_off + (kMaxE + 1);                         // [E] active experts
  int* s_run = s_active + kMaxE;                               // [E] next row of each expert
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, k = a.k, P = T * k;
  const int H = a.gu.H, F = a.gu.F;

  unsigned long long* const epoch_word = a.sync;
  unsigned long long* const abort_word = a.sync + 5;
  // the call's epoch (advanced by CTA 0 at the end of every completed call); a call after
  // one that gave up finds the sync words poisoned and does nothing but report it
  const unsigned long long epoch = *reinterpret_cast<volatile unsigned long long*>(epoch_word);
  if (*reinterpret_cast<volatile unsigned long long*>(abort_word) != 0ull) {
    if (threadIdx.x == 0) atomicOr(a.gu.err, (uint32_t)MOE_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kLayerSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---------------- x rows to f16, one per token ----------------
  // They do not depend on the routing: token t's row is converted by the last warp of CTA
  // G-1-t (a warp that routes no token while T < 20) while the CTAs route.
  if (warp == kLayerThreads / 32 - 1)
    for (int t = (int)gridDim.x - 1 - (int)blockIdx.x; t < T; t += (int)gridDim.x) {
      const int ex = x_row_f16_store(a.x + (size_t)t * H, H, lane, a.xg + (size_t)t * H);
      if (lane == 0) a.xe[t] = ex;
      __threadfence();
      __syncwarp();
      if (lane == 0) red_release_gpu(a.sync + 4);        // one more x row ready
    }

  // ---------------- routing: every CTA routes all T tokens ----------------
  // a warp per token: round j takes the largest key below the previous pick (keys are
  // distinct), so lane j ends with the j-th pick; weights as the routing kernel forms them
  auto finish_token = [&](int t, unsigned long long mine) {
    const float first_v = key_logit(__shfl_sync(0xffffffffu, mine, 0));
    const float ex = (lane < k) ? expf(key_logit(mine) - first_v) : 0.0f;
    // sum in ascending j so every lane sees the same value
    float denom = 0.0f;
    for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
      s_ids[t * k + lane] = key_id(mine);
      s_w[t * k + lane] = ex / denom;
    }
  };
  if (a.logits && E <= 512) {
    // each lane's 16 keys in registers, straight from global memory
    for (int t = warp; t < T; t += kLayerThreads / 32) {
      const float* lr = a.logits + (size_t)t * E;
      unsigned long long key[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? route_key(lr[e], e) : 0ull;
      }
      unsigned long long prev = ~0ull, mine = 0ull;
      for (int j = 0; j < k; ++j) {
        // four independent chains over the lane's keys, then their maximum
        unsigned long long b4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int i = 0; i < 16; ++i)
          b4[i & 3] = (key[i] < prev && key[i] > b4[i & 3]) ? key[i] : b4[i & 3];
        unsigned long long best = umax64(umax64(b4[0], b4[1]), umax64(b4[2], b4[3]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
        if (lane == j) mine = best;
        prev = best;
      }
      finish_token(t, mine);
    }
  } else if (a.logits) {
    // wider routers: the logits staged in the (not yet used) stage slots
    float* s_logits = reinterpret_cast<float*>(smem);
    for (int i = threadIdx.x; i < T * E; i += kLayerThreads) s_logits[i] = a.logits[i];
    __syncthreads();
    for (int t = warp; t < T; t += kLayerThreads / 32) {
      const float* lr = s_logits + (size_t)t * E;
      unsigned long long prev = ~0ull, mine = 0ull;
      for (int j = 0; j < k; ++j) {
        unsigned long long best = 0ull;
        for (int e = lane; e < E; e += 32) {
          const unsigned long long key = route_key(lr[e], e);
          if (key < prev && key > best) best = key;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
        if (lane == j) mine = best;
        prev = best;
      }
      finish_token(t, mine);
    }
  } else {
    for (int p = threadIdx.x; p < P; p += kLayerThreads) {
      s_ids[p] = a.ids[p];
      s_w[p] = a.w[p];
    }
  }
  for (int e = threadIdx.x; e <= E; e += kLayerThreads) s_off[e] = 0;
  __syncthreads();
  if (a.logits && blockIdx.x == 0)
    for (int p = threadIdx.x; p < P; p += kLayerThreads) {
      a.ids[p] = s_ids[p];
      a.w[p] = s_w[p];
    }

  // ---------------- CSR in shared memory ----------------
  for (int p = threadIdx.x; p < P; p += kLayerThreads) {
    const int e = s_ids[p];
    if (e >= 0 && e < E) atomicAdd(&s_off[e], 1);
    else if (blockIdx.x == 0) atomicOr(a.gu.err, (uint32_t)MOE_DEVERR_EXPERT_ID);
  }
  __syncthreads();
  if (warp == 0) {
    // counts -> exclusive offsets and the ascending active list; lane l owns a chunk
    const int ch = (E + 31) / 32, e0 = min(E, lane * ch), e1 = min(E, e0 + ch);
    int cnt[kMaxE / 32];
    int sum = 0, nact = 0;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      cnt[i] = e0 + i < e1 ? s_off[e0 + i] : 0;
      sum += cnt[i];
      nact += cnt[i] > 0 ? 1 : 0;
    }
    int isum = sum, iact = nact;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u1 = __shfl_up_sync(0xffffffffu, isum, o), u2 = __shfl_up_sync(0xffffffffu, iact, o);
      if (lane >= o) { isum += u1; iact += u2; }
    }
    int run = isum - sum, arun = iact - nact;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      if (e0 + i < e1) {
        s_off[e0 + i] = run;
        s_run[e0 + i] = run;
        if (cnt[i] > 0) s_active[arun++] = e0 + i;
      }
      run += cnt[i];
    }
    if (lane == 31) {
      s_off[E] = isum;
      s_misc[1] = iact;
    }
    __syncwarp();
    // rows in ascending p within an expert: 32 pairs at a time, equal experts matched
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + lane;
      const int e = p < P ? s_ids[p] : -1;
      const bool valid = e >= 0 && e < E;
      const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
      const int pos = valid ? s_run[e] + __popc(peers & ((1u << lane) - 1u)) : -1;
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) s_run[e] += __popc(peers);
      if (p < P) s_pos[p] = pos;
      if (valid) s_rowtok[pos] = p / k;
      __syncwarp();
    }
  }
  __syncthreads();

  GuTmaArgs gu = a.gu;
  gu.offsets = s_off;
  gu.active = s_active;
  gu.n_active = s_misc + 1;
  gu.row_tok = s_rowtok;
  DnTmaArgs dn = a.dn;
  dn.offsets = s_off;
  dn.active = s_active;
  dn.n_active = s_misc + 1;
  const int n_act = s_misc[1], nrows = s_off[E];
  // this CTA's contiguous (expert-major) ranges of the gate/up and down units
  const int gu_units = n_act * (F / 8), dn_units = n_act * (H / 16);
  const int gb = (int)((long long)blockIdx.x * gu_units / gridDim.x);
  const int ge = (int)((long long)(blockIdx.x + 1) * gu_units / gridDim.x);
  const int db = (int)((long long)blockIdx.x * dn_units / gridDim.x);
  const int de = (int)((long long)(blockIdx.x + 1) * dn_units / gridDim.x);
  const int nc = a.n_cons, slog = a.slog;

  constexpr int PER = kTmaWarps / kTmaProd;
  if (warp < kTmaProd) {
    // ---------------- producers: warp p feeds consumers p*PER .. p*PER+PER-1 ----------------
    if (lane == 0) {
      const int w0 = warp * PER;
      GuCursor gc[PER];
      DnCursor dc[PER];
      for (int i = 0; i < PER; ++i) gc[i] = GuCursor{gb + w0 + i, 0, 0, 0};
      bool more = true, ok = true, down = false;
      while (more && ok) {                           // every gate/up stage first
        more = false;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          if (!ok) break;
          if (w0 + i >= nc || gc[i].u >= ge) continue;
          more = true;
          ok = gu_issue(gu, &tmap_c, &tmap_s, gc[i], nc, smem, SB, full, empty,
                        Ring{(w0 + i) << slog, slog}, abort_flag);
        }
      }
      if (ok) {
        down = true;
        for (int i = 0; i < PER; ++i) dc[i] = DnCursor{db + w0 + i, 0, gc[i].q};
        more = true;
        while (more && ok) {                         // then the down stages, rings continuing
          more = false;
#pragma unroll
          for (int i = 0; i < PER; ++i) {
            if (!ok) break;
            if (w0 + i >= nc || dc[i].u >= de) continue;
            more = true;
            ok = dn_issue(dn, dc[i], nc, smem, SB, full, empty, Ring{(w0 + i) << slog, slog},
                          abort_flag);
          }
        }
      }
      // drain, bounded: every issued stage has landed before the CTA exits
      if (!ok)
        for (int i = 0; i < PER; ++i)
          if (w0 + i < nc)
            ring_drain(full, Ring{(w0 + i) << slog, slog}, down ? dc[i].q : gc[i].q);
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int cw = warp - kTmaProd;
  const int gw = blockIdx.x * kTmaWarps + cw, nw = gridDim.x * kTmaWarps;
  const Ring ring{cw << slog, slog};
  int q = 0;
  // every token's x row converted (one count each)
  if (threadIdx.x == 32 * kTmaProd) wait_count(a.sync + 4, (epoch + 1) * T, abort_word, abort_flag, gu.err);
  consumers_sync();
  if (cw < nc)
    for (int u = gb + cw; u < ge && !*abort_flag; u += nc)
      if (!gu_consume_unit<NB, ALPHA, false, true>(gu, u, smem, SB, full, empty, ring, q, abort_flag))
        break;
  grid_barrier(a.sync + 1, epoch, abort_word, abort_flag, gu.err);   // h complete
  // h rows to f16 (a warp per CSR row)
  for (int r = gw; r < nrows; r += nw)
    h_row_f16<kLayerMaxF / 128>(gu.h + (size_t)r * F, F, lane, a.hg + (size_t)r * F, a.he + r);
  grid_barrier(a.sync + 2, epoch, abort_word, abort_flag, gu.err);   // f16 h complete
  if (cw < nc)
    for (int u = db + cw; u < de && !*abort_flag; u += nc)
      if (!dn_consume_unit<false>(dn, u, smem, SB, full, empty, ring, q, abort_flag)) break;
  grid_barrier(a.sync + 3, epoch, abort_word, abort_flag, gu.err);   // partials complete
  // combine: four columns of one token per thread, in ascending j
  const int H4 = H / 4;
  for (int i = blockIdx.x * 32 * kTmaWarps + (threadIdx.x - 32 * kTmaProd); i < T * H4;
       i += gridDim.x * 32 * kTmaWarps) {
    const int t = i / H4, r = 4 * (i % H4);
    *reinterpret_cast<float4*>(a.y + (size_t)t * H + r) =
        combine4(dn.partial, s_pos + t * k, s_w + t * k, k, H, r);
  }
  // every CTA has passed the last barrier, so no wait of this call reads the epoch again:
  // CTA 0 opens the next one; a CTA that gave up poisons the words instead
  consumers_sync();
  if (threadIdx.x == 32 * kTmaProd) {
    if (*abort_flag) atomicExch(abort_word, 1ull);
    else if (blockIdx.x == 0) *reinterpret_cast<volatile unsigned long long*>(epoch_word) = epoch + 1;
  }
}

// K-chunking of the gate/up rows as in the per-call kernel: chunks of nb <= 2 boxes of 128
// bytes, H/256 = nh * nb
void gu_chunks(int H, int* nh, int* nb) {
  const int n256 = H / 256;
  int c = 1;
  while (n256 % c != 0 || n256 / c > 2) ++c;
  *nh = c;
  *nb = n256 / c;
}

int slot_bytes_for(int H, int F) {
  int nh, nb;
  gu_chunks(H, &nh, &nb);
  const int g = gu_stage_bytes(nb), d = dn_stage_bytes(F);
  return g > d ? g : d;
}

size_t layer_smem(int slot_bytes) {
  return 1024 + (size_t)kLayerSlots * slot_bytes + 2 * kLayerSlots * 8 + 16 +
         4 * kLayerMaxP * 4 + (3 * kMaxE + 1) * 4;
}

template <int NB, bool ALPHA>
cudaError_t run_layer(const CUtensorMap& mc, const CUtensorMap& ms, const LayerArgs& a,
                      size_t smem, cudaStream_t s) {
  auto kern = decode_layer_kernel<NB, ALPHA>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (st != cudaSuccess) return st;
  // every CTA must be resident at once (the grid waits on itself): one per SM
  int per_sm = 0;
  st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLayerThreads, smem);
  if (st != cudaSuccess) return st;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms());
  cfg.blockDim = dim3(kLayerThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mc, ms, a);
}

template <int NB>
cudaError_t run_layer_alpha(bool alpha, const CUtensorMap& mc, const CUtensorMap& ms,
                            const LayerArgs& a, size_t smem, cudaStream_t s) {
  return alpha ? run_layer<NB, true>(mc, ms, a, smem, s) : run_layer<NB, false>(mc, ms, a, smem, s);
}

}  // namespace

bool decode_layer_supported(int T, int H, int F, int E, int k) {
  const long long P = (long long)T * k;
  if (T < 1 || T > kLayerMaxT || P >= kLayerMaxP || decode_sliced(P)) return false;
  if (E > kMaxE || k > kMaxK || H % 256 != 0 || H > 4096) return false;
  if (F % 128 != 0 || F > kLayerMaxF) return false;
  const int sb = slot_bytes_for(H, F);
  // the logits of all tokens are staged in the slots
  if ((long long)T * E * 4 > (long long)kLayerSlots * sb) return false;
  return layer_smem(sb) <= 232448;
}

size_t decode_layer_sync_bytes() { return kLayerSyncWords * sizeof(unsigned long long); }

cudaError_t launch_decode_layer(const float* logits, int32_t* ids, float* w, const uint16_t* x,
                                int T, int H, int F, int k, const moe_nvfp4_bank& gub,
                                const moe_nvfp4_bank& dnb, const moe_ws_layout& L, char* ws,
                                float* y, cudaStream_t s) {
  const int E = gub.E;
  int nh, nb;
  gu_chunks(H, &nh, &nb);
  const int n256 = H / 256;
  // gate/up banks as [K-box][E*2 matrices][F rows][bytes of the K-box] (row pitch H/2, H/16)
  CUtensorMap mc, ms;
  const uint64_t cdims[4] = {128, (uint64_t)F, 2 * (uint64_t)E, (uint64_t)n256};
  const uint64_t cstr[3] = {(uint64_t)H / 2, (uint64_t)F * (H / 2), 128};
  const uint32_t cbox[4] = {128, 8, 2, (uint32_t)nb};
  const uint64_t sdims[4] = {16, (uint64_t)F, 2 * (uint64_t)E, (uint64_t)n256};
  const uint64_t sstr[3] = {(uint64_t)H / 16, (uint64_t)F * (H / 16), 16};
  const uint32_t sbox[4] = {16, 8, 2, (uint32_t)nb};
  if (!make_map4(&mc, gub.codes, cdims, cstr, cbox, true) ||
      !make_map4(&ms, gub.scales, sdims, sstr, sbox, false))
    return cudaErrorInvalidValue;

  LayerArgs a{};
  a.logits = logits;
  a.ids = ids;
  a.w = w;
  a.x = x;
  a.y = y;
  a.xg = reinterpret_cast<__half*>(ws + L.xg);
  a.xe = reinterpret_cast<int32_t*>(ws + L.xe);
  a.hg = reinterpret_cast<__half*>(ws + L.hg);
  a.he = reinterpret_cast<int32_t*>(ws + L.he);
  a.T = T;
  a.E = E;
  a.k = k;
  a.slot_bytes = slot_bytes_for(H, F);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws + L.error_word);
  a.gu = GuTmaArgs{a.xg, a.xe, H, F, nh, nb, nullptr, nullptr, nullptr,
                   reinterpret_cast<float*>(ws + L.h), err};
  a.gu.alpha = gub.alpha;
  a.dn = DnTmaArgs{a.hg, a.he, dnb.codes, dnb.scales, H, F, nullptr, nullptr, nullptr,
                   reinterpret_cast<float*>(ws + L.partial), err};
  a.dn.alpha = dnb.alpha;
  a.sync = reinterpret_cast<unsigned long long*>(ws + L.sync);
  // consumers that take units: few units per CTA go to fewer warps with longer rings, so
  // that most of the CTA's stages are in flight at once
  const long long P = (long long)T * k;
  const long long units = (P < E ? P : E) * (F / 8);
  const long long per_cta = (units + num_sms() - 1) / num_sms();
  a.n_cons = per_cta <= 4 ? 4 : per_cta <= 12 ? 8 : 16;
  a.slog = a.n_cons == 4 ? 3 : a.n_cons == 8 ? 2 : 1;

  const size_t smem = layer_smem(a.slot_bytes);
  const bool al = gub.alpha != nullptr;
  return nb == 1 ? run_layer_alpha<1>(al, mc, ms, a, smem, s)
                 : run_layer_alpha<2>(al, mc, ms, a, smem, s);
}

}  // namespace moe
