// Host side of the C ABI: argument validation, workspace layout and kernel launches.
#include <atomic>
#include <cstring>

#include "moe_internal.cuh"

namespace moe {

int num_sms() {
  constexpr int kCachedDevices = 64;
  static std::atomic<int> cache[kCachedDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  int n = (dev >= 0 && dev < kCachedDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 1;
  if (dev >= 0 && dev < kCachedDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool sizes_ok(int T, int H, int F, int E, int k) {
  if (T <= 0 || H <= 0 || F <= 0 || E <= 0 || k <= 0) return false;
  return true;
}

moe_status sizes_supported(int T, int H, int F, int E, int k) {
  if (!sizes_ok(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (k > E) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (H % 256 != 0 || H > 4096 || F % 64 != 0) return MOE_ERR_UNSUPPORTED;
  const long long P = (long long)T * k;
  const long long big = H > F ? H : F;
  if (P * big >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// A prepacked scale plane (sf_atoms) must be 16-byte aligned and written in the row order
// of the call it is passed to: `order`.
moe_status check_bank(const moe_nvfp4_bank* b, int E_expected, int rows, int in_f, int order) {
  if (!b || !b->codes || !b->scales) return MOE_ERR_INVALID_ARG;
  if (!aligned16(b->codes) || !aligned16(b->scales)) return MOE_ERR_INVALID_ARG;
  if (b->rows != rows || b->in_f != in_f || b->E <= 0) return MOE_ERR_INVALID_ARG;
  if (E_expected > 0 && b->E != E_expected) return MOE_ERR_INVALID_ARG;
  if (b->sf_atoms && (!aligned16(b->sf_atoms) || b->sf_atoms_order != order))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_csr(const moe_csr& c) {
  if (!c.expert_offsets || !c.pair_ids || !c.active_experts || !c.n_active)
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_ws(const void* ws, size_t ws_bytes, const moe_ws_layout& L) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

int resolve_path(int T, int k, int path) {
  if (path == MOE_PATH_DECODE || path == MOE_PATH_PREFILL) return path;
  return (long long)T * k >= kPrefillMinPairs ? MOE_PATH_PREFILL : MOE_PATH_DECODE;
}

// The per-path limit on F (the path AUTO resolves to for these sizes).
// The sliced down GEMM stages each weight row's F/16 scale bytes whole, through a tensor
// map whose rows are g consecutive scale rows (g the smallest power of two with g*F/16 a
// multiple of 16 and at least 32 bytes); a tensor-map box row holds at most 256 bytes.
bool sliced_down_supported(int F) {
  const int sfrow = F / 16;
  int g = 1;
  if (sfrow % 16 != 0)
    for (g = 2; (g * sfrow) % 16 != 0 || g * sfrow < 32; g *= 2) {
    }
  return 128 % g == 0 && g * sfrow <= 256 && 128 * sfrow <= 11264;
}

moe_status path_supported(int T, int F, int k, int path) {
  if (path != MOE_PATH_AUTO && path != MOE_PATH_DECODE && path != MOE_PATH_PREFILL)
    return MOE_ERR_INVALID_ARG;
  const int p = resolve_path(T, k, path);
  if (p == MOE_PATH_DECODE && F > kDecodeMaxF) return MOE_ERR_UNSUPPORTED;
  if (p == MOE_PATH_DECODE && decode_sliced((long long)T * k) && !sliced_down_supported(F))
    return MOE_ERR_UNSUPPORTED;                    // F = 1088, 1216, 1344
  if (p == MOE_PATH_PREFILL && F > kPrefillMaxF) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool compute_layout(int T, int H, int F, int E, int k, int path, moe_ws_layout* L) {
  std::memset(L, 0, sizeof(*L));
  if (sizes_supported(T, H, F, E, k) != MOE_OK) return false;
  if (path_supported(T, F, k, path) != MOE_OK) return false;
  path = resolve_path(T, k, path);
  const size_t P = (size_t)T * k;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L->error_word = take(sizeof(uint32_t));
  L->pair_pos = take(P * sizeof(int32_t));
  // both tile lists, written by the CSR call whatever the path (their place depends only on
  // P and E, so the CSR call finds them without knowing H, F or the path)
  L->tiles = take(tile_list_bytes((long long)P, 1, kTileRows, E));
  L->slice_tiles = take(tile_list_bytes((long long)P, kDecodeSlices, kSliceTileRows, E));
  L->h = take(P * F * sizeof(float));
  L->partial = take(P * H * sizeof(float));
  if (path == MOE_PATH_DECODE && !decode_sliced((long long)P)) {
    L->xg = take(P * H * 2);
    L->xe = take(P * sizeof(int32_t));
    L->hg = take(P * F * 2);
    L->he = take(P * sizeof(int32_t));
    L->row_tok = take(P * sizeof(int32_t));
    L->sync = take(decode_layer_sync_bytes());
  } else {
    // operand rows per pair: the sliced decode form keeps kDecodeSlices slices of each row
    const bool sl = path == MOE_PATH_DECODE;
    const size_t R = P * (sl ? kDecodeSlices : 1);
    L->qx_codes = take(R * (H / 2));
    L->qx_scales = take(R * (H / 16));
    L->qx_exp = take(R * sizeof(int32_t));
    L->qh_codes = take(R * (F / 2));
    L->qh_scales = take(R * qh_scale_pitch(F));
    L->qh_exp = take(R * sizeof(int32_t));
  }
  L->total = o;
  return true;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k, int32_t path) {
  moe_ws_layout L;
  if (!compute_layout(T, H, F, E, k, path, &L)) return 0;
  return L.total;
}

moe_status moe_workspace_layout(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k,
                                int32_t path, moe_ws_layout* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  moe_status st = sizes_supported(T, H, F, E, k);
  if (st != MOE_OK) return st;
  if ((st = path_supported(T, F, k, path)) != MOE_OK) return st;
  if (!compute_layout(T, H, F, E, k, path, out)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int32_t moe_prefill_min_pairs(void) { return kPrefillMinPairs; }

int32_t moe_decode_tensor_core_min_pairs(void) { return kSlicedMinPairs; }

int32_t moe_resolve_path(int32_t T, int32_t k, int32_t path) { return resolve_path(T, k, path); }

int32_t moe_kernel_launches(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k, int32_t path) {
  moe_ws_layout L;
  if (!compute_layout(T, H, F, E, k, path, &L)) return 0;
  const int P = T * k;
  const int csr = csr_scratch_bytes(P, E) ? 3 : 1;   // grid-wide build or one CTA
  if (resolve_path(T, k, path) == MOE_PATH_DECODE)
    return decode_sliced(P) ? csr + 2 /* x slices, gate/up */ + 3 /* h slices, down, combine */
                            : csr + 2 /* x gather, gate/up */ + 3 /* h prep, down, combine */;
  return csr + 2 /* Q(x), gate/up GEMM */ + 3 /* Q(h), down GEMM, combine */;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                          int32_t* topk_ids, float* topk_w, void* stream) {
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (T <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * E >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  return from_cuda(launch_route_topk(logits, T, E, k, topk_ids, topk_w,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status moe_build_expert_csr(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                                moe_csr csr, void* ws, size_t ws_bytes, void* stream) {
  if (!topk_ids) return MOE_ERR_INVALID_ARG;
  if (T <= 0 || k <= 0 || E <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  moe_status st = check_csr(csr);
  if (st != MOE_OK) return st;
  if ((long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  // the CSR needs only the error word and pair_pos, which sit at the same offsets for
  // every (H, F, path); validate against the smallest legal layout
  moe_ws_layout L;
  if (!compute_layout(T, 256, 64, E, k, MOE_PATH_DECODE, &L)) return MOE_ERR_UNSUPPORTED;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < L.h) return MOE_ERR_WORKSPACE;            // error word, pair_pos, tile lists
  // many pairs: the grid-wide build keeps per-chunk counts in the h region (written only
  // later, by the gate/up call); it needs that much workspace
  const size_t scratch = csr_scratch_bytes(T * k, E);
  if (scratch && ws_bytes < L.h + scratch) return MOE_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  return from_cuda(launch_build_csr(topk_ids, T * k, k, E, csr,
                                    reinterpret_cast<int32_t*>(w + L.pair_pos),
                                    reinterpret_cast<uint32_t*>(w + L.error_word),
                                    scratch ? reinterpret_cast<int32_t*>(w + L.h) : nullptr,
                                    reinterpret_cast<int32_t*>(w + L.tiles),
                                    reinterpret_cast<int32_t*>(w + L.slice_tiles),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gate_up_silu_nvfp4(const void* x_bf16, int32_t T, int32_t H, int32_t F,
                                          int32_t k, const moe_nvfp4_bank* w_gate_up,
                                          moe_csr csr, int32_t path, void* ws, size_t ws_bytes,
                                          void* stream) {
  if (!x_bf16 || !aligned16(x_bf16)) return MOE_ERR_INVALID_ARG;
  if (!w_gate_up) return MOE_ERR_INVALID_ARG;
  const int E = w_gate_up->E;
  moe_status st = sizes_supported(T, H, F, E, k);
  if (st != MOE_OK) return st;
  if ((st = path_supported(T, F, k, path)) != MOE_OK) return st;
  if ((st = check_bank(w_gate_up, E, 2 * F, H, MOE_SF_ATOMS_GATE_UP)) != MOE_OK) return st;
  if ((st = check_csr(csr)) != MOE_OK) return st;
  moe_ws_layout L;
  if (!compute_layout(T, H, F, E, k, path, &L)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, L)) != MOE_OK) return st;
  const int p = resolve_path(T, k, path);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p == MOE_PATH_PREFILL) {
    bool unsup = false;
    cudaError_t ce = launch_prefill_gate_up(static_cast<const uint16_t*>(x_bf16), T, H, F, k,
                                            *w_gate_up, csr, L, static_cast<char*>(ws), s, &unsup);
    if (unsup) return MOE_ERR_UNSUPPORTED;
    return from_cuda(ce);
  }
  if (decode_sliced((long long)T * k))
    return from_cuda(launch_sliced_gate_up(static_cast<const uint16_t*>(x_bf16), T, H, F, k,
                                           *w_gate_up, csr, L, static_cast<char*>(ws), s));
  return from_cuda(launch_decode_gate_up(static_cast<const uint16_t*>(x_bf16), T, H, F, k,
                                         *w_gate_up, csr, L, static_cast<char*>(ws), s));
}

moe_status moe_grouped_down_combine_nvfp4(const moe_nvfp4_bank* w_down, moe_csr csr,
                                          const float* topk_w, int32_t T, int32_t H, int32_t F,
                                          int32_t k, int32_t path, float* y, void* ws,
                                          size_t ws_bytes, void* stream) {
  if (!w_down || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y)) return MOE_ERR_INVALID_ARG;
  const int E = w_down->E;
  moe_status st = sizes_supported(T, H, F, E, k);
  if (st != MOE_OK) return st;
  if ((st = path_supported(T, F, k, path)) != MOE_OK) return st;
  if ((st = check_bank(w_down, E, H, F, MOE_SF_ATOMS_ROWS)) != MOE_OK) return st;
  if ((st = check_csr(csr)) != MOE_OK) return st;
  moe_ws_layout L;
  if (!compute_layout(T, H, F, E, k, path, &L)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, L)) != MOE_OK) return st;
  const int p = resolve_path(T, k, path);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  cudaError_t ce;
  if (p == MOE_PATH_PREFILL) {
    bool unsup = false;
    ce = launch_prefill_down(*w_down, csr, topk_w, T, H, F, k, L, w, y, s, &unsup);
    if (unsup) return MOE_ERR_UNSUPPORTED;
    return from_cuda(ce);
  }
  ce = decode_sliced((long long)T * k) ? launch_sliced_down(*w_down, csr, T, H, F, k, L, w, s)
                                       : launch_decode_down(*w_down, csr, T, H, F, k, L, w, s);
  if (ce != cudaSuccess) return MOE_ERR_CUDA;
  return from_cuda(launch_combine(topk_w, T, H, k, L, w, y, s));
}

int32_t moe_decode_layer_supported(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k) {
  if (sizes_supported(T, H, F, E, k) != MOE_OK) return 0;
  if (path_supported(T, F, k, MOE_PATH_DECODE) != MOE_OK) return 0;
  return decode_layer_supported(T, H, F, E, k) ? 1 : 0;
}

moe_status moe_decode_layer_nvfp4(const float* logits, int32_t* topk_ids, float* topk_w,
                                  const void* x_bf16, int32_t T, int32_t H, int32_t F, int32_t k,
                                  const moe_nvfp4_bank* w_gate_up, const moe_nvfp4_bank* w_down,
                                  float* y, void* ws, size_t ws_bytes, void* stream) {
  if (!topk_ids || !topk_w || !y || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  if (!x_bf16 || !aligned16(x_bf16)) return MOE_ERR_INVALID_ARG;
  if (!w_gate_up || !w_down) return MOE_ERR_INVALID_ARG;
  const int E = w_gate_up->E;
  moe_status st = sizes_supported(T, H, F, E, k);
  if (st != MOE_OK) return st;
  if ((st = check_bank(w_gate_up, E, 2 * F, H, MOE_SF_ATOMS_GATE_UP)) != MOE_OK) return st;
  if ((st = check_bank(w_down, E, H, F, MOE_SF_ATOMS_ROWS)) != MOE_OK) return st;
  if (!moe_decode_layer_supported(T, H, F, E, k)) return MOE_ERR_UNSUPPORTED;
  moe_ws_layout L;
  if (!compute_layout(T, H, F, E, k, MOE_PATH_DECODE, &L)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, L)) != MOE_OK) return st;
  return from_cuda(launch_decode_layer(logits, topk_ids, topk_w,
                                       static_cast<const uint16_t*>(x_bf16), T, H, F, k,
                                       *w_gate_up, *w_down, L, static_cast<char*>(ws), y,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_get_device_error(const void* ws, void* stream, int32_t* code) {
  if (!ws || !code) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  char* w = const_cast<char*>(static_cast<const char*>(ws));
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(w, 0, sizeof(uint32_t)) != cudaSuccess) return MOE_ERR_CUDA;
  *code = static_cast<int32_t>(v);
  return (v & MOE_DEVERR_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_OK;
}

}  // extern "C"
