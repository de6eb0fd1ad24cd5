/*
 * moe.h -- C ABI of the routed Mixture-of-Experts FFN with NVFP4 weights
 * (libmoe_gb300.so, hand-written CUDA for sm_103a).
 *
 * One layer runs four calls on one stream:
 *
 *   moe_route_topk                  top-k routing of router logits
 *   moe_build_expert_csr            expert-first grouping of the (token, expert) pairs
 *   moe_grouped_gate_up_silu_nvfp4  per expert: h = silu(W_gate a) * (W_up a)
 *   moe_grouped_down_combine_nvfp4  per expert: z = W_down h, then y[t] = sum_j w[t,j] z[t*k+j]
 *
 * or, for decode batches within moe_decode_layer_supported, the same four steps in one
 * call and one kernel (moe_decode_layer_nvfp4).
 *
 * Sources of the definitions (the pages the method is taken from):
 *   - "moe_sk_repro.rs" (fn main): pairs p = t*k + j grouped by expert in ascending p
 *     (buckets / ex_ids / ex_off / ex_pairs), token of a pair = p / k, three grouped
 *     projections per layer (gate, up, down);
 *   - "moe_union_probe.rs" (header comment and fn main): fused gate_up bank
 *     [E, 2*ff, hidden] (ff gate rows then ff up rows), down bank [E, hidden, ff], a row
 *     is in_f/2 E2M1 code bytes + in_f/16 UE4M3 scale bytes, each distinct expert's
 *     bytes read once per call (the union-of-experts gather);
 *   - "moe_sel_census.rs" (header constants): NVFP4 = E2M1 codes with one UE4M3 scale
 *     per 16 weights;
 *   - "Rank-local E256 MoE misses the Qwen K1 and K4 step budgets" (numeric check
 *     table and the paragraph after it): the atomic BF16 FC2 accumulation made replays
 *     differ; this library's combine uses no floating-point atomics and is bit-identical
 *     across replays.
 *
 * Conventions for every call:
 *   - Array pointers are DEVICE pointers owned by the caller; nothing is allocated or
 *     freed by the library, and no state survives a call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are asynchronous,
 *     do no host synchronisation and no allocation, so they can be captured in a CUDA
 *     graph (moe_get_device_error excepted).
 *   - Shapes are validated on the host before anything is launched; a bad argument
 *     returns an error status and launches nothing. No call prints, aborts or throws.
 *   - The workspace `ws` of moe_workspace_bytes(T, H, F, E, k, path) bytes (256-byte
 *     aligned) carries state from moe_build_expert_csr to the two projection calls:
 *     pass the SAME ws (and the same T, k, path) to the three calls of one layer.
 *     Zero-fill it once after allocating it (its first word is the device error word).
 *   - Problems only the device can see (an expert id outside [0, E)) set a sticky bit
 *     in the workspace's error word; the offending pair is skipped (it contributes
 *     nothing to y). moe_get_device_error reads and clears the word.
 *
 * NVFP4 bank layout (planar, row-major):
 *   codes  u8 [E][rows][in_f/2]  two E2M1 codes per byte, low nibble = even element
 *   scales u8 [E][rows][in_f/16] one UE4M3 byte per 16 consecutive elements of a row
 *   value(e, r, c) = E2M1(code) * UE4M3(scale[e][r][c/16]) (* alpha[e] when the bank has a
 *   per-expert second-level scale); scale bytes must be <= 0x7E.
 *   Both planes must be 16-byte aligned. Banks stored as the pages' interleaved 36-byte
 *   blocks convert with moe_nvfp4_from_interleaved.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, k > E, misalignment */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle (see limits) */
  MOE_ERR_WORKSPACE = 3,     /* ws smaller than moe_workspace_bytes() or misaligned */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5        /* a bounded device wait gave up (device error word) */
} moe_status;

/* Path selection: DECODE keeps the bf16 activations and a float32 h. Below
 * moe_decode_tensor_core_min_pairs() pairs it multiplies them exactly (as f16 with a
 * power-of-two row prescale) by weights dequantised in registers. From that many pairs it
 * writes each activation row as four residual NVFP4 slices for the block-scaled FP4
 * tensor cores; the sum of the slices is the row to ~6^-4 of each 16-block's largest
 * magnitude, far inside the tolerance. PREFILL quantises x and h to NVFP4 once (per-row
 * power-of-two scale, UE4M3 per 16, E2M1 codes; nearest-even) and runs block-scaled FP4
 * tensor-core GEMMs. AUTO picks PREFILL when T*k >= moe_prefill_min_pairs(). The paths
 * differ in numerics by design. */
enum { MOE_PATH_AUTO = 0, MOE_PATH_DECODE = 1, MOE_PATH_PREFILL = 2 };

/* Bits of the device error word. */
enum { MOE_DEVERR_EXPERT_ID = 1, MOE_DEVERR_TIMEOUT = 2 };

/* One NVFP4 weight bank. gate_up: rows = 2F (gate rows 0..F-1, up rows F..2F-1),
 * in_f = H. down: rows = H, in_f = F. A weight is E2M1(code) x UE4M3(scale of its
 * 16-group), times alpha[e] when `alpha` is not NULL: an optional per-expert float32
 * second-level scale (the two-level scaling of the ModelOpt NVFP4 checkpoints page 4 runs;
 * device array [E], finite, caller-owned). On the PREFILL path the
 * down bank's alpha must stay <= 2 (its f16 partials are scaled for |alpha| <= 2). */
typedef struct moe_nvfp4_bank {
  const uint8_t* codes;
  const uint8_t* scales;
  int32_t E, rows, in_f;
  const float* alpha;
  /* Optional: the scale plane rewritten by moe_nvfp4_prepack_sf (device, 16-byte aligned,
   * caller-owned) and the order it was written in; NULL and MOE_SF_ATOMS_NONE when the
   * bank has none. The tensor-core GEMMs (DECODE from moe_decode_tensor_core_min_pairs()
   * pairs, PREFILL) then copy each stage's weight scale factors straight into tensor memory
   * instead of rearranging `scales`; the results are bit-identical either way. `scales`
   * stays required (the other DECODE kernels read it). */
  const uint8_t* sf_atoms;
  int32_t sf_atoms_order;
} moe_nvfp4_bank;

/* Row orders of a prepacked scale plane: a gate/up bank's 128-row tiles interleave gate
 * row i and up row i (tile t, row m: gate row 64t + m/2 for even m, up row 64t + m/2 for
 * odd m); a down bank's tiles are rows 128t .. 128t + 127. */
enum { MOE_SF_ATOMS_NONE = 0, MOE_SF_ATOMS_GATE_UP = 1, MOE_SF_ATOMS_ROWS = 2 };

/* Expert-first CSR written by moe_build_expert_csr (all device arrays, caller-owned):
 *   expert_offsets i32 [E+1]  exclusive prefix sum of per-expert pair counts
 *   pair_ids       i32 [T*k]  pair indices p = t*k + j sorted by (expert, p); entries past
 *                             expert_offsets[E] are unspecified (pairs with invalid ids)
 *   active_experts i32 [E]    experts with at least one pair, ascending; first n_active valid
 *   n_active       i32 [1]    number of active experts (stays on the device) */
typedef struct moe_csr {
  int32_t* expert_offsets;
  int32_t* pair_ids;
  int32_t* active_experts;
  int32_t* n_active;
} moe_csr;

/* Byte offsets of the workspace regions (for tests and tools; the layout depends only
 * on the arguments of moe_workspace_bytes). A region of size 0 is absent. */
typedef struct moe_ws_layout {
  size_t total;
  size_t error_word;   /* u32 device error word */
  size_t pair_pos;     /* i32 [P]   CSR position of pair p, -1 if its expert id is invalid */
  size_t h;            /* f32 [P][F] h = silu(g) * u, rows in CSR order */
  size_t xg;           /* decode: f16 [T][H] each token's activation row times 2^-xe (the
                          region holds P rows; rows T..P-1 are unused) */
  size_t xe;           /* decode: i32 [T] power-of-two prescale of each token's row */
  size_t hg;           /* decode: f16 [P][F] h times 2^-he */
  size_t he;           /* decode: i32 [P] */
  size_t qx_codes;     /* prefill: u8 [P][H/2]  Q(x) in CSR order */
  size_t qx_scales;    /* prefill: u8 [P][H/16] */
  size_t qx_exp;       /* prefill: i32 [P] row exponents */
  size_t qh_codes;     /* prefill: u8 [P][F/2]  Q(h) in CSR order */
  size_t qh_scales;    /* prefill: u8 [P][S], S = F/16 rounded up to a multiple of 16 (bytes past F/16 unused) */
  size_t qh_exp;       /* prefill: i32 [P] */
  size_t partial;      /* per-pair down projections z, rows in CSR order: f32 [P][H] on the
                          decode path; on the prefill path f16 [P][H] holding
                          z * 2^-(qh_exp[row] + c_F), c_F the smallest shift with
                          F * 2688^2 * 2^-c_F < 2^15 */
  size_t tiles;        /* 128-row M-tiles of the prefill GEMMs (written by the CSR call): i32
                          count, pad to 16 B, then int4 {row0, rows, expert, 0} per tile */
  size_t slice_tiles;  /* the same for the sliced decode GEMMs: 32-row tiles over the 4 slice
                          rows of every pair (row0 and rows count slice rows) */
  size_t sync;         /* decode below moe_decode_tensor_core_min_pairs() pairs: u64 [6] sync
                          words of moe_decode_layer_nvfp4 (call counter, barrier counters) */
  size_t row_tok;      /* decode below moe_decode_tensor_core_min_pairs() pairs: i32 [P] token
                          of each CSR row (its xg / xe row) */
} moe_ws_layout;

/* Limits (MOE_ERR_UNSUPPORTED beyond them): 1 <= k <= min(E, 32); E <= 1024;
 * H % 256 == 0 and H <= 4096; F % 64 == 0; T*k < 2^31 / max(H, F); F <= 1408 on the
 * DECODE path, and from moe_decode_tensor_core_min_pairs() pairs on also F not in
 * {1088, 1216, 1344} (their weight-scale rows do not fit the down GEMM's staging); F <= 4096
 * on the PREFILL path (the path AUTO resolves to counts; moe_workspace_bytes returns 0 for
 * such sizes). */

/* Workspace size in bytes for one layer with these sizes (0 if the sizes are invalid). */
size_t moe_workspace_bytes(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k, int32_t path);

/* Fill *out with the workspace region offsets for these sizes. */
moe_status moe_workspace_layout(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k,
                                int32_t path, moe_ws_layout* out);

/* Path AUTO resolves to: PREFILL if T*k >= this value, else DECODE. */
int32_t moe_prefill_min_pairs(void);
/* On the DECODE path, from this many pairs (T*k) on the gate/up and down calls run the
 * tensor-core form: each activation row (x, then h) as four residual NVFP4 slices
 * multiplied by the block-scaled FP4 tensor cores; below it, the exact-f16 activations
 * against weights dequantised in registers. Both stay within the stated tolerance. */
int32_t moe_decode_tensor_core_min_pairs(void);
/* The path a call with these arguments runs (DECODE or PREFILL). */
int32_t moe_resolve_path(int32_t T, int32_t k, int32_t path);

/* Number of kernels one layer with these sizes launches in moe_build_expert_csr,
 * moe_grouped_gate_up_silu_nvfp4 and moe_grouped_down_combine_nvfp4 together (add one
 * for moe_route_topk); 0 if the sizes are invalid. */
int32_t moe_kernel_launches(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k, int32_t path);

/* Top-k routing of router logits (the pages' probes start from already-routed pairs;
 * this is the router that produces them). For each token t: the k experts with the largest
 * logits[t, :] in descending order, ties broken towards the lower expert id, comparing
 * the float32 values exactly; topk_w[t, j] = exp(l_j - l_0) / sum_j' exp(l_j' - l_0),
 * i.e. the softmax over the selected logits (equal to the full softmax renormalised
 * over the selection). logits f32 [T][E] (finite), topk_ids i32 [T][k], topk_w f32 [T][k]. */
moe_status moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                          int32_t* topk_ids, float* topk_w, void* stream);

/* Expert-first CSR of the P = T*k pairs ("moe_sk_repro.rs", fn main): a counting sort by
 * expert that keeps ascending p within an expert (placement by prefix sums, not by
 * atomic arrival order, so the result is bit-exact and deterministic). topk_ids i32
 * [T][k]. Writes `csr` and the workspace's pair_pos and both tile lists (tiles,
 * slice_tiles); ids outside [0, E) set MOE_DEVERR_EXPERT_ID and are left out. ws must hold
 * at least the regions before h (moe_workspace_layout with any H, F, path: they do not
 * depend on them). From T*k >= 4096 pairs it also keeps per-chunk counts in the
 * workspace's h region (which the gate/up call overwrites afterwards). */
moe_status moe_build_expert_csr(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                                moe_csr csr, void* ws, size_t ws_bytes, void* stream);

/* Grouped gate/up projection with SiLU(gate) * up over the active experts. Each active
 * expert's 2F x H NVFP4 rows are read from HBM once per call whatever its number of
 * pairs (the union-of-experts gather of "moe_union_probe.rs"). x_bf16 bf16 [T][H]
 * (16-byte aligned); w_gate_up: rows = 2F, in_f = H. Result h f32 [P][F] in the
 * workspace, rows in CSR order. Reads the CSR and the workspace's pair_pos written by
 * moe_build_expert_csr on this workspace. The DECODE path starts reading x_bf16 before
 * the CSR kernel has finished (its rows do not depend on the routing), so x_bf16 must be
 * complete in stream order when the call is made: a kernel that writes it and is launched
 * with programmatic dependent launch must not signal its dependents before its last write. */
moe_status moe_grouped_gate_up_silu_nvfp4(const void* x_bf16, int32_t T, int32_t H, int32_t F,
                                          int32_t k, const moe_nvfp4_bank* w_gate_up,
                                          moe_csr csr, int32_t path, void* ws, size_t ws_bytes,
                                          void* stream);

/* Grouped down projection z_p = W_down[e] h_p over the active experts, then the
 * deterministic combine y[t, :] = sum_{j=0..k-1} topk_w[t, j] * z_{t*k+j} summed in
 * ascending j with no floating-point atomics. w_down: rows = H, in_f = F; topk_w f32
 * [T][k]; y f32 [T][H] (overwritten; rows of tokens whose pairs are all invalid are 0). */
moe_status moe_grouped_down_combine_nvfp4(const moe_nvfp4_bank* w_down, moe_csr csr,
                                          const float* topk_w, int32_t T, int32_t H, int32_t F,
                                          int32_t k, int32_t path, float* y, void* ws,
                                          size_t ws_bytes, void* stream);

/* The whole decode layer in one call and one kernel: routing (or given picks), the CSR,
 * gate/up + SiLU, down and the combine of the four calls above. topk_ids and topk_w are
 * bit-identical to moe_route_topk's; every other step runs the arithmetic of the DECODE
 * path's TMA-fed kernels, so y is bit-identical to the four calls wherever those run them
 * (from 8 units per SM: min(T*k, E) * F/8 gate/up and min(T*k, E) * H/16 down units),
 * and agrees with them to rounding below that. One cooperative grid of one CTA per SM: every CTA routes the T tokens and
 * builds the CSR itself, the weight stream runs from the gate/up rows straight into the
 * down rows, and the steps are ordered by four grid-wide barriers, each wait bounded
 * (MOE_DEVERR_TIMEOUT on expiry). Sizes: moe_decode_layer_supported (T <= 32 tokens,
 * T*k below moe_decode_tensor_core_min_pairs(), H % 256 == 0, F % 128 == 0
 * and F <= 640, plus the limits above), else MOE_ERR_UNSUPPORTED.
 *   logits   f32 [T][E] (finite): routed as moe_route_topk does, the picks and weights
 *            written to topk_ids / topk_w; or NULL: topk_ids i32 [T][k] and topk_w f32
 *            [T][k] are inputs (ids outside [0, E) set MOE_DEVERR_EXPERT_ID and are left
 *            out, as in moe_build_expert_csr).
 *   x_bf16   bf16 [T][H], 16-byte aligned; w_gate_up rows = 2F, in_f = H; w_down rows = H,
 *            in_f = F (same E); y f32 [T][H], 16-byte aligned, overwritten.
 *   ws       moe_workspace_bytes(T, H, F, E, k, MOE_PATH_DECODE) bytes, zero-filled once
 *            after allocation like every workspace: its sync words hold a call counter and
 *            barrier counters that only grow, so no call resets them. A call whose wait
 *            gave up (MOE_DEVERR_TIMEOUT) marks them, and later calls on that workspace then
 *            only report MOE_DEVERR_TIMEOUT until it is zero-filled again. The call writes
 *            the regions the DECODE path uses (not a csr). */
moe_status moe_decode_layer_nvfp4(const float* logits, int32_t* topk_ids, float* topk_w,
                                  const void* x_bf16, int32_t T, int32_t H, int32_t F, int32_t k,
                                  const moe_nvfp4_bank* w_gate_up, const moe_nvfp4_bank* w_down,
                                  float* y, void* ws, size_t ws_bytes, void* stream);

/* 1 if moe_decode_layer_nvfp4 takes these sizes, else 0. */
int32_t moe_decode_layer_supported(int32_t T, int32_t H, int32_t F, int32_t E, int32_t k);

/* moe_build_expert_csr without a workspace, for callers that cannot allocate device
 * memory: a host engine or plugin that owns every device allocation and hands kernels only
 * its own tensors, or code on a path where a device allocation is not allowed because
 * cudaMalloc may block and synchronise the whole device. The paper the method comes from
 * has no counterpart to this entry point; it is an addition of this library.
 *
 * Same inputs and CSR outputs as moe_build_expert_csr (bit-identical results). Its scratch
 * (the per-pair CSR positions) lives in a fixed device array inside the library, 256 KiB
 * per GPU that loads the library, held until the process exits; nothing is allocated or
 * freed. Limits: T * k <= 65536 (else MOE_ERR_UNSUPPORTED), plus the limits above.
 * The first call on each device looks up the array's device address (once per device, on
 * the current device) and keeps it for the life of that device's primary context: make
 * that first call before any stream capture, and do not call this entry point again on a
 * device after resetting it (cudaDeviceReset). All calls share the one array: calls that
 * can overlap on the GPU (different streams, or different host threads, on the same
 * device) race, so serialise them. Invalid expert ids are left out as in
 * moe_build_expert_csr, but no error word is reported: expert_offsets[E] < T*k tells the
 * caller that some were dropped. The layer calls (gate/up, down/combine) also read the
 * per-pair positions that moe_build_expert_csr writes into their workspace, so they need
 * that entry point; this one serves callers that want the CSR alone. */
moe_status moe_build_expert_csr_static(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                                       moe_csr csr, void* stream);

/* Weight-layout import (not on the per-layer path): rows stored the way the pages' banks
 * are (mk_bank of "moe_sk_repro.rs" gives every 64 weights a 36-byte block; the BLK
 * constant of "moe_sel_census.rs" splits it into four UE4M3 scale bytes and thirty-two code
 * bytes) into the planar planes this library reads. Each
 * row of in_f weights is in_f/64 blocks; a block is its 4 scale bytes (scale i for weights
 * 16i..16i+15 of the block) followed by its 32 code bytes (low nibble = even weight).
 * blob u8 [rows][in_f/64*36] (4-byte aligned) -> codes u8 [rows][in_f/2] (16-byte aligned),
 * scales u8 [rows][in_f/16] (4-byte aligned); all device pointers, caller-owned; rows is
 * E times the rows of one expert for a whole bank. in_f % 64 == 0. Async on `stream`. */
moe_status moe_nvfp4_from_interleaved(const uint8_t* blob, int64_t rows, int32_t in_f,
                                      uint8_t* codes, uint8_t* scales, void* stream);

/* Scale-factor prepack (not on the per-layer path). The block-scaled MMA
 * (tcgen05.mma kind::mxf4nvf4, scale_vec::4X: one UE4M3 scale per 16 E2M1 weights, the
 * scaling the pages' NVFP4 format defines) reads a 128-row operand's scale factors for one
 * K-step of 64 weights from tensor memory: lane r, column x holds the four scale bytes of
 * row 32x + r. This writes a bank's planar scale plane in that order, one 512-byte atom per
 * (expert, 128-row tile, K-step): sf_atoms[((e * rows/128 + t) * in_f/64 + j) * 512 + 16r +
 * 4x + b] = scale byte 4j + b of tile row 32x + r (the tile rows of `order`, above), so a
 * GEMM stage's atoms are one contiguous copy that tcgen05.cp moves into tensor memory.
 *   scales    u8 [E][rows][in_f/16] (16-byte aligned, device)
 *   sf_atoms  u8 [moe_nvfp4_sf_atoms_bytes(E, rows, in_f)] (16-byte aligned, device,
 *             caller-owned; the same size as `scales`)
 *   order     MOE_SF_ATOMS_GATE_UP (rows = 2F) or MOE_SF_ATOMS_ROWS
 * Requires in_f % 64 == 0 and rows % 128 == 0; MOE_ERR_INVALID_ARG otherwise, for a null
 * or misaligned pointer, or for `bytes` below the size. Async on `stream`. */
size_t moe_nvfp4_sf_atoms_bytes(int32_t E, int32_t rows, int32_t in_f);
moe_status moe_nvfp4_prepack_sf(const uint8_t* scales, int32_t E, int32_t rows, int32_t in_f,
                                int32_t order, uint8_t* sf_atoms, size_t bytes, void* stream);

/* Human-readable name of a status (static string, never NULL). */
const char* moe_status_string(moe_status status);

/* Synchronise `stream`, read the workspace's device error word into *code and clear
 * it. For tests and diagnostics only: it blocks and cannot be graph-captured. */
moe_status moe_get_device_error(const void* ws, void* stream, int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
