// Internal declarations shared by the translation units of libmoe_gb300.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "moe.h"

namespace moe {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kPrefillMinPairs = 2048;
// Largest F per path: the decode down kernel keeps two 128-row weight tiles and eight f16
// h rows in shared memory; the prefill Q(h) kernel holds a row of h in registers.
constexpr int kDecodeMaxF = 1408;
constexpr int kPrefillMaxF = 4096;
// Slices per activation row in the decode form of the tensor-core path.
constexpr int kDecodeSlices = 4;
// The decode path runs the sliced tensor-core GEMMs from this many pairs on (below it, the
// TMA-fed mma.sync kernels of decode.cu, whose fixed costs are lower).
#ifndef MOE_SLICED_MIN_PAIRS
#define MOE_SLICED_MIN_PAIRS 256
#endif
constexpr int kSlicedMinPairs = MOE_SLICED_MIN_PAIRS;
inline bool decode_sliced(long long P) { return P >= kSlicedMinPairs; }
constexpr size_t kAlign = 256;
// Tile lists over the CSR: the prefill GEMMs cut an expert's rows into 128-row M-tiles; the
// sliced decode GEMMs cut its slice rows (kDecodeSlices per pair) into 32-row tiles.
constexpr int kTileRows = 128;
constexpr int kSliceTileRows = 32;
// Bytes of a tile list (count, pad to 16 B, then one int4 {row0, rows, expert, 0} per tile)
// for P pairs of rpp operand rows each: at most P*rpp/tile_rows full tiles plus one partial
// tile per active expert (at most min(E, P) of them).
inline size_t tile_list_bytes(long long P, int rpp, int tile_rows, int E) {
  const long long active = E < P ? E : P;
  return (size_t)(16 + 16 * (P * rpp / tile_rows + active + 1));
}

inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// Number of SMs of the current device (cached per device; grids are sized from it).
int num_sms();

// Row pitch of the Q(h) block scales in the prefill workspace: F/16 rounded up to a
// multiple of 16 bytes, so that the rows can be read by TMA.
inline int qh_scale_pitch(int F) { return (F / 16 + 15) / 16 * 16; }

// Workspace layout for one layer; pure function of the sizes (see moe_ws_layout).
bool compute_layout(int T, int H, int F, int E, int k, int path, moe_ws_layout* L);
int resolve_path(int T, int k, int path);

// Launchers (return cudaGetLastError() of the launch sequence).
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t s);
// With `scratch` (csr_scratch_bytes(P, E) bytes, nonzero from kCsrGridMinPairs pairs)
// the CSR is built by three grid-wide kernels, else by one CTA.
constexpr int kCsrGridMinPairs = 4096;
size_t csr_scratch_bytes(int P, int E);
// `tiles` / `slice_tiles` (either may be null) receive the two tile lists.
cudaError_t launch_build_csr(const int32_t* ids, int P, int k, int E, moe_csr csr,
                             int32_t* pair_pos, uint32_t* err, int32_t* scratch, int32_t* tiles,
                             int32_t* slice_tiles, cudaStream_t s);
cudaError_t launch_decode_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                  const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                  char* ws, cudaStream_t s);
cudaError_t launch_decode_down(const moe_nvfp4_bank& b, moe_csr csr, int T, int H, int F, int k,
                               const moe_ws_layout& L, char* ws, cudaStream_t s);
cudaError_t launch_combine(const float* w, int T, int H, int k, const moe_ws_layout& L, char* ws,
                           float* y, cudaStream_t s);
// The one-kernel decode layer (decode_layer.cu).
bool decode_layer_supported(int T, int H, int F, int E, int k);
size_t decode_layer_sync_bytes();
cudaError_t launch_decode_layer(const float* logits, int32_t* ids, float* w, const uint16_t* x,
                                int T, int H, int F, int k, const moe_nvfp4_bank& gu,
                                const moe_nvfp4_bank& dn, const moe_ws_layout& L, char* ws,
                                float* y, cudaStream_t s);
cudaError_t launch_sliced_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                  const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                  char* ws, cudaStream_t s);
cudaError_t launch_sliced_down(const moe_nvfp4_bank& b, moe_csr csr, int T, int H, int F, int k,
                               const moe_ws_layout& L, char* ws, cudaStream_t s);
cudaError_t launch_prefill_gate_up(const uint16_t* x_bf16, int T, int H, int F, int k,
                                   const moe_nvfp4_bank& b, moe_csr csr, const moe_ws_layout& L,
                                   char* ws, cudaStream_t s, bool* unsupported);
// Q(h), the down GEMM and the combine.
cudaError_t launch_prefill_down(const moe_nvfp4_bank& b, moe_csr csr, const float* w, int T, int H,
                                int F, int k, const moe_ws_layout& L, char* ws, float* y,
                                cudaStream_t s, bool* unsupported);
cudaError_t launch_quant_x(const uint16_t* x_bf16, int T, int H, int k, const int32_t* pair_pos,
                           uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s);
cudaError_t launch_quant_h(const float* h, int P, int F, int sf_pitch, const int32_t* offsets,
                           int E, uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s);
// Exponent c_F with F * 2688^2 * 2^-c_F < 2^15: the fixed shift of the f16 partials.
int down_shift_for(int F);
cudaError_t launch_prefill_combine(const float* w, int T, int H, int F, int k, int c0, int HS,
                                   const moe_ws_layout& L, char* ws, float* y, cudaStream_t s);
cudaError_t launch_slice_x(const uint16_t* x_bf16, int T, int H, int k, const int32_t* pair_pos,
                           uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s);
cudaError_t launch_slice_h(const float* h, int P, int F, int sf_pitch, const int32_t* offsets,
                           int E, uint8_t* qc, uint8_t* qs, int32_t* qe, cudaStream_t s);
// Programmatic dependent launch, device side: wait for the predecessor grid (complete,
// its memory visible), or allow the successor grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic dependent launch allowed: the kernel may start while its
// predecessor in the stream finishes, and must execute griddepcontrol.wait before it
// reads anything that predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// 2^e as a float, exact for -149 <= e <= 127 (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}


// Two E2M1 codes (one byte, low nibble = even element) to an f16x2 (low half = even).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r) : "r"(byte));
  return r;
}

// The four byte pairs of a 32-bit word of E2M1 codes as f16x2 (bytes 0..3 in order).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(w));
}

// Two UE4M3 bytes (low 16 bits of v) to f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Broadcast the low (hi=false) or high half of an f16x2 to both halves.
__device__ __forceinline__ uint32_t bcast_lo(uint32_t v) { return __byte_perm(v, v, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t v) { return __byte_perm(v, v, 0x3232); }

// D += A(16x16 f16, row) * B(16x8 f16, col), f32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Streaming 128-bit load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Routing key: unsigned order = (logit descending, id ascending); 0 is below every key.
// -0 and +0 share a key, as the float32 comparison makes them equal.
__device__ __forceinline__ unsigned long long route_key(float v, int id) {
  const uint32_t u = (v == 0.0f) ? 0u : __float_as_uint(v);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (0xffffffffu - (uint32_t)id);
}
__device__ __forceinline__ float key_logit(unsigned long long key) {
  const uint32_t o = (uint32_t)(key >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ int key_id(unsigned long long key) {
  return (int)(0xffffffffu - (uint32_t)key);
}

// Exponent e with |v| * 2^-e in [2^14, 2^15) for v != 0 (0 for v == 0): the power-of-two
// prescale that maps a row's largest magnitude into the top binade below f16's 2^15.
__device__ __forceinline__ int f16_prescale_exp(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e;
  frexpf(amax, &e);          // amax = m * 2^e, m in [0.5, 1)
  return (e - 1) - 14;
}

}  // namespace moe
