// Weight-layout conversions, one-time and off the per-layer path:
//   interleaved_to_planar_kernel  the pages' 36-byte blocks (4 UE4M3 scale bytes, then 32
//                                 code bytes for 64 weights) into the planar planes
//   prepack_sf_kernel             the planar scale plane into 512-byte tensor-memory atoms
//                                 (one per 128-row tile and K-step of 64)
#include "moe_internal.cuh"

namespace moe {

namespace {

// One thread per 36-byte block: nine 32-bit loads, one 4-byte scale store, two 16-byte code
// stores.  Block b of the whole bank is block b % bpr of row b / bpr.
__global__ void __launch_bounds__(256) interleaved_to_planar_kernel(const uint8_t* __restrict__ src,
                                                                    long long nblocks, int bpr,
                                                                    uint8_t* __restrict__ codes,
                                                                    uint8_t* __restrict__ scales) {
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  const uint32_t* s = reinterpret_cast<const uint32_t*>(src + b * 36);
  uint32_t w[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) w[i] = __ldg(s + i);
  // planar rows are contiguous and hold bpr blocks each, so block b lands at b*4 / b*32
  *reinterpret_cast<uint32_t*>(scales + b * 4) = w[0];
  uint4* c = reinterpret_cast<uint4*>(codes + b * 32);
  c[0] = make_uint4(w[1], w[2], w[3], w[4]);
  c[1] = make_uint4(w[5], w[6], w[7], w[8]);
}

// One thread per 16-byte atom row: atom a = (e * tiles + t) * kst + j, thread lane r writes
// bytes 16r .. 16r+15, the k-step j scale words of tile rows r, r+32, r+64, r+96.  Tile row
// m is bank row 128t + m, or (GATE_UP) gate row 64t + m/2 / up row F + 64t + m/2 for even
// / odd m.  The words are 4-byte aligned: rows are in_f/16 bytes, a multiple of 4.
template <bool GATE_UP>
__global__ void __launch_bounds__(256) prepack_sf_kernel(const uint8_t* __restrict__ scales,
                                                         int rows, int sfrow, int tiles, int kst,
                                                         long long n_rows16,
                                                         uint8_t* __restrict__ atoms) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows16) return;
  const long long a = i >> 5;
  const int r = (int)(i & 31);
  const int j = (int)(a % kst);
  const long long et = a / kst;
  const int t = (int)(et % tiles);
  const long long e = et / tiles;
  const int F = rows / 2;
  uint32_t w[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int m = 32 * x + r;
    const int row = GATE_UP ? ((m & 1) ? F : 0) + 64 * t + (m >> 1) : 128 * t + m;
    w[x] = __ldg(reinterpret_cast<const uint32_t*>(scales + (e * rows + row) * sfrow + 4 * j));
  }
  *reinterpret_cast<uint4*>(atoms + a * 512 + 16 * r) = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

}  // namespace moe

extern "C" moe_status moe_nvfp4_from_interleaved(const uint8_t* blob, int64_t rows, int32_t in_f,
                                                 uint8_t* codes, uint8_t* scales, void* stream) {
  using namespace moe;
  if (!blob || !codes || !scales || rows <= 0 || in_f <= 0) return MOE_ERR_INVALID_ARG;
  if (in_f % 64 != 0) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(blob) & 3) || (reinterpret_cast<uintptr_t>(codes) & 15) ||
      (reinterpret_cast<uintptr_t>(scales) & 3))
    return MOE_ERR_INVALID_ARG;
  const long long nblocks = (long long)rows * (in_f / 64);
  const long long grid = (nblocks + 255) / 256;
  if (grid > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  interleaved_to_planar_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      blob, nblocks, in_f / 64, codes, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" size_t moe_nvfp4_sf_atoms_bytes(int32_t E, int32_t rows, int32_t in_f) {
  if (E <= 0 || rows <= 0 || in_f <= 0 || rows % 128 != 0 || in_f % 64 != 0) return 0;
  return (size_t)E * (size_t)rows * (size_t)(in_f / 16);
}

extern "C" moe_status moe_nvfp4_prepack_sf(const uint8_t* scales, int32_t E, int32_t rows,
                                           int32_t in_f, int32_t order, uint8_t* sf_atoms,
                                           size_t bytes, void* stream) {
  using namespace moe;
  const size_t need = moe_nvfp4_sf_atoms_bytes(E, rows, in_f);
  if (!scales || !sf_atoms || need == 0 || bytes < need) return MOE_ERR_INVALID_ARG;
  if (order != MOE_SF_ATOMS_GATE_UP && order != MOE_SF_ATOMS_ROWS) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scales) & 15) || (reinterpret_cast<uintptr_t>(sf_atoms) & 15))
    return MOE_ERR_INVALID_ARG;
  const int tiles = rows / 128, kst = in_f / 64;
  const long long n_rows16 = (long long)(need / 16);
  const long long grid = (n_rows16 + 255) / 256;
  if (grid > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  auto kern = order == MOE_SF_ATOMS_GATE_UP ? prepack_sf_kernel<true> : prepack_sf_kernel<false>;
  kern<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(scales, rows, in_f / 16, tiles,
                                                                      kst, n_rows16, sf_atoms);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
