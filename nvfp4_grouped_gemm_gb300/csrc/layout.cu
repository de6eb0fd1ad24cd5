// Weight-layout import: the interleaved NVFP4 storage of the pages' banks (36-byte blocks,
// each 4 UE4M3 scale bytes then 32 code bytes for 64 weights) into the planar code and
// scale planes the kernels read.  A one-time conversion, off the per-layer path.
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
