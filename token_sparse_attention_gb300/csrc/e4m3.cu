// E4M3 encoding of a bf16 tensor for the fp8 K/V cache of the token-sparse
// kernel (the pages leave low-precision attention open: ai.info AI summary,
// "Future Directions").  E4M3 as the OCP 8-bit floating point specification
// defines it: bias 7, no infinities, largest finite magnitude 448.
//
// Each value is divided by the scale in fp32 (correctly rounded) and rounded
// to the nearest E4M3 value, ties to even, saturating at +-448.  An
// HBM-bound stream: 2 bytes read and 1 written per element; each thread
// handles 16 elements per step (two 16-byte loads, one 16-byte store), the
// grid a multiple of the SM count.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int kQThreads = 256;

__device__ __forceinline__ uint16_t encode2(uint32_t w, float scale) {
  const float lo = __fdiv_rn(__uint_as_float(w << 16), scale);
  const float hi = __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), scale);
  return f32x2_to_e4m3x2(lo, hi);
}

__global__ void __launch_bounds__(kQThreads)
    quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ x, size_t n, float scale,
                         uint8_t* __restrict__ x8) {
  const size_t n16 = n / 16;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride) {
    const uint4 a = ld_global_nc16(x + 16 * i);
    const uint4 b = ld_global_nc16(x + 16 * i + 8);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      o[k] = encode2(wa[2 * k], scale) | (static_cast<uint32_t>(encode2(wa[2 * k + 1], scale)) << 16);
      o[k + 2] =
          encode2(wb[2 * k], scale) | (static_cast<uint32_t>(encode2(wb[2 * k + 1], scale)) << 16);
    }
    *reinterpret_cast<uint4*>(x8 + 16 * i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  // the tail (n not a multiple of 16): one element per thread of block 0
  if (blockIdx.x == 0) {
    for (size_t i = 16 * n16 + threadIdx.x; i < n; i += blockDim.x) {
      const float v = __fdiv_rn(__bfloat162float(x[i]), scale);
      x8[i] = static_cast<uint8_t>(f32x2_to_e4m3x2(v, 0.f) & 0xFFu);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_e4m3(const __nv_bfloat16* x, size_t n, float scale, uint8_t* x8,
                                 cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t want = (n / 16 + kQThreads - 1) / kQThreads;
  const int blocks = static_cast<int>(std::max<size_t>(1, std::min<size_t>(want, 8 * static_cast<size_t>(sms))));
  quantize_e4m3_kernel<<<blocks, kQThreads, 0, stream>>>(x, n, scale, x8);
  return cudaGetLastError();
}

}  // namespace mcs
