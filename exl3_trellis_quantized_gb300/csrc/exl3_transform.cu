// exl3_transform.cu -- input rotation of the EXL3 linear layer.
//
// For every shard s, row r and 128-block b of k:
//   xh[s][r][128b+i] = fp16_rne(2^-4 * sum_j H[i][j] * (x[r][128b+j] * suh[s][128b+j]))
// (TensorFold PR #740, "Arithmetic" step 1: x*suh, the 128-point Hadamard in a
// fixed order of fp32 adds, times 2^-4, one rounding to fp16; cuda-exl3 README,
// "One op per layer": every shard in one launch, x read once, the bf16 -> fp16
// conversion folded into the same pass).
//
// One warp owns one (row, 128-block); lane l holds elements 4l..4l+3.  x is read
// once with one 8-byte load per lane and reused for every shard.  The kernel is
// HBM/L2-bound: 2 bytes in, 2*S bytes out per element.
#include "exl3_device.cuh"
#include "exl3_launch.h"

namespace exl3 {

template <bool X_BF16>
__global__ void __launch_bounds__(256) input_transform_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                              const uint16_t* __restrict__ suh, int num_shards,
                                                              uint16_t* __restrict__ xh) {
  const int lane = threadIdx.x & 31;
  const int64_t kb = k >> 7;
  const int64_t units = m * kb;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += warps_total) {
    const int64_t r = u / kb;
    const int64_t col = (u - r * kb) * 128 + 4 * lane;
    const uint2 raw = *reinterpret_cast<const uint2*>(x + r * k + col);
    float xv[4];
    const uint16_t e[4] = {(uint16_t)(raw.x & 0xFFFF), (uint16_t)(raw.x >> 16), (uint16_t)(raw.y & 0xFFFF),
                           (uint16_t)(raw.y >> 16)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xv[i] = X_BF16 ? __bfloat162float(__ushort_as_bfloat16(e[i])) : __half2float(__ushort_as_half(e[i]));
    }
    for (int s = 0; s < num_shards; ++s) {
      const uint2 sr = *reinterpret_cast<const uint2*>(suh + (int64_t)s * k + col);
      const uint16_t se[4] = {(uint16_t)(sr.x & 0xFFFF), (uint16_t)(sr.x >> 16), (uint16_t)(sr.y & 0xFFFF),
                              (uint16_t)(sr.y >> 16)};
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = xv[i] * __half2float(__ushort_as_half(se[i]));  // exact in fp32
      fwht128_warp(v, lane);
      uint16_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = __half_as_ushort(__float2half_rn(v[i] * 0.0625f));  // 2^-4 exact
      uint2 w;
      w.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
      w.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
      *reinterpret_cast<uint2*>(xh + ((int64_t)s * m + r) * k + col) = w;
    }
  }
}

cudaError_t launch_input_transform(const void* x, bool x_bf16, int64_t m, int64_t k, const uint16_t* suh,
                                   int num_shards, uint16_t* xh, cudaStream_t stream) {
  const int64_t units = m * (k >> 7);
  const int threads = 256;
  const int64_t want = (units + 7) / 8;
  const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
  if (x_bf16) {
    input_transform_kernel<true><<<blocks, threads, 0, stream>>>((const uint16_t*)x, m, k, suh, num_shards, xh);
  } else {
    input_transform_kernel<false><<<blocks, threads, 0, stream>>>((const uint16_t*)x, m, k, suh, num_shards, xh);
  }
  return cudaGetLastError();
}

}  // namespace exl3
