// exl3_transform.cu -- input rotation of the EXL3 linear layer.
//
// For every shard s, row r and 128-block b of k:
//   xh[s][r][128b+i] = fp16_rne(2^-4 * sum_j H[i][j] * (x[r][128b+j] * suh[s][128b+j]))
// (TensorFold PR #740, "Arithmetic" step 1: x*suh, the 128-point Hadamard in a
// fixed order of fp32 adds, times 2^-4, one rounding to fp16; cuda-exl3 README,
// "One op per layer": every shard in one launch, x read once, the bf16 -> fp16
// conversion folded into the same pass).
//
// Four lanes own one (row, 128-block): lane q of the four holds elements
// 32q..32q+31, so a warp covers eight blocks (2 KB of x) per pass with 16-byte
// loads and stores.  Butterfly stages of stride 1..16 stay in registers; the
// stride-32 and stride-64 stages exchange with lanes q^1 and q^2.  Each stage
// computes (a, b) -> (a + b, a - b) on the same pairs as the plain definition,
// so the order of fp32 adds is the fixed one.  x is read once and reused for
// every shard.  The kernel is HBM/L2-bound: 2 bytes in, 2*S bytes out per
// element.
#include "exl3_device.cuh"
#include "exl3_launch.h"
#include "exl3_sm100.cuh"

namespace exl3 {

namespace {

__device__ __forceinline__ void unpack8(const uint4 w, uint16_t (&e)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e[2 * i] = (uint16_t)(u[i] & 0xFFFFu);
    e[2 * i + 1] = (uint16_t)(u[i] >> 16);
  }
}

// The Hadamard butterfly of a lane's 32 values (stages of stride 1..16 in
// registers, 32 and 64 with lanes q^1 and q^2), times 2^-4, rounded to fp16
// and stored at dst (nothing is stored when dst is null; the lane still takes
// part in the exchanges).
__device__ __forceinline__ void rotate_store(float (&v)[32], int q, uint16_t* dst) {
#pragma unroll
  for (int st = 1; st < 32; st <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & st) == 0) {
        const float a = v[i], b = v[i + st];
        v[i] = a + b;
        v[i + st] = a - b;
      }
    }
  }
#pragma unroll
  for (int st = 1; st <= 2; st <<= 1) {  // element strides 32 and 64
    const bool upper = (q & st) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float p = __shfl_xor_sync(0xffffffffu, v[i], st);
      v[i] = upper ? (p - v[i]) : (v[i] + p);
    }
  }
  if (dst != nullptr) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint16_t lo = __half_as_ushort(__float2half_rn(v[8 * c + 2 * i] * 0.0625f));  // 2^-4 exact
        const uint16_t hi = __half_as_ushort(__float2half_rn(v[8 * c + 2 * i + 1] * 0.0625f));
        w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      *reinterpret_cast<uint4*>(dst + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

template <bool X_BF16>
__device__ __forceinline__ float to_f32(uint16_t e) {
  return X_BF16 ? __bfloat162float(__ushort_as_bfloat16(e)) : __half2float(__ushort_as_half(e));
}

template <bool X_BF16>
__global__ void __launch_bounds__(256) input_transform_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                              const uint16_t* __restrict__ suh, int num_shards,
                                                              uint16_t* __restrict__ xh) {
  // The GEMM that consumes xh may be scheduled now: it prefetches its weights
  // and waits for this grid to complete before it reads xh.
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int q = lane & 3;  // which 32 elements of the block
  const int64_t kb = k >> 7;
  const int64_t units = m * kb;
  const int64_t groups = (units + 7) / 8;  // eight blocks per warp and pass
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  // element offset of this lane's 32 values in group g (or -1 past the end)
  auto lane_offset = [&](int64_t g, int64_t* row) -> int64_t {
    const int64_t u = g * 8 + (lane >> 2);
    if (g >= groups || u >= units) return -1;
    *row = u / kb;
    return *row * k + (u - *row * kb) * 128 + 32 * q;
  };
  // x stays packed (bf16 / fp16 pairs) in registers; the next pass's words are
  // loaded before this pass computes, so two passes of loads are in flight
  int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int64_t row = 0;
  int64_t off = lane_offset(g, &row);
  uint4 cur[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) cur[c] = off >= 0 ? *reinterpret_cast<const uint4*>(x + off + 8 * c) : make_uint4(0, 0, 0, 0);
  for (; g < groups; g += warps_total) {
    int64_t nrow = 0;
    const int64_t noff = lane_offset(g + warps_total, &nrow);
    uint4 nxt[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      nxt[c] = noff >= 0 ? *reinterpret_cast<const uint4*>(x + noff + 8 * c) : make_uint4(0, 0, 0, 0);
    const int64_t col = off >= 0 ? off - row * k : 32 * q;
    for (int s = 0; s < num_shards; ++s) {
      float v[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint16_t e[8], se[8];
        unpack8(cur[c], e);
        unpack8(*reinterpret_cast<const uint4*>(suh + (int64_t)s * k + col + 8 * c), se);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[8 * c + i] = to_f32<X_BF16>(e[i]) * __half2float(__ushort_as_half(se[i]));  // exact
      }
      rotate_store(v, q, off >= 0 ? xh + (int64_t)s * m * k + off : nullptr);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) cur[c] = nxt[c];
    off = noff;
    row = nrow;
  }
}

// SwiGLU folded into the transform (cuda-exl3 README, "MoE throughput"): the
// input is a gated MLP's gate_up output [m][2k]; each element of the
// down-projection's input is h = silu(g) * u in fp32, silu(g) = g / (1 + e^-g),
// with g from the first k columns and u from the last k, and h then takes the
// place of x above.  Same lane layout; the next pass's words are prefetched.
template <bool X_BF16>
__global__ void __launch_bounds__(256) input_transform_swiglu_kernel(const uint16_t* __restrict__ gu, int64_t m,
                                                                     int64_t k, const uint16_t* __restrict__ suh,
                                                                     int num_shards, uint16_t* __restrict__ xh) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int q = lane & 3;
  const int64_t kb = k >> 7;
  const int64_t units = m * kb;
  const int64_t groups = (units + 7) / 8;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  // (row, column) of this lane's 32 values in group g; false past the end
  auto lane_pos = [&](int64_t g, int64_t* row, int64_t* col) -> bool {
    const int64_t u = g * 8 + (lane >> 2);
    if (g >= groups || u >= units) return false;
    *row = u / kb;
    *col = (u - *row * kb) * 128 + 32 * q;
    return true;
  };
  auto load = [&](bool ok, int64_t row, int64_t col, uint4 (&gw)[4], uint4 (&uw)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      gw[c] = ok ? *reinterpret_cast<const uint4*>(gu + row * 2 * k + col + 8 * c) : make_uint4(0, 0, 0, 0);
      uw[c] = ok ? *reinterpret_cast<const uint4*>(gu + row * 2 * k + k + col + 8 * c) : make_uint4(0, 0, 0, 0);
    }
  };
  int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int64_t row = 0, col = 0;
  bool ok = lane_pos(g, &row, &col);
  uint4 cg[4], cu[4];
  load(ok, row, col, cg, cu);
  for (; g < groups; g += warps_total) {
    int64_t nrow = 0, ncol = 0;
    const bool nok = lane_pos(g + warps_total, &nrow, &ncol);
    uint4 ng[4], nu[4];
    load(nok, nrow, ncol, ng, nu);
    float h[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint16_t ge[8], ue[8];
      unpack8(cg[c], ge);
      unpack8(cu[c], ue);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float gv = to_f32<X_BF16>(ge[i]);
        h[8 * c + i] = gv / (1.0f + expf(-gv)) * to_f32<X_BF16>(ue[i]);
      }
    }
    const int64_t c0 = ok ? col : 32 * q;
    for (int s = 0; s < num_shards; ++s) {
      float v[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint16_t se[8];
        unpack8(*reinterpret_cast<const uint4*>(suh + (int64_t)s * k + c0 + 8 * c), se);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[8 * c + i] = h[8 * c + i] * __half2float(__ushort_as_half(se[i]));
      }
      rotate_store(v, q, ok ? xh + ((int64_t)s * m + row) * k + col : nullptr);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      cg[c] = ng[c];
      cu[c] = nu[c];
    }
    ok = nok;
    row = nrow;
    col = ncol;
  }
}

// Mixture-of-experts gather (cuda-exl3 README, "What is supported": suh is per
// expert, so the rotation happens after routing; each routed row is gathered and
// rotated with its own expert's scales in one pass).  Padded row r of the
// block-aligned routing belongs to block r / block of expert block_expert[..]
// and to pair sorted_ids[r] = token * topk + slot (or a padding id).  Rows of a
// block with no expert (-1, or an id past the last) are not written; padding
// rows of live blocks get zeros.  Same lane layout as the plain transform.
template <bool X_BF16>
__global__ void __launch_bounds__(256) moe_input_transform_kernel(
    const uint16_t* __restrict__ x, int64_t num_tokens, int64_t k, const int32_t* __restrict__ sorted_ids,
    int64_t rows, int32_t topk, const int32_t* __restrict__ block_expert, int32_t block,
    const uint16_t* __restrict__ suh, int num_shards, int num_experts, uint16_t* __restrict__ xh) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int q = lane & 3;
  const int64_t kb = k >> 7;
  const int64_t units = rows * kb;
  const int64_t groups = (units + 7) / 8;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t pairs = num_tokens * topk;
  for (int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < groups; g += warps_total) {
    const int64_t u = g * 8 + (lane >> 2);
    const bool in_range = u < units;
    const int64_t r = in_range ? u / kb : 0;
    const int64_t col = (in_range ? (u - r * kb) * 128 : 0) + 32 * q;
    const int e = in_range ? block_expert[r / block] : -1;
    const bool live = e >= 0 && e < num_experts;
    const int64_t id = live ? (int64_t)sorted_ids[r] : -1;
    const int64_t tok = (id >= 0 && id < pairs) ? id / topk : -1;
    uint4 xw[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      xw[c] = tok >= 0 ? *reinterpret_cast<const uint4*>(x + tok * k + col + 8 * c) : make_uint4(0, 0, 0, 0);
    for (int s = 0; s < num_shards; ++s) {
      float v[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint16_t xe[8], se[8];
        unpack8(xw[c], xe);
        unpack8(tok >= 0 ? *reinterpret_cast<const uint4*>(suh + ((int64_t)e * num_shards + s) * k + col + 8 * c)
                         : make_uint4(0, 0, 0, 0),
                se);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[8 * c + i] = to_f32<X_BF16>(xe[i]) * __half2float(__ushort_as_half(se[i]));  // exact; 0 on padding
      }
      rotate_store(v, q, live ? xh + ((int64_t)s * rows + r) * k + col : nullptr);
    }
  }
}

namespace {

// Blocks that stay resident on the device at once (read once per device and
// kernel variant): the grid is exactly that, so every warp streams through many
// passes with the next pass's loads in flight.
template <int ID, typename Kernel>
int resident_blocks(Kernel kern, int threads) {
  static int cache[64] = {};  // one cache per ID (one ID per kernel)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152 * 2;
  if (cache[dev] == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
    cache[dev] = (sms > 0 ? sms : 152) * (per_sm > 0 ? per_sm : 1);  // benign race: same value
  }
  return cache[dev];
}

}  // namespace

cudaError_t launch_input_transform(const void* x, bool x_bf16, int64_t m, int64_t k, const uint16_t* suh,
                                   int num_shards, uint16_t* xh, cudaStream_t stream) {
  const int64_t groups = (m * (k >> 7) + 7) / 8;  // one warp pass each
  const int threads = 256;
  const int64_t want = (groups + 7) / 8;
  const int cap = x_bf16 ? resident_blocks<0>(input_transform_kernel<true>, threads)
                         : resident_blocks<1>(input_transform_kernel<false>, threads);
  const int blocks = (int)(want < cap ? want : cap);
  if (x_bf16) {
    input_transform_kernel<true><<<blocks, threads, 0, stream>>>((const uint16_t*)x, m, k, suh, num_shards, xh);
  } else {
    input_transform_kernel<false><<<blocks, threads, 0, stream>>>((const uint16_t*)x, m, k, suh, num_shards, xh);
  }
  return cudaGetLastError();
}

cudaError_t launch_input_transform_swiglu(const void* gate_up, bool bf16, int64_t m, int64_t k, const uint16_t* suh,
                                          int num_shards, uint16_t* xh, cudaStream_t stream) {
  const int64_t groups = (m * (k >> 7) + 7) / 8;
  const int threads = 256;
  const int64_t want = (groups + 7) / 8;
  const int cap = bf16 ? resident_blocks<2>(input_transform_swiglu_kernel<true>, threads)
                       : resident_blocks<3>(input_transform_swiglu_kernel<false>, threads);
  const int blocks = (int)(want < cap ? want : cap);
  if (bf16) {
    input_transform_swiglu_kernel<true><<<blocks, threads, 0, stream>>>((const uint16_t*)gate_up, m, k, suh,
                                                                        num_shards, xh);
  } else {
    input_transform_swiglu_kernel<false><<<blocks, threads, 0, stream>>>((const uint16_t*)gate_up, m, k, suh,
                                                                         num_shards, xh);
  }
  return cudaGetLastError();
}

cudaError_t launch_moe_input_transform(const void* x, bool x_bf16, int64_t num_tokens, int64_t k,
                                       const int32_t* sorted_ids, int64_t rows, int32_t topk,
                                       const int32_t* block_expert, int32_t block, const uint16_t* suh,
                                       int num_shards, int num_experts, uint16_t* xh, cudaStream_t stream) {
  const int64_t groups = (rows * (k >> 7) + 7) / 8;
  const int threads = 256;
  const int64_t want = (groups + 7) / 8;
  const int cap = x_bf16 ? resident_blocks<4>(moe_input_transform_kernel<true>, threads)
                         : resident_blocks<5>(moe_input_transform_kernel<false>, threads);
  const int blocks = (int)(want < cap ? want : cap);
  if (x_bf16) {
    moe_input_transform_kernel<true><<<blocks, threads, 0, stream>>>((const uint16_t*)x, num_tokens, k, sorted_ids,
                                                                     rows, topk, block_expert, block, suh, num_shards,
                                                                     num_experts, xh);
  } else {
    moe_input_transform_kernel<false><<<blocks, threads, 0, stream>>>((const uint16_t*)x, num_tokens, k, sorted_ids,
                                                                      rows, topk, block_expert, block, suh,
                                                                      num_shards, num_experts, xh);
  }
  return cudaGetLastError();
}

}  // namespace exl3
