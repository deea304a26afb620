// exl3_transform.cu -- input rotation of the EXL3 linear layer.
//
// For every shard s, row r and 128-block b of k:
//   xh[s][r][128b+i] = fp16_rne(2^-4 * sum_j H[i][j] * (x[r][128b+j] * suh[s][128b+j]))
// (TensorFold PR #740, "Arithmetic" step 1: x*suh, the 128-point Hadamard in a
// fixed order of fp32 adds, times 2^-4, one rounding to fp16; cuda-exl3 README,
// "One op per layer": every shard in one launch, x read once, the bf16 -> fp16
// conversion folded into the same pass).
//
// The plain transform gives eight lanes to one (row, 128-block): lane p of the
// eight holds elements 16p..16p+15, so a warp covers four blocks (1 KB of x)
// per pass with 16-byte loads.  Butterfly stages of stride 1..8 stay in
// registers; for the stride-16, -32 and -64 stages the warp regroups its blocks
// once through shared memory (rotate_store16).  The SwiGLU and grouped-expert
// transforms use the same layout.
// Each stage computes (a, b) -> (a + b, a - b) on the same pairs as the plain
// definition, so the order of fp32 adds is the fixed one.  x is read once and reused for
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

// The Hadamard butterfly of a block over eight lanes, 16 values a lane
// (elements 16p..16p+15 of lane p of the eight), times 2^-4, rounded to fp16
// and stored at dst (nothing is stored when dst is null; the lane still takes
// part in the exchange).  74 registers in the plain transform against 110-127
// for a four-lane form (32 values a lane), so three blocks of eight warps stay
// resident per SM instead of two (measured 3-17% faster, most at m <= 512).
// Strides 1..8 run in registers; one pass through the
// warp's shared-memory area (four blocks of 128 floats, 144 apart so the two
// blocks of a half-warp land on different banks) regroups each lane to
// elements 16t + 2p + e (t = 0..7, e = 0, 1), whose stride-16, -32 and -64
// partners it then holds; the 16-byte chunks are written with their slot XORed
// by p / 2, so a quarter-warp's writes cover all 32 banks.  Every stage maps
// the same pairs (a, b) -> (a + b, a - b) in the same stride order, so the fp32
// sums are the definition's.  Each lane stores 4 bytes per t, a block 32
// contiguous bytes per t.
__device__ __forceinline__ void rotate_store16(float (&v)[16], int p, float* xp, uint16_t* dst) {
#pragma unroll
  for (int st = 1; st < 16; st <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & st) == 0) {
        const float a = v[i], b = v[i + st];
        v[i] = a + b;
        v[i + st] = a - b;
      }
    }
  }
  float* blk = xp + ((threadIdx.x & 31) >> 3) * 144;
  __syncwarp();  // the previous pass's reads of xp are done
#pragma unroll
  for (int i4 = 0; i4 < 4; ++i4) {
    const int slot = i4 ^ (p >> 1);
    *reinterpret_cast<float4*>(blk + 16 * p + 4 * slot) = make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]);
  }
  __syncwarp();
  float w[8][2];  // w[t][e] = element 16t + 2p + e
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const float2 f = *reinterpret_cast<const float2*>(blk + 16 * t + 4 * ((p >> 1) ^ (t >> 1)) + 2 * (p & 1));
    w[t][0] = f.x;
    w[t][1] = f.y;
  }
#pragma unroll
  for (int st = 1; st < 8; st <<= 1) {  // element strides 16, 32, 64
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      if ((t & st) == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float a = w[t][e], b = w[t + st][e];
          w[t][e] = a + b;
          w[t + st][e] = a - b;
        }
      }
    }
  }
  if (dst != nullptr) {
    uint16_t* base = dst - 16 * p + 2 * p;  // element 2p of the block
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      // 2^-4 is exact; both values rounded to fp16 by one conversion
      const __half2 hv = __floats2half2_rn(w[t][0] * 0.0625f, w[t][1] * 0.0625f);
      *reinterpret_cast<uint32_t*>(base + 16 * t) = *reinterpret_cast<const uint32_t*>(&hv);
    }
  }
}

}  // namespace

template <bool X_BF16>
__device__ __forceinline__ float to_f32(uint16_t e) {
  return X_BF16 ? __bfloat162float(__ushort_as_bfloat16(e)) : __half2float(__ushort_as_half(e));
}

// Both elements of a packed pair (low half first) as fp32, exactly: bf16 by
// moving its bits to the top of the word, fp16 by the paired conversion.
template <bool X_BF16>
__device__ __forceinline__ float2 pair_to_f32(uint32_t w) {
  if (X_BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// v[0..7] = x * suh for one 16-byte chunk of each (exact in fp32).
template <bool X_BF16>
__device__ __forceinline__ void scale_chunk(const uint4 xw, const uint4 sw, float* v) {
  const uint32_t xs[4] = {xw.x, xw.y, xw.z, xw.w};
  const uint32_t ss[4] = {sw.x, sw.y, sw.z, sw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 xf = pair_to_f32<X_BF16>(xs[i]);
    const float2 sf = pair_to_f32<false>(ss[i]);
    v[2 * i] = xf.x * sf.x;
    v[2 * i + 1] = xf.y * sf.y;
  }
}

template <bool X_BF16>
__global__ void __launch_bounds__(256) input_transform_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                              const uint16_t* __restrict__ suh, int num_shards,
                                                              uint16_t* __restrict__ xh) {
  // The GEMM that consumes xh may be scheduled now: it prefetches its weights
  // and waits for this grid to complete before it reads xh.
  pdl_launch_dependents();
  __shared__ __align__(16) float xpose[8][4 * 144];  // per warp: its four blocks for the stride-16..64 stages
  float* const xp = xpose[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const int p = lane & 7;  // which 16 elements of the block
  const int64_t kb = k >> 7;
  const int64_t units = m * kb;
  const int64_t groups = (units + 3) / 4;  // four blocks per warp and pass
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  // The lane's unit u = g * 4 + lane / 8 advances by 4 * warps_total units a
  // pass; its (row, block) is stepped, not divided out, each pass.
  int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t step = 4 * warps_total;
  const int64_t step_rows = step / kb, step_blk = step - step_rows * kb;
  int64_t u = g * 4 + (lane >> 3);
  int64_t row = u / kb, blk = u - row * kb;
  // x stays packed (bf16 / fp16 pairs) in registers; the next pass's words are
  // loaded before this pass computes, so two passes of loads are in flight
  uint4 cur[2];
#pragma unroll
  for (int c = 0; c < 2; ++c)
    cur[c] = (g < groups && u < units) ? *reinterpret_cast<const uint4*>(x + row * k + blk * 128 + 16 * p + 8 * c)
                                       : make_uint4(0, 0, 0, 0);
  for (; g < groups; g += warps_total, u += step) {
    int64_t nrow = row + step_rows, nblk = blk + step_blk;
    if (nblk >= kb) {
      nblk -= kb;
      nrow += 1;
    }
    const bool nok = g + warps_total < groups && u + step < units;
    uint4 nxt[2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
      nxt[c] = nok ? *reinterpret_cast<const uint4*>(x + nrow * k + nblk * 128 + 16 * p + 8 * c) : make_uint4(0, 0, 0, 0);
    const bool ok = u < units;
    const int64_t col = ok ? blk * 128 + 16 * p : 16 * p;
    for (int s = 0; s < num_shards; ++s) {
      float v[16];
#pragma unroll
      for (int c = 0; c < 2; ++c)
        scale_chunk<X_BF16>(cur[c], *reinterpret_cast<const uint4*>(suh + (int64_t)s * k + col + 8 * c), v + 8 * c);
      rotate_store16(v, p, xp, ok ? xh + ((int64_t)s * m + row) * k + col : nullptr);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) cur[c] = nxt[c];
    row = nrow;
    blk = nblk;
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
  __shared__ __align__(16) float xpose[8][4 * 144];  // per warp: its four blocks for the stride-16..64 stages
  float* const xp = xpose[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const int p = lane & 7;  // which 16 elements of the block
  const int64_t kb = k >> 7;
  const int64_t units = m * kb;
  const int64_t groups = (units + 3) / 4;  // four blocks per warp and pass
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  // the lane's unit advances by 4 * warps_total a pass: (row, block) stepped
  const int64_t step = 4 * warps_total;
  const int64_t step_rows = step / kb, step_blk = step - step_rows * kb;
  auto load = [&](bool ok, int64_t row, int64_t col, uint4 (&gw)[2], uint4 (&uw)[2]) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      gw[c] = ok ? *reinterpret_cast<const uint4*>(gu + row * 2 * k + col + 8 * c) : make_uint4(0, 0, 0, 0);
      uw[c] = ok ? *reinterpret_cast<const uint4*>(gu + row * 2 * k + k + col + 8 * c) : make_uint4(0, 0, 0, 0);
    }
  };
  int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int64_t u = g * 4 + (lane >> 3);
  int64_t row = u / kb, blk = u - row * kb;
  uint4 cg[2], cu[2];
  load(g < groups && u < units, row, blk * 128 + 16 * p, cg, cu);
  for (; g < groups; g += warps_total, u += step) {
    int64_t nrow = row + step_rows, nblk = blk + step_blk;
    if (nblk >= kb) {
      nblk -= kb;
      nrow += 1;
    }
    const bool nok = g + warps_total < groups && u + step < units;
    uint4 ng[2], nu[2];
    load(nok, nrow, nblk * 128 + 16 * p, ng, nu);
    float h[16];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint16_t ge[8], ue[8];
      unpack8(cg[c], ge);
      unpack8(cu[c], ue);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float gv = to_f32<X_BF16>(ge[i]);
        h[8 * c + i] = gv / (1.0f + expf(-gv)) * to_f32<X_BF16>(ue[i]);
      }
    }
    const bool ok = u < units;
    const int64_t col = ok ? blk * 128 + 16 * p : 16 * p;
    for (int s = 0; s < num_shards; ++s) {
      float v[16];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint16_t se[8];
        unpack8(*reinterpret_cast<const uint4*>(suh + (int64_t)s * k + col + 8 * c), se);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[8 * c + i] = h[8 * c + i] * __half2float(__ushort_as_half(se[i]));
      }
      rotate_store16(v, p, xp, ok ? xh + ((int64_t)s * m + row) * k + col : nullptr);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      cg[c] = ng[c];
      cu[c] = nu[c];
    }
    row = nrow;
    blk = nblk;
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
  __shared__ __align__(16) float xpose[8][4 * 144];  // per warp: its four blocks for the stride-16..64 stages
  float* const xp = xpose[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const int p = lane & 7;  // which 16 elements of the block
  const int64_t kb = k >> 7;
  const int64_t units = rows * kb;
  const int64_t groups = (units + 3) / 4;  // four blocks per warp and pass
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t pairs = num_tokens * topk;
  const int block_shift = block == 16 ? 4 : block == 32 ? 5 : 7;  // block is 16, 32 or 128 rows
  // the lane's unit advances by 4 * warps_total a pass: (row, block) stepped
  const int64_t step = 4 * warps_total;
  const int64_t step_rows = step / kb, step_blk = step - step_rows * kb;
  int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int64_t u = g * 4 + (lane >> 3);
  int64_t ur = u / kb, ub = u - ur * kb;
  for (; g < groups; g += warps_total, u += step) {
    const bool in_range = u < units;
    const int64_t r = in_range ? ur : 0;
    const int64_t col = (in_range ? ub * 128 : 0) + 16 * p;
    ub += step_blk;
    ur += step_rows;
    if (ub >= kb) {
      ub -= kb;
      ur += 1;
    }
    const int e = in_range ? block_expert[r >> block_shift] : -1;
    const bool live = e >= 0 && e < num_experts;
    const int64_t id = live ? (int64_t)sorted_ids[r] : -1;
    // pair ids stay below num_tokens * topk <= 2^28: a 32-bit division
    const int64_t tok = (id >= 0 && id < pairs) ? (int64_t)((uint32_t)id / (uint32_t)topk) : -1;
    uint4 xw[2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
      xw[c] = tok >= 0 ? *reinterpret_cast<const uint4*>(x + tok * k + col + 8 * c) : make_uint4(0, 0, 0, 0);
    for (int s = 0; s < num_shards; ++s) {
      float v[16];
#pragma unroll
      for (int c = 0; c < 2; ++c)  // 0 on padding rows
        scale_chunk<X_BF16>(xw[c],
                            tok >= 0 ? *reinterpret_cast<const uint4*>(suh + ((int64_t)e * num_shards + s) * k + col + 8 * c)
                                     : make_uint4(0, 0, 0, 0),
                            v + 8 * c);
      rotate_store16(v, p, xp, live ? xh + ((int64_t)s * rows + r) * k + col : nullptr);
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
  const int64_t groups = (m * (k >> 7) + 3) / 4;  // one warp pass each (four blocks)
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
  const int64_t groups = (m * (k >> 7) + 3) / 4;  // one warp pass each (four blocks)
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
  const int64_t groups = (rows * (k >> 7) + 3) / 4;  // one warp pass each (four blocks)
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
