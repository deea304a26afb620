// exl3_gemm_mma.cuh -- EXL3 GEMM on warp-level mma.sync (m16n8k16, fp16 x fp16 -> fp32).
//
// A CTA owns one 128-column block (one output Hadamard block) and BM = 16*MT
// rows, over a contiguous range of whole 128-row blocks of k (the whole k
// extent unless split-k).  Warp w decodes the 16-column trellis tile strip w of
// the block: for every k16 step the lane reads its window words of tile
// (kt, nt), decodes its 8 values straight into the two B fragments of the n8
// halves, and multiplies them against every 16-row A fragment of the CTA's rows,
// so each tile is decoded exactly once per CTA (cuda-exl3 README, "What
// profiling found": a warp tile one tile wide avoids decoding a tile twice;
// "Why custom kernels": a block covering all of k streams its trellis once).  The activations xh stream through shared memory with
// cp.async in 128-wide chunks, double-buffered.
//
// Epilogue (parts == 1): fp32 z -> shared -> per-row 128-point butterfly ->
// *2^-3 * svh -> bf16/fp16.  With parts > 1 the fp32 partial goes to the split-k
// workspace instead (cuda-exl3 README, "One op per layer", split-k).
//
// The fp32 sum over k is a sequence of mma.sync k16 steps in ascending k,
// identical for every row whatever m is, so rows are byte-equal across batch
// sizes (TensorFold PR #740, "Arithmetic": rows never mix).
#pragma once

#include "exl3_device.cuh"
#include "exl3_launch.h"
#include "exl3_ptx.cuh"

namespace exl3 {

constexpr int kMmaThreads = 256;  // 8 warps = 8 tile columns = one 128-column block
constexpr int kChunkK = 128;      // k per shared-memory chunk
constexpr int kLdsHalves = kChunkK + 8;  // padded row stride of the xh chunk (halves)
constexpr int kZStride = 128 + 8;        // padded row stride of the fp32 z tile (floats)

template <int MT>
constexpr int mma_smem_bytes() {
  return 2 * 16 * MT * kLdsHalves * 2 > 16 * MT * kZStride * 4 ? 2 * 16 * MT * kLdsHalves * 2
                                                                 : 16 * MT * kZStride * 4;
}

template <int BITS, int CB, int MT>
__global__ void __launch_bounds__(kMmaThreads, 1) gemm_mma_kernel(const GemmArgs a) {
  constexpr int BM = 16 * MT;
  constexpr int TW = 8 * BITS;  // 32-bit words per tile
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t c0 = (int64_t)blockIdx.x * 128;
  const int64_t r0 = (int64_t)blockIdx.y * BM;

  int shard = 0;
  while (shard + 1 < a.num_shards && c0 >= a.shard_cols[shard + 1]) ++shard;
  const uint16_t* xsrc = a.xh + (int64_t)shard * a.m * a.k;

  const int64_t kblocks = a.k >> 7;
  const int64_t kb0 = ((int64_t)blockIdx.z * kblocks) / a.parts;
  const int64_t kb1 = ((int64_t)(blockIdx.z + 1) * kblocks) / a.parts;
  const int nchunks = (int)(kb1 - kb0);

  const int64_t NT = a.n >> 4;
  const int64_t nt = (c0 >> 4) + warp;
  const uint32_t* tr32 = reinterpret_cast<const uint32_t*>(a.trellis);
  const LaneWindow<BITS> lw(lane);
  const MulConsts mc(a.one);
  const int64_t kt_begin = kb0 * 8;
  const int64_t kt_last = kb1 * 8 - 1;

  auto load_chunk = [&](int chunk, int buf) {
    const int64_t kbase = (kb0 + chunk) * kChunkK;
    uint16_t* dst = xs + buf * BM * kLdsHalves;
    for (int i = threadIdx.x; i < BM * 16; i += kMmaThreads) {
      const int row = i >> 4;
      const int piece = i & 15;
      const int64_t gr = r0 + row;
      const bool valid = gr < a.m;
      const uint16_t* src = xsrc + (valid ? gr : 0) * a.k + kbase + piece * 8;
      cp_async16(smem_u32(dst + row * kLdsHalves + piece * 8), src, valid ? 16 : 0);
    }
    cp_async_commit();
  };

  auto load_words = [&](int64_t kt, uint32_t (&w)[3]) {
    const int64_t ktc = kt < kt_last ? kt : kt_last;
    const uint32_t* t = tr32 + (ktc * NT + nt) * TW;
    w[0] = ldg_nc_u32(t + lw.idx[0]);
    w[1] = ldg_nc_u32(t + lw.idx[1]);
    w[2] = (LaneWindow<BITS>::kNeed == 3) ? ldg_nc_u32(t + lw.idx[2]) : 0u;
  };

  float acc[MT][2][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][h][i] = 0.f;

  uint32_t wr[4][3];
#pragma unroll
  for (int d = 0; d < 4; ++d) load_words(kt_begin + d, wr[d]);
  load_chunk(0, 0);

  for (int c = 0; c < nchunks; ++c) {
    if (c + 1 < nchunks) {
      load_chunk(c + 1, (c + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t* xb = xs + (c & 1) * BM * kLdsHalves;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t kt = kt_begin + (int64_t)c * 8 + j;
      const Aligned al = align_window<BITS>(wr[j & 3][0], wr[j & 3][1], wr[j & 3][2], lw.off);
      load_words(kt + 4, wr[j & 3]);
      uint32_t b[4];
      decode_lane<BITS, CB>(al, mc, b);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t af[4];
        ldmatrix_x4(af, smem_u32(xb + (mt * 16 + (lane & 15)) * kLdsHalves + j * 16 + (lane >> 4) * 8));
        mma_16816(acc[mt][0], af, b[0], b[1]);
        mma_16816(acc[mt][1], af, b[2], b[3]);
      }
    }
    __syncthreads();
  }

  const int g = lane >> 2;
  const int q = lane & 3;
  if (a.parts > 1) {
    float* dst = a.acc + (int64_t)blockIdx.z * a.m * a.n;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t col = c0 + warp * 16 + h * 8 + 2 * q;
        const int64_t ra = r0 + mt * 16 + g;
        if (ra < a.m) *reinterpret_cast<float2*>(dst + ra * a.n + col) = make_float2(acc[mt][h][0], acc[mt][h][1]);
        if (ra + 8 < a.m)
          *reinterpret_cast<float2*>(dst + (ra + 8) * a.n + col) = make_float2(acc[mt][h][2], acc[mt][h][3]);
      }
    return;
  }

  float* zs = reinterpret_cast<float*>(smem_raw);
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float* p0 = zs + (mt * 16 + g) * kZStride + warp * 16 + h * 8 + 2 * q;
      *reinterpret_cast<float2*>(p0) = make_float2(acc[mt][h][0], acc[mt][h][1]);
      *reinterpret_cast<float2*>(p0 + 8 * kZStride) = make_float2(acc[mt][h][2], acc[mt][h][3]);
    }
  __syncthreads();

  const uint2 sv = *reinterpret_cast<const uint2*>(a.svh + c0 + 4 * lane);
  const float svf[4] = {__half2float(__ushort_as_half((uint16_t)(sv.x & 0xFFFF))),
                        __half2float(__ushort_as_half((uint16_t)(sv.x >> 16))),
                        __half2float(__ushort_as_half((uint16_t)(sv.y & 0xFFFF))),
                        __half2float(__ushort_as_half((uint16_t)(sv.y >> 16)))};
  const bool bf16 = a.y_bf16 != 0;
  uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
  for (int row = warp; row < BM; row += kMmaThreads / 32) {
    const int64_t gr = r0 + row;
    if (gr >= a.m) break;
    const float4 z4 = *reinterpret_cast<const float4*>(zs + row * kZStride + 4 * lane);
    float v[4] = {z4.x, z4.y, z4.z, z4.w};
    fwht128_warp(v, lane);
    uint16_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = f32_to_out((v[i] * 0.125f) * svf[i], bf16);
    uint2 w;
    w.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
    w.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
    *reinterpret_cast<uint2*>(y + gr * a.n + c0 + 4 * lane) = w;
  }
}

template <int BITS, int CB, int MT>
cudaError_t launch_mma_variant(const GemmArgs& a, cudaStream_t stream) {
  constexpr int smem = mma_smem_bytes<MT>();
  auto kern = gemm_mma_kernel<BITS, CB, MT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)(a.n / 128), (unsigned)((a.m + 16 * MT - 1) / (16 * MT)), (unsigned)a.parts);
  kern<<<grid, kMmaThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int BITS, int CB>
cudaError_t launch_mma_cb(const GemmArgs& a, cudaStream_t stream) {
  if (a.m <= 16) return launch_mma_variant<BITS, CB, 1>(a, stream);
  if (a.m <= 32) return launch_mma_variant<BITS, CB, 2>(a, stream);
  if (a.m <= 64) return launch_mma_variant<BITS, CB, 4>(a, stream);
  return launch_mma_variant<BITS, CB, 8>(a, stream);
}

template <int BITS>
cudaError_t launch_gemm_mma_bits(const GemmArgs& a, int cb, cudaStream_t stream) {
  switch (cb) {
    case CB_3INST:
      return launch_mma_cb<BITS, CB_3INST>(a, stream);
    case CB_MCG:
      return launch_mma_cb<BITS, CB_MCG>(a, stream);
    default:
      return launch_mma_cb<BITS, CB_MUL1>(a, stream);
  }
}

}  // namespace exl3
