// exl3_kernels_misc.cu -- the split-k epilogue, the MoE combine and the test-only decode kernels.
#include "exl3_device.cuh"
#include "exl3_launch.h"
#include "exl3_sm100.cuh"

namespace exl3 {

// Split-k epilogue (cuda-exl3 README, "One op per layer": a second kernel turns
// the fp32 partials into outputs and leaves the buffer zeroed for the next call;
// TensorFold PR #740, "Arithmetic": parts are summed in a fixed part order).  One warp per (row, 128-column block); lane l owns
// columns 4l..4l+3 of the block: z = ((p0 + p1) + p2) + ..., then the same
// butterfly, scale and rounding as the fused epilogue, then zeros written back.
// P is a template argument, so a thread holds exactly P partials.  When the
// parts' GEMM triggers it (a.trigger_dependents == 2) it is launched as a
// programmatic dependent of that GEMM, scheduled before the GEMM ends: then
// nothing is read or written before the GEMM has completed (pdl_wait, which
// returns at once after a plain launch).
template <int P>
__global__ void __launch_bounds__(256) splitk_epilogue_kernel(const GemmArgs a) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t cb = a.n >> 7;
  const int64_t units = a.m * cb;
  const int64_t plane = a.m * a.n;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const bool bf16 = a.y_bf16 != 0;
  uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += warps_total) {
    const int64_t r = u / cb;
    const int64_t col = (u - r * cb) * 128 + 4 * lane;
    float* p = a.acc + r * a.n + col;
    // every part's partial first (all loads in flight together; a zero store
    // between them would order each load after the previous store), then the
    // sum in part order, then the zeros
    float4 t[P];
#pragma unroll
    for (int part = 0; part < P; ++part) t[part] = __ldcs(reinterpret_cast<const float4*>(p + part * plane));
    float4 s = t[0];
#pragma unroll
    for (int part = 1; part < P; ++part) {
      s.x = s.x + t[part].x;
      s.y = s.y + t[part].y;
      s.z = s.z + t[part].z;
      s.w = s.w + t[part].w;
    }
#pragma unroll
    for (int part = 0; part < P; ++part) __stcs(reinterpret_cast<float4*>(p + part * plane), make_float4(0.f, 0.f, 0.f, 0.f));
    float v[4] = {s.x, s.y, s.z, s.w};
    fwht128_warp(v, lane);
    const uint2 sv = *reinterpret_cast<const uint2*>(a.svh + col);
    const float svf[4] = {__half2float(__ushort_as_half((uint16_t)(sv.x & 0xFFFF))),
                          __half2float(__ushort_as_half((uint16_t)(sv.x >> 16))),
                          __half2float(__ushort_as_half((uint16_t)(sv.y & 0xFFFF))),
                          __half2float(__ushort_as_half((uint16_t)(sv.y >> 16)))};
    uint16_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = f32_to_out((v[i] * 0.125f) * svf[i], bf16);
    uint2 w;
    w.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
    w.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
    *reinterpret_cast<uint2*>(y + r * a.n + col) = w;
  }
}

cudaError_t launch_splitk_epilogue(const GemmArgs& a, cudaStream_t stream) {
  const int64_t units = a.m * (a.n >> 7);
  const int64_t want = (units + 7) / 8;
  const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
  void (*kern)(const GemmArgs) = nullptr;
  switch (a.parts) {  // exl3_splitk_parts returns 2..16 whenever this runs
#define EXL3_SPLITK_CASE(P) \
  case P: kern = splitk_epilogue_kernel<P>; break;
    EXL3_SPLITK_CASE(2) EXL3_SPLITK_CASE(3) EXL3_SPLITK_CASE(4) EXL3_SPLITK_CASE(5) EXL3_SPLITK_CASE(6)
    EXL3_SPLITK_CASE(7) EXL3_SPLITK_CASE(8) EXL3_SPLITK_CASE(9) EXL3_SPLITK_CASE(10) EXL3_SPLITK_CASE(11)
    EXL3_SPLITK_CASE(12) EXL3_SPLITK_CASE(13) EXL3_SPLITK_CASE(14) EXL3_SPLITK_CASE(15) EXL3_SPLITK_CASE(16)
#undef EXL3_SPLITK_CASE
    default: return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1u, 1u);
  cfg.blockDim = dim3(256u, 1u, 1u);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.trigger_dependents == 2 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// ---------------------------------------------------------------------------
// MoE combine: the weighted sum of each token's top-k expert rows (the pages
// run the routed experts as a grouped GEMM and leave this sum to the caller:
// cuda-exl3 README, "MoE notes").  Two launches, no atomics:
//   1. every row of a live block whose pair id p lies in [0, tokens * topk)
//      records pair_rows[p] = row;
//   2. per token and 8-column chunk, the slots in ascending order: a slot's
//      entry counts only when it names a row of a live block that holds this
//      very pair, so entries never written in this call (left from an earlier
//      call, or garbage) are ignored and the table needs no clearing; the sum
//      is fp32, w * y added with one fma per slot in slot order, then one
//      rounding to the output type.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_pair_rows_kernel(const int32_t* __restrict__ sorted_ids, int64_t rows,
                                                            const int32_t* __restrict__ block_expert,
                                                            int block_shift, int num_experts, int64_t pairs,
                                                            int32_t* __restrict__ pair_rows) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += stride) {
    const int e = block_expert[r >> block_shift];
    const int64_t p = sorted_ids[r];
    if (e >= 0 && e < num_experts && p >= 0 && p < pairs) pair_rows[p] = (int32_t)r;
  }
}

template <bool Y_BF16>
__device__ __forceinline__ float row_elem_to_f32(uint32_t e) {
  return Y_BF16 ? __bfloat162float(__ushort_as_bfloat16((uint16_t)e)) : __half2float(__ushort_as_half((uint16_t)e));
}

template <bool Y_BF16>
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint16_t* __restrict__ y, int64_t rows, int64_t n,
                                                          const int32_t* __restrict__ sorted_ids,
                                                          const int32_t* __restrict__ block_expert, int block_shift,
                                                          int num_experts, const float* __restrict__ weights,
                                                          int64_t num_tokens, int topk,
                                                          const int32_t* __restrict__ pair_rows,
                                                          uint16_t* __restrict__ out, bool out_bf16) {
  const int64_t chunks = n >> 3;
  const int64_t units = num_tokens * chunks;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
    const int64_t t = u / chunks;
    const int64_t c = (u - t * chunks) << 3;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // eight slots at a time: their table entries, then their checks, then
    // their rows are each loaded together (three rounds of independent loads
    // instead of three dependent loads per slot); the sum stays in slot order
    for (int s0 = 0; s0 < topk; s0 += 8) {
      int32_t r[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) r[j] = s0 + j < topk ? pair_rows[t * topk + s0 + j] : -1;
      bool live[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        live[j] = r[j] >= 0 && r[j] < rows;
        if (live[j]) {
          const int e = block_expert[r[j] >> block_shift];
          live[j] = (int64_t)sorted_ids[r[j]] == t * topk + s0 + j && e >= 0 && e < num_experts;
        }
      }
      uint4 v[8];
      float w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (live[j]) {
          v[j] = *reinterpret_cast<const uint4*>(y + (int64_t)r[j] * n + c);
          w[j] = weights[t * topk + s0 + j];
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (!live[j]) continue;
        const uint32_t vw[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(w[j], row_elem_to_f32<Y_BF16>(vw[i] & 0xFFFFu), acc[2 * i]);
          acc[2 * i + 1] = fmaf(w[j], row_elem_to_f32<Y_BF16>(vw[i] >> 16), acc[2 * i + 1]);
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = (uint32_t)f32_to_out(acc[2 * i], out_bf16) | ((uint32_t)f32_to_out(acc[2 * i + 1], out_bf16) << 16);
    *reinterpret_cast<uint4*>(out + t * n + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_moe_combine(const void* y, bool y_bf16, int64_t rows, int64_t n, const int32_t* sorted_ids,
                               const int32_t* block_expert, int32_t block, int num_experts, const float* weights,
                               int64_t num_tokens, int32_t topk, int32_t* pair_rows, void* out, bool out_bf16,
                               cudaStream_t stream) {
  const int shift = block == 16 ? 4 : block == 32 ? 5 : 7;
  if (rows > 0) {
    const int64_t want = (rows + 255) / 256;
    const int blocks = (int)(want < 152 * 8 ? want : 152 * 8);
    moe_pair_rows_kernel<<<blocks, 256, 0, stream>>>(sorted_ids, rows, block_expert, shift, num_experts,
                                                     num_tokens * topk, pair_rows);
  }
  if (num_tokens > 0) {
    const int64_t want = (num_tokens * (n >> 3) + 255) / 256;
    const int blocks = (int)(want < 152 * 8 ? want : 152 * 8);
    const uint16_t* yy = static_cast<const uint16_t*>(y);
    uint16_t* oo = static_cast<uint16_t*>(out);
    if (y_bf16) {
      moe_combine_kernel<true><<<blocks, 256, 0, stream>>>(yy, rows, n, sorted_ids, block_expert, shift, num_experts,
                                                           weights, num_tokens, topk, pair_rows, oo, out_bf16);
    } else {
      moe_combine_kernel<false><<<blocks, 256, 0, stream>>>(yy, rows, n, sorted_ids, block_expert, shift,
                                                            num_experts, weights, num_tokens, topk, pair_rows, oo,
                                                            out_bf16);
    }
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Test-only kernels: the same device decode as the GEMM, written out densely.
// ---------------------------------------------------------------------------
template <int CB>
__global__ void test_codebook_kernel(uint16_t* out, const DecodeConsts dc) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;  // states 2t, 2t+1
  if (t >= 32768) return;
  // Both decoders of a state pair: the table holds their common value, or
  // 0xFFFF (a NaN, which no state decodes to) where they disagree.
  const uint32_t v = decode_pair<CB>(2u * t, 2u * t + 1u);
  const uint32_t w = decode_pair_balanced<CB>(2u * t, 2u * t + 1u, dc);
  const uint32_t lo = (v & 0xFFFFu) == (w & 0xFFFFu) ? (v & 0xFFFFu) : 0xFFFFu;
  const uint32_t hi = (v >> 16) == (w >> 16) ? (v >> 16) : 0xFFFFu;
  reinterpret_cast<uint32_t*>(out)[t] = lo | (hi << 16);
}

cudaError_t launch_test_codebook(int cb, uint16_t* out, cudaStream_t stream) {
  DecodeConsts dc;
  fill_decode_consts(&dc);
  if (cb == CB_3INST) test_codebook_kernel<CB_3INST><<<128, 256, 0, stream>>>(out, dc);
  else if (cb == CB_MCG) test_codebook_kernel<CB_MCG><<<128, 256, 0, stream>>>(out, dc);
  else test_codebook_kernel<CB_MUL1><<<128, 256, 0, stream>>>(out, dc);
  return cudaGetLastError();
}

// One warp per tile; lane l writes its 8 values at their (k, n) positions.
template <int BITS, int CB>
__global__ void test_unpack_kernel(const int16_t* __restrict__ trellis, int64_t k, int64_t n, uint16_t* wq,
                                   const DecodeConsts dc) {
  DecodeConsts mc;
#pragma unroll
  for (int i = 0; i <= 16; ++i) mc.pow2[i] = dc.pow2[i];
  const int lane = threadIdx.x & 31;
  const int64_t NT = n >> 4;
  const int64_t tiles = (k >> 4) * NT;
  const int64_t tile = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (tile >= tiles) return;
  const int64_t kt = tile / NT, nt = tile - kt * NT;
  const LaneWindow<BITS> lw(lane);
  const uint32_t* tw = reinterpret_cast<const uint32_t*>(trellis) + tile * (8 * BITS);
  const Aligned al = load_lane_window<BITS>(tw, lw);
  uint32_t b[4];
  decode_lane<BITS, CB>(al, mc, b);
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t kk = kt * 16 + 2 * q + ((r & 1) ? 8 : 0);
    const int64_t nn = nt * 16 + g + ((r & 2) ? 8 : 0);
    wq[kk * n + nn] = (uint16_t)(b[r] & 0xFFFF);
    wq[(kk + 1) * n + nn] = (uint16_t)(b[r] >> 16);
  }
}

template <int BITS>
static cudaError_t launch_unpack_bits(const int16_t* t, int cb, int64_t k, int64_t n, uint16_t* wq,
                                      cudaStream_t stream) {
  DecodeConsts dc;
  fill_decode_consts(&dc);
  const int64_t tiles = (k >> 4) * (n >> 4);
  const unsigned blocks = (unsigned)((tiles + 7) / 8);
  if (cb == CB_3INST) test_unpack_kernel<BITS, CB_3INST><<<blocks, 256, 0, stream>>>(t, k, n, wq, dc);
  else if (cb == CB_MCG) test_unpack_kernel<BITS, CB_MCG><<<blocks, 256, 0, stream>>>(t, k, n, wq, dc);
  else test_unpack_kernel<BITS, CB_MUL1><<<blocks, 256, 0, stream>>>(t, k, n, wq, dc);
  return cudaGetLastError();
}

cudaError_t launch_test_unpack(const int16_t* trellis, int bits, int cb, int64_t k, int64_t n, uint16_t* wq,
                               cudaStream_t stream) {
  switch (bits) {
    case 1: return launch_unpack_bits<1>(trellis, cb, k, n, wq, stream);
    case 2: return launch_unpack_bits<2>(trellis, cb, k, n, wq, stream);
    case 3: return launch_unpack_bits<3>(trellis, cb, k, n, wq, stream);
    case 4: return launch_unpack_bits<4>(trellis, cb, k, n, wq, stream);
    case 5: return launch_unpack_bits<5>(trellis, cb, k, n, wq, stream);
    case 6: return launch_unpack_bits<6>(trellis, cb, k, n, wq, stream);
    case 7: return launch_unpack_bits<7>(trellis, cb, k, n, wq, stream);
    default: return launch_unpack_bits<8>(trellis, cb, k, n, wq, stream);
  }
}

}  // namespace exl3
