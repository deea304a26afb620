// exl3_kernels_misc.cu -- the split-k epilogue and the test-only decode kernels.
#include "exl3_device.cuh"
#include "exl3_launch.h"

namespace exl3 {

// Split-k epilogue (cuda-exl3 README, "One op per layer": a second kernel turns
// the fp32 partials into outputs and leaves the buffer zeroed for the next call;
// TensorFold PR #740, "Arithmetic": parts are summed in a fixed part order).  One warp per (row, 128-column block); lane l owns
// columns 4l..4l+3 of the block: z = ((p0 + p1) + p2) + ..., then the same
// butterfly, scale and rounding as the fused epilogue, then zeros written back.
// P is a template argument, so a thread holds exactly P partials.
template <int P>
__global__ void __launch_bounds__(256) splitk_epilogue_kernel(const GemmArgs a) {
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
  switch (a.parts) {  // exl3_splitk_parts returns 2..16 whenever this runs
#define EXL3_SPLITK_CASE(P) \
  case P: splitk_epilogue_kernel<P><<<blocks, 256, 0, stream>>>(a); break;
    EXL3_SPLITK_CASE(2) EXL3_SPLITK_CASE(3) EXL3_SPLITK_CASE(4) EXL3_SPLITK_CASE(5) EXL3_SPLITK_CASE(6)
    EXL3_SPLITK_CASE(7) EXL3_SPLITK_CASE(8) EXL3_SPLITK_CASE(9) EXL3_SPLITK_CASE(10) EXL3_SPLITK_CASE(11)
    EXL3_SPLITK_CASE(12) EXL3_SPLITK_CASE(13) EXL3_SPLITK_CASE(14) EXL3_SPLITK_CASE(15) EXL3_SPLITK_CASE(16)
#undef EXL3_SPLITK_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Test-only kernels: the same device decode as the GEMM, written out densely.
// ---------------------------------------------------------------------------
template <int CB>
__global__ void test_codebook_kernel(uint16_t* out) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;  // states 2t, 2t+1
  if (t < 32768) reinterpret_cast<uint32_t*>(out)[t] = decode_pair<CB>(2u * t, 2u * t + 1u);
}

cudaError_t launch_test_codebook(int cb, uint16_t* out, cudaStream_t stream) {
  if (cb == CB_3INST) test_codebook_kernel<CB_3INST><<<128, 256, 0, stream>>>(out);
  else if (cb == CB_MCG) test_codebook_kernel<CB_MCG><<<128, 256, 0, stream>>>(out);
  else test_codebook_kernel<CB_MUL1><<<128, 256, 0, stream>>>(out);
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
