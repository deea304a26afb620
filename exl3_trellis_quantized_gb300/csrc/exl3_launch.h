// exl3_launch.h -- internal host-side launchers (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace exl3 {

constexpr int kMaxShards = 8;

// Everything one GEMM launch needs; passed by value as a kernel parameter.
struct GemmArgs {
  const uint16_t* xh;      // fp16 [S][m][k]
  const int16_t* trellis;  // int16 [k/16][n/16][16*bits]
  const uint16_t* svh;     // fp16 [n]
  void* y;                 // [m][n], bf16 or fp16
  float* acc;              // split-k workspace fp32 [P][m][n], or nullptr
  int64_t m, k, n;
  int32_t shard_cols[kMaxShards + 1];
  int32_t num_shards;
  int32_t parts;  // P (1 = no split)
  int32_t y_bf16;
  uint32_t one;  // always 1: seeds the decoder's multiplier constants at run time
};

cudaError_t launch_input_transform(const void* x, bool x_bf16, int64_t m, int64_t k, const uint16_t* suh,
                                   int num_shards, uint16_t* xh, cudaStream_t stream);

// mma.sync GEMM mainloop; with args.parts > 1 it writes fp32 partials to args.acc.
cudaError_t launch_gemm_mma(const GemmArgs& args, int bits, int cb, cudaStream_t stream);

// Sum the P partials in part order, rotate, scale, store y, zero the workspace.
cudaError_t launch_splitk_epilogue(const GemmArgs& args, cudaStream_t stream);

cudaError_t launch_test_codebook(int cb, uint16_t* out, cudaStream_t stream);
cudaError_t launch_test_unpack(const int16_t* trellis, int bits, int cb, int64_t k, int64_t n, uint16_t* wq,
                               cudaStream_t stream);

// tcgen05 GEMM (one translation unit per width); parts > 1 is not handled here.
constexpr int kTcBK = 64;  // k per pipeline stage (one 128-byte swizzle row of fp16)
struct TcParams {
  GemmArgs a;
  int32_t box_rows;  // rows per xh tile copy (<= 128)
};
cudaError_t launch_gemm_tc(const GemmArgs& args, int bits, int cb, cudaStream_t stream);
template <int BITS>
cudaError_t launch_gemm_tc_bits(const CUtensorMap& xmap, const TcParams& p, int cb, int bn, int rg,
                                cudaStream_t stream);
// Read and clear the wait-timeout flags of every kernel translation unit (synchronous).
cudaError_t take_device_errors(uint32_t* flags);
template <int BITS>
cudaError_t take_device_error_tc(uint32_t* flags);

// Per-width instantiations of the mma.sync GEMM (one translation unit per width).
template <int BITS>
cudaError_t launch_gemm_mma_bits(const GemmArgs& args, int cb, cudaStream_t stream);

}  // namespace exl3
