// exl3_gemm_tc_inst.cu -- the tcgen05 GEMM for one trellis width; the build
// compiles this file once per EXL3_INST_BITS in 1..8.
#include "exl3_gemm_tc.cuh"

#ifndef EXL3_INST_BITS
#error "compile with -DEXL3_INST_BITS=<1..8>"
#endif

namespace exl3 {
template cudaError_t launch_gemm_tc_bits<EXL3_INST_BITS>(const TcMaps&, const TcParams&, int, TcShape,
                                                         cudaStream_t);
template cudaError_t launch_moe_gemm_tc_bits<EXL3_INST_BITS>(const TcMaps&, const TcParams&, int, int,
                                                             cudaStream_t);

// This translation unit's wait-timeout flag (see exl3_sm100.cuh).
template <>
cudaError_t take_device_error_tc<EXL3_INST_BITS>(uint32_t* flags) {
  return take_tu_device_error(flags);
}

#if EXL3_INST_BITS == 1
namespace {
// The failure path of a bounded wait, on purpose: one CTA waits on an
// mbarrier that nothing ever arrives on.  The wait gives up after
// kWaitTimeoutNs, records kErrWaitTimeout in this translation unit's flag (which
// exl3_device_status reads) and returns; *out = 1 would mean it had returned
// normally.
__global__ void test_wait_timeout_kernel(uint32_t* out) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0u);
  if (threadIdx.x == 0) *out = ok ? 1u : 0u;
}
}  // namespace

cudaError_t launch_test_wait_timeout(uint32_t* out, cudaStream_t stream) {
  test_wait_timeout_kernel<<<1, 32, 0, stream>>>(out);
  return cudaGetLastError();
}
#endif
}  // namespace exl3
