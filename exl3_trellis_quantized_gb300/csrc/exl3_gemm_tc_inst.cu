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
}  // namespace exl3
