// exl3_gemm_mma_inst.cu -- one translation unit per trellis width; the build
// compiles this file once for each EXL3_INST_BITS in 1..8 so the 96 kernel
// instantiations (8 widths x 3 codebooks x 4 row tiles) compile in parallel.
#include "exl3_gemm_mma.cuh"

#ifndef EXL3_INST_BITS
#error "compile with -DEXL3_INST_BITS=<1..8>"
#endif

namespace exl3 {
template cudaError_t launch_gemm_mma_bits<EXL3_INST_BITS>(const GemmArgs&, int, cudaStream_t);
}  // namespace exl3
