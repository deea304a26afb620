// exl3_noalloc.cu -- split-k GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device workspace: a plugin running inside
// a host program that owns the allocator and exposes no allocation hook, or
// code that must not call cudaMalloc because it would synchronise the device or
// fragment a carefully budgeted memory pool.  exl3_gemm_splitk_noalloc gives
// them the split-k GEMM without a workspace argument: its fp32 partials live in
// a fixed array compiled into this library.  The array occupies
// EXL3_NOALLOC_SCRATCH_BYTES on every GPU that loads the library, for as long as
// the process runs.
#include "../../include/exl3.h"

namespace {

constexpr size_t kScratchFloats = EXL3_NOALLOC_SCRATCH_BYTES / sizeof(float);

// The scratch buffer.  In host code this name is only a stand-in for the symbol,
// not a device address: the address is obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

// Device address of the scratch array in the current device's context.  It is
// looked up on every call (a table lookup that allocates nothing), so a context
// torn down and rebuilt by cudaDeviceReset never leaves a stale address behind.
exl3_status_t scratch_for_current_device(float** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return EXL3_ECUDA;
  *out = static_cast<float*>(p);
  return EXL3_OK;
}

}  // namespace

extern "C" exl3_status_t exl3_gemm_splitk_noalloc(const uint16_t* xh, int64_t m, int64_t k, const int16_t* trellis,
                                                  int32_t bits, exl3_codebook_t cb, const uint16_t* svh,
                                                  const int32_t* shard_cols, int32_t num_shards, void* y,
                                                  exl3_dtype_t y_dtype, int64_t n, void* stream) {
  if (m < 0 || exl3_splitk_parts(k, n) <= 0) return EXL3_EINVAL;
  if (exl3_splitk_workspace_bytes(m, k, n) > EXL3_NOALLOC_SCRATCH_BYTES) return EXL3_EWORKSPACE;
  float* scratch = nullptr;
  const exl3_status_t st = scratch_for_current_device(&scratch);
  if (st != EXL3_OK) return st;
  // The parts overwrite every partial the epilogue reads, so leftovers from an
  // earlier call are never used; the epilogue also leaves the array zeroed.
  return exl3_gemm_splitk(xh, m, k, trellis, bits, cb, svh, shard_cols, num_shards, y, y_dtype, n, scratch,
                          EXL3_NOALLOC_SCRATCH_BYTES, stream);
}
