// exl3_tc_host.cu -- host side of the tcgen05 GEMM: the TMA tensor map of the
// rotated activations, the tile-shape choice and the width dispatch.
#include <cudaTypedefs.h>

#include <mutex>

#include "exl3_launch.h"

namespace exl3 {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// xh is fp16 [S][m][k]; tiles are 64 (k) x box_rows (rows) x 1 (shard), 128-byte
// swizzled, out-of-range rows read as zeros.
cudaError_t make_xh_map(CUtensorMap* map, const uint16_t* xh, int64_t m, int64_t k, int num_shards, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)k, (cuuint64_t)m, (cuuint64_t)num_shards};
  cuuint64_t strides[2] = {(cuuint64_t)k * 2, (cuuint64_t)(m * k * 2)};
  cuuint32_t box[3] = {(cuuint32_t)kTcBK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(xh), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(const GemmArgs& a, int bits, int cb, cudaStream_t stream) {
  TcParams p;
  p.a = a;
  p.box_rows = a.m >= 128 ? 128 : (int)((a.m + 7) / 8 * 8);
  CUtensorMap map;
  cudaError_t e = make_xh_map(&map, a.xh, a.m, a.k, a.num_shards, p.box_rows);
  if (e != cudaSuccess) return e;
  const int bn = 128, rg = 1;
  switch (bits) {
    case 1: return launch_gemm_tc_bits<1>(map, p, cb, bn, rg, stream);
    case 2: return launch_gemm_tc_bits<2>(map, p, cb, bn, rg, stream);
    case 3: return launch_gemm_tc_bits<3>(map, p, cb, bn, rg, stream);
    case 4: return launch_gemm_tc_bits<4>(map, p, cb, bn, rg, stream);
    case 5: return launch_gemm_tc_bits<5>(map, p, cb, bn, rg, stream);
    case 6: return launch_gemm_tc_bits<6>(map, p, cb, bn, rg, stream);
    case 7: return launch_gemm_tc_bits<7>(map, p, cb, bn, rg, stream);
    default: return launch_gemm_tc_bits<8>(map, p, cb, bn, rg, stream);
  }
}

cudaError_t take_device_errors(uint32_t* flags) {
  *flags = 0;
  cudaError_t e = cudaSuccess;
  cudaError_t (*fns[8])(uint32_t*) = {take_device_error_tc<1>, take_device_error_tc<2>, take_device_error_tc<3>,
                                      take_device_error_tc<4>, take_device_error_tc<5>, take_device_error_tc<6>,
                                      take_device_error_tc<7>, take_device_error_tc<8>};
  for (auto f : fns) {
    cudaError_t r = f(flags);
    if (r != cudaSuccess) e = r;
  }
  return e;
}

}  // namespace exl3
