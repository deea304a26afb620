// exl3_api.cu -- the C ABI declared in include/exl3.h: host-side validation,
// the shape-only split-k policy, and dispatch to the kernels.  Nothing here
// allocates device memory or synchronises the host.
#include <stdio.h>
#include <string.h>

#include "../../include/exl3.h"
#include "exl3_launch.h"

namespace {

thread_local char g_last_error[256] = "";

// Largest batch a call accepts (keeps every grid dimension within CUDA's limits).
constexpr int64_t kMaxRows = int64_t(1) << 22;

exl3_status_t cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return EXL3_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  return EXL3_ECUDA;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_kn(int64_t v) { return v >= 128 && v % 128 == 0 && v <= (int64_t(1) << 31); }

bool valid_cb(int cb) { return cb == EXL3_CB_3INST || cb == EXL3_CB_MCG || cb == EXL3_CB_MUL1; }

bool valid_dtype(int d) { return d == EXL3_F16 || d == EXL3_BF16; }

// Shard edges: 0 = c_0 < c_1 < ... < c_S = n, every edge a multiple of 128
// (cuda-exl3 README, "Loading into a dim vLLM has padded": Hadamard blocks are
// whole 128-column blocks; "Notes on the format": one suh row per shard).
bool valid_shards(const int32_t* cols, int32_t s, int64_t n) {
  if (cols == nullptr || s < 1 || s > EXL3_MAX_SHARDS) return false;
  if (cols[0] != 0 || cols[s] != n) return false;
  for (int i = 0; i < s; ++i) {
    if (cols[i + 1] <= cols[i] || cols[i + 1] % 128 != 0) return false;
  }
  return true;
}

// Validates everything exl3_gemm and exl3_gemm_splitk share and fills `a`.
// Grouped row blocks: 16 (the pages' floor for few tokens per expert), 32 or 128 rows.
bool valid_moe_block(int32_t block) { return block == 16 || block == 32 || block == 128; }

exl3_status_t check_gemm(const uint16_t* xh, int64_t m, int64_t k, const int16_t* trellis, int32_t bits,
                         exl3_codebook_t cb, const uint16_t* svh, const int32_t* shard_cols, int32_t num_shards,
                         void* y, exl3_dtype_t y_dtype, int64_t n, exl3::GemmArgs* a) {
  if (m < 0 || m > kMaxRows) return EXL3_EINVAL;
  if (!valid_kn(k) || !valid_kn(n)) return EXL3_EINVAL;
  if (bits < 1 || bits > 8 || !valid_cb(cb) || !valid_dtype(y_dtype)) return EXL3_EINVAL;
  if (!valid_shards(shard_cols, num_shards, n)) return EXL3_EINVAL;
  if (!aligned16(trellis) || !aligned16(svh)) return EXL3_EINVAL;
  // an empty batch dereferences no activation or output, which may then be NULL
  if (m > 0 && (!aligned16(xh) || !aligned16(y))) return EXL3_EINVAL;
  memset(a, 0, sizeof(*a));
  a->xh = xh;
  a->trellis = trellis;
  a->svh = svh;
  a->y = y;
  a->m = m;
  a->k = k;
  a->n = n;
  a->num_shards = num_shards;
  for (int i = 0; i <= num_shards; ++i) a->shard_cols[i] = shard_cols[i];
  a->parts = 1;
  a->part_atoms = 2;
  a->y_bf16 = (y_dtype == EXL3_BF16) ? 1 : 0;
  exl3::fill_decode_consts(&a->dc);
  return EXL3_OK;
}

}  // namespace

extern "C" {

exl3_status_t exl3_input_transform(const void* x, exl3_dtype_t x_dtype, int64_t m, int64_t k, const uint16_t* suh,
                                   int32_t num_shards, uint16_t* xh, void* stream) {
  if (m < 0 || m > kMaxRows || !valid_kn(k) || !valid_dtype(x_dtype)) return EXL3_EINVAL;
  if (num_shards < 1 || num_shards > EXL3_MAX_SHARDS) return EXL3_EINVAL;
  if (!aligned16(suh)) return EXL3_EINVAL;
  if (m == 0) return EXL3_OK;  // empty batch: x and xh may be NULL
  if (!aligned16(x) || !aligned16(xh)) return EXL3_EINVAL;
  return cuda_status(exl3::launch_input_transform(x, x_dtype == EXL3_BF16, m, k, suh, num_shards, xh,
                                                  static_cast<cudaStream_t>(stream)),
                     "exl3_input_transform");
}

exl3_status_t exl3_input_transform_swiglu(const void* gate_up, exl3_dtype_t dtype, int64_t m, int64_t k,
                                          const uint16_t* suh, int32_t num_shards, uint16_t* xh, void* stream) {
  if (m < 0 || m > kMaxRows || !valid_kn(k) || !valid_dtype(dtype)) return EXL3_EINVAL;
  if (num_shards < 1 || num_shards > EXL3_MAX_SHARDS) return EXL3_EINVAL;
  if (!aligned16(suh)) return EXL3_EINVAL;
  if (m == 0) return EXL3_OK;
  if (!aligned16(gate_up) || !aligned16(xh)) return EXL3_EINVAL;
  return cuda_status(exl3::launch_input_transform_swiglu(gate_up, dtype == EXL3_BF16, m, k, suh, num_shards, xh,
                                                         static_cast<cudaStream_t>(stream)),
                     "exl3_input_transform_swiglu");
}

exl3_status_t exl3_moe_input_transform(const void* x, exl3_dtype_t x_dtype, int64_t num_tokens, int64_t k,
                                       const int32_t* sorted_ids, int64_t rows, int32_t topk,
                                       const int32_t* block_expert, int32_t block, const uint16_t* suh,
                                       int32_t num_shards, int32_t num_experts, uint16_t* xh, void* stream) {
  if (num_tokens < 0 || num_tokens > kMaxRows || rows < 0 || rows > kMaxRows || !valid_kn(k)) return EXL3_EINVAL;
  if (!valid_dtype(x_dtype) || topk < 1 || topk > 64 || !valid_moe_block(block) || rows % block) {
    return EXL3_EINVAL;
  }
  if (num_shards < 1 || num_shards > EXL3_MAX_SHARDS || num_experts < 1) return EXL3_EINVAL;
  if (!aligned16(suh)) return EXL3_EINVAL;
  if (rows == 0) return EXL3_OK;
  if (!aligned16(xh) || sorted_ids == nullptr || block_expert == nullptr) return EXL3_EINVAL;
  if (num_tokens > 0 && !aligned16(x)) return EXL3_EINVAL;
  return cuda_status(exl3::launch_moe_input_transform(x, x_dtype == EXL3_BF16, num_tokens, k, sorted_ids, rows, topk,
                                                      block_expert, block, suh, num_shards, num_experts, xh,
                                                      static_cast<cudaStream_t>(stream)),
                     "exl3_moe_input_transform");
}

exl3_status_t exl3_moe_gemm(const uint16_t* xh, int64_t rows, int64_t k, const int16_t* trellis, int32_t bits,
                            exl3_codebook_t cb, const uint16_t* svh, const int32_t* shard_cols, int32_t num_shards,
                            const int32_t* block_expert, int32_t block, int32_t num_experts, void* y,
                            exl3_dtype_t y_dtype, int64_t n, void* stream) {
  exl3::GemmArgs a;
  exl3_status_t st = check_gemm(xh, rows, k, trellis, bits, cb, svh, shard_cols, num_shards, y, y_dtype, n, &a);
  if (st != EXL3_OK) return st;
  if (!valid_moe_block(block) || rows % block || num_experts < 1) return EXL3_EINVAL;
  // the expert index times one expert's trellis bytes must fit the tensor map's strides
  if ((int64_t)num_experts * (k / 16) * (n / 16) * 32 * bits > (int64_t(1) << 40)) return EXL3_EINVAL;
  if (rows == 0) return EXL3_OK;
  if (block_expert == nullptr) return EXL3_EINVAL;
  a.block_expert = block_expert;
  a.num_experts = num_experts;
  a.moe_block = block;
  return cuda_status(exl3::launch_moe_gemm_tc(a, bits, cb, block, static_cast<cudaStream_t>(stream)), "exl3_moe_gemm");
}

exl3_status_t exl3_moe_combine(const void* y, exl3_dtype_t y_dtype, int64_t rows, int64_t n,
                               const int32_t* sorted_ids, const int32_t* block_expert, int32_t block,
                               int32_t num_experts, const float* weights, int64_t num_tokens, int32_t topk,
                               int32_t* pair_rows, void* out, exl3_dtype_t out_dtype, void* stream) {
  if (rows < 0 || rows > kMaxRows || num_tokens < 0 || num_tokens > kMaxRows || !valid_kn(n)) return EXL3_EINVAL;
  if (!valid_dtype(y_dtype) || !valid_dtype(out_dtype) || topk < 1 || topk > 64) return EXL3_EINVAL;
  if (!valid_moe_block(block) || rows % block || num_experts < 1) return EXL3_EINVAL;
  if (num_tokens == 0) return EXL3_OK;
  if (!aligned16(out) || weights == nullptr || pair_rows == nullptr) return EXL3_EINVAL;
  if (rows > 0 && (!aligned16(y) || sorted_ids == nullptr || block_expert == nullptr)) return EXL3_EINVAL;
  return cuda_status(exl3::launch_moe_combine(y, y_dtype == EXL3_BF16, rows, n, sorted_ids, block_expert, block,
                                              num_experts, weights, num_tokens, topk, pair_rows, out,
                                              out_dtype == EXL3_BF16, static_cast<cudaStream_t>(stream)),
                     "exl3_moe_combine");
}

exl3_status_t exl3_gemm(const uint16_t* xh, int64_t m, int64_t k, const int16_t* trellis, int32_t bits,
                        exl3_codebook_t cb, const uint16_t* svh, const int32_t* shard_cols, int32_t num_shards,
                        void* y, exl3_dtype_t y_dtype, int64_t n, void* stream) {
  exl3::GemmArgs a;
  exl3_status_t st = check_gemm(xh, m, k, trellis, bits, cb, svh, shard_cols, num_shards, y, y_dtype, n, &a);
  if (st != EXL3_OK) return st;
  if (m == 0) return EXL3_OK;
  return cuda_status(exl3::launch_gemm_tc(a, bits, cb, static_cast<cudaStream_t>(stream)), "exl3_gemm");
}

// Shape-only split policy: the number of parts P makes (n/128) * P work units
// fill the 152 SMs of a GB300 in whole waves as evenly as possible.  It is the
// smallest P whose wave efficiency units / (152 * ceil(units / 152)) reaches
// 0.85, else the most efficient P; P <= k/128 (every part holds at least one
// 128-row block; split_part_atoms picks whole 256-row units where k/128 is
// even and P <= k/256) and P <= 16.  It never depends on m, so rows are
// byte-equal across batches.
int32_t exl3_splitk_parts(int64_t k, int64_t n) {
  if (!valid_kn(k) || !valid_kn(n)) return 0;
  const int64_t nb = n / 128;
  const int64_t kb = k / 128;
  const int64_t sms = 152;
  const int64_t pmax = kb < 16 ? kb : 16;
  int64_t best = 1;
  double best_eff = -1.0;
  for (int64_t p = 1; p <= pmax; ++p) {
    const int64_t units = nb * p;
    const double eff = (double)units / (double)(sms * ((units + sms - 1) / sms));
    if (eff >= 0.85) return (int32_t)p;
    if (eff > best_eff + 1e-12) {
      best_eff = eff;
      best = p;
    }
  }
  return (int32_t)best;
}

size_t exl3_splitk_workspace_bytes(int64_t m, int64_t k, int64_t n) {
  const int32_t p = exl3_splitk_parts(k, n);
  if (p <= 0 || m < 0) return 0;
  return (size_t)p * (size_t)m * (size_t)n * sizeof(float);
}

exl3_status_t exl3_gemm_splitk(const uint16_t* xh, int64_t m, int64_t k, const int16_t* trellis, int32_t bits,
                               exl3_codebook_t cb, const uint16_t* svh, const int32_t* shard_cols,
                               int32_t num_shards, void* y, exl3_dtype_t y_dtype, int64_t n, float* acc,
                               size_t acc_bytes, void* stream) {
  return exl3_test_gemm_shape(-1, xh, m, k, trellis, bits, cb, svh, shard_cols, num_shards, y, y_dtype, n, acc,
                              acc_bytes, stream);
}

exl3_status_t exl3_test_gemm_shape(int32_t tile_shape, const uint16_t* xh, int64_t m, int64_t k,
                                   const int16_t* trellis, int32_t bits, exl3_codebook_t cb, const uint16_t* svh,
                                   const int32_t* shard_cols, int32_t num_shards, void* y, exl3_dtype_t y_dtype,
                                   int64_t n, float* acc, size_t acc_bytes, void* stream) {
  // tile_shape -1 (only from exl3_gemm_splitk): the library's own choice
  const bool split = acc != nullptr || tile_shape < 0;
  exl3::GemmArgs a;
  exl3_status_t st = check_gemm(xh, m, k, trellis, bits, cb, svh, shard_cols, num_shards, y, y_dtype, n, &a);
  if (st != EXL3_OK) return st;
  if (tile_shape < -1 || tile_shape >= EXL3_TEST_TILE_SHAPES) return EXL3_EINVAL;
  if (split) {
    if (m > 0 && !aligned16(acc)) return EXL3_EINVAL;
    if (acc_bytes < exl3_splitk_workspace_bytes(m, k, n)) return EXL3_EWORKSPACE;
    a.acc = acc;
    a.parts = exl3_splitk_parts(k, n);
    a.part_atoms = exl3::split_part_atoms(k, a.parts);
  }
  if (tile_shape >= 0 && !exl3::tc_shape_supported(tile_shape, a)) return EXL3_EUNSUPPORTED;
  if (m == 0) return EXL3_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.parts == 1) {
    // no split (or one part: the fused epilogue does everything; acc untouched)
    return cuda_status(exl3::launch_gemm_tc(a, bits, cb, s, tile_shape), "exl3_gemm");
  }
  // Up to 16 rows the epilogue follows as a programmatic dependent, scheduled
  // once every CTA of the parts' GEMM has reached its own epilogue: 0.3-0.7
  // us faster on seven split layers on GB300.  From 32 rows on the same
  // launch measured up to 10% slower than a plain one (as did a trigger with
  // the activations, earlier still, at 16-64 rows), so there the epilogue is
  // a plain launch after the GEMM.
  a.trigger_dependents = m <= 16 ? 2 : 0;
  st = cuda_status(exl3::launch_gemm_tc(a, bits, cb, s, tile_shape), "exl3_gemm_splitk parts");
  if (st != EXL3_OK) return st;
  return cuda_status(exl3::launch_splitk_epilogue(a, s), "exl3_gemm_splitk epilogue");
}

exl3_status_t exl3_test_codebook(exl3_codebook_t cb, uint16_t* out, void* stream) {
  if (!valid_cb(cb) || !aligned16(out)) return EXL3_EINVAL;
  return cuda_status(exl3::launch_test_codebook(cb, out, static_cast<cudaStream_t>(stream)), "exl3_test_codebook");
}

exl3_status_t exl3_test_unpack(const int16_t* trellis, int32_t bits, exl3_codebook_t cb, int64_t k, int64_t n,
                               uint16_t* wq, void* stream) {
  if (bits < 1 || bits > 8 || !valid_cb(cb)) return EXL3_EINVAL;
  if (k < 16 || n < 16 || k % 16 || n % 16 || k > (int64_t(1) << 31) || n > (int64_t(1) << 31)) return EXL3_EINVAL;
  if (!aligned16(trellis) || !aligned16(wq)) return EXL3_EINVAL;
  return cuda_status(exl3::launch_test_unpack(trellis, bits, cb, k, n, wq, static_cast<cudaStream_t>(stream)),
                     "exl3_test_unpack");
}

exl3_status_t exl3_test_tile_plan(int64_t m, int64_t k, int64_t n, const int32_t* shard_cols, int32_t num_shards,
                                  int32_t split, int64_t* out) {
  if (m < 1 || m > kMaxRows || !valid_kn(k) || !valid_kn(n) || out == nullptr) return EXL3_EINVAL;
  if (num_shards < 1 || num_shards > EXL3_MAX_SHARDS || !valid_shards(shard_cols, num_shards, n)) return EXL3_EINVAL;
  if (split != 0 && split != 1) return EXL3_EINVAL;
  exl3::GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.m = m;
  a.k = k;
  a.n = n;
  a.num_shards = num_shards;
  for (int i = 0; i <= num_shards; ++i) a.shard_cols[i] = shard_cols[i];
  a.parts = split ? exl3_splitk_parts(k, n) : 1;
  a.part_atoms = exl3::split_part_atoms(k, a.parts);
  exl3::tc_plan(a, out);
  return EXL3_OK;
}

exl3_status_t exl3_set_autotune(int32_t enable) {
  if (enable != 0 && enable != 1) return EXL3_EINVAL;
  exl3::tc_set_autotune(enable == 1);
  return EXL3_OK;
}

exl3_status_t exl3_clear_autotune(void) {
  exl3::tc_clear_autotune();
  return EXL3_OK;
}

int64_t exl3_autotune_entries(void) { return exl3::tc_autotune_entries(); }

const char* exl3_status_string(exl3_status_t status) {
  switch (status) {
    case EXL3_OK: return "ok";
    case EXL3_EINVAL: return "invalid argument";
    case EXL3_EUNSUPPORTED: return "unsupported";
    case EXL3_EWORKSPACE: return "split-k workspace too small";
    case EXL3_ECUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* exl3_last_error(void) { return g_last_error; }

exl3_status_t exl3_test_wait_timeout(uint32_t* out, void* stream) {
  if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 3u) != 0) return EXL3_EINVAL;
  return cuda_status(exl3::launch_test_wait_timeout(out, static_cast<cudaStream_t>(stream)),
                     "exl3_test_wait_timeout");
}

exl3_status_t exl3_device_status(uint32_t* flags) {
  if (flags == nullptr) return EXL3_EINVAL;
  return cuda_status(exl3::take_device_errors(flags), "exl3_device_status");
}

}  // extern "C"
