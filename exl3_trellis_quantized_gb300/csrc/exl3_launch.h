// exl3_launch.h -- internal host-side launchers (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace exl3 {

constexpr int kMaxShards = 8;

// Powers of two the decoder multiplies by when it runs shifts on the integer
// multiply pipe (the ALU pipe that executes shifts, masks and permutes is the
// decoder's bottleneck).  They arrive as kernel parameters, so the compiler
// cannot fold them back into shifts; kernels copy them into registers once.
struct DecodeConsts {
  uint32_t pow2[17];  // pow2[i] = 1 << i, filled on the host
};
inline void fill_decode_consts(DecodeConsts* dc) {
  for (int i = 0; i <= 16; ++i) dc->pow2[i] = 1u << i;
}

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
  int32_t parts;       // P (1 = no split)
  int32_t part_atoms;  // a part is whole units of this many 64-wide k atoms (2 or 4)
  int32_t y_bf16;
  DecodeConsts dc;
  // grouped (mixture-of-experts) GEMM only: expert of each row block, or -1
  const int32_t* block_expert;
  int32_t num_experts;
  // Tile placement of one launch (zero: the whole output).  CTAs cover rows
  // from row_base and columns from col_base; pair shapes number their pair
  // tiles linearly, row pair major with tile_cols column tiles per row pair,
  // and launch pair_tiles of them.  trigger_dependents: let the next launch
  // in the stream start once every CTA has its activations (1: the tail of a
  // split launch, see exl3_tc_host.cu) or has reached its epilogue (2: the
  // split-k epilogue).
  int64_t row_base, col_base;
  int32_t tile_cols, pair_tiles;
  int32_t trigger_dependents;
  int32_t moe_block;  // grouped GEMM: rows per block (16, 32 or 128)
};

// Split-k parts are whole units of four 64-wide k atoms (256 rows of k) when
// k/128 is even and every part gets at least one such unit, else whole
// 128-row blocks (two atoms); like P itself a function of the shape only.
inline int32_t split_part_atoms(int64_t k, int32_t parts) {
  const int64_t kb = k / 128;
  return (parts > 1 && kb % 2 == 0 && parts <= kb / 2) ? 4 : 2;
}

cudaError_t launch_input_transform(const void* x, bool x_bf16, int64_t m, int64_t k, const uint16_t* suh,
                                   int num_shards, uint16_t* xh, cudaStream_t stream);

// The same with the input computed as silu(gate) * up from gate_up [m][2k].
cudaError_t launch_input_transform_swiglu(const void* gate_up, bool bf16, int64_t m, int64_t k, const uint16_t* suh,
                                          int num_shards, uint16_t* xh, cudaStream_t stream);

// Gather each block-aligned routed row of x and rotate it with its block's
// expert's suh (rows of -1 blocks untouched, padding rows zero).
cudaError_t launch_moe_input_transform(const void* x, bool x_bf16, int64_t num_tokens, int64_t k,
                                       const int32_t* sorted_ids, int64_t rows, int32_t topk,
                                       const int32_t* block_expert, int32_t block, const uint16_t* suh,
                                       int num_shards, int num_experts, uint16_t* xh, cudaStream_t stream);
// Grouped GEMM over row blocks of `block` rows (32 or 128), one expert per block.
cudaError_t launch_moe_gemm_tc(const GemmArgs& args, int bits, int cb, int block, cudaStream_t stream);

// Sum the P partials in part order, rotate, scale, store y, zero the workspace.
cudaError_t launch_splitk_epilogue(const GemmArgs& args, cudaStream_t stream);
// Weighted sum of each token's top-k rows of a grouped GEMM's output (pair_rows:
// int32 [tokens * topk] scratch, rewritten by the call, never needs clearing).
cudaError_t launch_moe_combine(const void* y, bool y_bf16, int64_t rows, int64_t n, const int32_t* sorted_ids,
                               const int32_t* block_expert, int32_t block, int num_experts, const float* weights,
                               int64_t num_tokens, int32_t topk, int32_t* pair_rows, void* out, bool out_bf16,
                               cudaStream_t stream);

cudaError_t launch_test_codebook(int cb, uint16_t* out, cudaStream_t stream);
cudaError_t launch_test_unpack(const int16_t* trellis, int bits, int cb, int64_t k, int64_t n, uint16_t* wq,
                               cudaStream_t stream);

// tcgen05 GEMM (one translation unit per width).
constexpr int kTcBK = 64;  // k per swizzle atom (one 128-byte row of fp16)
struct TcParams {
  GemmArgs a;
  int32_t box_rows;  // rows per xh tile copy (<= 128)
};
// The tensor maps one tcgen05 launch reads through.
struct TcMaps {
  CUtensorMap xh;       // fp16 xh, 4-D {64, m, k/64, S}: KA atoms (1 when box_rows < XR) of box_rows rows per copy
  CUtensorMap trellis;  // int16 trellis, 3-D {16*bits, n/16, k/16}: a stage's tile rows per copy
};
// Tile shapes of the tcgen05 GEMM: columns per CTA (BN), row groups of 128
// (RG), 64-wide k atoms per pipeline stage (KA) and activation rows held per
// atom (XR).  Shapes whose BN is not a multiple of 128 run as clusters of
// 128/gcd(BN, 128) CTAs that span whole Hadamard blocks; pair shapes
// (P) as clusters of two CTAs on neighbouring rows that decode half of the
// columns each and share the decoded operand.
enum class TcShape : int {
  kN32Small,   // BN=32,  RG=1, KA=4, XR=32   (m <= 32, narrow layers)
  kN64Small,   // BN=64,  RG=1, KA=2, XR=32   (m <= 32, wide layers)
  kN128Small,  // BN=128, RG=1, KA=2, XR=32   (m <= 32, wide layers with odd k/128, split-k parts)
  kN128,       // BN=128, RG=1, KA=2, XR=128  (m <= 128)
  kN128R2,     // BN=128, RG=2, KA=1, XR=128  (large m)
  kN256R2,     // BN=256, RG=2, KA=1, XR=128  (large m, 256-aligned shard edges)
  kN128R2P,    // BN=128, RG=2, KA=1, XR=128, pair (large m)
  kN256R2P,    // BN=256, RG=2, KA=1, XR=128, pair (large m, 256-aligned shard edges)
  kN128SmallK4,  // BN=128, RG=1, KA=4, XR=32  (m <= 32, wide layers, even k/128, no split-k)
  kN96SmallK4,   // BN=96,  RG=1, KA=4, XR=32  (m <= 32, n and shard edges multiples of 384, even k/128,
                 //                             no split-k; clusters of 4 CTAs over 3 Hadamard blocks)
  kN96,          // BN=96,  RG=1, KA=2, XR=128 (n and shard edges multiples of 384)
  kN96R2,        // BN=96,  RG=2, KA=2, XR=128 (n and shard edges multiples of 384)
  kN32SmallK8,   // BN=32,  RG=1, KA=8, XR=32  (m <= 32, k a multiple of 512, no split-k)
  kN64SmallK4,   // BN=64,  RG=1, KA=4, XR=32  (m <= 32, k/128 even, no split-k)
  kN96M64K4,     // BN=96,  RG=1, KA=4, XR=64  (m <= 64, k/128 even, no split-k, 384-aligned edges)
  kN64M64K4,     // BN=64,  RG=1, KA=4, XR=64  (m <= 64, k/128 even, no split-k)
  kN64K4,        // BN=64,  RG=1, KA=4, XR=128 (m <= 128, split-off tails; k/128 even, no split-k)
  kN32K4,        // BN=32,  RG=1, KA=4, XR=128 (m <= 128 on narrow layers, split-off tails; k/128 even,
                 //                             no split-k)
  // Decoded weights as the tensor core's A operand (M = 128 weight columns),
  // the XR activation rows as B (N = XR): kT* keep A in tensor memory
  // (exl3_gemm_tm.cuh), kS* in shared memory (strips in clusters of four).
  kT128K4,       // BN=128, KA=4, XR=32 (m <= 32, k/128 even; split-k only on 256-row parts)
  kT128,         // BN=128, KA=2, XR=32 (m <= 32)
  kS96K4,        // BN=96,  KA=4, XR=32 (m <= 32, k/128 even, no split-k, n and shard edges multiples of 384)
  kT128K4X16,    // BN=128, KA=4, XR=16 (m <= 16, k/128 even; split-k only on 256-row parts)
  kS96K4X16,     // BN=96,  KA=4, XR=16 (m <= 16, k/128 even, no split-k, 384-aligned edges)
  kT128X16,      // BN=128, KA=2, XR=16 (m <= 16)
  kT128K4X64,    // BN=128, KA=4, XR=64 (m <= 64, k/128 even; split-k only on 256-row parts)
  kT128X64,      // BN=128, KA=2, XR=64 (m <= 64)
  kT128X128,     // BN=128, KA=2, XR=128 (m <= 128)
  kS96K4X64,     // BN=96,  KA=4, XR=64 (m <= 64, k/128 even, no split-k, 384-aligned edges)
  kT128K4X128,   // BN=128, KA=4 (2 at 7-8 bits), XR=128 (m <= 128, k/128 even; split-k only on 256-row parts)
  kLast = kT128K4X128,
};
// Runs the whole GEMM (parts == 1) or writes the fp32 partials of every part
// (parts > 1) for the split-k epilogue.
// shape < 0: chosen from the sizes; otherwise a TcShape value that
// tc_shape_supported() accepted.
cudaError_t launch_gemm_tc(const GemmArgs& args, int bits, int cb, cudaStream_t stream, int shape = -1);
// The cost model's plan for a call (host only, no launch): out[0] the tile
// shape; for a pair shape whose last wave is split off, out[1] the second
// launch's shape, out[2] the pair tiles of the first, out[3] / out[4] the
// first row / column of the second; else out[1] = -1.
void tc_plan(const GemmArgs& args, int64_t out[5]);
// Whether tile shape `shape` can run the call described by `args`.
bool tc_shape_supported(int shape, const GemmArgs& args);
// Tile-shape autotune (see exl3_tc_host.cu): switch, cache reset, cache size.
void tc_set_autotune(bool on);
void tc_clear_autotune();
int64_t tc_autotune_entries();
template <int BITS>
cudaError_t launch_gemm_tc_bits(const TcMaps& maps, const TcParams& p, int cb, TcShape shape,
                                cudaStream_t stream);
// Grouped GEMM tiles: 32-row blocks with two or four k atoms per stage (or in
// 96-column strips with four), 128-row blocks.
// Grouped GEMM tiles: the persistent tensor-memory kernel over (row block,
// 128-column block) items holding 16, 32 or 128 rows, four k atoms a stage
// (16 and 32 rows with k/128 even) or two.
// Atoms a stage of the 128-row four-atom tensor-memory tiles (dense and
// grouped): two 64 KB activation slots leave room for three trellis slots of
// four atoms only up to 6 bits.  The host's tensor maps and the kernel's
// instantiation both follow this.
constexpr int tm128_k4_atoms(int bits) { return bits <= 6 ? 4 : 2; }

enum MoeTile : int {
  kMoeTileTm16K4 = 0,
  kMoeTileTm16 = 1,
  kMoeTileTm32K4 = 2,
  kMoeTileTm32 = 3,
  kMoeTileTm128 = 4,
  kMoeTileTm128K4 = 5,  // four atoms a stage (two at 7-8 bits, where three trellis slots would not fit)
};
template <int BITS>
cudaError_t launch_moe_gemm_tc_bits(const TcMaps& maps, const TcParams& p, int cb, int tile, cudaStream_t stream);
// Read and clear the wait-timeout flags of every kernel translation unit (synchronous).
cudaError_t take_device_errors(uint32_t* flags);
// exl3_test_wait_timeout's kernel (in the 1-bit instantiation unit).
cudaError_t launch_test_wait_timeout(uint32_t* out, cudaStream_t stream);
template <int BITS>
cudaError_t take_device_error_tc(uint32_t* flags);


}  // namespace exl3
