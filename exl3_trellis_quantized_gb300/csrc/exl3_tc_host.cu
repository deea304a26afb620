// exl3_tc_host.cu -- host side of the tcgen05 GEMM: the TMA tensor maps of the
// rotated activations and of the trellis, the tile-shape choice and the width
// dispatch.
#include <cudaTypedefs.h>

#include <map>
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

namespace {

// xh is fp16 [S][m][k], viewed as 4-D {64 (k inside an atom), m, k/64 (atoms), S}
// so that one copy brings KA atoms of box_rows rows each, laid out atom after
// atom in shared memory, 128-byte swizzled; rows past m read as zeros.
cudaError_t make_xh_map(CUtensorMap* map, const uint16_t* xh, int64_t m, int64_t k, int num_shards, int box_rows,
                        int atoms) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[4] = {(cuuint64_t)kTcBK, (cuuint64_t)m, (cuuint64_t)(k / kTcBK), (cuuint64_t)num_shards};
  cuuint64_t strides[3] = {(cuuint64_t)k * 2, (cuuint64_t)kTcBK * 2, (cuuint64_t)(m * k * 2)};
  cuuint32_t box[4] = {(cuuint32_t)kTcBK, (cuuint32_t)box_rows, (cuuint32_t)atoms, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<uint16_t*>(xh), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// trellis is int16 [k/16][n/16][16*bits], viewed as 3-D {16*bits, n/16, k/16}; one
// copy brings the bn/16 tiles a CTA decodes for the k16 rows of a stage, stored
// row after row.
cudaError_t make_trellis_map(CUtensorMap* map, const int16_t* trellis, int64_t k, int64_t n, int bits, int bn,
                             int rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)(16 * bits), (cuuint64_t)(n / 16), (cuuint64_t)(k / 16)};
  cuuint64_t strides[2] = {(cuuint64_t)(32 * bits), (cuuint64_t)((n / 16) * 32 * bits)};
  cuuint32_t box[3] = {(cuuint32_t)(16 * bits), (cuuint32_t)(bn / 16), (cuuint32_t)rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<int16_t*>(trellis), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Experts' trellises stacked as [E][k/16][n/16][16*bits], viewed as 4-D
// {16*bits, n/16, k/16, E}: a copy takes one expert's tiles of a stage.
cudaError_t make_moe_trellis_map(CUtensorMap* map, const int16_t* trellis, int64_t k, int64_t n, int bits, int bn,
                                 int rows, int experts) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[4] = {(cuuint64_t)(16 * bits), (cuuint64_t)(n / 16), (cuuint64_t)(k / 16), (cuuint64_t)experts};
  cuuint64_t strides[3] = {(cuuint64_t)(32 * bits), (cuuint64_t)((n / 16) * 32 * bits),
                           (cuuint64_t)((k / 16) * (n / 16) * 32 * bits)};
  cuuint32_t box[4] = {(cuuint32_t)(16 * bits), (cuuint32_t)(bn / 16), (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<int16_t*>(trellis), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct ShapeDims {
  int bn, ka, xr, pair, rg;
};

ShapeDims dims_of(TcShape s) {
  switch (s) {
    case TcShape::kN32Small: return {32, 4, 32, 1, 1};
    case TcShape::kN64Small: return {64, 2, 32, 1, 1};
    case TcShape::kN128Small: return {128, 2, 32, 1, 1};
    case TcShape::kN128: return {128, 2, 128, 1, 1};
    case TcShape::kN128R2: return {128, 1, 128, 1, 2};
    case TcShape::kN128R2P: return {128, 1, 128, 2, 2};
    case TcShape::kN256R2P: return {256, 1, 128, 2, 2};
    case TcShape::kN128SmallK4: return {128, 4, 32, 1, 1};
    case TcShape::kN96SmallK4: return {96, 4, 32, 1, 1};
    case TcShape::kN96: return {96, 2, 128, 1, 1};
    case TcShape::kN96R2: return {96, 2, 128, 1, 2};
    case TcShape::kN32SmallK8: return {32, 8, 32, 1, 1};
    case TcShape::kN64SmallK4: return {64, 4, 32, 1, 1};
    case TcShape::kN96M64K4: return {96, 4, 64, 1, 1};
    case TcShape::kN64M64K4: return {64, 4, 64, 1, 1};
    case TcShape::kN64K4: return {64, 4, 128, 1, 1};
    case TcShape::kN32K4: return {32, 4, 128, 1, 1};
    case TcShape::kT128K4: return {128, 4, 32, 1, 1};
    case TcShape::kT128: return {128, 2, 32, 1, 1};
    case TcShape::kS96K4: return {96, 4, 32, 1, 1};
    case TcShape::kT128K4X16: return {128, 4, 16, 1, 1};
    case TcShape::kS96K4X16: return {96, 4, 16, 1, 1};
    case TcShape::kT128X16: return {128, 2, 16, 1, 1};
    case TcShape::kT128K4X64: return {128, 4, 64, 1, 1};
    case TcShape::kT128X64: return {128, 2, 64, 1, 1};
    case TcShape::kT128X128: return {128, 2, 128, 1, 1};
    case TcShape::kT128K4X128: return {128, 4, 128, 1, 1};  // 2 atoms at 7-8 bits (launch_one)
    case TcShape::kS96K4X64: return {96, 4, 64, 1, 1};
    default: return {256, 1, 128, 1, 2};
  }
}

// Tile shape for a call.  Every shape computes each output element with the
// same sequence of k16 steps, so this choice never changes the result; it only
// trades parallelism (small batches need many CTAs to reach every SM) against
// reuse of each decoded tile across rows (large batches).
// Decode throughput a small-batch CTA reaches on its SM relative to a
// 128-column CTA, measured on GB300 (q_proj-like layer, m = 1 to 32): narrow
// strips spend more of each SM on the cluster, per-stage synchronisation and
// the tensor core's 128-row operand reads.
constexpr double kRel96 = 0.81;
// m <= 32, per CTA against a 128-column tensor-memory CTA (kT128*) in one
// wave, measured on GB300 with the tensor-core instructions issued by an
// elected lane (5120 x 12288, 5120 x 6144, 4096 x 8192, 12288 x 4096,
// 2048 x 4096, m = 1 to 32): 96-column strips with the decoded weights as the
// tensor core's 128-row operand, 64- and 32-column strips with two or four
// (64) and four or eight (32) k atoms per stage.
constexpr double kRel96S = 0.85, kRel64 = 0.52, kRel64K4 = 0.68, kRel32 = 0.50, kRel32K8 = 0.55;
// The tensor-memory kernel is persistent: its per-CTA start and epilogue are
// paid once per SM, not once per wave, so its rate per CTA grows with the
// waves a layer needs (5120 x 34816: 2 waves, 4096 x 154880: 8 waves).
double rel_tm(int64_t waves) { return waves <= 1 ? 1.02 : waves == 2 ? 1.06 : waves == 3 ? 1.15 : 1.3; }
// The tensor-memory kernel holding 64 rows (four k atoms a stage) at
// 32 < m <= 64 measured at the same per-SM rates as at m <= 32 (5120 x 12288:
// 1.03 in one wave, 5120 x 34816: 1.07 in two, 4096 x 154880: 1.41 in eight);
// holding 128 rows on two k atoms at 64 < m <= 128, about 0.89 of them (0.91,
// 0.94, 1.22 on the same layers); on four atoms (k/128 even), about 0.92 of
// them (4096 x 154880: 178.5 against 165 us at m = 64, 5120 x 34816: 61.8
// against 56.5 us; 10-17% faster than on two atoms).
constexpr double kRelTm128 = 0.89;
constexpr double kRelTm128K4 = 0.92;
// 256-column, 256-row tiles at 32 < m <= 128 against 128 columns, per column
// (5120 x 34816, 4096 x 154880): fewer CTAs in whole waves.
constexpr double kRel256Mid = 1.07;
// 64-column strips of 128 rows on four k atoms at 64 < m <= 128 against 128
// columns (12288 x 4096, 4096 x 8192, 5120 x 6144: 0.68 to 0.78).
constexpr double kRel64Full = 0.7;
// 32-column strips of 128 rows on four k atoms at 32 < m <= 128, per SM
// against a 128-column CTA: layers with few 128-column blocks get twice the
// CTAs of the 64-column strips (12288 x 4096: 43.6 to 43.9 us against 49.7 to
// 53.1 at m = 48 to 128; where 64-column strips already fill the GPU, as on
// 4096 x 8192 and 5120 x 6144, they stay faster).
constexpr double kRel32Full = 0.4;
// The same for the full-row (128-row) tiles at 32 < m <= 128: 96 columns
// against 128 (5120 x 12288, m = 48 to 128).
constexpr double kRel96Full = 0.76;

constexpr double kCost128 = 0.87, kCost128P = 0.93, kCost256 = 1.49, kCost256P = 1.33, kCost96R2 = 0.91;
// A 128-row, 64-column strip CTA in the split-off last wave of a pair launch,
// where it runs alone and its decode sets its time: about half of a 128 x 128
// CTA (GB300, 5120 x 12288 at m = 4096: 64 such CTAs in place of 32 of 128 x
// 128 took the call from 345.5 to 337.2 us).
constexpr double kCost64K4 = 0.5;
// The same for 32-column strips (5120 x 12288 at m = 4096: 128 of them in place
// of 64 of 64 columns, 339.0 to 334.5 us; wider tails lose, as their grids
// need several waves).
constexpr double kCost32K4 = 0.3;

// Split-k at m <= 128: a 256-column CTA over a k part costs this many 128-column
// CTAs (decode-bound; its per-stage synchronisation, prologue and epilogue are
// shared by twice the columns), measured on GB300 (17408 x 5120, 6 bits, 7
// parts, m = 1 to 128).
constexpr double kCost256Split = 1.75;

// Split-k at 33 to 128 rows takes the tensor-memory kernel when each CTA's
// items hold at least this much k in all.
constexpr int64_t kTmSplitDepth = 1024;

// SMs of the current device, read once per device.
int64_t sm_count() {
  static std::mutex mu;
  static int64_t cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int v = 0;
    cache[dev] = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0 ? v : 152;
  }
  return cache[dev];
}

// Average number of busy SMs over the waves of a grid (one CTA per SM), times
// its per-SM rate.
double small_batch_rate(int64_t ctas, double rel) {
  const int64_t sms = sm_count();
  const int64_t waves = (ctas + sms - 1) / sms;
  return rel * (double)ctas / (double)waves;
}

// Whole waves of a grid times the cost of one of its CTAs.
double large_batch_time(int64_t ctas, double cost) {
  const int64_t sms = sm_count();
  return (double)((ctas + sms - 1) / sms) * cost;
}

int64_t lcm_128(int64_t bn) {
  int64_t x = bn, y = 128;
  while (y != 0) {
    const int64_t t = x % y;
    x = y;
    y = t;
  }
  return bn / x * 128;
}

bool edges_multiple_of(const GemmArgs& a, int64_t span) {
  if (a.n % span != 0) return false;
  for (int i = 0; i <= a.num_shards; ++i)
    if (a.shard_cols[i] % span != 0) return false;
  return true;
}

// Pair launches split off their partial last wave.  A pair shape's grid of C
// CTAs fills ceil(C / SMs) waves; when the last is partial its R CTAs (R / 2
// pair tiles, the last ones in row-pair-major order, so the final columns of
// the final row pair) can instead run as a second launch of smaller tiles
// (or of 128-column pairs, which still share the decode of each weight over
// 512 rows) that spread over the whole GPU.  Every shape computes each element with the
// same k16 steps, so the split changes no byte.  The plan is taken when the
// smaller tiles' waves cost less than the pair wave they replace (costs as in
// choose_shape).
struct TailPlan {
  bool split = false;
  int64_t primary_tiles = 0;  // pair tiles of the first launch
  int64_t row_base = 0, col_base = 0;
  TcShape tail = TcShape::kN128;
  double time = 0.0;  // modelled time of both launches
};

TailPlan plan_tail(const GemmArgs& a, TcShape shape) {
  const ShapeDims d = dims_of(shape);
  TailPlan t;
  const int64_t sms = sm_count();
  const int64_t ncol = a.n / d.bn, rows_per_tile = 2 * 128 * d.rg;
  const int64_t nrp = (a.m + rows_per_tile - 1) / rows_per_tile;
  const int64_t ctas = 2 * ncol * nrp * a.parts;
  const double cost = d.bn == 256 ? kCost256P : kCost128P;
  t.time = large_batch_time(ctas, cost);
  const int64_t rem = ctas % sms;
  const int64_t tail_tiles = rem / 2;
  if (a.parts != 1 || sms % 2 != 0 || ctas <= sms || rem == 0 || tail_tiles > ncol) return t;
  GemmArgs ta = a;
  ta.row_base = (nrp - 1) * rows_per_tile;
  ta.col_base = (ncol - tail_tiles) * d.bn;
  const int64_t rows = a.m - ta.row_base, cols = tail_tiles * d.bn;
  // the tail's tiles: 128 x 128, 256 x 128, 256 x 256, pairs of 256 x 128
  // (each CTA of a pair decodes half of the 128 columns for 512 rows), or
  // 128-row strips of 64 or 32 columns (four k atoms a stage; k/128 even)
  struct Option {
    TcShape shape;
    int64_t rows_per_cta, bn, pair;
    double cost;
  };
  const Option opts[6] = {{TcShape::kN128, 128, 128, 1, kCost128},
                          {TcShape::kN128R2, 256, 128, 1, 1.0},
                          {TcShape::kN256R2, 256, 256, 1, kCost256},
                          {TcShape::kN128R2P, 256, 128, 2, kCost128P},
                          {TcShape::kN64K4, 128, 64, 1, kCost64K4},
                          {TcShape::kN32K4, 128, 32, 1, kCost32K4}};
  double best = 1e300;
  for (const Option& o : opts) {
    if (cols % o.bn != 0 || ta.col_base % o.bn != 0 || !tc_shape_supported((int)o.shape, ta)) continue;
    const int64_t span = o.rows_per_cta * o.pair;
    const double tt = large_batch_time((rows + span - 1) / span * o.pair * (cols / o.bn), o.cost);
    if (tt < best) {
      best = tt;
      t.tail = o.shape;
    }
  }
  if (best >= 0.95 * cost) return t;
  t.split = true;
  t.primary_tiles = ctas / 2 - tail_tiles;
  t.row_base = ta.row_base;
  t.col_base = ta.col_base;
  t.time = large_batch_time(ctas - rem, cost) + best;
  return t;
}

TcShape choose_shape(const GemmArgs& a) {
  const bool edges256 = edges_multiple_of(a, 256);
  if (a.parts > 1 && a.m <= 128) {
    // The tensor-memory kernel over (128-column block, k part) items.  Forced
    // shapes, whole split-k calls on GB300 (seven layers from 1024 x 512 to
    // 17408 x 5120, 3 to 16 parts): at m <= 32 it led or tied every layer,
    // by up to 16%; at 33-128 rows it wins where a CTA's items hold at least
    // 1024 k in all (4-10% on 5120 x 6144, 12288 x 4096, 17408 x 5120) and
    // loses below that (4-15% on 2048 x 4096 and smaller), where its longer
    // prologue is not amortised.
    const int64_t items = a.n / 128 * a.parts;
    const int64_t sms = sm_count();
    const int64_t depth = (items + sms - 1) / sms * (a.k / a.parts);
    if (a.m <= 32 || depth >= kTmSplitDepth) {
      // four atoms a stage when the parts are whole four-atom units
      if (a.part_atoms == 4)
        return a.m <= 16 ? TcShape::kT128K4X16 : a.m <= 32 ? TcShape::kT128K4 : a.m <= 64 ? TcShape::kT128K4X64
                                                                             : TcShape::kT128K4X128;
      return a.m <= 16 ? TcShape::kT128X16 : a.m <= 32 ? TcShape::kT128 : a.m <= 64 ? TcShape::kT128X64
                                                                          : TcShape::kT128X128;
    }
    // whole waves of 128-column CTAs against fewer, wider ones
    if (edges256 && large_batch_time(a.n / 256 * a.parts, kCost256Split) < large_batch_time(a.n / 128 * a.parts, 1.0))
      return TcShape::kN256R2;
    return a.m <= 32 ? TcShape::kN128Small : TcShape::kN128;
  }
  if (a.m <= 32) {
    // pick the column width whose grid keeps the most decode throughput busy
    const int64_t sms = sm_count();
    const int64_t blocks = a.n / 128;
    const double rt = rel_tm((blocks + sms - 1) / sms) * (double)(blocks < sms ? blocks : sms);
    // four k atoms per stage halve the per-stage synchronisation (k must hold
    // an even number of 128-blocks); 32-column strips take eight once k holds
    // four or more such stages
    const bool k4 = (a.k / 128) % 2 == 0;
    const bool k8 = a.k % 512 == 0 && a.k >= 2048;
    const double r64 = small_batch_rate(a.n / 64, k4 ? kRel64K4 : kRel64);
    const double r32 = k8 ? small_batch_rate(a.n / 32, kRel32K8) : k4 ? small_batch_rate(a.n / 32, kRel32) : 0.0;
    // 96-column strips: clusters of four over three Hadamard blocks
    const double r96 = k4 && edges_multiple_of(a, 384) ? small_batch_rate(a.n / 96, kRel96S) : 0.0;
    const bool x16 = a.m <= 16;  // the 16-row tiles read half the activations
    if (rt >= r96 && rt >= r64 && rt >= r32)
      return k4 ? (x16 ? TcShape::kT128K4X16 : TcShape::kT128K4) : (x16 ? TcShape::kT128X16 : TcShape::kT128);
    if (r96 >= r64 && r96 >= r32) return x16 ? TcShape::kS96K4X16 : TcShape::kS96K4;
    if (r64 >= r32) return k4 ? TcShape::kN64SmallK4 : TcShape::kN64Small;
    return k8 ? TcShape::kN32SmallK8 : TcShape::kN32Small;
  }
  const bool edges384 = edges_multiple_of(a, 384);
  if (a.m <= 64 && (a.k / 128) % 2 == 0) {
    // 33 to 64 rows: the narrow strips hold 64 rows on four k atoms a stage,
    // measured at the small-batch strips' per-SM rates (5120 x 12288 and
    // 5120 x 6144, m = 33 to 64); 128 columns keep the 128-row tile
    const double r128 = small_batch_rate(a.n / 128, 1.0);
    const double r256 = edges256 ? small_batch_rate(a.n / 256, kRel256Mid) : 0.0;
    const double r96 = edges_multiple_of(a, 384) ? small_batch_rate(a.n / 96, kRel96) : 0.0;
    const double r64 = small_batch_rate(a.n / 64, kRel64K4);
    const double r32 = small_batch_rate(a.n / 32, kRel32Full);  // 128-row strips
    const int64_t sms = sm_count();
    const int64_t blocks = a.n / 128;
    const double rt = rel_tm((blocks + sms - 1) / sms) * (double)(blocks < sms ? blocks : sms);
    if (rt >= r128 && rt >= r256 && rt >= r96 && rt >= r64 && rt >= r32) return TcShape::kT128K4X64;
    if (r256 > r128 && r256 >= r96 && r256 >= r64 && r256 >= r32) return TcShape::kN256R2;
    if (r128 >= r96 && r128 >= r64 && r128 >= r32) return TcShape::kN128;
    if (r32 > r96 && r32 > r64) return TcShape::kN32K4;
    // the 96-column strips with swapped operands: the 64 rows are the narrow
    // operand, not half of a padded 128-row one (5120 x 12288, m = 33 to 64:
    // 2-4% faster than the unswapped strips)
    return r96 >= r64 ? TcShape::kS96K4X64 : TcShape::kN64M64K4;
  }
  if (a.m <= 128) {
    // as for small batches: 96-column tiles put a 96-block layer on 128 SMs
    const double r128 = small_batch_rate(a.n / 128, 1.0);
    const double r256 = edges256 ? small_batch_rate(a.n / 256, kRel256Mid) : 0.0;
    const double r96 = edges384 ? small_batch_rate(a.n / 96, kRel96Full) : 0.0;
    const double r64 = (a.k / 128) % 2 == 0 ? small_batch_rate(a.n / 64, kRel64Full) : 0.0;
    const double r32 = (a.k / 128) % 2 == 0 ? small_batch_rate(a.n / 32, kRel32Full) : 0.0;
    const int64_t sms = sm_count();
    const int64_t blocks = a.n / 128;
    const bool k4 = (a.k / 128) % 2 == 0;
    const double rt =
        (k4 ? kRelTm128K4 : kRelTm128) * rel_tm((blocks + sms - 1) / sms) * (double)(blocks < sms ? blocks : sms);
    if (rt >= r128 && rt >= r256 && rt >= r96 && rt >= r64 && rt >= r32)
      return k4 ? TcShape::kT128K4X128 : TcShape::kT128X128;
    if (r256 > r128 && r256 >= r96 && r256 >= r64 && r256 >= r32) return TcShape::kN256R2;
    if (r32 > r128 && r32 > r96 && r32 > r64) return TcShape::kN32K4;
    if (r64 > r128 && r64 > r96) return TcShape::kN64K4;
    return r96 > r128 ? TcShape::kN96 : TcShape::kN128;
  }
  // Larger batches: least estimated time over whole waves.  Per-CTA costs are
  // relative to a 256-row, 128-column CTA over the same k, measured on GB300
  // (5120 x 12288 at 6 bits, 5120 x 34816 at 5 bits, 12288 x 4096 at 5 bits,
  // m = 256 to 4096).  Pair shapes decode half of the columns per CTA; their
  // grid pads the row blocks to an even count, and a partial last wave may be
  // split off (plan_tail).
  // split-k parts multiply every grid
  const int64_t g128 = (a.m + 127) / 128 * a.parts, g256 = (a.m + 255) / 256 * a.parts;
  struct Option {
    TcShape shape;
    double time;
  };
  const Option opts[6] = {
      {TcShape::kN128R2, large_batch_time(a.n / 128 * g256, 1.0)},
      {TcShape::kN96R2, edges384 ? large_batch_time(a.n / 96 * g256, kCost96R2) : 1e300},
      {TcShape::kN128, large_batch_time(a.n / 128 * g128, kCost128)},
      {TcShape::kN128R2P, plan_tail(a, TcShape::kN128R2P).time},
      {TcShape::kN256R2, edges256 ? large_batch_time(a.n / 256 * g256, kCost256) : 1e300},
      {TcShape::kN256R2P, edges256 ? plan_tail(a, TcShape::kN256R2P).time : 1e300},
  };
  Option best = opts[0];
  for (const Option& o : opts)
    if (o.time < best.time) best = o;
  return best.shape;
}

}  // namespace

void tc_plan(const GemmArgs& a, int64_t out[5]) {
  const TcShape s = choose_shape(a);
  out[0] = (int64_t)s;
  out[1] = -1;
  out[2] = out[3] = out[4] = 0;
  if (dims_of(s).pair > 1) {
    const TailPlan t = plan_tail(a, s);
    if (t.split) {
      out[1] = (int64_t)t.tail;
      out[2] = t.primary_tiles;
      out[3] = t.row_base;
      out[4] = t.col_base;
    }
  }
}

// The persistent tensor-memory kernel's shapes: one row group of XR rows, the
// grid over column items only.
static bool tm_shape(TcShape s) {
  return s == TcShape::kT128K4 || s == TcShape::kT128 || s == TcShape::kT128K4X16 || s == TcShape::kT128X16 ||
         s == TcShape::kT128K4X64 || s == TcShape::kT128X64 || s == TcShape::kT128X128 || s == TcShape::kT128K4X128;
}

bool tc_shape_supported(int shape, const GemmArgs& a) {
  if (shape < 0 || shape > (int)TcShape::kLast) return false;
  const TcShape s = (TcShape)shape;
  const ShapeDims d = dims_of(s);
  // small-batch shapes hold XR rows; the tensor-memory kernel holds XR rows
  // whatever XR is (it has no row groups)
  if ((d.xr < 128 || tm_shape(s)) && a.m > d.xr) return false;
  // several atoms per stage: k must hold whole stages, and split-k parts
  // only the tensor-memory kernel's four-atom stages, on four-atom parts
  if (d.ka > 2 && ((a.k / 128) % (d.ka / 2) != 0 ||
                   (a.parts > 1 && !(tm_shape(s) && d.ka == 4 && a.part_atoms == 4))))
    return false;
  // n and every shard edge fall on whole CTA spans: lcm(BN, 128) columns (a
  // cluster's span when BN is not a multiple of 128)
  return edges_multiple_of(a, lcm_128(d.bn));
}

namespace {

// One launch of the GEMM kernel with a given tile shape over the rows and
// columns from a.row_base / a.col_base (all pair tiles unless a.pair_tiles).
cudaError_t launch_one(const GemmArgs& a, int bits, int cb, TcShape shape, cudaStream_t stream) {
  TcParams p;
  p.a = a;
  ShapeDims d = dims_of(shape);
  if (shape == TcShape::kT128K4X128) d.ka = tm128_k4_atoms(bits);
  p.a.tile_cols = (int32_t)((a.n - a.col_base) / d.bn);
  if (d.pair > 1 && p.a.pair_tiles == 0) {
    const int64_t rows_per_tile = 2 * 128 * d.rg;
    p.a.pair_tiles = (int32_t)((a.m - a.row_base + rows_per_tile - 1) / rows_per_tile * p.a.tile_cols);
  }
  // rows per activation copy: just the rows in use, rounded up to 8 (copies
  // of every allocated row, zero-filled past m, made 1-4 row calls of a
  // 12288 x 4096 layer 23-39% slower on GB300); a copy brings all KA atoms of
  // a stage when it fills their regions, which sit back to back, else one atom
  // (the kernel then issues KA copies)
  p.box_rows = a.m >= d.xr ? d.xr : (int)((a.m + 7) / 8 * 8);
  TcMaps maps;
  cudaError_t e = make_xh_map(&maps.xh, a.xh, a.m, a.k, a.num_shards, p.box_rows, p.box_rows == d.xr ? d.ka : 1);
  if (e != cudaSuccess) return e;
  e = make_trellis_map(&maps.trellis, a.trellis, a.k, a.n, bits, d.bn / d.pair, 4 * d.ka);
  if (e != cudaSuccess) return e;
  switch (bits) {
    case 1: return launch_gemm_tc_bits<1>(maps, p, cb, shape, stream);
    case 2: return launch_gemm_tc_bits<2>(maps, p, cb, shape, stream);
    case 3: return launch_gemm_tc_bits<3>(maps, p, cb, shape, stream);
    case 4: return launch_gemm_tc_bits<4>(maps, p, cb, shape, stream);
    case 5: return launch_gemm_tc_bits<5>(maps, p, cb, shape, stream);
    case 6: return launch_gemm_tc_bits<6>(maps, p, cb, shape, stream);
    case 7: return launch_gemm_tc_bits<7>(maps, p, cb, shape, stream);
    default: return launch_gemm_tc_bits<8>(maps, p, cb, shape, stream);
  }
}

// The GEMM with a given tile shape: one launch, or for a pair shape whose
// last wave is better split off, the whole waves of pair tiles followed by a
// launch of smaller tiles over the rest (plan_tail).  The second launch may
// be scheduled as soon as every CTA of the first has its activations.
cudaError_t launch_shape(const GemmArgs& a, int bits, int cb, TcShape shape, cudaStream_t stream) {
  if (dims_of(shape).pair > 1) {
    const TailPlan t = plan_tail(a, shape);
    if (t.split) {
      GemmArgs first = a;
      first.pair_tiles = (int32_t)t.primary_tiles;
      first.trigger_dependents = 1;
      cudaError_t e = launch_one(first, bits, cb, shape, stream);
      if (e != cudaSuccess) return e;
      GemmArgs rest = a;
      rest.row_base = t.row_base;
      rest.col_base = t.col_base;
      return launch_one(rest, bits, cb, t.tail, stream);
    }
  }
  return launch_one(a, bits, cb, shape, stream);
}

// Tile-shape autotune (off by default).  A call's key is its device, width,
// codebook, k, n, shard edges, split-k parts and batch bucket (m <= 32, else
// the next power of two of m).  On a miss outside stream capture, every shape
// that can run the call is timed with CUDA events on the caller's stream (the
// host waits on them): two rounds over the candidates, a warm-up launch in the
// first, two timed launches in each, a shape's time the lower of its rounds so
// a clock or power swing during one round does not decide.  The cost model's
// shape is kept unless another is more than 2% faster.  Every shape gives the
// same bytes, so the choice never changes a result.  Under capture the cache
// is read but never filled: a key tuned in an eager warm-up reaches captured
// work, any other key takes the cost model's shape.
struct TuneKey {
  int dev, bits, cb, parts, num_shards;
  int64_t k, n, bucket;
  int32_t cols[kMaxShards + 1];
  bool operator<(const TuneKey& o) const {
    if (dev != o.dev) return dev < o.dev;
    if (bits != o.bits) return bits < o.bits;
    if (cb != o.cb) return cb < o.cb;
    if (parts != o.parts) return parts < o.parts;
    if (k != o.k) return k < o.k;
    if (n != o.n) return n < o.n;
    if (bucket != o.bucket) return bucket < o.bucket;
    if (num_shards != o.num_shards) return num_shards < o.num_shards;
    for (int i = 0; i <= num_shards; ++i)
      if (cols[i] != o.cols[i]) return cols[i] < o.cols[i];
    return false;
  }
};
std::mutex g_tune_mu;
bool g_tune_on = false;
std::map<TuneKey, TcShape> g_tune;

int64_t batch_bucket(int64_t m) {
  if (m <= 32) return 32;
  int64_t b = 64;
  while (b < m) b <<= 1;
  return b;
}

// The tuned shape for this call, or the cost model's when tuning is off, the
// key is untuned under capture, or the timing fails.
TcShape tuned_shape(const GemmArgs& a, int bits, int cb, cudaStream_t stream) {
  const TcShape model = choose_shape(a);
  {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    if (!g_tune_on) return model;
  }
  TuneKey key = {};
  if (cudaGetDevice(&key.dev) != cudaSuccess) return model;
  key.bits = bits;
  key.cb = cb;
  key.parts = a.parts;
  key.k = a.k;
  key.n = a.n;
  key.bucket = batch_bucket(a.m);
  key.num_shards = a.num_shards;
  for (int i = 0; i <= a.num_shards; ++i) key.cols[i] = a.shard_cols[i];
  {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    auto it = g_tune.find(key);
    if (it != g_tune.end()) return it->second;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return model;
  constexpr int kShapes = (int)TcShape::kLast + 1;
  float best_ms[kShapes];
  for (int s = 0; s < kShapes; ++s) best_ms[s] = 1e30f;
  cudaEvent_t ev[2];
  if (cudaEventCreate(&ev[0]) != cudaSuccess) return model;
  if (cudaEventCreate(&ev[1]) != cudaSuccess) {
    cudaEventDestroy(ev[0]);
    return model;
  }
  for (int round = 0; round < 2; ++round) {
    for (int s = 0; s < kShapes; ++s) {
      if (!tc_shape_supported(s, a)) continue;
      const TcShape shape = (TcShape)s;
      bool ok = round > 0 || launch_shape(a, bits, cb, shape, stream) == cudaSuccess;  // warm-up
      ok = ok && cudaEventRecord(ev[0], stream) == cudaSuccess;
      for (int r = 0; ok && r < 2; ++r) ok = launch_shape(a, bits, cb, shape, stream) == cudaSuccess;
      ok = ok && cudaEventRecord(ev[1], stream) == cudaSuccess && cudaEventSynchronize(ev[1]) == cudaSuccess;
      float ms = 0.f;
      if (ok && cudaEventElapsedTime(&ms, ev[0], ev[1]) == cudaSuccess) best_ms[s] = fminf(best_ms[s], ms);
    }
  }
  cudaEventDestroy(ev[0]);
  cudaEventDestroy(ev[1]);
  TcShape best = model;
  const float bar = 0.98f * best_ms[(int)model];
  for (int s = 0; s < kShapes; ++s)
    if (best_ms[s] < bar && best_ms[s] < best_ms[(int)best]) best = (TcShape)s;
  std::lock_guard<std::mutex> lock(g_tune_mu);
  g_tune[key] = best;
  return best;
}

}  // namespace

void tc_set_autotune(bool on) {
  std::lock_guard<std::mutex> lock(g_tune_mu);
  g_tune_on = on;
}

void tc_clear_autotune() {
  std::lock_guard<std::mutex> lock(g_tune_mu);
  g_tune.clear();
}

int64_t tc_autotune_entries() {
  std::lock_guard<std::mutex> lock(g_tune_mu);
  return (int64_t)g_tune.size();
}

cudaError_t launch_gemm_tc(const GemmArgs& a, int bits, int cb, cudaStream_t stream, int forced) {
  const TcShape shape = forced >= 0 ? (TcShape)forced : tuned_shape(a, bits, cb, stream);
  return launch_shape(a, bits, cb, shape, stream);
}

cudaError_t launch_moe_gemm_tc(const GemmArgs& a, int bits, int cb, int block, cudaStream_t stream) {
  TcParams p;
  p.a = a;
  // The persistent tensor-memory kernel over (row block, 128-column block)
  // items, holding exactly the block's rows (each activation copy brings
  // them), four k atoms a stage when k holds an even number of 128-blocks
  // (128-row blocks only up to 6 bits).  Measured on 128 experts, top-8,
  // hidden 2048, gate_up 2 x 768, 4-bit mcg: 1.2-1.4x faster than one CTA per
  // (block, column tile) at 1 to 256 tokens, 1.1x with 128-row blocks on two
  // atoms at 1024 tokens, and four atoms there 163 -> 151 us.
  const bool k4 = (a.k / 128) % 2 == 0;
  const int tile = block <= 32 ? (block == 16 ? (k4 ? kMoeTileTm16K4 : kMoeTileTm16)
                                              : (k4 ? kMoeTileTm32K4 : kMoeTileTm32))
                               : (k4 ? kMoeTileTm128K4 : kMoeTileTm128);
  p.box_rows = block;
  const int ka = (tile == kMoeTileTm16K4 || tile == kMoeTileTm32K4) ? 4
                 : tile == kMoeTileTm128K4                          ? tm128_k4_atoms(bits)
                                                                    : 2;
  const int bn = 128;
  TcMaps maps;
  cudaError_t e = make_xh_map(&maps.xh, a.xh, a.m, a.k, a.num_shards, p.box_rows, ka);
  if (e != cudaSuccess) return e;
  e = make_moe_trellis_map(&maps.trellis, a.trellis, a.k, a.n, bits, bn, 4 * ka, a.num_experts);
  if (e != cudaSuccess) return e;
  switch (bits) {
    case 1: return launch_moe_gemm_tc_bits<1>(maps, p, cb, tile, stream);
    case 2: return launch_moe_gemm_tc_bits<2>(maps, p, cb, tile, stream);
    case 3: return launch_moe_gemm_tc_bits<3>(maps, p, cb, tile, stream);
    case 4: return launch_moe_gemm_tc_bits<4>(maps, p, cb, tile, stream);
    case 5: return launch_moe_gemm_tc_bits<5>(maps, p, cb, tile, stream);
    case 6: return launch_moe_gemm_tc_bits<6>(maps, p, cb, tile, stream);
    case 7: return launch_moe_gemm_tc_bits<7>(maps, p, cb, tile, stream);
    default: return launch_moe_gemm_tc_bits<8>(maps, p, cb, tile, stream);
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
