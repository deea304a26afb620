// exl3_gemm_tc.cuh -- EXL3 GEMM on the 5th-generation tensor cores (tcgen05).
//
// One CTA owns BN output columns and RG*128 rows over the whole k extent (or
// over one shape-fixed part of k under split-k).  Owning all of k lets a block
// stream its share of the trellis a single time and apply the output Hadamard
// and svh in its epilogue (cuda-exl3 README, "Why custom kernels").  When
// BN < 128 a thread-block cluster of 128/BN CTAs spans one 128-column Hadamard
// block: each CTA accumulates its own columns and the epilogue reads the
// partners' fp32 tiles through distributed shared memory, so the arithmetic is
// the same whatever BN is.
//
// Warp roles:
//   warp 0      TMA producer: per stage (KA swizzle atoms of 64 k), one 3-D
//               tensor copy of the CTA's trellis tiles for the stage's k16 rows
//               and one 4-D tensor copy of the rotated activations xh (KA
//               atoms, 128-byte swizzle) per row group, all completing on full[s];
//   warp 1      TMEM allocator and MMA issuer: one thread issues tcgen05.mma
//               kind::f16 (M=128, N=BN, K=16) per row group and k16 step, fp32
//               accumulators in tensor memory;
//   warps 2..17 decoders: each lane decodes its 8 values of a 16x16 tile
//               (bitshift trellis + procedural codebook, TensorFold PR #740,
//               "Arithmetic" step 2) into registers in mma B-fragment order and
//               stmatrix stores them into the 128-byte-swizzled K-major B
//               operand; then the epilogue.
//
// Small batches: the activation region of an atom holds only XR rows.  The
// tensor core still reads 128 rows; rows past XR land on later bytes of the
// same stage (decoded weights, trellis words), which only feed accumulator
// rows that are never stored.  The read span always stays inside the stage.
//
// Each tile is decoded exactly once per CTA.  The fp32 sum over k is a fixed
// sequence of tcgen05 k16 steps in ascending k for every row, whatever m or the
// tiling, so rows are byte-equal across batch sizes.  Every wait is bounded: a
// kernel that gives up records kErrWaitTimeout and skips its stores.
#pragma once

#include "exl3_device.cuh"
#include "exl3_launch.h"
#include "exl3_sm100.cuh"

namespace exl3 {

constexpr int kTcDecodeWarps = 16;  // decoder / epilogue warps
constexpr int kTcThreads = 32 * (2 + kTcDecodeWarps);
constexpr int kTcSmemBudget = 227 * 1024;

template <int BITS, int BN, int RG, int KA, int XR>
struct TcCfg {
  static constexpr int kCluster = BN < 128 ? 128 / BN : 1;
  static constexpr int kXAtom = XR * 128;                        // one atom of one row group
  static constexpr int kXBytes = RG * KA * kXAtom;
  static constexpr int kWAtom = BN * 128;                        // decoded B operand, one atom
  static constexpr int kWBytes = KA * kWAtom;
  static constexpr int kTrRowBytes = (BN / 16) * 32 * BITS;      // one k16 row of BN/16 tiles
  static constexpr int kTrRows = 4 * KA;
  static constexpr int kTrBytes = kTrRows * kTrRowBytes;
  static constexpr int kStageBytes = ((kXBytes + kWBytes + kTrBytes) + 1023) / 1024 * 1024;
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kStages0 = (kTcSmemBudget - 1024 - kCtrlBytes) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  static constexpr int kSmem = 1024 + kCtrlBytes + kStages * kStageBytes;
  static constexpr int kTmemCols =
      RG * BN <= 32 ? 32 : RG * BN <= 64 ? 64 : RG * BN <= 128 ? 128 : RG * BN <= 256 ? 256 : 512;
  static constexpr int kTiles = kTrRows * (BN / 16);    // tiles decoded per stage
  static constexpr int kTpw = kTiles / kTcDecodeWarps;  // per decoder warp
  static constexpr int kZStride = BN + 4;               // epilogue staging row stride (floats)
  static_assert(RG * BN <= 512, "accumulators exceed tensor memory");
  static_assert(kStages >= 2, "not enough shared memory for two stages");
  static_assert(kTiles % kTcDecodeWarps == 0, "tiles per stage must split evenly over the decoders");
  static_assert(XR == 128 || RG == 1, "partial activation regions need a single row group");
  static_assert(XR == 128 || (KA - 1) * kXAtom + 16384 <= kStageBytes,
                "the tensor core's 128-row read of the last atom must stay inside the stage");
  static_assert(128 * kZStride * 4 <= kStages * kStageBytes, "epilogue tile must fit in the stage buffers");
};

template <int BITS, int CB, int BN, int RG, int KA, int XR>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
  using C = TcCfg<BITS, BN, RG, KA, XR>;
  constexpr int ST = C::kStages;
  constexpr int CL = C::kCluster;
  constexpr uint32_t kIdesc = idesc_f16_f32(128, BN);
  const GemmArgs& a = p.a;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by pointer arithmetic so that
  // the compiler keeps every access in the shared address space (an integer
  // round trip would turn the window loads into generic loads).
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* wfull = full + ST;
  uint64_t* empty = wfull + ST;
  uint64_t* accfull = empty + ST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfull + 1);
  volatile uint32_t* failed = tmem_slot + 1;  // set by the MMA issuer if any wait gave up
  uint8_t* stages = base + C::kCtrlBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t c0 = (int64_t)blockIdx.x * BN;
  const int64_t row0 = (int64_t)blockIdx.y * (128 * RG);
  const int part = (int)blockIdx.z;
  // this CTA's k range in 64-wide atoms: whole 128-row blocks of k per part
  const int64_t kb0 = (int64_t)part * (a.k >> 7) / a.parts * 2;
  const int64_t kb1 = (int64_t)(part + 1) * (a.k >> 7) / a.parts * 2;
  const int nk = (int)((kb1 - kb0) / KA);  // pipeline stages (the host keeps KA a divisor of every part)

  int shard = 0;
#pragma unroll
  for (int i = 1; i < kMaxShards; ++i)
    if (i < a.num_shards && c0 >= a.shard_cols[i]) shard = i;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&wfull[s], kTcDecodeWarps);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accfull, 1);
    *failed = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&maps.xh);
      prefetch_tensormap(&maps.trellis);
      const int nt0 = (int)(c0 >> 4);
      const uint32_t tx = (uint32_t)C::kTrBytes + (uint32_t)(RG * KA) * (uint32_t)p.box_rows * 128u;
      int s = 0;
      uint32_t ph = 0;
      for (int it = 0; it < nk; ++it) {
        if (!mbar_wait(&empty[s], ph ^ 1u)) break;
        mbar_arrive_expect_tx(&full[s], tx);
        uint8_t* st = stages + s * C::kStageBytes;
        const int atom0 = (int)(kb0 + (int64_t)it * KA);  // first 64-wide k atom of the stage
        tma_tile3d_g2s(st + C::kXBytes + C::kWBytes, &maps.trellis, 0, nt0, atom0 * 4, &full[s]);
#pragma unroll
        for (int r = 0; r < RG; ++r)
          tma_tile4d_g2s(st + r * KA * C::kXAtom, &maps.xh, 0, (int)(row0 + r * 128), atom0, shard, &full[s]);
        if (++s == ST) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      int s = 0;
      uint32_t ph = 0;
      const uint64_t desc0 = sdesc_sw128(smem_u32(stages));
      for (int it = 0; it < nk; ++it) {
        ok = mbar_wait(&full[s], ph) && mbar_wait(&wfull[s], ph);
        if (!ok) break;
        tc_fence_after();
        // descriptors of this stage's operands; an operand at byte offset o
        // from the stage has descriptor da + (o >> 4) (start-address field)
        const uint64_t da = desc0 + (uint64_t)((s * C::kStageBytes) >> 4);
#pragma unroll
        for (int at = 0; at < KA; ++at) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int r = 0; r < RG; ++r) {
              tc_mma_f16(tmem + r * BN, da + (uint64_t)((((r * KA + at) * C::kXAtom) + j * 32) >> 4),
                         da + (uint64_t)((C::kXBytes + at * C::kWAtom + j * 32) >> 4), kIdesc, (it | at | j) != 0);
            }
          }
        }
        tc_commit(&empty[s]);
        if (++s == ST) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) *failed = 1u;
      tc_commit(accfull);
    }
    __syncwarp();
  } else {
    // ---------------- decoders ----------------
    const int dw = warp - 2;
    const LaneWindow<BITS> lw(lane);
    // the multipliers, copied once from parameter memory into registers
    // (read in place, each use would become a constant-bank load)
    DecodeConsts mc;
#pragma unroll
    for (int i = 0; i <= 16; ++i) mc.pow2[i] = a.dc.pow2[i];
    // Per-warp constant byte offsets, so that a tile costs only its loads, its
    // decode and its store: the lane's three window words inside a tile, and
    // where each of this warp's tiles lands in the decoded operand.
    constexpr int kTilesN = BN / 16;
    constexpr int kTileBytes = 32 * BITS;
    const uint32_t word_off[3] = {dw * (uint32_t)kTileBytes + 4u * lw.idx[0], dw * (uint32_t)kTileBytes + 4u * lw.idx[1],
                                  dw * (uint32_t)kTileBytes + 4u * lw.idx[2]};
    uint32_t w_off[C::kTpw];
    {
      const int row_in = (lane & 7) + ((lane >> 4) << 3);  // stmatrix row of this lane within a 16-row tile
      const int chunk_hi = (lane >> 3) & 1;                // second 8-wide k half of a k16 step
#pragma unroll
      for (int i = 0; i < C::kTpw; ++i) {
        const int t = dw + i * kTcDecodeWarps;
        const int kt_l = t / kTilesN;  // k16 row within the stage
        const int row = (t - kt_l * kTilesN) * 16 + row_in;
        const int chunk = 2 * (kt_l & 3) + chunk_hi;
        w_off[i] = (uint32_t)((kt_l >> 2) * C::kWAtom + row * 128 + ((chunk ^ (row & 7)) << 4));
      }
    }
    const uint32_t stages_u32 = smem_u32(stages);
    int s = 0;
    uint32_t ph = 0;
    for (int it = 0; it < nk; ++it) {
      if (!mbar_wait(&full[s], ph)) break;
      const uint32_t st = stages_u32 + (uint32_t)(s * C::kStageBytes);
      const uint32_t trbase = st + C::kXBytes + C::kWBytes;
      const uint32_t wbase = st + C::kXBytes;
      // all window words of this warp's tiles first, so their latency overlaps
      uint32_t wv[C::kTpw][3];
#pragma unroll
      for (int i = 0; i < C::kTpw; ++i) {
        constexpr int kStep = kTcDecodeWarps * kTileBytes;  // tiles of one warp are kTcDecodeWarps apart
        wv[i][0] = ld_shared_u32(trbase + word_off[0] + i * kStep);
        wv[i][1] = ld_shared_u32(trbase + word_off[1] + i * kStep);
        wv[i][2] = (LaneWindow<BITS>::kNeed == 3) ? ld_shared_u32(trbase + word_off[2] + i * kStep) : 0u;
      }
#pragma unroll
      for (int i = 0; i < C::kTpw; ++i) {
        const Aligned al = align_window<BITS>(wv[i][0], wv[i][1], wv[i][2], lw.off);
        uint32_t b[4];
        decode_lane<BITS, CB>(al, mc, b);
        stmatrix_x4(wbase + w_off[i], b[0], b[1], b[2], b[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&wfull[s]);
      if (++s == ST) {
        s = 0;
        ph ^= 1u;
      }
    }
  }

  // ---------------- epilogue ----------------
  // Decoder warps wait for the accumulators; every warp takes part in the
  // block / cluster barriers below.
  const int dw = warp - 2;
  bool ok = true;
  if (warp >= 2) {
    ok = mbar_wait(accfull, 0) && *failed == 0u;
    tc_fence_after();
  }
  const bool bf16 = a.y_bf16 != 0;
  uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
  float* zs = reinterpret_cast<float*>(stages);
  constexpr int kZ = C::kZStride;

  if (a.parts > 1) {
    // split-k: this part's fp32 sums go straight to acc[part][row][col]
    if (warp >= 2) {
      const int quarter = warp & 3;
      float* dst = a.acc + (int64_t)part * a.m * a.n;
      for (int r = 0; r < RG; ++r) {
        for (int cc = dw >> 2; cc < BN / 32; cc += kTcDecodeWarps / 4) {
          uint32_t q[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(r * BN + cc * 32), q);
          tmem_ld_wait();
          const int64_t row = row0 + r * 128 + quarter * 32 + lane;
          if (ok && row < a.m) {
            float4* o = reinterpret_cast<float4*>(dst + row * a.n + c0 + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              o[i] = make_float4(__uint_as_float(q[4 * i]), __uint_as_float(q[4 * i + 1]),
                                 __uint_as_float(q[4 * i + 2]), __uint_as_float(q[4 * i + 3]));
          }
        }
      }
    }
  } else {
    const uint32_t rank = (CL > 1) ? cluster_ctarank() : 0u;
    const int64_t cbase = c0 - (int64_t)rank * BN;  // first column of the cluster's span
    constexpr int kSpan = BN < 128 ? 128 : BN;
    for (int r = 0; r < RG; ++r) {
      // 1. tensor memory -> this CTA's fp32 tile zs[128][BN]
      if (warp >= 2) {
        const int quarter = warp & 3;
        for (int cc = dw >> 2; cc < BN / 32; cc += kTcDecodeWarps / 4) {
          uint32_t q[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(r * BN + cc * 32), q);
          tmem_ld_wait();
          float* dst = zs + (quarter * 32 + lane) * kZ + cc * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(__uint_as_float(q[i]), __uint_as_float(q[i + 1]),
                                                              __uint_as_float(q[i + 2]), __uint_as_float(q[i + 3]));
        }
      }
      if (CL > 1) {
        cluster_sync();
      } else {
        __syncthreads();
      }
      // 2. rows: lane l owns columns 4l..4l+3 of each 128-column block of the span
      if (warp >= 2) {
        for (int hb = 0; hb < kSpan / 128; ++hb) {
          const int span_col = hb * 128 + 4 * lane;
          const uint32_t src_rank = (uint32_t)(span_col / BN);
          const int local_col = span_col - (int)src_rank * BN;
          const int64_t col = cbase + span_col;
          const uint2 sv = *reinterpret_cast<const uint2*>(a.svh + col);
          const float svf[4] = {__half2float(__ushort_as_half((uint16_t)(sv.x & 0xFFFF))),
                                __half2float(__ushort_as_half((uint16_t)(sv.x >> 16))),
                                __half2float(__ushort_as_half((uint16_t)(sv.y & 0xFFFF))),
                                __half2float(__ushort_as_half((uint16_t)(sv.y >> 16)))};
          const uint32_t zsrc = (CL > 1) ? mapa_shared(smem_u32(zs), src_rank) : smem_u32(zs);
          for (int rr = (int)rank + CL * dw; rr < 128; rr += CL * kTcDecodeWarps) {
            const int64_t row = row0 + r * 128 + rr;
            if (!ok || row >= a.m) break;  // rows ascend with rr
            float4 z4;
            if (CL > 1) {
              z4 = ld_shared_cluster_f4(zsrc + (uint32_t)((rr * kZ + local_col) * 4));
            } else {
              z4 = *reinterpret_cast<const float4*>(zs + rr * kZ + local_col);
            }
            float v[4] = {z4.x, z4.y, z4.z, z4.w};
            fwht128_warp(v, lane);
            uint16_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = f32_to_out((v[i] * 0.125f) * svf[i], bf16);
            uint2 w;
            w.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
            w.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
            *reinterpret_cast<uint2*>(y + row * a.n + col) = w;
          }
        }
      }
      // the tile is reused by the next row group, and partners may still read it
      if (CL > 1) {
        cluster_sync();
      } else {
        __syncthreads();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int BITS, int CB, int BN, int RG, int KA, int XR>
cudaError_t launch_tc_variant(const TcMaps& maps, const TcParams& p, cudaStream_t stream) {
  using C = TcCfg<BITS, BN, RG, KA, XR>;
  auto kern = gemm_tc_kernel<BITS, CB, BN, RG, KA, XR>;
  static bool configured = false;  // benign race: every thread sets the same attribute
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.a.n / BN), (unsigned)((p.a.m + 128 * RG - 1) / (128 * RG)), (unsigned)p.a.parts);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

// Tile shapes compiled for every width and codebook (see TcShape in exl3_launch.h).
template <int BITS, int CB>
cudaError_t launch_tc_cb(const TcMaps& maps, const TcParams& p, TcShape shape, cudaStream_t stream) {
  switch (shape) {
    case TcShape::kN32Small: return launch_tc_variant<BITS, CB, 32, 1, 4, 32>(maps, p, stream);
    case TcShape::kN64Small: return launch_tc_variant<BITS, CB, 64, 1, 2, 32>(maps, p, stream);
    case TcShape::kN128Small: return launch_tc_variant<BITS, CB, 128, 1, 2, 32>(maps, p, stream);
    case TcShape::kN128: return launch_tc_variant<BITS, CB, 128, 1, 1, 128>(maps, p, stream);
    case TcShape::kN128R2: return launch_tc_variant<BITS, CB, 128, 2, 1, 128>(maps, p, stream);
    default: return launch_tc_variant<BITS, CB, 256, 2, 1, 128>(maps, p, stream);
  }
}

template <int BITS>
cudaError_t launch_gemm_tc_bits(const TcMaps& maps, const TcParams& p, int cb, TcShape shape,
                                cudaStream_t stream) {
  switch (cb) {
    case CB_3INST: return launch_tc_cb<BITS, CB_3INST>(maps, p, shape, stream);
    case CB_MCG: return launch_tc_cb<BITS, CB_MCG>(maps, p, shape, stream);
    default: return launch_tc_cb<BITS, CB_MUL1>(maps, p, shape, stream);
  }
}

}  // namespace exl3
