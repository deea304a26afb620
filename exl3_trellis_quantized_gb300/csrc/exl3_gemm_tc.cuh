// exl3_gemm_tc.cuh -- EXL3 GEMM on the 5th-generation tensor cores (tcgen05).
//
// One CTA owns BN output columns (BN/128 output Hadamard blocks) and RG*128
// rows over the whole k extent.  Owning all of k lets a block stream its share
// of the trellis a single time and apply the output Hadamard and svh in its
// epilogue (cuda-exl3 README, "Why custom kernels").  Warp roles:
//
//   warp 0      TMA producer: per 64-wide k stage, four 1-D bulk copies of the
//               stage's trellis tile rows and RG tiled copies of the rotated
//               activations xh (128-byte swizzle), all completing on full[s];
//   warp 1      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma kind::f16 (M=128, N=BN, K=16) per row group and
//               16-wide k step into the fp32 accumulators in tensor memory;
//   warps 2..9  decoders: each lane decodes its 8 values of a 16x16 tile
//               (bitshift trellis + procedural codebook, TensorFold PR #740,
//               "Arithmetic" step 2) into registers in mma B-fragment order and
//               stmatrix writes them into the swizzled K-major B operand; then
//               the epilogue: tcgen05.ld of a row's 128 accumulators, the
//               128-point butterfly in registers, *2^-3 * svh, bf16/fp16 store.
//
// Each tile is decoded exactly once per CTA.  The fp32 sum over k is a fixed
// sequence of tcgen05 k16 steps in ascending k for every row, whatever m is, so
// rows are byte-equal across batch sizes.  Every wait is bounded: a kernel that
// gives up records kErrWaitTimeout and skips its stores.
#pragma once

#include "exl3_device.cuh"
#include "exl3_launch.h"
#include "exl3_sm100.cuh"

namespace exl3 {

constexpr int kTcDecodeWarps = 16;  // decoder / epilogue warps
constexpr int kTcThreads = 32 * (2 + kTcDecodeWarps);
constexpr int kTcSmemBudget = 227 * 1024;

template <int BITS, int BN, int RG>
struct TcCfg {
  static constexpr int kXBytes = 128 * 128;                 // one row group of xh per stage (16 KB)
  static constexpr int kWBytes = BN * 128;                  // decoded B operand per stage
  static constexpr int kTrRowBytes = (BN / 16) * 32 * BITS;  // one k16 row of BN/16 tiles
  static constexpr int kTrBytes = 4 * kTrRowBytes;          // four k16 rows per stage
  static constexpr int kStageBytes = RG * kXBytes + kWBytes + kTrBytes;
  static constexpr int kZStride = 128 + 4;  // fp32 row stride of the epilogue staging tile
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kStages0 = (kTcSmemBudget - 1024 - kCtrlBytes) / kStageBytes;
  static constexpr int kStages = kStages0 > 6 ? 6 : kStages0;
  static constexpr int kSmem = 1024 + kCtrlBytes + kStages * kStageBytes;
  static constexpr int kTmemCols = RG * BN <= 128 ? 128 : (RG * BN <= 256 ? 256 : 512);
  static_assert(RG * BN <= 512, "accumulators exceed tensor memory");
  static_assert(kStages >= 2, "not enough shared memory for two stages");
  static_assert(128 * kZStride * 4 <= kStages * kStageBytes, "epilogue tile must fit in the stage buffers");
};


template <int BITS, int CB, int BN, int RG>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ TcParams p) {
  using C = TcCfg<BITS, BN, RG>;
  constexpr int ST = C::kStages;
  constexpr uint32_t kIdesc = idesc_f16_f32(128, BN);
  const GemmArgs& a = p.a;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base);
  uint64_t* wfull = full + ST;
  uint64_t* empty = wfull + ST;
  uint64_t* accfull = empty + ST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfull + 1);
  volatile uint32_t* failed = tmem_slot + 1;  // set by the MMA issuer if any wait gave up
  uint8_t* stages = base + C::kCtrlBytes;
  auto xs_stage = [&](int s) { return stages + s * C::kStageBytes; };
  auto w_stage = [&](int s) { return stages + s * C::kStageBytes + RG * C::kXBytes; };
  auto tr_stage = [&](int s) { return stages + s * C::kStageBytes + RG * C::kXBytes + C::kWBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t c0 = (int64_t)blockIdx.x * BN;
  const int64_t row0 = (int64_t)blockIdx.y * (128 * RG);
  const int nk = (int)(a.k / kTcBK);

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
      prefetch_tensormap(&xmap);
      const int64_t NT = a.n >> 4;
      const int64_t nt0 = c0 >> 4;
      const uint32_t tx = 4u * C::kTrRowBytes + (uint32_t)RG * (uint32_t)p.box_rows * 128u;
      for (int it = 0; it < nk; ++it) {
        const int s = it % ST;
        const uint32_t ph = (uint32_t)(it / ST) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u)) break;
        mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t kt = (int64_t)it * 4 + j;
          const int16_t* src = a.trellis + (kt * NT + nt0) * (16 * BITS);
          tma_bulk_g2s(tr_stage(s) + j * C::kTrRowBytes, src, C::kTrRowBytes, &full[s]);
        }
#pragma unroll
        for (int r = 0; r < RG; ++r)
          tma_tile3d_g2s(xs_stage(s) + r * C::kXBytes, &xmap, it * kTcBK, (int)(row0 + r * 128), shard, &full[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      for (int it = 0; it < nk && ok; ++it) {
        const int s = it % ST;
        const uint32_t ph = (uint32_t)(it / ST) & 1u;
        ok = mbar_wait(&full[s], ph) && mbar_wait(&wfull[s], ph);
        if (!ok) break;
        tc_fence_after();
        const uint32_t xa = smem_u32(xs_stage(s));
        const uint32_t wa = smem_u32(w_stage(s));
#pragma unroll
        for (int j = 0; j < kTcBK / 16; ++j) {
#pragma unroll
          for (int r = 0; r < RG; ++r) {
            tc_mma_f16(tmem + r * BN, sdesc_sw128(xa + r * C::kXBytes + j * 32), sdesc_sw128(wa + j * 32), kIdesc,
                       (it | j) != 0);
          }
        }
        tc_commit(&empty[s]);
      }
      if (!ok) *failed = 1u;
      tc_commit(accfull);
    }
    __syncwarp();
  } else {
    // ---------------- decoders ----------------
    const int dw = warp - 2;
    const LaneWindow<BITS> lw(lane);
    const MulConsts mc(a.one);
    const int row_in = (lane & 7) + ((lane >> 4) << 3);  // stmatrix row of this lane within a 16-row tile
    const int chunk_hi = (lane >> 3) & 1;                // second 8-wide k half
    constexpr int kTilesN = BN / 16;
    for (int it = 0; it < nk; ++it) {
      const int s = it % ST;
      const uint32_t ph = (uint32_t)(it / ST) & 1u;
      if (!mbar_wait(&full[s], ph)) break;
      const uint32_t* trw = reinterpret_cast<const uint32_t*>(tr_stage(s));
      const uint32_t wbase = smem_u32(w_stage(s));
      // all window words of this warp's tiles first, so their latency overlaps
      constexpr int kTpw = 4 * kTilesN / kTcDecodeWarps;  // tiles per warp per stage
      uint32_t wv[kTpw][3];
#pragma unroll
      for (int i = 0; i < kTpw; ++i) {
        const int t = dw + i * kTcDecodeWarps;
        const uint32_t* tile = trw + t * (8 * BITS);
        wv[i][0] = tile[lw.idx[0]];
        wv[i][1] = tile[lw.idx[1]];
        wv[i][2] = (LaneWindow<BITS>::kNeed == 3) ? tile[lw.idx[2]] : 0u;
      }
#pragma unroll
      for (int i = 0; i < kTpw; ++i) {
        const int t = dw + i * kTcDecodeWarps;
        const int kt_l = t / kTilesN;
        const int nt_l = t - kt_l * kTilesN;
        const Aligned al = align_window<BITS>(wv[i][0], wv[i][1], wv[i][2], lw.off);
        uint32_t b[4];
        decode_lane<BITS, CB>(al, mc, b);
        const int row = nt_l * 16 + row_in;
        const int chunk = 2 * kt_l + chunk_hi;
        stmatrix_x4(wbase + row * 128 + ((chunk ^ (row & 7)) << 4), b[0], b[1], b[2], b[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&wfull[s]);
    }

    // ---------------- epilogue ----------------
    // Per 128x128 accumulator block: every decoder warp copies a 32-row x
    // 32-column piece of tensor memory into a shared fp32 tile (the pipeline
    // stages are free once the accumulators are final), then each warp takes
    // whole rows, lane l holding columns 4l..4l+3, and runs the same 128-point
    // butterfly, scale and rounding as the other epilogues.
    bool ok = mbar_wait(accfull, 0) && *failed == 0u;
    tc_fence_after();
    float* zs = reinterpret_cast<float*>(stages);
    const int quarter = warp & 3;          // tensor-memory lanes this warp may read
    const int cchunk = dw >> 2;            // which 32-column piece it copies
    constexpr int kZ = C::kZStride;
    const bool bf16 = a.y_bf16 != 0;
    uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
    constexpr int kBlocks = RG * (BN / 128);
    for (int blk = 0; blk < kBlocks; ++blk) {
      const int r = blk / (BN / 128);
      const int hb = blk - r * (BN / 128);
      {
        uint32_t q[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(r * BN + hb * 128 + cchunk * 32), q);
        tmem_ld_wait();
        float* dst = zs + (quarter * 32 + lane) * kZ + cchunk * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(__uint_as_float(q[i]), __uint_as_float(q[i + 1]),
                                                            __uint_as_float(q[i + 2]), __uint_as_float(q[i + 3]));
      }
      named_barrier(1, 32 * kTcDecodeWarps);
      const int64_t col = c0 + hb * 128 + 4 * lane;
      const uint2 sv = *reinterpret_cast<const uint2*>(a.svh + col);
      const float svf[4] = {__half2float(__ushort_as_half((uint16_t)(sv.x & 0xFFFF))),
                            __half2float(__ushort_as_half((uint16_t)(sv.x >> 16))),
                            __half2float(__ushort_as_half((uint16_t)(sv.y & 0xFFFF))),
                            __half2float(__ushort_as_half((uint16_t)(sv.y >> 16)))};
      for (int rr = dw; rr < 128; rr += kTcDecodeWarps) {
        const int64_t row = row0 + r * 128 + rr;
        if (!ok || row >= a.m) break;  // rows ascend with rr
        const float4 z4 = *reinterpret_cast<const float4*>(zs + rr * kZ + 4 * lane);
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
      named_barrier(1, 32 * kTcDecodeWarps);  // the tile is reused by the next block
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int BITS, int CB, int BN, int RG>
cudaError_t launch_tc_variant(const CUtensorMap& xmap, const TcParams& p, cudaStream_t stream) {
  using C = TcCfg<BITS, BN, RG>;
  auto kern = gemm_tc_kernel<BITS, CB, BN, RG>;
  static bool configured = false;  // benign race: every thread sets the same attribute
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const dim3 grid((unsigned)(p.a.n / BN), (unsigned)((p.a.m + 128 * RG - 1) / (128 * RG)), 1);
  kern<<<grid, kTcThreads, C::kSmem, stream>>>(xmap, p);
  return cudaGetLastError();
}

template <int BITS, int CB>
cudaError_t launch_tc_cb(const CUtensorMap& xmap, const TcParams& p, int bn, int rg, cudaStream_t stream) {
  (void)bn;
  (void)rg;
  return launch_tc_variant<BITS, CB, 128, 1>(xmap, p, stream);
}

template <int BITS>
cudaError_t launch_gemm_tc_bits(const CUtensorMap& xmap, const TcParams& p, int cb, int bn, int rg,
                                cudaStream_t stream) {
  switch (cb) {
    case CB_3INST:
      return launch_tc_cb<BITS, CB_3INST>(xmap, p, bn, rg, stream);
    case CB_MCG:
      return launch_tc_cb<BITS, CB_MCG>(xmap, p, bn, rg, stream);
    default:
      return launch_tc_cb<BITS, CB_MUL1>(xmap, p, bn, rg, stream);
  }
}

}  // namespace exl3
