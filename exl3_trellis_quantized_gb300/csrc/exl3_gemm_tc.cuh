// exl3_gemm_tc.cuh -- EXL3 GEMM on the 5th-generation tensor cores (tcgen05).
//
// One CTA owns BN output columns and RG*128 rows over the whole k extent (or
// over one shape-fixed part of k under split-k).  Owning all of k lets a block
// stream its share of the trellis a single time and apply the output Hadamard
// and svh in its epilogue (cuda-exl3 README, "Why custom kernels").  When BN
// is not a multiple of 128, a thread-block cluster of 128/gcd(BN, 128) CTAs
// spans whole 128-column Hadamard blocks (32 columns: 4 CTAs over one block;
// 96 columns: 4 CTAs over three): each CTA accumulates its own columns and the
// epilogue reads the partners' fp32 tiles through distributed shared memory,
// so the arithmetic is the same whatever BN is.  With PAIR = 2 two CTAs that
// own the same columns and neighbouring rows form a cluster {2, 1, 1}: each
// decodes half of the columns and copies its half of the decoded operand into
// the partner's shared memory, so every decoded weight feeds 2*RG*128 rows.
// A pair launch may cover only whole waves of pair tiles (numbered row pair
// major), the rest going to a second launch of smaller tiles or 128-column
// pairs (row_base / col_base), see exl3_tc_host.cu.
//
// Shared memory holds three rings, each with its own depth: rotated
// activations (NX slots, RG row groups of KA swizzle atoms of 64 k), decoded
// weights (NW slots, the tensor core's B operand) and trellis words (NT slots).
// The trellis ring is deep, so the copies of the compressed weights run far
// ahead of the decoders, and activation copies never wait for a decode.
//
// Warp roles:
//   warp 0      trellis producer: one 3-D tensor copy per stage of the CTA's
//               tiles for the stage's k16 rows (thread 0 issues the first
//               ring-full before the block synchronises);
//   warp 1      TMEM allocator and MMA issuer: the warp runs the loop and
//               one elected lane issues tcgen05.mma kind::f16 (M=128, N=BN,
//               K=16) per row group and k16 step, fp32 accumulators in tensor
//               memory (with SWAP, M=128 weight columns and N=XR rows);
//   warp 2      activation producer: one 4-D tensor copy of xh (KA atoms,
//               128-byte swizzle) per row group and stage, or one per atom of
//               just the rows in use when the batch is smaller than a slot;
//   warp 3      with PAIR = 2, sends the CTA's decoded half of each stage to
//               the partner (bulk copy into its shared memory);
//   warps 4..19 decoders: each lane decodes its 8 values of a 16x16 tile
//               (bitshift trellis + procedural codebook, TensorFold PR #740,
//               "Arithmetic" step 2) into registers in mma B-fragment order and
//               stmatrix stores them into the 128-byte-swizzled K-major B
//               operand; then the epilogue.
//
// Small batches: the activation region of an atom holds only XR rows, and the
// copies leave rows past the batch unwritten.  The tensor core still reads 128
// (or, for the 64-row MMA, 64) rows; rows past the batch, or past XR on later
// bytes of the rings, only feed accumulator rows that are never stored.  The
// read span always stays inside the rings.
//
// Each tile is decoded exactly once per CTA (per pair with PAIR = 2).  The fp32
// sum over k is a fixed sequence of tcgen05 k16 steps in ascending k for every
// row, whatever m or the tiling, so rows are byte-equal across batch sizes.
// Every wait is bounded: a kernel that gives up records kErrWaitTimeout and
// skips its stores.
#pragma once

#include "exl3_device.cuh"
#include "exl3_gemm_tm.cuh"
#include "exl3_launch.h"
#include "exl3_sm100.cuh"

namespace exl3 {

constexpr int kTcDecodeWarps = 16;  // decoder / epilogue warps
constexpr int kTcFirstDecoder = 4;  // warps 0..3: trellis producer, MMA issuer, activation producer, sender
constexpr int kTcThreads = 32 * (kTcFirstDecoder + kTcDecodeWarps);
constexpr int kTcSmemBudget = 227 * 1024;

constexpr int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }

// SWAP: the decoded weights are the tensor core's A operand (M = 128 weight
// columns per instruction, the CTA's BN columns in its first rows) and the XR
// activation rows its B operand (N = XR), so a small batch costs the tensor
// core XR rows instead of 128.  The accumulator then holds one weight column
// per tensor-memory lane and one batch row per tensor-memory column.
template <int BITS, int BN, int RG, int KA, int XR, int PAIR, bool SWAP = false>
struct TcCfg {
  static constexpr int kClusterX = 128 / gcd_int(BN, 128);  // CTAs spanning whole Hadamard blocks
  static constexpr int kCluster = kClusterX * PAIR;
  static constexpr int kXAtom = XR * 128;                     // one atom of one row group
  static constexpr int kXSlot = RG * KA * kXAtom;             // activations of a stage
  static constexpr int kWAtom = BN * 128;                     // decoded B operand, one atom
  static constexpr int kWSlot = KA * kWAtom;                  // decoded operand of a stage
  static constexpr int kBNL = BN / PAIR;                      // columns this CTA decodes
  static constexpr int kWHalfAtom = kBNL * 128;               // its rows of one atom
  static constexpr int kTrRows = 4 * KA;                      // k16 rows per stage
  static constexpr int kTrCopy = kTrRows * (kBNL / 16) * 32 * BITS;  // bytes of one trellis copy
  static constexpr int kTSlot = (kTrCopy + 127) / 128 * 128;
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kAvail = kTcSmemBudget - 1024 - kCtrlBytes;
  // Ring depths: three decoded-operand slots when two activation slots and
  // four trellis slots still fit (three for small batches, whose stages are
  // long enough that two copies in flight cover the memory latency), else
  // two; then four activation slots for small batches (they are small),
  // otherwise three, if four trellis slots still fit, else two; the trellis
  // ring takes the rest.
  static constexpr int kNW = (kAvail - 2 * kXSlot - 3 * kWSlot >= (XR < 128 ? 3 : 4) * kTSlot) ? 3 : 2;
  static constexpr int kNX = (kAvail - (XR < 128 ? 4 : 3) * kXSlot - kNW * kWSlot >= 4 * kTSlot) ? (XR < 128 ? 4 : 3) : 2;
  static constexpr int kNT0 = (kAvail - kNX * kXSlot - kNW * kWSlot) / kTSlot;
  static constexpr int kNT = kNT0 > 16 ? 16 : kNT0;
  static constexpr int kXRing = 0;  // byte offsets of the rings
  static constexpr int kWRing = kNX * kXSlot;
  static constexpr int kTRing = kWRing + kNW * kWSlot;
  static constexpr int kRingBytes = kTRing + kNT * kTSlot;
  static constexpr int kSmem = 1024 + kCtrlBytes + kRingBytes;
  static constexpr int kMmaHalves = (BN + 127) / 128;  // SWAP: M = 128 instructions per k16 step
  // Unswapped tiles holding at most 64 batch rows use the 64-row MMA: it reads
  // half the activation operand of a 128-row one, most of which would be
  // padding.  Its accumulator puts row r in tensor-memory lane
  // (r % 16) + 32 (r / 16): lanes 32q..32q+15 of quarter q hold rows
  // 16q..16q+15.  Measured on GB300 at m <= 32: 32-column strips 4-7% faster
  // (12288 x 4096, 2048 x 4096, 5120 x 12288), 64-column strips on two k atoms
  // 9% faster, 32-row grouped-expert tiles 1%; 64-column strips on four atoms
  // neutral to 3% slower (17408 x 5120), so they keep the 128-row MMA.
  static constexpr int kMmaM = (!SWAP && XR <= 64 && RG == 1 && !(BN == 64 && KA == 4)) ? 64 : 128;
  static constexpr int kAccCols = SWAP ? kMmaHalves * XR : RG * BN;
  static constexpr int kTmemCols =
      kAccCols <= 32 ? 32 : kAccCols <= 64 ? 64 : kAccCols <= 128 ? 128 : kAccCols <= 256 ? 256 : 512;
  static constexpr int kTiles = kTrRows * (kBNL / 16);  // tiles decoded per stage
  static constexpr int kTpw = kTiles / kTcDecodeWarps;  // per decoder warp
  static constexpr int kZStride = BN + 4;               // epilogue staging row stride (floats)
  // Decoders decode a stage into registers before waiting for its operand
  // slot, except in the single-row-group, full-row shape, where that order
  // measured slower on GB300.
  static constexpr bool kDecodeFirst = !(RG == 1 && XR == 128);
  static_assert(RG * BN <= 512, "accumulators exceed tensor memory");
  static_assert(kNT >= 2, "not enough shared memory for two trellis slots");
  static_assert(kTiles % kTcDecodeWarps == 0 && kTpw >= 1, "tiles per stage must split evenly over the decoders");
  static_assert(XR == 128 || RG == 1, "partial activation regions need a single row group");
  static_assert(kXSlot % 1024 == 0 && kWSlot % 1024 == 0, "operand slots must keep 1024-byte swizzle alignment");
  static_assert(SWAP || XR == 128 || kWRing - kXAtom + 16384 <= kRingBytes,
                "the tensor core's 128-row read of the last atom must stay inside the rings");
  static_assert(!SWAP || BN % 128 == 0 || kWRing + kNW * kWSlot - kWAtom + 16384 <= kRingBytes,
                "the tensor core's 128-row read of the last weight atom must stay inside the rings");
  static_assert(!SWAP || (RG == 1 && PAIR == 1 && XR % 16 == 0 && XR <= 64 && BN % 32 == 0),
                "swapped operands: one row group of 16 to 64 rows, no pairs, whole 32-column quarters");
  static_assert(PAIR == 1 || (BN >= 128 && XR == 128), "pairs share whole 128-column blocks of full row groups");
  static_assert(kWHalfAtom % 1024 == 0, "each CTA's half of an atom must be whole 8-row swizzle groups");
  static_assert(128 * kZStride * 4 <= kRingBytes, "epilogue tile must fit in the rings");
  static_assert((2 * kNT + 2 * kNX + 3 * kNW + 1) * 8 + 8 <= kCtrlBytes, "barriers exceed the control area");
};

template <int BITS, int CB, int BN, int RG, int KA, int XR, int PAIR, bool SWAP = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
  using C = TcCfg<BITS, BN, RG, KA, XR, PAIR, SWAP>;
  constexpr int NT = C::kNT;
  constexpr int NX = C::kNX;
  constexpr int NW = C::kNW;
  constexpr int CLX = C::kClusterX;
  constexpr uint32_t kIdesc = SWAP ? idesc_f16_f32(128, XR) : idesc_f16_f32(C::kMmaM, BN);
  // the row of the row group that a lane of accumulator quarter q holds (-1: none)
  constexpr int kRowsPerQuarter = C::kMmaM / 4;
  const GemmArgs& a = p.a;
  const uint16_t* const svh = a.svh;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by pointer arithmetic so that
  // the compiler keeps every access in the shared address space (an integer
  // round trip would turn the window loads into generic loads).
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* tfull = reinterpret_cast<uint64_t*>(base);  // trellis slot landed (TMA bytes)
  uint64_t* tempty = tfull + NT;                        // trellis slot decoded by every decoder warp
  uint64_t* xfull = tempty + NT;                        // activation slot landed (TMA bytes)
  uint64_t* xempty = xfull + NX;                        // activation slot consumed by the MMA
  uint64_t* wfull = xempty + NX;                        // decoded operand complete
  uint64_t* wdone = wfull + NW;                         // this CTA's decoders done (PAIR = 2)
  uint64_t* wempty = wdone + NW;                        // decoded operand consumed by the MMA(s)
  uint64_t* accfull = wempty + NW;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfull + 1);
  volatile uint32_t* failed = tmem_slot + 1;  // set by the MMA issuer if any wait gave up
  uint8_t* rings = base + C::kCtrlBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A pair is a cluster {2, 1, 1}: blockIdx.x = 2 * pair tile + rank, pair
  // tiles numbered row pair major (a.tile_cols per row pair).
  const uint32_t prank = PAIR > 1 ? cluster_ctarank() : 0u;
  int64_t c0, row0;
  if constexpr (PAIR > 1) {
    const int64_t t = (int64_t)(blockIdx.x >> 1);
    const int64_t rp = t / a.tile_cols;
    c0 = a.col_base + (t - rp * a.tile_cols) * BN;
    row0 = a.row_base + (rp * 2 + prank) * (128 * RG);
  } else {
    c0 = a.col_base + (int64_t)blockIdx.x * BN;
    row0 = a.row_base + (int64_t)blockIdx.y * (128 * RG);
  }
  const int part = (int)blockIdx.z;
  // this CTA's k range in 64-wide atoms: whole units of part_atoms atoms per
  // part (part_atoms = 2 without a split)
  const int64_t units = (a.k >> 6) / a.part_atoms;
  const int64_t kb0 = (int64_t)part * units / a.parts * a.part_atoms;
  const int64_t kb1 = (int64_t)(part + 1) * units / a.parts * a.part_atoms;
  const int nk = (int)((kb1 - kb0) / KA);  // pipeline stages (the host keeps KA a divisor of every part)

  int shard = 0;
#pragma unroll
  for (int i = 1; i < kMaxShards; ++i)
    if (i < a.num_shards && c0 >= a.shard_cols[i]) shard = i;
  // the first tile column of this CTA's trellis copies (a pair's CTAs decode
  // one half of the columns each)
  const int nt0 = (int)(c0 >> 4) + (int)prank * (C::kBNL / 16);
  // trellis copies issued before the block synchronises (by thread 0, the
  // producer): the first min(nk, NT) stages, whose slots start empty
  const int npre = nk < NT ? nk : NT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NT; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], kTcDecodeWarps);
    }
    // The first trellis copies go out now, while the tensor memory is
    // allocated and the block (or pair) synchronises: they need only this
    // CTA's own trellis barriers, initialised just above.
    fence_mbar_init();
    fence_proxy_async_smem();
    prefetch_tensormap(&maps.trellis);
    for (int it = 0; it < npre; ++it) {
      mbar_arrive_expect_tx(&tfull[it], (uint32_t)C::kTrCopy);
      tma_tile3d_g2s(rings + C::kTRing + it * C::kTSlot, &maps.trellis, 0, nt0, (int)(kb0 + (int64_t)it * KA) * 4,
                     &tfull[it]);
    }
    for (int s = 0; s < NX; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int s = 0; s < NW; ++s) {
      // PAIR = 2: the sender arrives once and the partner's copy brings its bytes
      mbar_init(&wfull[s], PAIR > 1 ? 1 : kTcDecodeWarps);
      mbar_init(&wdone[s], kTcDecodeWarps);
      mbar_init(&wempty[s], PAIR);  // one commit per MMA issuer of the pair
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
  // the partner arrives on this CTA's barriers: they must be initialised first
  if (PAIR > 1) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- trellis producer ----------------
    if (lane == 0) {
      // the first npre stages went out before the block synchronised
      int s = npre == NT ? 0 : npre;
      uint32_t ph = npre == NT ? 1u : 0u;
      int it = npre;
      for (; it < nk; ++it) {
        if (!mbar_wait(&tempty[s], ph ^ 1u)) break;
        mbar_arrive_expect_tx(&tfull[s], (uint32_t)C::kTrCopy);
        const int atom0 = (int)(kb0 + (int64_t)it * KA);  // first 64-wide k atom of the stage
        tma_tile3d_g2s(rings + C::kTRing + s * C::kTSlot, &maps.trellis, 0, nt0, atom0 * 4, &tfull[s]);
        if (++s == NT) {
          s = 0;
          ph ^= 1u;
        }
      }
      drain_ring(tfull, NT, it);  // it copies issued
    }
  } else if (warp == 2) {
    // ---------------- activation producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&maps.xh);
      // The activations may come from the kernel just before this one in the
      // stream (the input transform, which lets this grid start early): wait
      // for it here.  Everything else this kernel reads before the wait (the
      // trellis, svh) is weights, which no kernel of this library writes.
      pdl_wait();
      // a split launch's tail may now be scheduled onto SMs as they free up
      if (a.trigger_dependents == 1) pdl_launch_dependents();
      const uint32_t tx = (uint32_t)(RG * KA) * (uint32_t)p.box_rows * 128u;
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      for (; it < nk; ++it) {
        if (!mbar_wait(&xempty[s], ph ^ 1u)) break;
        mbar_arrive_expect_tx(&xfull[s], tx);
        const int atom0 = (int)(kb0 + (int64_t)it * KA);
        uint8_t* o = rings + C::kXRing + s * C::kXSlot;
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          if (KA == 1 || p.box_rows == XR) {
            tma_tile4d_g2s(o + r * KA * C::kXAtom, &maps.xh, 0, (int)(row0 + r * 128), atom0, shard, &xfull[s]);
          } else {
            // fewer rows than an atom region holds: one copy per atom (the
            // map's box is one atom), the rows past box_rows left unwritten
#pragma unroll
            for (int at = 0; at < KA; ++at)
              tma_tile4d_g2s(o + (r * KA + at) * C::kXAtom, &maps.xh, 0, (int)(row0 + r * 128), atom0 + at, shard,
                             &xfull[s]);
          }
        }
        if (++s == NX) {
          s = 0;
          ph ^= 1u;
        }
      }
      drain_ring(xfull, NX, it);  // it copies issued
    }
  } else if (warp == 3) {
    // ---------------- sender (pairs) ----------------
    if (PAIR > 1 && lane == 0) {
      const uint32_t wring_u32 = smem_u32(rings + C::kWRing);
      const uint32_t peer = prank ^ 1u;
      int s = 0;
      uint32_t ph = 0;
      for (int it = 0; it < nk; ++it) {
        if (!mbar_wait(&wdone[s], ph)) break;
        // this CTA's half is complete: expect the partner's half and send ours
        mbar_arrive_expect_tx(&wfull[s], (uint32_t)(KA * C::kWHalfAtom));
#pragma unroll
        for (int at = 0; at < KA; ++at) {
          const uint32_t src = wring_u32 + (uint32_t)(s * C::kWSlot + at * C::kWAtom + (int)prank * C::kWHalfAtom);
          bulk_s2cluster(mapa_shared(src, peer), src, (uint32_t)C::kWHalfAtom, mapa_shared(smem_u32(&wfull[s]), peer));
        }
        if (++s == NW) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // The whole warp runs the loop and one elected lane issues (see elect_one).
    {
      const uint32_t leader = elect_one();
      bool ok = true;
      int xs = 0, ws = 0;
      uint32_t xph = 0, wph = 0;
      const uint64_t xdesc0 = sdesc_sw128(smem_u32(rings + C::kXRing));
      const uint64_t wdesc0 = sdesc_sw128(smem_u32(rings + C::kWRing));
      for (int it = 0; it < nk; ++it) {
        // every lane waits; the vote keeps the warp's decision uniform
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&xfull[xs], xph) && mbar_wait(&wfull[ws], wph));
        if (!ok) break;
        tc_fence_after();
        // descriptors of this stage's operands; an operand at byte offset o
        // from a ring has descriptor desc0 + (o >> 4) (start-address field)
        const uint64_t dx = xdesc0 + (uint64_t)((xs * C::kXSlot) >> 4);
        const uint64_t dwb = wdesc0 + (uint64_t)((ws * C::kWSlot) >> 4);
#pragma unroll
        for (int at = 0; at < KA; ++at) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if constexpr (SWAP) {
              // A: 128 decoded weight rows (columns of W) from the atom, B: the XR activation rows
#pragma unroll
              for (int h = 0; h < C::kMmaHalves; ++h) {
                if (leader)
                  tc_mma_f16(tmem + h * XR, dwb + (uint64_t)((at * C::kWAtom + h * 16384 + j * 32) >> 4),
                             dx + (uint64_t)((at * C::kXAtom + j * 32) >> 4), kIdesc, (it | at | j) != 0);
                __syncwarp();
              }
            } else {
#pragma unroll
              for (int r = 0; r < RG; ++r) {
                if (leader)
                  tc_mma_f16(tmem + r * BN, dx + (uint64_t)((((r * KA + at) * C::kXAtom) + j * 32) >> 4),
                             dwb + (uint64_t)((at * C::kWAtom + j * 32) >> 4), kIdesc, (it | at | j) != 0);
                __syncwarp();
              }
            }
          }
        }
        if (leader) {
          tc_commit(&xempty[xs]);
          if (PAIR > 1) {
            tc_commit_multicast(&wempty[ws], (uint16_t)3u);
          } else {
            tc_commit(&wempty[ws]);
          }
        }
        __syncwarp();
        if (++xs == NX) {
          xs = 0;
          xph ^= 1u;
        }
        if (++ws == NW) {
          ws = 0;
          wph ^= 1u;
        }
      }
      if (leader) {
        if (!ok) *failed = 1u;
        tc_commit(accfull);
      }
    }
    __syncwarp();
  } else {
    // ---------------- decoders ----------------
    const int dw = warp - kTcFirstDecoder;
    const LaneWindow<BITS> lw(lane);
    // the multipliers, copied once from parameter memory into registers
    // (read in place, each use would become a constant-bank load)
    DecodeConsts mc;
#pragma unroll
    for (int i = 0; i <= 16; ++i) {
      // an opaque register copy: the compiler can neither fold the multiply
      // back into a shift nor re-read the value from constant memory per use
      uint32_t v = a.dc.pow2[i];
      asm volatile("" : "+r"(v));
      mc.pow2[i] = v;
    }
    // Per-warp constant byte offsets, so that a tile costs only its loads, its
    // decode and its store: the lane's three window words inside a tile, and
    // where each of this warp's tiles lands in the decoded operand.
    constexpr int kTilesN = C::kBNL / 16;
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
        const int row = (int)prank * C::kBNL + (t - kt_l * kTilesN) * 16 + row_in;
        const int chunk = 2 * (kt_l & 3) + chunk_hi;
        w_off[i] = (uint32_t)((kt_l >> 2) * C::kWAtom + row * 128 + ((chunk ^ (row & 7)) << 4));
      }
    }
    const uint32_t tring_u32 = smem_u32(rings + C::kTRing);
    const uint32_t wring_u32 = smem_u32(rings + C::kWRing);
    uint64_t* const wready = PAIR > 1 ? wdone : wfull;
    int ts = 0, ws = 0;
    uint32_t tph = 0, wph = 0;
    constexpr int kStep = kTcDecodeWarps * kTileBytes;  // tiles of one warp are kTcDecodeWarps apart
    for (int it = 0; it < nk; ++it) {
      if (!mbar_wait(&tfull[ts], tph)) break;
      const uint32_t trbase = tring_u32 + (uint32_t)(ts * C::kTSlot);
      const uint32_t wbase = wring_u32 + (uint32_t)(ws * C::kWSlot);
      if constexpr (XR < 128) {
        // Small batches: one tile at a time, the next tile's window words
        // loaded before this tile's decode and its store right after it.
        // Every decoder warp starts a stage at about the same time: loading
        // a whole stage's words first and storing all of its tiles last
        // queued them on the shared-memory pipe in two bursts that left the
        // warps waiting (measured 4-6% slower on 128-column tiles).
        if (!mbar_wait(&wempty[ws], wph ^ 1u)) break;
        uint32_t wn[3];
        wn[0] = ld_shared_u32(trbase + word_off[0]);
        wn[1] = ld_shared_u32(trbase + word_off[1]);
        wn[2] = (LaneWindow<BITS>::kNeed == 3) ? ld_shared_u32(trbase + word_off[2]) : 0u;
#pragma unroll
        for (int i = 0; i < C::kTpw; ++i) {
          const uint32_t w0 = wn[0], w1 = wn[1], w2 = wn[2];
          if (i + 1 < C::kTpw) {
            const uint32_t o = (uint32_t)((i + 1) * kStep);
            wn[0] = ld_shared_u32(trbase + word_off[0] + o);
            wn[1] = ld_shared_u32(trbase + word_off[1] + o);
            wn[2] = (LaneWindow<BITS>::kNeed == 3) ? ld_shared_u32(trbase + word_off[2] + o) : 0u;
          }
          const Aligned al = align_window<BITS>(w0, w1, w2, lw.off);
          uint32_t b[4];
          decode_lane<BITS, CB>(al, mc, b);
          stmatrix_x4(wbase + w_off[i], b[0], b[1], b[2], b[3]);
        }
      } else {
        // all window words of this warp's tiles first, so their latency overlaps
        uint32_t wv[C::kTpw][3];
#pragma unroll
        for (int i = 0; i < C::kTpw; ++i) {
          wv[i][0] = ld_shared_u32(trbase + word_off[0] + i * kStep);
          wv[i][1] = ld_shared_u32(trbase + word_off[1] + i * kStep);
          wv[i][2] = (LaneWindow<BITS>::kNeed == 3) ? ld_shared_u32(trbase + word_off[2] + i * kStep) : 0u;
        }
        if constexpr (C::kDecodeFirst) {
          // decode into registers first, so that waiting for the decoded-operand
          // slot (consumed by the MMA(s) of its last use) overlaps the arithmetic
          uint32_t b[C::kTpw][4];
#pragma unroll
          for (int i = 0; i < C::kTpw; ++i) {
            const Aligned al = align_window<BITS>(wv[i][0], wv[i][1], wv[i][2], lw.off);
            decode_lane<BITS, CB>(al, mc, b[i]);
          }
          if (!mbar_wait(&wempty[ws], wph ^ 1u)) break;
#pragma unroll
          for (int i = 0; i < C::kTpw; ++i) stmatrix_x4(wbase + w_off[i], b[i][0], b[i][1], b[i][2], b[i][3]);
        } else {
          if (!mbar_wait(&wempty[ws], wph ^ 1u)) break;
#pragma unroll
          for (int i = 0; i < C::kTpw; ++i) {
            const Aligned al = align_window<BITS>(wv[i][0], wv[i][1], wv[i][2], lw.off);
            uint32_t b[4];
            decode_lane<BITS, CB>(al, mc, b);
            stmatrix_x4(wbase + w_off[i], b[0], b[1], b[2], b[3]);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&wready[ws]);
        // The decode above consumed every window word, so the loads have
        // returned: the trellis slot can go back to the producer.  (An arrive
        // issued right after the loads, before their values are used, let the
        // next copy overwrite words that were still being read.)
        mbar_arrive(&tempty[ts]);
      }
      if (++ts == NT) {
        ts = 0;
        tph ^= 1u;
      }
      if (++ws == NW) {
        ws = 0;
        wph ^= 1u;
      }
    }
  }

  // ---------------- epilogue ----------------
  // Decoder warps wait for the accumulators; every warp takes part in the
  // block / cluster barriers below.
  const int dw = warp - kTcFirstDecoder;
  bool ok = true;
  // The output scales of this lane's columns (pass 2 below), loaded before
  // the wait for the accumulators so that their latency hides behind the
  // last MMAs instead of stalling the epilogue.
  constexpr int kSpanBlocks = C::kClusterX * BN / 128;
  const uint32_t rank = (C::kClusterX > 1) ? cluster_ctarank() : 0u;
  const int64_t cbase = c0 - (int64_t)rank * BN;  // first column of the cluster's span
  // Without a cluster, pass 2 gives lane j = lane & 7 columns 4j..4j+3 of
  // each 32-column quarter (four adjacent outputs per store); across a
  // cluster's partner tiles it keeps one column per lane and quarter (scalar
  // distributed-shared-memory loads measured faster there).
  constexpr bool kPackedRows = C::kClusterX == 1;
  float svf[kSpanBlocks][4];  // one column per lane and quarter
  uint2 svw[kSpanBlocks][4];  // four adjacent columns per lane and quarter, fp16 packed
  uint2 svs[kSpanBlocks];  // SWAP: columns 4l..4l+3 of each 128-column block of the span, fp16 packed
  if (SWAP && warp >= kTcFirstDecoder && a.parts == 1) {
#pragma unroll
    for (int hb = 0; hb < kSpanBlocks; ++hb) svs[hb] = *reinterpret_cast<const uint2*>(svh + cbase + hb * 128 + 4 * lane);
  }
  if (!SWAP && warp >= kTcFirstDecoder && a.parts == 1) {
#pragma unroll
    for (int hb = 0; hb < kSpanBlocks; ++hb)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (kPackedRows) {
          svw[hb][i] = *reinterpret_cast<const uint2*>(svh + cbase + hb * 128 + 32 * i + 4 * (lane & 7));
        } else {
          svf[hb][i] = __half2float(__ushort_as_half(svh[cbase + hb * 128 + lane + 32 * i]));
        }
      }
  }
  if (warp >= kTcFirstDecoder) {
    ok = mbar_wait(accfull, 0) && *failed == 0u;
    // the split-k epilogue may be scheduled once every CTA is this far
    if (a.trigger_dependents == 2 && warp == kTcFirstDecoder && lane == 0) pdl_launch_dependents();
    if (PAIR > 1) {
      // This CTA's copies of its decoded halves into the partner read the
      // operand ring, which the epilogue below overwrites: they are complete
      // once the partner's MMAs have consumed them, i.e. when every slot's
      // final phase (which also takes the partner's commit) has completed.
      // That also retires the partner's last arrivals on this CTA's barriers.
      if (lane < NW && lane < nk) {
        const int uses = (nk - lane + NW - 1) / NW;
        ok = mbar_wait(&wempty[lane], (uint32_t)(uses - 1) & 1u) && ok;
      }
      ok = __all_sync(0xFFFFFFFFu, ok);
    }
    tc_fence_after();
  }
  const bool bf16 = a.y_bf16 != 0;
  // rows this CTA stores: everything below m
  const int64_t row_end = a.m;
  uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
  float* zs = reinterpret_cast<float*>(rings);
  constexpr int kZ = C::kZStride;

  if constexpr (SWAP) {
    // Thread (quarter, h) of a decoder warp holds weight column h*128 +
    // 32*quarter + lane of the CTA and its XR batch rows.
    const int quarter = warp & 3;
    const int h = dw >> 2;
    const int col = h * 128 + quarter * 32 + lane;
    const bool holds = warp >= kTcFirstDecoder && h < C::kMmaHalves && h * 128 + quarter * 32 < BN;
    if (a.parts > 1) {
      // split-k: this part's fp32 sums go straight to acc[part][row][col]
      if (holds) {
        uint32_t q[XR];
        tmem_ld_32x32b_cols<XR>(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(h * XR), q);
        tmem_ld_wait();
        float* dst = a.acc + (int64_t)part * a.m * a.n + c0 + col;
        if (ok) {
#pragma unroll
          for (int r = 0; r < XR; ++r)
            if (row0 + r < row_end) dst[(row0 + r) * a.n] = __uint_as_float(q[r]);
        }
      }
    } else {
      // 1. tensor memory -> zs[row][col], raw fp32 sums
      if (holds) {
        uint32_t q[XR];
        tmem_ld_32x32b_cols<XR>(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(h * XR), q);
        tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < XR; ++r) zs[r * kZ + col] = __uint_as_float(q[r]);
      }
      if (CLX > 1) {
        cluster_sync();
      } else {
        __syncthreads();
      }
      // 2. one warp per (row, 128-column block of the span): lane l takes
      // columns 4l..4l+3 (from whichever CTA of the cluster holds them), the
      // full butterfly (strides 1, 2 in registers, 4..64 across lanes), scale
      // and store four adjacent outputs.  The CTAs of a cluster split the rows.
      if (warp >= kTcFirstDecoder) {
        constexpr int kBlocks = CLX * BN / 128;
        const int64_t live = row_end - row0 < XR ? row_end - row0 : XR;
        for (int u = dw;; u += kTcDecodeWarps) {
          const int rr = (int)rank + CLX * (u / kBlocks);
          const int hb = u % kBlocks;
          if (rr >= live) break;
          const int span_col = hb * 128 + 4 * lane;
          const uint32_t src_rank = (uint32_t)(span_col / BN);
          const int local_col = span_col - (int)src_rank * BN;
          const uint32_t zaddr = ((CLX > 1) ? mapa_shared(smem_u32(zs), src_rank) : smem_u32(zs)) +
                                 (uint32_t)((rr * kZ + local_col) * 4);
          const float4 t = (CLX > 1) ? ld_shared_cluster_v4f(zaddr) : ld_shared_v4f(zaddr);
          float v[4] = {t.x, t.y, t.z, t.w};
          fwht128_warp(v, lane);
          uint2 sv = svs[0];
#pragma unroll
          for (int i = 1; i < kSpanBlocks; ++i)
            if (hb == i) sv = svs[i];
          const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sv.x));
          const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&sv.y));
          const uint32_t o0 = f32_to_out((v[0] * 0.125f) * s01.x, bf16), o1 = f32_to_out((v[1] * 0.125f) * s01.y, bf16);
          const uint32_t o2 = f32_to_out((v[2] * 0.125f) * s23.x, bf16), o3 = f32_to_out((v[3] * 0.125f) * s23.y, bf16);
          if (ok)
            *reinterpret_cast<uint2*>(y + (row0 + rr) * a.n + cbase + span_col) = make_uint2(o0 | (o1 << 16), o2 | (o3 << 16));
        }
      }
    }
  } else {
    if (a.parts > 1) {
      // split-k: this part's fp32 sums go straight to acc[part][row][col]
      if (warp >= kTcFirstDecoder) {
        const int quarter = warp & 3;
        float* dst = a.acc + (int64_t)part * a.m * a.n;
        for (int r = 0; r < RG; ++r) {
          for (int cc = dw >> 2; cc < BN / 32; cc += kTcDecodeWarps / 4) {
            uint32_t q[32];
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(r * BN + cc * 32), q);
            tmem_ld_wait();
            const int64_t row = row0 + r * 128 + quarter * kRowsPerQuarter + lane;
            if (ok && lane < kRowsPerQuarter && row < row_end) {
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
      constexpr int kSpan = CLX * BN;  // whole 128-column blocks
      for (int r = 0; r < RG; ++r) {
        // 1. tensor memory -> zs[128][BN].  Each thread holds one row's 32
        // consecutive columns after a load and runs the Hadamard stages of
        // stride 1..16 on them in registers (those pairs never leave a 32-column
        // chunk), so only the stride-32 and stride-64 stages remain.
        if (warp >= kTcFirstDecoder) {
          const int quarter = warp & 3;
          const bool live = row0 + r * 128 + quarter * kRowsPerQuarter < row_end;  // this quarter holds stored rows
          for (int cc = dw >> 2; live && cc < BN / 32; cc += kTcDecodeWarps / 4) {
            uint32_t q[32];
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(r * BN + cc * 32), q);
            tmem_ld_wait();
            float v[32];
  #pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(q[e]);
            fwht32_regs(v);
            float* dst = zs + (quarter * kRowsPerQuarter + lane) * kZ + cc * 32;
            if (lane < kRowsPerQuarter) {  // with the 64-row MMA, lanes 16..31 of a quarter hold no row
  #pragma unroll
              for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            }
          }
        }
        if (CLX > 1) {
          cluster_sync();
        } else {
          __syncthreads();
        }
        if constexpr (kPackedRows) {
          // 2. rows: eight lanes per row, four rows per warp step.  Lane j of a
          // row owns columns 4j..4j+3 of each 32-column quarter of a 128-column
          // block of the span: the stride-32 and stride-64 stages, then scale and
          // store four adjacent outputs (8 bytes) per quarter.
          if (warp >= kTcFirstDecoder) {
            const int j = lane & 7, sr = lane >> 3;
    #pragma unroll
            for (int hb = 0; hb < kSpan / 128; ++hb) {
              uint32_t zsrc[4];
              int64_t col[4];
              float sv[4][4];
    #pragma unroll
              for (int i = 0; i < 4; ++i) {
                // a quarter never straddles two CTAs: BN is a multiple of 32
                const int span_col = hb * 128 + 32 * i + 4 * j;
                const uint32_t src_rank = (uint32_t)(span_col / BN);
                const int local_col = span_col - (int)src_rank * BN;
                col[i] = cbase + span_col;
                zsrc[i] = ((CLX > 1) ? mapa_shared(smem_u32(zs), src_rank) : smem_u32(zs)) + (uint32_t)(local_col * 4);
                const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&svw[hb][i].x));
                const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&svw[hb][i].y));
                sv[i][0] = s01.x;
                sv[i][1] = s01.y;
                sv[i][2] = s23.x;
                sv[i][3] = s23.y;
              }
              for (int rb = (int)rank + CLX * 4 * dw; rb < 128; rb += CLX * 4 * kTcDecodeWarps) {
                const int rr = rb + CLX * sr;  // < 128: rb + 3 * CLX stays inside the group
                const int64_t row = row0 + r * 128 + rr;
                float v[4][4];
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint32_t addr = zsrc[i] + (uint32_t)(rr * kZ * 4);
                  const float4 t = (CLX > 1) ? ld_shared_cluster_v4f(addr) : ld_shared_v4f(addr);
                  v[i][0] = t.x;
                  v[i][1] = t.y;
                  v[i][2] = t.z;
                  v[i][3] = t.w;
                }
                if (ok && row < row_end) {
                  uint16_t* yr = y + row * a.n;
    #pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    // stride 32: (0,1), (2,3); stride 64: (0,2), (1,3)
                    const float a0 = v[0][e] + v[1][e], a1 = v[0][e] - v[1][e];
                    const float a2 = v[2][e] + v[3][e], a3 = v[2][e] - v[3][e];
                    v[0][e] = a0 + a2;
                    v[2][e] = a0 - a2;
                    v[1][e] = a1 + a3;
                    v[3][e] = a1 - a3;
                  }
    #pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    uint32_t o[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = f32_to_out((v[i][e] * 0.125f) * sv[i][e], bf16);
                    *reinterpret_cast<uint2*>(yr + col[i]) = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
                  }
                }
              }
            }
          }
        } else {
          // 2. rows: lane l owns columns l, l+32, l+64, l+96 of each 128-column
          // block of the span: the stride-32 and stride-64 stages, then scale and
          // store (each store instruction writes 32 consecutive columns)
          if (warp >= kTcFirstDecoder) {
    #pragma unroll
            for (int hb = 0; hb < kSpan / 128; ++hb) {
              uint32_t zsrc[4];
              int64_t col[4];
    #pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int span_col = hb * 128 + lane + 32 * i;
                const uint32_t src_rank = (uint32_t)(span_col / BN);
                const int local_col = span_col - (int)src_rank * BN;
                col[i] = cbase + span_col;
                zsrc[i] = ((CLX > 1) ? mapa_shared(smem_u32(zs), src_rank) : smem_u32(zs)) + (uint32_t)(local_col * 4);
              }
              for (int rr = (int)rank + CLX * dw; rr < 128; rr += CLX * kTcDecodeWarps) {
                const int64_t row = row0 + r * 128 + rr;
                if (!ok || row >= row_end) break;  // rows ascend with rr
                float v[4];
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint32_t addr = zsrc[i] + (uint32_t)(rr * kZ * 4);
                  v[i] = (CLX > 1) ? ld_shared_cluster_f32(addr) : ld_shared_f32(addr);
                }
                // stride 32: (0,1), (2,3); stride 64: (0,2), (1,3)
                const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
                v[0] = a0 + a2;
                v[2] = a0 - a2;
                v[1] = a1 + a3;
                v[3] = a1 - a3;
                uint16_t* yr = y + row * a.n;
    #pragma unroll
                for (int i = 0; i < 4; ++i) yr[col[i]] = f32_to_out((v[i] * 0.125f) * svf[hb][i], bf16);
              }
            }
          }
        }
        // the tile is reused by the next row group, and partners may still read it
        if (CLX > 1) {
          cluster_sync();
        } else {
          __syncthreads();
        }
      }
    }

  }
  tc_fence_before();
  if (C::kCluster > 1) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int BITS, int CB, int BN, int RG, int KA, int XR, int PAIR = 1, bool SWAP = false>
cudaError_t launch_tc_variant(const TcMaps& maps, const TcParams& p, cudaStream_t stream) {
  using C = TcCfg<BITS, BN, RG, KA, XR, PAIR, SWAP>;
  auto kern = gemm_tc_kernel<BITS, CB, BN, RG, KA, XR, PAIR, SWAP>;
  // the shared-memory opt-in, once per device (benign race: every thread sets
  // the same attribute)
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  // a pair's second CTA may own only rows past m: it still decodes its half
  if (PAIR > 1) {
    cfg.gridDim = dim3((unsigned)(2 * p.a.pair_tiles), 1u, (unsigned)p.a.parts);
  } else {
    const int64_t row_blocks = (p.a.m - p.a.row_base + 128 * RG - 1) / (128 * RG);
    cfg.gridDim = dim3((unsigned)((p.a.n - p.a.col_base) / BN), (unsigned)row_blocks, (unsigned)p.a.parts);
  }
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::kClusterX * PAIR;  // strips (BN < 128) and pairs never combine
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel (the input transform) still runs;
  // the activation producer waits for it (pdl_wait) before reading xh
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

// Tile shapes compiled for every width and codebook (see TcShape in exl3_launch.h).
template <int BITS, int CB>
cudaError_t launch_tc_cb(const TcMaps& maps, const TcParams& p, TcShape shape, cudaStream_t stream) {
  switch (shape) {
    case TcShape::kN32Small: return launch_tc_variant<BITS, CB, 32, 1, 4, 32>(maps, p, stream);
    case TcShape::kN64Small: return launch_tc_variant<BITS, CB, 64, 1, 2, 32>(maps, p, stream);
    case TcShape::kN128Small: return launch_tc_variant<BITS, CB, 128, 1, 2, 32>(maps, p, stream);
    case TcShape::kN128: return launch_tc_variant<BITS, CB, 128, 1, 2, 128>(maps, p, stream);
    case TcShape::kN128R2: return launch_tc_variant<BITS, CB, 128, 2, 1, 128>(maps, p, stream);
    case TcShape::kN128R2P: return launch_tc_variant<BITS, CB, 128, 2, 1, 128, 2>(maps, p, stream);
    case TcShape::kN256R2P: return launch_tc_variant<BITS, CB, 256, 2, 1, 128, 2>(maps, p, stream);
    case TcShape::kN128SmallK4: return launch_tc_variant<BITS, CB, 128, 1, 4, 32>(maps, p, stream);
    case TcShape::kN96SmallK4: return launch_tc_variant<BITS, CB, 96, 1, 4, 32>(maps, p, stream);
    case TcShape::kN96: return launch_tc_variant<BITS, CB, 96, 1, 2, 128>(maps, p, stream);
    case TcShape::kN96R2: return launch_tc_variant<BITS, CB, 96, 2, 2, 128>(maps, p, stream);
    case TcShape::kN32SmallK8: return launch_tc_variant<BITS, CB, 32, 1, 8, 32>(maps, p, stream);
    case TcShape::kN64SmallK4: return launch_tc_variant<BITS, CB, 64, 1, 4, 32>(maps, p, stream);
    case TcShape::kN96M64K4: return launch_tc_variant<BITS, CB, 96, 1, 4, 64>(maps, p, stream);
    case TcShape::kN64M64K4: return launch_tc_variant<BITS, CB, 64, 1, 4, 64>(maps, p, stream);
    case TcShape::kN64K4: return launch_tc_variant<BITS, CB, 64, 1, 4, 128>(maps, p, stream);
    case TcShape::kN32K4: return launch_tc_variant<BITS, CB, 32, 1, 4, 128>(maps, p, stream);
    case TcShape::kT128K4: return launch_tm_variant<BITS, CB, 4, 32>(maps, p, stream);
    case TcShape::kT128: return launch_tm_variant<BITS, CB, 2, 32>(maps, p, stream);
    case TcShape::kS96K4: return launch_tc_variant<BITS, CB, 96, 1, 4, 32, 1, true>(maps, p, stream);
    case TcShape::kT128K4X16: return launch_tm_variant<BITS, CB, 4, 16>(maps, p, stream);
    case TcShape::kS96K4X16: return launch_tc_variant<BITS, CB, 96, 1, 4, 16, 1, true>(maps, p, stream);
    case TcShape::kT128X16: return launch_tm_variant<BITS, CB, 2, 16>(maps, p, stream);
    case TcShape::kT128K4X64: return launch_tm_variant<BITS, CB, 4, 64>(maps, p, stream);
    case TcShape::kT128X64: return launch_tm_variant<BITS, CB, 2, 64>(maps, p, stream);
    case TcShape::kT128X128: return launch_tm_variant<BITS, CB, 2, 128>(maps, p, stream);
    case TcShape::kT128K4X128: return launch_tm_variant<BITS, CB, tm128_k4_atoms(BITS), 128>(maps, p, stream);
    case TcShape::kS96K4X64: return launch_tc_variant<BITS, CB, 96, 1, 4, 64, 1, true>(maps, p, stream);
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

// Grouped GEMM tiles: the persistent tensor-memory kernel, one item per row
// block and 128-column block, holding the block's 16, 32 or 128 rows.
template <int BITS, int CB>
cudaError_t launch_moe_cb(const TcMaps& maps, const TcParams& p, int tile, cudaStream_t stream) {
  if (tile == kMoeTileTm16K4) return launch_tm_variant<BITS, CB, 4, 16, true>(maps, p, stream);
  if (tile == kMoeTileTm16) return launch_tm_variant<BITS, CB, 2, 16, true>(maps, p, stream);
  if (tile == kMoeTileTm32K4) return launch_tm_variant<BITS, CB, 4, 32, true>(maps, p, stream);
  if (tile == kMoeTileTm32) return launch_tm_variant<BITS, CB, 2, 32, true>(maps, p, stream);
  if (tile == kMoeTileTm128K4) return launch_tm_variant<BITS, CB, tm128_k4_atoms(BITS), 128, true>(maps, p, stream);
  return launch_tm_variant<BITS, CB, 2, 128, true>(maps, p, stream);  // kMoeTileTm128
}

template <int BITS>
cudaError_t launch_moe_gemm_tc_bits(const TcMaps& maps, const TcParams& p, int cb, int tile, cudaStream_t stream) {
  switch (cb) {
    case CB_3INST: return launch_moe_cb<BITS, CB_3INST>(maps, p, tile, stream);
    case CB_MCG: return launch_moe_cb<BITS, CB_MCG>(maps, p, tile, stream);
    default: return launch_moe_cb<BITS, CB_MUL1>(maps, p, tile, stream);
  }
}

}  // namespace exl3
