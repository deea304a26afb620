// exl3_gemm_tm.cuh -- small-batch EXL3 GEMM with the decoded weights in tensor
// memory.
//
// A work item is 128 output columns (one Hadamard block) and at most XR batch
// rows (XR = 16, 32, 64 or 128), over all of k or one shape-fixed part of it;
// in the grouped (MOE) mode, one expert block's rows.  The tensor core
// takes the decoded weights as its A operand (M = 128 weight columns) straight
// from tensor memory and the rotated activations as B (N = XR rows) from
// shared memory: the accumulator holds one weight column per tensor-memory
// lane and one batch row per column, and every element is the same fp32 sum
// of k16 steps in ascending k as in the shared-memory kernels, so the bytes of
// a row do not depend on which kernel ran it.
//
// The decoders write each k16 step of A with tcgen05.st: thread t of a warp on
// SM sub-partition q owns tensor-memory lane 32q + t, i.e. weight column
// 32q + t of the CTA, and decodes that column's 16 values of the k16 step (the
// 16 states of one column of a 16x16 tile lie in 28 consecutive values of the
// tile's bit stream), packs them as 8 k pairs and stores them.  Compared with
// decoding into the shared-memory operand layout, the decoded weights never
// touch shared memory (no stores, no proxy fence, no operand reads by the
// tensor core), which is what bounded the shared-memory kernels at small m.
//
// The kernel is persistent: CTA c takes the work items (128-column block,
// k part) c, c + G, c + 2G, ... of a grid of G <= #SMs CTAs, its rings running
// on from one item to the next, so the trellis copies of the next item start
// while the current one finishes, and its epilogue overlaps the next item's
// decode (two accumulator buffers in tensor memory).
//
// Warp roles: 0 trellis producer (3-D tensor copies into a deep ring), 1 MMA
// issuer (one elected lane), 2 activation producer, 3 idle, 4..19 decoders,
// 20..23 the epilogue.  Decoder warp dw serves lane quarter dw & 3 (a warp
// reaches only the tensor-memory lanes of its sub-partition) and the stage's
// k16 rows (dw >> 2) + 4i; epilogue warp e reads lane quarter e.  Tensor
// memory: two accumulators of max(32, XR) columns from column 0, then NW slots
// of decoded A (32*KA columns each) from column max(128, 2 * max(32, XR)).
#pragma once

#include "exl3_device.cuh"
#include "exl3_launch.h"
#include "exl3_sm100.cuh"

namespace exl3 {

constexpr int kTmDecodeWarps = 16;
constexpr int kTmFirstDecoder = 4;
constexpr int kTmFirstEpilogue = kTmFirstDecoder + kTmDecodeWarps;
constexpr int kTmThreads = 32 * (kTmFirstEpilogue + 4);
constexpr int kTmSmemBudget = 227 * 1024;

// A thread's bit window: the states of values v0 + d, d in {0..3, 8..11,
// 16..19, 24..27}, i.e. 27 * BITS + 16 bits from the state of v0.
template <int BITS>
struct ColWindow {
  static constexpr int kSpan = 27 * BITS + 16;
  static constexpr int kViews = (kSpan + 31) / 32;  // aligned 32-bit views of the window
  static constexpr int kWords = kViews + 1;         // words loaded (the window starts anywhere in word 0)
  static constexpr int kTileWords = 8 * BITS;
};

template <int BITS, int KA, int XR>
struct TmCfg {
  static constexpr int kTiles = 4 * KA * 8;                          // 16x16 tiles per stage
  static constexpr int kTrCopy = kTiles * 32 * BITS;                 // bytes of one trellis copy
  static constexpr int kTSlot = (kTrCopy + 127) / 128 * 128;
  static constexpr int kXSlot = KA * XR * 128;                       // activation rows of a stage
  // four activation slots while they are small, three, or two when a slot
  // is 64 KB (128 rows, four atoms)
  static constexpr int kNX = XR <= 32 ? 4 : (kXSlot >= 64 * 1024 ? 2 : 3);
  // tensor memory: two accumulator buffers of max(32, XR) columns (one batch
  // row per column, one weight column per lane), then the A slots
  static constexpr int kAccCols = XR < 32 ? 32 : XR;
  static constexpr int kABase = 2 * kAccCols > 128 ? 2 * kAccCols : 128;
  static constexpr int kACols = 32 * KA;                             // tensor-memory columns of a stage's A
  static constexpr int kNW = (512 - kABase) / kACols > 4 ? 4 : (512 - kABase) / kACols;
  // the epilogue stages up to 32 accumulator rows at a time
  static constexpr int kZRows = XR < 32 ? XR : 32;
  static constexpr int kZChunks = XR / kZRows;
  static constexpr int kZStride = 128 + 4;                           // epilogue staging row stride (floats)
  static constexpr int kZBytes = (kZRows * kZStride * 4 + 1023) / 1024 * 1024;
  static constexpr int kCtrlBytes = 1024;
  static constexpr int kAvail = kTmSmemBudget - 1024 - kCtrlBytes - kNX * kXSlot - kZBytes - 128;
  static constexpr int kNT0 = kAvail / kTSlot;
  static constexpr int kNT = kNT0 > 12 ? 12 : kNT0;
  static constexpr int kXRing = 0;
  static constexpr int kZRing = kNX * kXSlot;
  static constexpr int kTRing = kZRing + kZBytes;
  // 128 bytes of slack after the trellis ring: a window's last word may lie
  // one word past the last tile of the last slot (it is loaded, never used)
  static constexpr int kRingBytes = kTRing + kNT * kTSlot + 128;
  // more than half of the shared memory, so one CTA per SM (each allocates all
  // 512 tensor-memory columns)
  static constexpr int kSmemRaw = 1024 + kCtrlBytes + kRingBytes;
  static constexpr int kSmem = kSmemRaw > 120 * 1024 ? kSmemRaw : 120 * 1024;
  static_assert(XR == 16 || XR == 32 || XR == 64 || XR == 128, "16, 32, 64 or 128 batch rows");
  static_assert(kNW >= 2 && kNT >= 3, "rings too shallow");
  static_assert(kABase + kNW * kACols <= 512, "tensor memory overflow");
  static_assert(kXSlot % 1024 == 0, "activation slots keep 1024-byte swizzle alignment");
  // the rings' full and empty barriers, accfull[2], accempty[2], zfull, zdone
  // and mdrain, then the tensor-memory address and the failure flag
  static_assert((2 * kNT + 2 * kNX + 2 * kNW + 7) * 8 + 8 <= kCtrlBytes, "barriers exceed the control area");
};

// State of relative value D of a thread's window from its aligned views
// (r[i] = window bits [32 i, 32 i + 32), h[i] = bits [32 i + 16, 32 i + 48)).
// One operation when the state sits at bit 0, 8 or 16 of a view; a state that
// straddles two aligned views elsewhere is one funnel shift of the pair plus a
// mask (so no half view is built for it); otherwise the bits above it are
// dropped by a multiply with 2^(16 - q) on the integer multiply pipe (the
// hashes of 3inst and mcg leave that pipe room) or, for mul1, whose byte sums
// already load it, by a shift on the ALU pipe, and the bits below by a right
// shift of 16.
template <int BITS, int D, int CB, int V>
__device__ __forceinline__ uint32_t col_state(const uint32_t (&r)[V], const uint32_t (&h)[V], const DecodeConsts& mc) {
  constexpr int p = D * BITS;
  constexpr int v = p / 32, q0 = p % 32;
  constexpr bool half = q0 > 16;               // inside the half-offset view h[v]
  constexpr int q = half ? q0 - 16 : q0;       // offset inside the chosen view
  static_assert(v < V && (!half || v + 1 < V), "state outside the views");
  if constexpr (half && q != 0 && q != 8) return __funnelshift_r(r[v], r[v + 1], q0) & 0xFFFFu;
  const uint32_t x = half ? h[v] : r[v];
  if constexpr (q == 0) {
    return x & 0xFFFFu;
  } else if constexpr (q == 16) {
    return x >> 16;
  } else if constexpr (q == 8) {
    return __byte_perm(x, 0u, 0x4421);
  } else if constexpr (CB == CB_MUL1) {
    return (x >> q) & 0xFFFFu;
  } else {
    return (x * mc.pow2[16 - q]) >> 16;
  }
}

// The thread's 16 values as 8 k pairs of its column: register c holds k = 2c
// (low half) and 2c + 1 of the k16 step, i.e. relative values 8c, 8c + 1 for
// c < 4 and 8(c - 4) + 2, 8(c - 4) + 3 for c >= 4 (the tile's value order:
// TensorFold PR #740, "Arithmetic" step 2, the mma.m16n8k16 B-fragment order).
template <int BITS, int CB>
__device__ __forceinline__ void decode_column(const uint32_t* w, uint32_t off, const DecodeConsts& mc, uint32_t out[8]) {
  using W = ColWindow<BITS>;
  uint32_t r[W::kViews], h[W::kViews];
#pragma unroll
  for (int i = 0; i < W::kViews; ++i) r[i] = __funnelshift_r(w[i], w[i + 1], off);
#pragma unroll
  for (int i = 0; i + 1 < W::kViews; ++i) h[i] = __byte_perm(r[i], r[i + 1], 0x5432);
  h[W::kViews - 1] = 0u;  // never used: no state spans past the last view
  out[0] = decode_pair_balanced<CB>(col_state<BITS, 0, CB>(r, h, mc), col_state<BITS, 1, CB>(r, h, mc), mc);
  out[1] = decode_pair_balanced<CB>(col_state<BITS, 8, CB>(r, h, mc), col_state<BITS, 9, CB>(r, h, mc), mc);
  out[2] = decode_pair_balanced<CB>(col_state<BITS, 16, CB>(r, h, mc), col_state<BITS, 17, CB>(r, h, mc), mc);
  out[3] = decode_pair_balanced<CB>(col_state<BITS, 24, CB>(r, h, mc), col_state<BITS, 25, CB>(r, h, mc), mc);
  out[4] = decode_pair_balanced<CB>(col_state<BITS, 2, CB>(r, h, mc), col_state<BITS, 3, CB>(r, h, mc), mc);
  out[5] = decode_pair_balanced<CB>(col_state<BITS, 10, CB>(r, h, mc), col_state<BITS, 11, CB>(r, h, mc), mc);
  out[6] = decode_pair_balanced<CB>(col_state<BITS, 18, CB>(r, h, mc), col_state<BITS, 19, CB>(r, h, mc), mc);
  out[7] = decode_pair_balanced<CB>(col_state<BITS, 26, CB>(r, h, mc), col_state<BITS, 27, CB>(r, h, mc), mc);
}

// The work item w of a call: its 128-column block, its k part, the first
// column and the first 64-wide k atom and stage count of the part; for the
// grouped GEMM also its row block, that block's first row and expert, and
// whether the block has an expert at all (live).
struct TmItem {
  int64_t c0;
  int64_t kb0;
  int64_t row0;
  int nk;
  int part;
  int expert;
  bool live;
};
template <int KA, bool MOE>
__device__ __forceinline__ TmItem tm_item(const GemmArgs& a, int64_t w64) {
  TmItem t;
  if constexpr (MOE) {
    // items are (row block, 128-column block), row block major
    const int64_t nblk = a.n >> 7;
    const int64_t blk = w64 / nblk;
    t.c0 = (w64 - blk * nblk) * 128;
    t.part = 0;
    t.kb0 = 0;
    t.nk = (int)((a.k >> 7) * 2 / KA);
    t.row0 = blk * a.moe_block;
    t.expert = a.block_expert[blk];
    t.live = t.expert >= 0 && t.expert < a.num_experts;
    return t;
  } else {
    // 32-bit index arithmetic (every warp calls this once per item): k and n
    // are at most 2^31, so n/128 and the k units (2 or 4 atoms of 64) are at
    // most 2^24, and there are at most 16 parts, so every product below stays
    // under 2^28 before its scaling by part_atoms
    const uint32_t nblk = (uint32_t)((a.n - a.col_base) >> 7);
    const uint32_t pa = (uint32_t)a.part_atoms;
    const uint32_t kunits = (uint32_t)(a.k >> 6) / pa;
    const uint32_t parts = (uint32_t)a.parts;
    const uint32_t w = (uint32_t)w64;
    const uint32_t part = w / nblk;
    t.c0 = a.col_base + (int64_t)(w - part * nblk) * 128;
    t.part = (int)part;
    // whole units of part_atoms atoms of k per part
    const uint32_t kb0 = part * kunits / parts * pa;
    const uint32_t kb1 = (part + 1) * kunits / parts * pa;
    t.kb0 = (int64_t)kb0;
    t.nk = (int)((kb1 - kb0) / KA);  // the host keeps KA a divisor of every part
    t.row0 = a.row_base;
    t.expert = 0;
    t.live = true;
    return t;
  }
}

template <int BITS, int CB, int KA, int XR, bool MOE = false>
__global__ void __launch_bounds__(kTmThreads, 1)
    gemm_tm_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcParams p) {
  using C = TmCfg<BITS, KA, XR>;
  using W = ColWindow<BITS>;
  constexpr int NT = C::kNT;
  constexpr int NX = C::kNX;
  constexpr int NW = C::kNW;
  constexpr uint32_t kIdesc = idesc_f16_f32(128, XR);
  const GemmArgs& a = p.a;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* tfull = reinterpret_cast<uint64_t*>(base);  // trellis slot landed (TMA bytes)
  uint64_t* tempty = tfull + NT;                        // trellis slot decoded by every decoder warp
  uint64_t* xfull = tempty + NT;                        // activation slot landed (TMA bytes)
  uint64_t* xempty = xfull + NX;                        // activation slot consumed by the MMAs
  uint64_t* afull = xempty + NX;                        // decoded A of a stage stored in tensor memory
  uint64_t* aempty = afull + NW;                        // decoded A of a stage consumed by the MMAs
  uint64_t* accfull = aempty + NW;                      // [2] an item's accumulator complete
  uint64_t* accempty = accfull + 2;                     // [2] an item's accumulator read by the epilogue
  uint64_t* zfull = accempty + 2;                       // the epilogue staging tile written by all four warps
  uint64_t* zdone = zfull + 1;                          // the epilogue staging tile read by all four warps
  uint64_t* mdrain = zdone + 1;                         // the MMAs issued before a wait gave up are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdrain + 1);
  volatile uint32_t* failed = tmem_slot + 1;  // set by the MMA issuer if a wait gave up
  uint8_t* rings = base + C::kCtrlBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // grouped GEMM: every (row block, 128-column block); a block of no expert
  // is skipped by every warp alike
  const int64_t items = MOE ? (a.m / a.moe_block) * (a.n >> 7) : ((a.n - a.col_base) >> 7) * a.parts;
  const int64_t stride = gridDim.x;
  // this CTA's items: blockIdx.x, blockIdx.x + G, ...
  const int64_t count = (items - blockIdx.x + stride - 1) / stride;
  // Dense calls: the trellis copies of the first min(nk, NT) stages of this
  // CTA's first item (item blockIdx.x, always live) are issued by thread 0,
  // the producer, before the block synchronises; their slots start empty.
  int npre = 0;
  int64_t first_c0 = 0, first_kb0 = 0;
  if constexpr (!MOE) {
    const TmItem first = tm_item<KA, false>(a, blockIdx.x);
    npre = first.nk < NT ? first.nk : NT;
    first_c0 = first.c0;
    first_kb0 = first.kb0;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < NT; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], kTmDecodeWarps);
    }
    if constexpr (!MOE) {
      // they need only the trellis barriers, initialised just above, and
      // overlap the tensor-memory allocation and the block barrier
      fence_mbar_init();
      fence_proxy_async_smem();
      prefetch_tensormap(&maps.trellis);
      for (int it = 0; it < npre; ++it) {
        mbar_arrive_expect_tx(&tfull[it], (uint32_t)C::kTrCopy);
        tma_tile3d_g2s(rings + C::kTRing + it * C::kTSlot, &maps.trellis, 0, (int)(first_c0 >> 4),
                       (int)(first_kb0 + (int64_t)it * KA) * 4, &tfull[it]);
      }
    }
    for (int s = 0; s < NX; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int s = 0; s < NW; ++s) {
      mbar_init(&afull[s], kTmDecodeWarps);
      mbar_init(&aempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 4);  // the four epilogue warps
    }
    mbar_init(zfull, 4);
    mbar_init(zdone, 4);
    mbar_init(mdrain, 1);
    *failed = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- trellis producer ----------------
    if (lane == 0) {
      if constexpr (MOE) prefetch_tensormap(&maps.trellis);
      // the first npre stages went out before the block synchronised
      int s = npre == NT ? 0 : npre;
      uint32_t ph = npre == NT ? 1u : 0u;
      int64_t issued = npre;  // copies put into the ring so far
      bool ok = true;
      for (int64_t i = 0; ok && i < count; ++i) {
        const TmItem t = tm_item<KA, MOE>(a, blockIdx.x + i * stride);
        if (!t.live) continue;
        const int nt0 = (int)(t.c0 >> 4);
        for (int it = i == 0 ? npre : 0; it < t.nk; ++it) {
          if (!mbar_wait(&tempty[s], ph ^ 1u)) {
            ok = false;
            break;
          }
          ++issued;
          mbar_arrive_expect_tx(&tfull[s], (uint32_t)C::kTrCopy);
          if constexpr (MOE) {
            tma_tile4d_g2s(rings + C::kTRing + s * C::kTSlot, &maps.trellis, 0, nt0,
                           (int)(t.kb0 + (int64_t)it * KA) * 4, t.expert, &tfull[s]);
          } else {
            tma_tile3d_g2s(rings + C::kTRing + s * C::kTSlot, &maps.trellis, 0, nt0,
                           (int)(t.kb0 + (int64_t)it * KA) * 4, &tfull[s]);
          }
          if (++s == NT) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      drain_ring(tfull, NT, issued);
    }
  } else if (warp == 2) {
    // ---------------- activation producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&maps.xh);
      // the activations may come from the kernel just before this one (the
      // input transform, which lets this grid start early): wait for it here;
      // the trellis and svh read before are weights, which no kernel writes
      pdl_wait();
      const uint32_t tx = (uint32_t)KA * (uint32_t)p.box_rows * 128u;
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;  // copies put into the ring so far
      bool ok = true;
      for (int64_t i = 0; ok && i < count; ++i) {
        const TmItem t = tm_item<KA, MOE>(a, blockIdx.x + i * stride);
        if (!t.live) continue;
        int shard = 0;
#pragma unroll
        for (int j = 1; j < kMaxShards; ++j)
          if (j < a.num_shards && t.c0 >= a.shard_cols[j]) shard = j;
        for (int it = 0; it < t.nk; ++it) {
          if (!mbar_wait(&xempty[s], ph ^ 1u)) {
            ok = false;
            break;
          }
          ++issued;
          mbar_arrive_expect_tx(&xfull[s], tx);
          const int atom0 = (int)(t.kb0 + (int64_t)it * KA);
          if (p.box_rows == XR) {
            tma_tile4d_g2s(rings + C::kXRing + s * C::kXSlot, &maps.xh, 0, (int)t.row0, atom0, shard, &xfull[s]);
          } else {
            // fewer rows than a slot's atom holds: one copy per atom (the
            // map's box is one atom), the rows past box_rows left unwritten
#pragma unroll
            for (int at = 0; at < KA; ++at)
              tma_tile4d_g2s(rings + C::kXRing + s * C::kXSlot + at * XR * 128, &maps.xh, 0, (int)t.row0, atom0 + at,
                             shard, &xfull[s]);
          }
          if (++s == NX) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      drain_ring(xfull, NX, issued);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // The whole warp runs the loop and one elected lane issues (see
    // elect_one).  A k16 step's A is the 8 tensor-memory columns 8r of its
    // stage's slot, B its rows of the activation slot (descriptor start
    // advanced 32 bytes per k16 inside an atom); item i accumulates in buffer
    // i & 1 once the epilogue has read that buffer's previous item.
    {
      const uint32_t leader = elect_one();
      bool ok = true;
      int xs = 0, as = 0;
      uint32_t xph = 0, aph = 0;
      const uint64_t xdesc0 = sdesc_sw128(smem_u32(rings + C::kXRing));
      uint32_t li = 0;  // live items so far: they alternate the accumulator buffers
      for (int64_t i = 0; ok && i < count; ++i) {
        const TmItem t = tm_item<KA, MOE>(a, blockIdx.x + i * stride);
        if (!t.live) continue;
        const int buf = (int)(li & 1u);
        // (every lane waits; the vote keeps the warp's decision uniform)
        if (li >= 2 && !__all_sync(0xFFFFFFFFu, mbar_wait(&accempty[buf], ((li >> 1) - 1) & 1u))) {
          ok = false;
          break;
        }
        const uint32_t dacc = tmem + (uint32_t)(C::kAccCols * buf);
        for (int it = 0; it < t.nk; ++it) {
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(&xfull[xs], xph) && mbar_wait(&afull[as], aph));
          if (!ok) break;
          tc_fence_after();
          const uint64_t dx = xdesc0 + (uint64_t)((xs * C::kXSlot) >> 4);
          const uint32_t acol = tmem + (uint32_t)C::kABase + (uint32_t)(as * C::kACols);
#pragma unroll
          for (int at = 0; at < KA; ++at) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (leader)
                tc_mma_f16_ta(dacc, acol + (uint32_t)(8 * (4 * at + j)), dx + (uint64_t)((at * XR * 128 + j * 32) >> 4),
                              kIdesc, (it | at | j) != 0);
              __syncwarp();
            }
          }
          if (leader) {
            tc_commit(&xempty[xs]);
            tc_commit(&aempty[as]);
          }
          __syncwarp();
          if (++xs == NX) {
            xs = 0;
            xph ^= 1u;
          }
          if (++as == NW) {
            as = 0;
            aph ^= 1u;
          }
        }
        if (ok && leader) tc_commit(&accfull[buf]);
        __syncwarp();
        ++li;
      }
      if (!ok) {
        // a wait gave up: the MMAs issued so far may still be running, so
        // wait (bounded) for them before the tensor memory is freed
        if (leader) {
          *failed = 1u;
          tc_commit(mdrain);
        }
        __syncwarp();
        mbar_wait(mdrain, 0u);
      }
    }
    __syncwarp();
  } else if (warp >= kTmFirstDecoder && warp < kTmFirstEpilogue) {
    // ---------------- decoders ----------------
    const int dw = warp - kTmFirstDecoder;
    // the powers of two, copied once from parameter memory into registers
    // (opaque, so the multiplies stay multiplies and are not re-read per use)
    DecodeConsts mc;
#pragma unroll
    for (int i = 0; i <= 16; ++i) {
      uint32_t v = a.dc.pow2[i];
      asm volatile("" : "+r"(v));
      mc.pow2[i] = v;
    }
    const int quarter = dw & 3;  // this warp's sub-partition: tensor-memory lanes 32q..32q+31
    const int rsel = dw >> 2;    // the stage's k16 rows rsel + 4i
    // this thread's column: 32q + lane of the block, column lane & 15 of tile 2q + (lane >> 4)
    const int ctile = 2 * quarter + (lane >> 4);
    const int v0 = 32 * (lane & 7) + 4 * ((lane >> 3) & 1);  // first of its 16 values in the tile
    int start = (v0 + 1) * BITS - 16;                          // bit where that value's state starts
    if (start < 0) start += 256 * BITS;                        // circular: wraps to the tile's end
    const uint32_t off = (uint32_t)(start & 31);
    // Byte offsets of the window's words inside a tile: the first may wrap to
    // the tile's last word, the others follow one another from the next word
    // (the window never runs past the tile's end), so they load at constant
    // offsets from one base.
    constexpr int kRowBytes = 8 * 32 * BITS;  // the 8 tiles of one k16 row
    const uint32_t col_off = (uint32_t)(ctile * 32 * BITS + rsel * kRowBytes);
    const uint32_t wo0 = col_off + (uint32_t)(4 * (start >> 5));
    const uint32_t wo1 = col_off + (uint32_t)(4 * (((start >> 5) + 1) % W::kTileWords));
    const uint32_t tring_u32 = smem_u32(rings + C::kTRing);
    const uint32_t tlane = tmem + ((uint32_t)(32 * quarter) << 16);
    int ts = 0, as = 0;
    uint32_t tph = 0, aph = 0;
    bool ok = true;
    for (int64_t i = 0; ok && i < count; ++i) {
      const TmItem t = tm_item<KA, MOE>(a, blockIdx.x + i * stride);
      if (!t.live) continue;
      const int nk = t.nk;
      for (int it = 0; it < nk; ++it) {
        if (!mbar_wait(&tfull[ts], tph) || !mbar_wait(&aempty[as], aph ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tring_u32 + (uint32_t)(ts * C::kTSlot);
        const uint32_t b0 = tb + wo0, b1 = tb + wo1;
        const uint32_t acol = tlane + (uint32_t)C::kABase + (uint32_t)(as * C::kACols);
        // the next row's words are loaded before this row's decode
        uint32_t wn[W::kWords];
        wn[0] = ld_shared_u32(b0);
#pragma unroll
        for (int k = 1; k < W::kWords; ++k) wn[k] = ld_shared_u32(b1 + 4u * (k - 1));
#pragma unroll
        for (int u = 0; u < KA; ++u) {
          uint32_t w[W::kWords];
#pragma unroll
          for (int k = 0; k < W::kWords; ++k) w[k] = wn[k];
          if (u + 1 < KA) {
            constexpr uint32_t kNext = 4 * kRowBytes;
            wn[0] = ld_shared_u32(b0 + (uint32_t)(u + 1) * kNext);
#pragma unroll
            for (int k = 1; k < W::kWords; ++k) wn[k] = ld_shared_u32(b1 + (uint32_t)(u + 1) * kNext + 4u * (k - 1));
          }
          uint32_t out[8];
          decode_column<BITS, CB>(w, off, mc, out);
          tmem_st_32x32b_x8(acol + (uint32_t)(8 * (rsel + 4 * u)), out);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&afull[as]);
          // the decode consumed every window word of the stage, so the loads
          // have returned and the trellis slot can go back to the producer
          mbar_arrive(&tempty[ts]);
        }
        if (++ts == NT) {
          ts = 0;
          tph ^= 1u;
        }
        if (++as == NW) {
          as = 0;
          aph ^= 1u;
        }
      }
    }
  } else if (warp >= kTmFirstEpilogue) {
    // ---------------- epilogue ----------------
    // Warp e reads lane quarter e (its 32 columns' rows) of the item's
    // accumulator and hands the buffer back to the MMA issuer; then, after the
    // four have staged their columns, each takes rows e, e + 4, ...: the
    // 128-point butterfly (strides 1, 2 in registers, 4..64 across lanes),
    // scale and store four adjacent outputs per lane.
    const int e = warp - kTmFirstEpilogue;
    const bool bf16 = a.y_bf16 != 0;
    // rows stored: a grouped block owns exactly its rows (padding rows of a
    // live block included); otherwise every held row below m
    const int64_t live =
        MOE ? (int64_t)a.moe_block : (a.m - a.row_base < XR ? a.m - a.row_base : XR);
    uint16_t* y = reinterpret_cast<uint16_t*>(a.y);
    float* zs = reinterpret_cast<float*>(rings + C::kZRing);
    constexpr int kZ = C::kZStride;
    uint32_t li = 0;  // live items so far (accumulator buffer and staging phases)
    for (int64_t i = 0; i < count; ++i) {
      const TmItem t = tm_item<KA, MOE>(a, blockIdx.x + i * stride);
      if (!t.live) continue;
      const int buf = (int)(li & 1u);
      const uint16_t* svh = MOE ? a.svh + (int64_t)t.expert * a.n : a.svh;
      uint2 sv = make_uint2(0u, 0u);
      if (a.parts == 1) sv = *reinterpret_cast<const uint2*>(svh + t.c0 + 4 * lane);
      // every wait here is bounded: a warp that gives up leaves, and the others
      // then give up on their next wait instead of hanging
      if (!mbar_wait(&accfull[buf], (li >> 1) & 1u)) break;
      // the split-k epilogue may be scheduled once every CTA has begun the
      // epilogue of its last item
      if (a.trigger_dependents == 2 && i + 1 == count && e == 0 && lane == 0) pdl_launch_dependents();
      tc_fence_after();
      const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sv.x));
      const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&sv.y));
      bool ok = true;
      // the accumulator in chunks of kZRows batch rows (tensor-memory columns)
#pragma unroll 1
      for (int c = 0; ok && c < C::kZChunks; ++c) {
        constexpr int ZR = C::kZRows;
        const int r0 = c * ZR;
        uint32_t q[ZR];
        tmem_ld_32x32b_cols<ZR>(tmem + ((uint32_t)(32 * e) << 16) + (uint32_t)(C::kAccCols * buf + r0), q);
        tmem_ld_wait();
        if (c + 1 == C::kZChunks) {
          // every chunk of the buffer has been read: the MMAs may reuse it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[buf]);
        }
        if (a.parts > 1) {
          // split-k: this part's fp32 sums go straight to acc[part][row][col]
          float* dst = a.acc + (int64_t)t.part * a.m * a.n + t.c0 + 32 * e + lane;
#pragma unroll
          for (int r = 0; r < ZR; ++r)
            if (r0 + r < live) dst[(t.row0 + r0 + r) * a.n] = __uint_as_float(q[r]);
        } else {
          // staging-tile use number z of this CTA: the previous use's rows have
          // been read before the tile is rewritten
          const uint32_t z = li * (uint32_t)C::kZChunks + (uint32_t)c;
          if (z > 0 && !mbar_wait(zdone, (z - 1u) & 1u)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int r = 0; r < ZR; ++r) zs[r * kZ + 32 * e + lane] = __uint_as_float(q[r]);
          __syncwarp();
          if (lane == 0) mbar_arrive(zfull);
          if (!mbar_wait(zfull, z & 1u)) {
            ok = false;
            break;
          }
          for (int rr = e; rr < ZR && r0 + rr < live; rr += 4) {
            const float4 zv = ld_shared_v4f(smem_u32(zs) + (uint32_t)((rr * kZ + 4 * lane) * 4));
            float v[4] = {zv.x, zv.y, zv.z, zv.w};
            fwht128_warp(v, lane);
            const uint32_t o0 = f32_to_out((v[0] * 0.125f) * s01.x, bf16), o1 = f32_to_out((v[1] * 0.125f) * s01.y, bf16);
            const uint32_t o2 = f32_to_out((v[2] * 0.125f) * s23.x, bf16), o3 = f32_to_out((v[3] * 0.125f) * s23.y, bf16);
            *reinterpret_cast<uint2*>(y + (t.row0 + r0 + rr) * a.n + t.c0 + 4 * lane) =
                make_uint2(o0 | (o1 << 16), o2 | (o3 << 16));
          }
          // the staging tile is rewritten by the next chunk or item
          __syncwarp();
          if (lane == 0) mbar_arrive(zdone);
        }
      }
      if (!ok) break;
      ++li;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int BITS, int CB, int KA, int XR, bool MOE = false>
cudaError_t launch_tm_variant(const TcMaps& maps, const TcParams& p, cudaStream_t stream) {
  using C = TmCfg<BITS, KA, XR>;
  auto kern = gemm_tm_kernel<BITS, CB, KA, XR, MOE>;
  // the shared-memory opt-in and the SM count, once per device (benign race:
  // every thread writes the same values)
  static bool configured[64] = {};
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms[dev] = v > 0 ? v : 1;
    configured[dev] = true;
  }
  const int64_t items =
      MOE ? (p.a.m / p.a.moe_block) * (p.a.n >> 7) : ((p.a.n - p.a.col_base) >> 7) * p.a.parts;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(items < sms[dev] ? items : sms[dev]), 1u, 1u);
  cfg.blockDim = dim3(kTmThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // may start while the previous kernel (the input transform) still runs; the
  // activation producer waits for it (pdl_wait) before reading xh
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

}  // namespace exl3
