// exl3_device.cuh -- device-side building blocks shared by the EXL3 kernels:
// trellis windows, the three procedural codebooks, packed half2 output in
// mma.m16n8k16 B-fragment order, and the 128-point butterfly.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "exl3_launch.h"

namespace exl3 {

// ---------------------------------------------------------------------------
// Codebook constants.
// mcg multiplier: cuda-exl3 README, "GLM-5.3-Flash" (multiplier 0xCBAC1FED).
// 3inst / mul1: the pages print no constants; this library reads 3inst as the
// mcg multiply with an increment of 1 and mul1 as the same multiplier followed
// by a byte sum and one fp16 fused multiply-add (TensorFold PR #740,
// "Arithmetic" step 2).  The half mask/xor put each 16-bit half in +-[2^-3, 2),
// so every state decodes to a finite value, as the cuda-exl3 README requires of
// all 65,536 states ("Loading into a dim vLLM has padded").
// ---------------------------------------------------------------------------
constexpr uint32_t kMcgMult = 0xCBAC1FEDu;
constexpr uint32_t k3instMult = 0xCBAC1FEDu;
constexpr uint32_t k3instAdd = 1u;
constexpr uint32_t kMul1Mult = 0xCBAC1FEDu;
constexpr uint32_t kHalfMask = 0x8FFF8FFFu;
constexpr uint32_t kHalfXor = 0x30003000u;
// fp16 bit patterns of the mul1 coefficients: 0x1EEE = 1774 * 2^-18 (nearest
// fp16 to 1/147.8) and 0xC2E7 = -1767 * 2^-9 (nearest fp16 to -510/147.8).
constexpr uint32_t kMul1ScaleH2 = 0x1EEE1EEEu;
constexpr uint32_t kMul1BiasH2 = 0xC2E7C2E7u;
// 1024.0 in both fp16 lanes: 0x6400 + t is the fp16 number 1024 + t for t < 1024.
constexpr uint32_t kH2_1024 = 0x64006400u;

enum Codebook { CB_3INST = 0, CB_MCG = 1, CB_MUL1 = 2 };

__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// (u & kHalfMask) ^ kHalfXor as one three-input logic op (truth table 0x6A:
// a & b ^ c), written out so that it is never split into two operations.
__device__ __forceinline__ uint32_t lop3_mask_xor(uint32_t u) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(u), "n"(kHalfMask), "n"(kHalfXor));
  return d;
}

// Two states -> one half2 register {value(s0) in bits 0..15, value(s1) in bits 16..31}.
template <int CB>
__device__ __forceinline__ uint32_t decode_pair(uint32_t s0, uint32_t s1) {
  if constexpr (CB == CB_MUL1) {
    const uint32_t u0 = s0 * kMul1Mult;
    const uint32_t u1 = s1 * kMul1Mult;
    // byte sums t0, t1 (0..1020), biased by the fp16 pattern of 1024.0
    const uint32_t t0 = __dp4a(u0, 0x01010101u, 0x6400u);
    const uint32_t t1 = __dp4a(u1, 0x01010101u, 0x6400u);
    const uint32_t p = __byte_perm(t0, t1, 0x5410);  // {1024+t0, 1024+t1}, exact
    const uint32_t t = hsub2_u32(p, kH2_1024);        // {t0, t1}, exact
    return hfma2_u32(t, kMul1ScaleH2, kMul1BiasH2);   // one rounding each
  } else {
    uint32_t u0, u1;
    if constexpr (CB == CB_3INST) {
      u0 = s0 * k3instMult + k3instAdd;
      u1 = s1 * k3instMult + k3instAdd;
    } else {
      u0 = s0 * kMcgMult;
      u1 = s1 * kMcgMult;
    }
    u0 = lop3_mask_xor(u0);
    u1 = lop3_mask_xor(u1);
    // {u0.lo, u1.lo} + {u0.hi, u1.hi}: each lane sums the two halves of one state
    const uint32_t lo = __byte_perm(u0, u1, 0x5410);
    const uint32_t hi = __byte_perm(u0, u1, 0x7632);
    return hadd2_u32(lo, hi);
  }
}

// The same two values with the integer work spread over the ALU, multiply and
// fp16 pipes (identical results, pinned against decode_pair over all states by
// the codebook test).  mcg / 3inst: after the hash and mask, each value's two
// halves are added by one fp16 fma per value, fma(hi, 1, lo) = lo + hi rounded
// once, whose other lane computes hi * -1 + hi = +0 exactly, so the two partial
// words {v0, +0} and {+0, v1} merge with one exact fp16 add instead of two byte
// permutes.  mul1: the two biased byte sums merge with a multiply-add by 2^16
// (each is below 2^16) instead of a byte permute.
template <int CB>
__device__ __forceinline__ uint32_t decode_pair_balanced(uint32_t s0, uint32_t s1, const DecodeConsts& mc) {
  if constexpr (CB == CB_MUL1) {
    const uint32_t u0 = s0 * kMul1Mult;
    const uint32_t u1 = s1 * kMul1Mult;
    const uint32_t t0 = __dp4a(u0, 0x01010101u, 0x6400u);
    const uint32_t t1 = __dp4a(u1, 0x01010101u, 0x6400u);
    uint32_t pk;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(pk) : "r"(t1), "r"(mc.pow2[16]), "r"(t0));
    const uint32_t t = hsub2_u32(pk, kH2_1024);     // {t0, t1}, exact
    return hfma2_u32(t, kMul1ScaleH2, kMul1BiasH2);  // one rounding each
  } else {
    uint32_t u0, u1;
    if constexpr (CB == CB_3INST) {
      u0 = s0 * k3instMult + k3instAdd;
      u1 = s1 * k3instMult + k3instAdd;
    } else {
      u0 = s0 * kMcgMult;
      u1 = s1 * kMcgMult;
    }
    u0 = lop3_mask_xor(u0);
    u1 = lop3_mask_xor(u1);
    const __half2 h0 = *reinterpret_cast<const __half2*>(&u0);
    const __half2 h1 = *reinterpret_cast<const __half2*>(&u1);
    const uint32_t k1u = 0xBC003C00u, k2u = 0x3C00BC00u;  // {1, -1}, {-1, 1}
    const __half2 k1 = *reinterpret_cast<const __half2*>(&k1u);
    const __half2 k2 = *reinterpret_cast<const __half2*>(&k2u);
    const __half2 t0 = __hfma2(__high2half2(h0), k1, h0);  // {lo0 + hi0, +0}
    const __half2 t1 = __hfma2(__low2half2(h1), k2, h1);   // {+0, lo1 + hi1}
    const __half2 r = __hadd2(t0, t1);                     // {v0, v1}, exact
    return *reinterpret_cast<const uint32_t*>(&r);
  }
}

// ---------------------------------------------------------------------------
// Trellis windows.
//
// A tile is 16*BITS int16 words = 8*BITS 32-bit words forming one circular,
// little-endian bit stream of 256*BITS bits.  Value v's 16-bit state is the 16
// bits ending just before position (v+1)*BITS (cuda-exl3 README, "Where the time
// goes": 58-bit window for 8 values at 6 bits, index wrap modulo the tile).
// Lane l decodes values 8l..8l+7 (lane*8 alignment), i.e. the window of bits
// [8*l*BITS + BITS - 16, 8*l*BITS + 8*BITS), at most three 32-bit words.
// ---------------------------------------------------------------------------
template <int BITS>
struct LaneWindow {
  static constexpr int kWords = 8 * BITS;            // 32-bit words per tile
  static constexpr int kBytes = 32 * BITS;           // bytes per tile
  static constexpr int kNeed = (BITS <= 4) ? 2 : 3;  // words a lane reads
  int idx[3];  // word indices within the tile (already wrapped)
  int off;     // bit offset of the window start within word idx[0]

  __device__ __forceinline__ explicit LaneWindow(int lane) {
    int s = 8 * lane * BITS + BITS - 16;
    if (s < 0) s += 256 * BITS;
    const int w = s >> 5;
    off = s & 31;
    idx[0] = w;
    idx[1] = (w + 1) % kWords;
    idx[2] = (w + 2) % kWords;
  }
};

// Aligned views of a lane's window: r[i] holds window bits [16*i, 16*i + 32).
// r[0], r[2], r[4] are funnel shifts of the stream words by the lane's offset;
// r[1], r[3] are byte permutes of their neighbours.
struct Aligned {
  uint32_t r[5];
};

template <int BITS>
__device__ __forceinline__ Aligned align_window(uint32_t w0, uint32_t w1, uint32_t w2, int off) {
  Aligned a;
  a.r[0] = __funnelshift_r(w0, w1, off);
  a.r[2] = (BITS >= 3) ? __funnelshift_r(w1, w2, off) : 0u;
  a.r[4] = (BITS >= 7) ? (w2 >> off) : 0u;
  a.r[1] = (BITS >= 3) ? __byte_perm(a.r[0], a.r[2], 0x5432) : 0u;
  a.r[3] = (BITS >= 6) ? __byte_perm(a.r[2], a.r[4], 0x5432) : 0u;
  return a;
}

// State of the lane's J-th value (J = 0..7): bits [J*BITS, J*BITS+16) of the
// window, read from the view r[i] that holds it at offset q = J*BITS - 16*i in
// 0..16.  q = 0 is one mask and q = 16 one shift.  Otherwise the bits above the
// state are dropped either by a shift (ALU pipe) or by a multiply with 2^(16-q)
// (integer multiply pipe), and those below by a right shift of 16.  The
// codebooks that hash with a multiply only (3inst, mcg) take the multiply form
// so both half-rate pipes carry about the same load; mul1, whose byte sum and
// fp16 fma already load the multiply pipe, takes the shift form.
template <int BITS, int J, int CB>
__device__ __forceinline__ uint32_t window_state(const Aligned& a, const DecodeConsts& mc) {
  constexpr int p = J * BITS;
  constexpr int i = (p % 16 == 0 && p >= 16) ? (p / 16 - 1) : (p / 16);  // prefer q = 16 over q = 0
  constexpr int q = p - 16 * i;
  static_assert(q >= 0 && q <= 16 && i <= 4, "state outside the window views");
  const uint32_t v = a.r[i];
  if constexpr (q == 16) {
    return v >> 16;
  } else if constexpr (q == 0) {
    return v & 0xFFFFu;
  } else if constexpr (CB == CB_MUL1) {
    return (v >> q) & 0xFFFFu;
  } else {
    return (v * mc.pow2[16 - q]) >> 16;
  }
}

// The lane's 8 values as 4 half2 registers, in mma.m16n8k16 B-fragment order:
// b[0] = {k=2q, 2q+1; n=g}, b[1] = {k=2q+8, 2q+9; n=g}, b[2], b[3] = same for n=g+8
// (TensorFold PR #740, "Arithmetic" step 2: tiles decode directly into the B
// fragments of two mma.m16n8k16, which fixes the order of a tile's values).
template <int BITS, int CB>
__device__ __forceinline__ void decode_lane(const Aligned& a, const DecodeConsts& mc, uint32_t b[4]) {
  b[0] = decode_pair<CB>(window_state<BITS, 0, CB>(a, mc), window_state<BITS, 1, CB>(a, mc));
  b[1] = decode_pair<CB>(window_state<BITS, 2, CB>(a, mc), window_state<BITS, 3, CB>(a, mc));
  b[2] = decode_pair<CB>(window_state<BITS, 4, CB>(a, mc), window_state<BITS, 5, CB>(a, mc));
  b[3] = decode_pair<CB>(window_state<BITS, 6, CB>(a, mc), window_state<BITS, 7, CB>(a, mc));
}

// Load the lane's window words of one tile (tile_words = first 32-bit word of the tile).
template <int BITS>
__device__ __forceinline__ Aligned load_lane_window(const uint32_t* tile_words, const LaneWindow<BITS>& lw) {
  const uint32_t w0 = tile_words[lw.idx[0]];
  const uint32_t w1 = tile_words[lw.idx[1]];
  const uint32_t w2 = (LaneWindow<BITS>::kNeed == 3) ? tile_words[lw.idx[2]] : 0u;
  return align_window<BITS>(w0, w1, w2, lw.off);
}

// ---------------------------------------------------------------------------
// 128-point Hadamard butterfly over one row held as 4 consecutive values per
// lane (lane l holds elements 4l..4l+3).  Stages run in the fixed order of
// strides 1, 2, 4, ..., 64; each stage maps (a, b) -> (a + b, a - b) for the
// pair at indices (i, i + stride), i.e. H[i][j] = (-1)^popcount(i & j).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fwht128_warp(float v[4], int lane) {
  float t0 = v[0] + v[1], t1 = v[0] - v[1];
  float t2 = v[2] + v[3], t3 = v[2] - v[3];
  v[0] = t0 + t2;
  v[2] = t0 - t2;
  v[1] = t1 + t3;
  v[3] = t1 - t3;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = __shfl_xor_sync(0xffffffffu, v[i], s);
      v[i] = upper ? (p - v[i]) : (v[i] + p);
    }
  }
}

// The first five stages (strides 1, 2, 4, 8, 16) of the same butterfly on 32
// consecutive elements held by one thread.
__device__ __forceinline__ void fwht32_regs(float (&v)[32]) {
#pragma unroll
  for (int st = 1; st < 32; st <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & st) == 0) {
        const float a = v[i], b = v[i + st];
        v[i] = a + b;
        v[i + st] = a - b;
      }
    }
  }
}

__device__ __forceinline__ uint16_t f32_to_out(float v, bool bf16) {
  if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}

}  // namespace exl3
