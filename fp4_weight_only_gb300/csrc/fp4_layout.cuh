// Repacked weight layout and the in-register FP4 -> BF16 decode shared by the
// repack, dequant-hook and GEMM kernels.
//
// The decode turns an E2M1 code into BF16 with shifts and masks only (the
// pages' "dequantise in registers with bit tricks"; Petit blog, "Efficient
// dequantization via preprocessing", where an offline shuffle puts the bits
// where the decode wants them).  Placing a code's two exponent bits on the two
// lowest BF16 exponent bits and its mantissa bit on the top BF16 mantissa bit
// gives the BF16 number value(code) * 2^-126 exactly -- including code 0.5,
// which becomes the BF16 subnormal 2^-127.  One BF16x2 multiply by the block
// scale (pre-multiplied by 2^118, exact for every E4M3 value) then yields
// value * scale * 2^-8, exactly representable; the GEMM epilogue multiplies
// the FP32 sum by g * 2^8.  MXFP4 uses one exact multiply by 2^(c-1) when
// every E8M0 code c of a chunk is at most 128 (recorded by the repack in the
// chunk), and otherwise two (by 2^126, then by 2^(c-127)), because E8M0
// covers 2^-127..2^127 and BF16 only up to 2^127.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace petit {

constexpr int kLayoutVersion = 4;
constexpr int kTileN = 128;   // weight rows per tile (the MMA M side)
constexpr int kStageK = 128;  // k elements per repacked chunk / pipeline stage
constexpr int kWChunkBytes = kTileN * kStageK / 2;  // 8192
constexpr int kGroupsPerRow = kStageK / 32;         // 16-byte groups per row per chunk

// kNVFP4F16: NVFP4 codes and scales packed for the FP16-activation GEMM
// (same chunk layout and sizes, FP16 bit positions; see pack_word_f16)
enum : int { kNVFP4 = 0, kMXFP4 = 1, kNVFP4F16 = 2 };

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<kNVFP4> {
  static constexpr int kBlock = 16;                          // k per scale
  static constexpr int kSChunkBytes = kTileN * kStageK / 16; // 1024
  static constexpr int kScaleBytesPerHalf = 4;               // 64 k / 16
  static constexpr int kChunkBytes = kWChunkBytes + kSChunkBytes;  // 9216
};
template <>
struct FmtTraits<kNVFP4F16> : FmtTraits<kNVFP4> {};
template <>
struct FmtTraits<kMXFP4> {
  static constexpr int kBlock = 32;
  static constexpr int kSChunkBytes = kTileN * kStageK / 32; // 512
  static constexpr int kScaleBytesPerHalf = 2;               // 64 k / 32
  // after the scales: byte 0 = 1 when every E8M0 code of the chunk is at
  // most 128 (scale <= 2), so the decode may use one multiply (see
  // decode_group); bytes 1..15 zero
  static constexpr int kFlagBytes = 16;
  static constexpr int kChunkBytes = kWChunkBytes + kSChunkBytes + kFlagBytes;  // 8720
};

// ---------------------------------------------------------------- layout
// One repacked buffer holds, for every (tile t of 128 rows, stage s of 128
// k), a chunk of kChunkBytes at byte (t * stages + s) * kChunkBytes: 8192
// bytes of codes followed by the chunk's scales, so one contiguous bulk copy
// brings both (and consecutive stages of a tile are adjacent, so a copy may
// span several chunks).
// Codes: the 16-byte group g (k = 32g .. 32g+31 of the stage) of row r
// (0..127) sits at byte (g * 128 + r) * 16, so a warp reading one group for
// 32 consecutive rows touches 512 consecutive bytes (no bank conflicts).
// Word w of a group holds k = 8w .. 8w+7 in the bit order of pack_word().
// Scales (at byte 8192 of the chunk): half h (k = 64h .. 64h+63) of row r
// sits at (h * 128 + r) * kScaleBytesPerHalf, byte j holding block j of that
// half.  MXFP4 chunks end with a 16-byte flag field (FmtTraits<kMXFP4>).
template <int FMT>
__host__ __device__ constexpr size_t chunk_offset(int64_t tile, int64_t stage, int64_t stages) {
  return static_cast<size_t>((tile * stages + stage) * FmtTraits<FMT>::kChunkBytes);
}

// Bit positions of each code's bits (m, e0, e1, s) in a 32-bit word:
//   c0:  6  7  8 15     c1: 22 23 24 31     (decode: q & M)
//   c2:  0  1  2  9     c3: 16 17 18 25     (decode: (q << 6) & M)
//   c4: 26 27 28  3     c5: 10 11 12 19     (decode: rotl(q, 12) & M)
//   c6:  4  5 30 13     c7: 20 21 14 29     (decode: (q << 2) & M' | rotl(q, 10) & M'')
// with M = 0x81C081C0 selecting BF16 bits {15, 8, 7, 6} of both halves,
// M' = 0x80C080C0 and M'' = 0x01000100.  Nine integer operations per word, two
// of them rotates (funnel shifts): an exhaustive search shows that no four
// rotated copies of M tile the word, so one output merges two rotations.
__host__ __device__ inline uint32_t pack_word(const uint32_t (&c)[8]) {
  constexpr int pos[8][4] = {{6, 7, 8, 15},   {22, 23, 24, 31}, {0, 1, 2, 9},     {16, 17, 18, 25},
                             {26, 27, 28, 3}, {10, 11, 12, 19}, {4, 5, 30, 13},   {20, 21, 14, 29}};
  uint32_t q = 0;
  for (int i = 0; i < 8; ++i)
    for (int b = 0; b < 4; ++b) q |= ((c[i] >> b) & 1u) << pos[i][b];
  return q;
}

// FP16 variant.  FP16 has its exponent's two low bits at 11 and 10 and its top
// mantissa bit at 9, so sign/e1/e0/m on bits 15/11/10/9 give the FP16 number
// value(code) * 2^-14 exactly (code 0.5 -> the FP16 subnormal 2^-15).  The
// 8 codes of a word sit where two shifted copies and two two-part merges
// put them (decode_word_raw_f16); code bits (m, e0, e1, s) at:
//   c0:  5  6  7 11    c1: 21 22 23 27    (decode: (q << 4) & M16)
//   c2:  2  3  4  8    c3: 18 19 20 24    (decode: (q << 7) & M16)
//   c4: 30 10  0 15    c5: 14 26 16 31    (decode: q & K | rot(q, 11) & K')
//   c6:  9 28 29  1    c7: 25 12 13 17    (decode: q & K | rot(q, 14) & K')
// with M16 = 0x8E008E00 selecting FP16 bits {15, 11, 10, 9} of both halves.
__host__ __device__ inline uint32_t pack_word_f16(const uint32_t (&c)[8]) {
  // bit positions of (m, e0, e1, s) for each code
  constexpr int pos[8][4] = {{5, 6, 7, 11},   {21, 22, 23, 27}, {2, 3, 4, 8},     {18, 19, 20, 24},
                             {30, 10, 0, 15}, {14, 26, 16, 31}, {9, 28, 29, 1},   {25, 12, 13, 17}};
  uint32_t q = 0;
  for (int i = 0; i < 8; ++i)
    for (int b = 0; b < 4; ++b) q |= ((c[i] >> b) & 1u) << pos[i][b];
  return q;
}

// ---------------------------------------------------------------- decode
// Four BF16x2 words value(c_i) * 2^-126 for the pairs (c0,c1) .. (c6,c7).
__device__ __forceinline__ void decode_word_raw(uint32_t q, uint32_t (&p)[4]) {
  constexpr uint32_t M = 0x81C081C0u;
  p[0] = q & M;
  p[1] = (q << 6) & M;
  p[2] = __funnelshift_l(q, q, 12) & M;
  p[3] = ((q << 2) & 0x80C080C0u) | (__funnelshift_l(q, q, 10) & 0x01000100u);
}

// Four FP16x2 words value(c_i) * 2^-14 for the pairs (c0,c1) .. (c6,c7) of a
// word packed by pack_word_f16.
__device__ __forceinline__ void decode_word_raw_f16(uint32_t q, uint32_t (&p)[4]) {
  constexpr uint32_t M16 = 0x8E008E00u;
  p[0] = (q << 4) & M16;
  p[1] = (q << 7) & M16;
  p[2] = (q & 0x84008400u) | (__funnelshift_l(q, q, 11) & 0x0A000A00u);
  p[3] = (q & 0x02000200u) | (__funnelshift_l(q, q, 14) & 0x8C008C00u);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

constexpr uint32_t kF16x2_2p7 = 0x58005800u;  // 2^7 in both halves

// Two E4M3 bytes -> FP16x2 splats of scale * 2^7 (exact: E4M3 -> FP16 is
// exact and 448 * 2^7 < 65504).
__device__ __forceinline__ void nv_scale_splats_f16(uint32_t v, uint32_t& s0, uint32_t& s1) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(v & 0xFFFFu)));
  h2 = hmul2(h2, kF16x2_2p7);
  s0 = __byte_perm(h2, 0, 0x1010);
  s1 = __byte_perm(h2, 0, 0x3232);
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_splat_f32(float f) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(f));
  return d;
}

// Two E4M3 bytes (low 16 bits of v: byte 0 = first block) -> BF16x2 splats of
// scale * 2^118.  The hardware E4M3 -> F16 conversion is exact (subnormal
// scales included); F16 -> F32 is exact; * 2^118 stays below 2^127.
__device__ __forceinline__ void nv_scale_splats(uint32_t v, uint32_t& s0, uint32_t& s1) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(v & 0xFFFFu)));
  const float f0 = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
  const float f1 = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
  s0 = bf16x2_splat_f32(f0 * 0x1p118f);
  s1 = bf16x2_splat_f32(f1 * 0x1p118f);
}

// E8M0 byte c <= 128 -> BF16x2 splat of 2^(c-1): BF16 exponent field c + 126,
// one multiply-add (FMA pipe).  value(code) * 2^-126 * 2^(c-1) = Wq exactly
// (a power-of-two scaling; the smallest product, 2^-128, is a BF16
// subnormal with room to spare).
__device__ __forceinline__ uint32_t mx_fast_splat(uint32_t c) { return c * 0x00800080u + 0x3F003F00u; }

// E8M0 byte -> BF16x2 splat of 2^(c-127) (c = 0 is the BF16 subnormal 2^-127).
__device__ __forceinline__ uint32_t mx_scale_splat(uint32_t c) {
  uint32_t b = (c & 0xFFu) << 7;
  b = b > 0x40u ? b : 0x40u;
  return b | (b << 16);
}

constexpr uint32_t kBf16x2_2p126 = 0x7E807E80u;  // 2^126 in both halves
constexpr uint32_t kBf16x2_2p8 = 0x43804380u;    // 2^8 in both halves

// Decode one 16-byte group (32 codes) into 16 BF16x2 words: out[j] holds k =
// 2j (low half) and 2j+1 (high half).  NVFP4: sc holds the two E4M3 bytes of
// the group (k 0-15, 16-31); result = Wq * 2^-8.  MXFP4: sc holds the E8M0
// byte; result = Wq (kMxFast: sc <= 128, one multiply per word instead of
// two).  NVFP4F16: FP16x2 words, result = Wq * 2^-7.
template <int FMT, bool kMxFast = false>
__device__ __forceinline__ void decode_group(const uint4& g, uint32_t sc, uint32_t (&out)[16]) {
  const uint32_t w[4] = {g.x, g.y, g.z, g.w};
  if constexpr (FMT == kNVFP4F16) {
    // FP16: value * 2^-14 times (scale * 2^7) = Wq * 2^-7, exact (the
    // smallest product, 2^-17, is an FP16 subnormal with room to spare)
    uint32_t s0, s1;
    nv_scale_splats_f16(sc, s0, s1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t p[4];
      decode_word_raw_f16(w[i], p);
      const uint32_t s = i < 2 ? s0 : s1;
#pragma unroll
      for (int j = 0; j < 4; ++j) out[4 * i + j] = hmul2(p[j], s);
    }
  } else if constexpr (FMT == kNVFP4) {
    uint32_t s0, s1;
    nv_scale_splats(sc, s0, s1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t p[4];
      decode_word_raw(w[i], p);
      const uint32_t s = i < 2 ? s0 : s1;
#pragma unroll
      for (int j = 0; j < 4; ++j) out[4 * i + j] = bmul2(p[j], s);
    }
  } else if constexpr (kMxFast) {
    const uint32_t s = mx_fast_splat(sc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t p[4];
      decode_word_raw(w[i], p);
#pragma unroll
      for (int j = 0; j < 4; ++j) out[4 * i + j] = bmul2(p[j], s);
    }
  } else {
    const uint32_t s = mx_scale_splat(sc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t p[4];
      decode_word_raw(w[i], p);
#pragma unroll
      for (int j = 0; j < 4; ++j) out[4 * i + j] = bmul2(bmul2(p[j], kBf16x2_2p126), s);
    }
  }
}

}  // namespace petit
