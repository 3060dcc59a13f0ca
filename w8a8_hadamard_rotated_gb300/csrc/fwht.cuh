// Shared device helpers of the rotate + quantize step (sm_103a): the
// Walsh-Hadamard butterflies and the int8 rounding.
//
// Page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX",
// section "What changed in the computation": X_rot = X H with H the Kronecker
// power of 4x4 Hadamards divided by 16 (groups of 256 along K); with the
// Sylvester 4x4 base, x H is the fast Walsh-Hadamard transform (8 stages of
// a + b, a - b) times 1/16, and Q = clamp(round(X_rot / s), -128, 127),
// s = max |X_rot| / 127 per row.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace convrot {

// ---------------------------------------------------------------------------
// Butterfly helpers.
// ---------------------------------------------------------------------------

// In-register Walsh-Hadamard butterflies over the index bits of v[0..N).
template <int N>
__device__ __forceinline__ void fwht_regs(float (&v)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
}

// One butterfly stage across lanes: partner = lane ^ mask.  The lane whose
// `mask` bit is 0 keeps a + b, the other keeps a - b (a = lower index value).
template <int N>
__device__ __forceinline__ void fwht_xlane(float (&v)[N], int lane, int mask) {
  const float sgn = (lane & mask) ? -1.0f : 1.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float other = __shfl_xor_sync(0xffffffffu, v[i], mask);
    v[i] = fmaf(sgn, v[i], other);  // lower: v + other; upper: other - v
  }
}

// Integer rounding through the fp32 adder.  kRoundMagic = 2^23 + 2^22 + 25728
// (bit pattern 0x4B406480).  For |t| < 2^21 the sum t + kRoundMagic lies in
// [2^23, 2^24), where consecutive fp32 values are 1 apart, so
// fmaf(v, inv, kRoundMagic) rounds the exact product v * inv once, to the
// nearest integer with ties to even, and the low byte of the result's bit
// pattern is (q + 128) mod 256.  The quantizers call it with |v * inv| <=
// 127 (1 + 2^-24), so q lies in [-127, 127]; a NaN product (non-finite input)
// gives the canonical NaN, whose low byte 0 reads as q = -128, so every code
// stays in the int8 range.  No float <-> int conversion instruction is used.
constexpr float kRoundMagic = 12608640.0f;

__device__ __forceinline__ uint32_t round_magic(float v, float inv) {
  return __float_as_uint(fmaf(v, inv, kRoundMagic));
}

// Two rounded values -> the fp16 pair (q0, q1): 0x6400 | byte is the fp16
// bit pattern of 1024 + byte = 1152 + q, and 1152 + q - 1152 is exact in fp16.
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t r0, uint32_t r1) {
  const uint32_t b = (__byte_perm(r0, r1, 0x0400) & 0x00ff00ffu) | 0x64006400u;
  const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&b), k1152);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four rounded values -> four packed int8 codes (byte ^ 0x80 = q).
__device__ __forceinline__ uint32_t codes_s8x4(uint32_t r0, uint32_t r1, uint32_t r2,
                                               uint32_t r3) {
  const uint32_t lo = __byte_perm(r0, r1, 0x0040);  // bytes r0.b0, r1.b0
  const uint32_t hi = __byte_perm(r2, r3, 0x0040);
  return __byte_perm(lo, hi, 0x5410) ^ 0x80808080u;
}

// Negates v[i] where bit i of `bits` is set (the input signs of a
// non-Sylvester base), by flipping the fp32 sign bit.
template <int N>
__device__ __forceinline__ void apply_signs(float (&v)[N], uint32_t bits) {
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(__float_as_uint(v[i]) ^ ((bits >> i) << 31));
}

// ---------------------------------------------------------------------------
// Packed form: the values of a lane as float2 pairs w[k] = (v[2k], v[2k+1]),
// transformed with the paired fp32 instructions of sm_100+ (two IEEE fp32
// operations per instruction, each rounded exactly like its scalar form), so
// the results are bit-identical to the scalar helpers above.
// ---------------------------------------------------------------------------

// a - b, exactly as the scalar subtraction: fma(b, -1, a) rounds once.
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}

// In-register butterflies over the element index bits of v[0..2*N2): the
// first stage pairs the two halves of each float2 (scalar), the others pair
// whole float2 values (packed).
template <int N2>
__device__ __forceinline__ void fwht_regs2(float2 (&w)[N2]) {
#pragma unroll
  for (int k = 0; k < N2; ++k) {
    const float a = w[k].x, b = w[k].y;
    w[k] = make_float2(a + b, a - b);
  }
#pragma unroll
  for (int h = 1; h < N2; h <<= 1) {
#pragma unroll
    for (int k = 0; k < N2; ++k) {
      if ((k & h) == 0) {
        const float2 a = w[k], b = w[k + h];
        w[k] = __fadd2_rn(a, b);
        w[k + h] = fsub2(a, b);
      }
    }
  }
}

// One butterfly stage across lanes (partner = lane ^ mask), packed.
template <int N2>
__device__ __forceinline__ void fwht_xlane2(float2 (&w)[N2], int lane, int mask) {
  const float sg = (lane & mask) ? -1.0f : 1.0f;
  const float2 sgn = make_float2(sg, sg);
#pragma unroll
  for (int k = 0; k < N2; ++k) {
    float2 other;
    other.x = __shfl_xor_sync(0xffffffffu, w[k].x, mask);
    other.y = __shfl_xor_sync(0xffffffffu, w[k].y, mask);
    w[k] = __ffma2_rn(sgn, w[k], other);  // lower: w + other; upper: other - w
  }
}

// Negates the elements of w (element 2k is w[k].x, 2k + 1 is w[k].y) whose
// bit is set in `bits` (the input signs of a non-Sylvester base).
template <int N2>
__device__ __forceinline__ void apply_signs2(float2 (&w)[N2], uint64_t bits) {
#pragma unroll
  for (int k = 0; k < N2; ++k) {
    const uint32_t b = static_cast<uint32_t>(bits >> (2 * k));
    w[k].x = __uint_as_float(__float_as_uint(w[k].x) ^ (b << 31));
    w[k].y = __uint_as_float(__float_as_uint(w[k].y) ^ ((b >> 1) << 31));
  }
}

// Two codes at once: the packed form of round_magic + codes_f16x2.
__device__ __forceinline__ uint32_t codes_f16x2_packed(float2 w, float2 inv2) {
  const float2 r = __ffma2_rn(w, inv2, make_float2(kRoundMagic, kRoundMagic));
  return codes_f16x2(__float_as_uint(r.x), __float_as_uint(r.y));
}

// load_swizzled_row, into float2 pairs.
// kBf16: the row holds bf16 values (widened exactly: a bf16 is the top half
// of an fp32 bit pattern).
template <int N2, bool kBf16 = false>
__device__ __forceinline__ void load_swizzled_row2(const uint8_t* rowp, int r, int c0,
                                                   float2 (&w)[N2]) {
#pragma unroll
  for (int j = 0; j < N2 / 4; ++j) {
    const int phys = (c0 + j) ^ (r & 7);
    const uint4 raw = *reinterpret_cast<const uint4*>(rowp + phys * 16);
    if constexpr (kBf16) {
      const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[j * 4 + e] = make_float2(__uint_as_float(u[e] << 16), __uint_as_float(u[e] & 0xffff0000u));
    } else {
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) w[j * 4 + e] = __half22float2(h2[e]);
    }
  }
}

// Reads N consecutive fp16 values of one 128-byte row of a 128-byte-swizzled
// shared-memory tile (16-byte chunk c of row r sits at chunk c ^ (r % 8)),
// starting at chunk c0, and widens them to fp32 (exact).
template <int N>
__device__ __forceinline__ void load_swizzled_row(const uint8_t* rowp, int r, int c0,
                                                  float (&v)[N]) {
#pragma unroll
  for (int j = 0; j < N / 8; ++j) {
    const int phys = (c0 + j) ^ (r & 7);
    const uint4 raw = *reinterpret_cast<const uint4*>(rowp + phys * 16);
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h2[e]);
      v[j * 8 + 2 * e] = f.x;
      v[j * 8 + 2 * e + 1] = f.y;
    }
  }
}

}  // namespace convrot
