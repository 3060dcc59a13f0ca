// Scale-restore epilogue shared by the GEMM kernels of the INT8ConvRot library.
//
// Page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX",
// section "What changed in the computation": Y = A (.) s_X s_W^T, A the exact
// int32 product.  Evaluated in fp32 as ((float)A * s_X[m]) * s_W[n], then the
// optional bias and unmerged LoRA term of the page "[PR #249] Add an mps
// backend: weight-only INT8 and W4A8/W6A8 linears for Apple GPUs" (section
// "What"; "applies the up weight in fp32", bias "in eager's order" and bf16
// "with torch's cast" under "Design") follow in fp32 before the single
// rounding to fp16 or bf16:
//   y = fl(fl((float)A * s_X) * s_W);  y = fl(y + bias[n]);
//   y += lora_scale * S[m,n],  S[m,n] = sum_r T[m,r] * lora_up[n,r] in fp32
//   (computed once per call by the LoRA up kernel, lora.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kernels.h"

namespace convrot {

// Two 16-bit floats of one 32-bit word (element 0 in the low half), widened
// exactly: fp16, or bf16 (the top half of an fp32 pattern).
__device__ __forceinline__ float2 widen2(uint32_t w, bool bf16) {
  if (bf16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

__device__ __forceinline__ float widen1(uint16_t h, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

// Scale restore and bias of output column n, each its own IEEE rounding (no
// contraction into a fused multiply-add).  Columns at or past N (clipped on
// store) read no bias.
__device__ __forceinline__ float scale_bias(float a, float sx, float sw, const float* bias, int n,
                                            int N) {
  float y = __fmul_rn(__fmul_rn(a, sx), sw);
  if (bias) y = __fadd_rn(y, n < N ? __ldg(bias + n) : 0.0f);
  return y;
}

// fp32 outputs of columns [n0, n0 + NC) of row m from the exact sums `sum`
// (columns at or beyond N give 0).  kLora selects the variant that adds the
// LoRA term and kExt the one that honours the bias and bf16 fields (separate
// instantiations keep the plain fp16 path lean: the runtime branches of the
// extended epilogue, replicated through the unrolled loops, grew the GEMM
// kernels' code by half and slowed them through instruction fetch).
template <int NC, bool kLora, bool kExt = false>
__device__ __forceinline__ void epilogue_values(const EpilogueArgs& e, int N, int64_t m, int n0,
                                                const int32_t (&sum)[NC], float (&y)[NC]) {
  const float sx = e.sX[m];
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int n = n0 + i;
    if constexpr (kExt)
      y[i] = (n < N) ? scale_bias(static_cast<float>(sum[i]), sx, e.sW[n], e.bias, n, N) : 0.0f;
    else
      y[i] = (static_cast<float>(sum[i]) * sx) * ((n < N) ? e.sW[n] : 0.0f);
  }
  if (kLora && e.R > 0) {
    // The LoRA sums S = T up^T come precomputed (launch_lora_up).
    const float* srow = e.S + m * N;
#pragma unroll
    for (int i = 0; i < NC; ++i)
      if (n0 + i < N) y[i] = y[i] + e.lora_scale * srow[n0 + i];
  }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Two outputs as fp16 or bf16 (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack_out2(float a, float b, bool bf16) {
  if (bf16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  return pack_half2(a, b);
}

__device__ __forceinline__ uint16_t pack_out1(float a, bool bf16) {
  if (bf16) {
    const __nv_bfloat16 h = __float2bfloat16_rn(a);
    return *reinterpret_cast<const uint16_t*>(&h);
  }
  const __half h = __float2half_rn(a);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// Writes columns [n0, n0 + NC) of row m to global memory from the exact sums.
// Columns at or beyond N are skipped.
template <int NC, bool kLora, bool kExt = false>
__device__ __forceinline__ void epilogue_store(const EpilogueArgs e, int N, int64_t m, int n0,
                                               const int32_t (&sum)[NC]) {
  const bool full = (n0 + NC <= N);
  if (e.mode == kOutI32) {
    int32_t* dst = e.A + m * N + n0;
    if (full && (N % 4) == 0) {
#pragma unroll
      for (int i = 0; i < NC; i += 4)
        *reinterpret_cast<int4*>(dst + i) = make_int4(sum[i], sum[i + 1], sum[i + 2], sum[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < NC; ++i)
        if (n0 + i < N) dst[i] = sum[i];
    }
    return;
  }
  float y[NC];
  epilogue_values<NC, kLora, kExt>(e, N, m, n0, sum, y);
  uint16_t* dst = e.Y + m * N + n0;
  const bool bf16 = kExt && e.out_bf16 != 0;
  if (full && (N % 8) == 0) {
#pragma unroll
    for (int i = 0; i < NC; i += 8) {
      uint4 o;
      o.x = pack_out2(y[i + 0], y[i + 1], bf16);
      o.y = pack_out2(y[i + 2], y[i + 3], bf16);
      o.z = pack_out2(y[i + 4], y[i + 5], bf16);
      o.w = pack_out2(y[i + 6], y[i + 7], bf16);
      *reinterpret_cast<uint4*>(dst + i) = o;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NC; ++i)
      if (n0 + i < N) dst[i] = pack_out1(y[i], bf16);
  }
}

}  // namespace convrot
