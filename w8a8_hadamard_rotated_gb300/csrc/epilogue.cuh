// Scale-restore epilogue shared by the GEMM kernels of the INT8ConvRot library.
//
// Page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX",
// section "What changed in the computation": Y = A (.) s_X s_W^T, A the exact
// int32 product.  Evaluated in fp32 as ((float)A * s_X[m]) * s_W[n], then the
// optional unmerged LoRA term of the page "[PR #249] Add an mps backend:
// weight-only INT8 and W4A8/W6A8 linears for Apple GPUs" (section "What";
// "applies the up weight in fp32" under "Design") is added in fp32 before the
// single rounding to fp16:  y += lora_scale * sum_r T[m,r] * lora_up[n,r].
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kernels.h"

namespace convrot {

// fp32 outputs of columns [n0, n0 + NC) of row m from the exact sums `sum`
// (columns at or beyond N give 0).  kLora selects the variant that adds the
// LoRA term (a separate instantiation keeps the plain path lean).
template <int NC, bool kLora>
__device__ __forceinline__ void epilogue_values(const EpilogueArgs& e, int N, int64_t m, int n0,
                                                const int32_t (&sum)[NC], float (&y)[NC]) {
  const float sx = e.sX[m];
#pragma unroll
  for (int i = 0; i < NC; ++i) {
    const int n = n0 + i;
    const float sw = (n < N) ? e.sW[n] : 0.0f;
    y[i] = (static_cast<float>(sum[i]) * sx) * sw;
  }
  if (kLora && e.R > 0) {
    float l[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) l[i] = 0.0f;
    const float* trow = e.T + m * e.R;
    if ((e.R % 8) == 0) {
      for (int r0 = 0; r0 < e.R; r0 += 8) {
        float t[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) t[j] = trow[r0 + j];
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          const int n = n0 + i;
          if (n < N) {
            const uint4 raw =
                *reinterpret_cast<const uint4*>(e.up + static_cast<int64_t>(n) * e.R + r0);
            const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 u = __half22float2(h2[j]);
              l[i] = fmaf(t[2 * j], u.x, l[i]);
              l[i] = fmaf(t[2 * j + 1], u.y, l[i]);
            }
          }
        }
      }
    } else {
      for (int r = 0; r < e.R; ++r) {
        const float t = trow[r];
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          const int n = n0 + i;
          if (n < N)
            l[i] = fmaf(t,
                        __half2float(reinterpret_cast<const __half*>(
                            e.up)[static_cast<int64_t>(n) * e.R + r]),
                        l[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NC; ++i) y[i] = y[i] + e.lora_scale * l[i];
  }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Writes columns [n0, n0 + NC) of row m to global memory from the exact sums.
// Columns at or beyond N are skipped.
template <int NC, bool kLora>
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
  epilogue_values<NC, kLora>(e, N, m, n0, sum, y);
  uint16_t* dst = e.Y + m * N + n0;
  if (full && (N % 8) == 0) {
#pragma unroll
    for (int i = 0; i < NC; i += 8) {
      uint4 o;
      o.x = pack_half2(y[i + 0], y[i + 1]);
      o.y = pack_half2(y[i + 2], y[i + 3]);
      o.z = pack_half2(y[i + 4], y[i + 5]);
      o.w = pack_half2(y[i + 6], y[i + 7]);
      *reinterpret_cast<uint4*>(dst + i) = o;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NC; ++i)
      if (n0 + i < N) {
        const __half h = __float2half_rn(y[i]);
        dst[i] = *reinterpret_cast<const uint16_t*>(&h);
      }
  }
}

}  // namespace convrot
