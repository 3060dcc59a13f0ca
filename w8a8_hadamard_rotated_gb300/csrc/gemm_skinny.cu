// Small-M variant of the exact int8 GEMM: A = Q_X Q_W^T (int32), then the
// scale restore Y = A (.) s_X s_W^T (page "INT8ConvRot GEMM vs fp16 on M1 Max
// with Metal, MPSMatrix, and MLX", section "What changed in the computation").
//
// For M <= 64 the layer is a stream over the weight (N*K int8 bytes).  This
// kernel reads Q_W once, as int8, with 16-byte loads, and multiplies on the
// integer mma.sync path (m16n8k32, s8 x s8 -> s32, exact).  The K range is
// split across CTAs; each CTA reduces its 4 warps in shared memory and adds
// its exact partial into a zeroed int32 workspace with atomics (integer adds
// commute: deterministic).  The last CTA to finish a 32-column block applies
// the epilogue for that block.
//
// Operand fragments.  For one 64-wide K step, lane (g = lane/4, t = lane%4)
// loads 16 consecutive bytes k0 + 16t .. k0 + 16t + 15 of a weight row and of
// the activation rows g and g + 8.  The two m16n8k32 MMAs of the step take
// bytes [8s, 8s + 8) of those (s = 0, 1): the MMA's K positions 4t..4t+3 and
// 16+4t..16+4t+3 map to the same real k for A and for B, so the products are
// the right ones (a sum over k does not depend on the order of k).
#include <cuda_fp16.h>
#include <stdint.h>

#include "epilogue.cuh"
#include "kernels.h"

namespace convrot {

__device__ __forceinline__ void mma_s8_16832(int32_t (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const int8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

constexpr int kSkinnyWarps = 4;
constexpr int kSkinnyCols = 32;  // 4 n8 tiles per warp

template <int MT>
__global__ void __launch_bounds__(kSkinnyWarps * 32) gemm_skinny_kernel(const GemmSkinnyArgs p) {
  __shared__ int32_t red[MT * 16][kSkinnyCols];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int n0 = blockIdx.x * kSkinnyCols;
  const int k_begin = blockIdx.y * p.k_per_split;
  const int k_end = min(p.K, k_begin + p.k_per_split);

  for (int i = threadIdx.x; i < MT * 16 * kSkinnyCols; i += blockDim.x)
    (&red[0][0])[i] = 0;

  int32_t acc[MT][4][4];
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[a][j][e] = 0;

  const int8_t* wrow[4];
  bool wok[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n = n0 + 8 * j + g;
    wok[j] = n < p.N;
    wrow[j] = p.QW + static_cast<int64_t>(wok[j] ? n : 0) * p.K + 16 * t;
  }
  const int8_t* xrow[MT][2];
  bool xok[MT][2];
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = a * 16 + g + 8 * h;
      xok[a][h] = m < p.M;
      xrow[a][h] = p.QX + static_cast<int64_t>(xok[a][h] ? m : 0) * p.K + 16 * t;
    }

  const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll 2
  for (int k = k_begin + warp * 64; k < k_end; k += kSkinnyWarps * 64) {
    uint4 bq[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) bq[j] = wok[j] ? ldg_stream(wrow[j] + k) : zero;
    uint4 aq[MT][2];
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        aq[a][h] = xok[a][h] ? *reinterpret_cast<const uint4*>(xrow[a][h] + k) : zero;
#pragma unroll
    for (int a = 0; a < MT; ++a) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mma_s8_16832(acc[a][j], aq[a][0].x, aq[a][1].x, aq[a][0].y, aq[a][1].y, bq[j].x, bq[j].y);
        mma_s8_16832(acc[a][j], aq[a][0].z, aq[a][1].z, aq[a][0].w, aq[a][1].w, bq[j].z, bq[j].w);
      }
    }
  }
  __syncthreads();  // red[] zeroed
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = a * 16 + g;
      const int c = 8 * j + 2 * t;
      atomicAdd(&red[r][c], acc[a][j][0]);
      atomicAdd(&red[r][c + 1], acc[a][j][1]);
      atomicAdd(&red[r + 8][c], acc[a][j][2]);
      atomicAdd(&red[r + 8][c + 1], acc[a][j][3]);
    }
  __syncthreads();
  for (int i = threadIdx.x; i < p.M * kSkinnyCols; i += blockDim.x) {
    const int m = i / kSkinnyCols;
    const int c = i % kSkinnyCols;
    if (n0 + c < p.N) atomicAdd(&p.acc[static_cast<int64_t>(m) * p.N + n0 + c], red[m][c]);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(&p.counters[blockIdx.x], 1) == gridDim.y - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < p.M * (kSkinnyCols / 8); i += blockDim.x) {
    const int m = i / (kSkinnyCols / 8);
    const int nn = n0 + 8 * (i % (kSkinnyCols / 8));
    int32_t s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      s[e] = (nn + e < p.N) ? __ldcg(&p.acc[static_cast<int64_t>(m) * p.N + nn + e]) : 0;
    epilogue_store<8, true>(p.ep, p.N, m, nn, s);
  }
}

cudaError_t launch_gemm_skinny(const GemmSkinnyArgs& a, cudaStream_t stream) {
  const dim3 grid((a.N + kSkinnyCols - 1) / kSkinnyCols, a.splits);
  const int mt = (a.M + 15) / 16;
  switch (mt) {
    case 1: gemm_skinny_kernel<1><<<grid, kSkinnyWarps * 32, 0, stream>>>(a); break;
    case 2: gemm_skinny_kernel<2><<<grid, kSkinnyWarps * 32, 0, stream>>>(a); break;
    case 3: gemm_skinny_kernel<3><<<grid, kSkinnyWarps * 32, 0, stream>>>(a); break;
    case 4: gemm_skinny_kernel<4><<<grid, kSkinnyWarps * 32, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace convrot
