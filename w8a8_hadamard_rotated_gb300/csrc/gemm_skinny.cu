// Small-M variant of the exact int8 GEMM: A = Q_X Q_W^T (int32), then the
// scale restore Y = A (.) s_X s_W^T (page "INT8ConvRot GEMM vs fp16 on M1 Max
// with Metal, MPSMatrix, and MLX", section "What changed in the computation").
//
// For M <= 64 the layer is a stream over the weight (N*K int8 bytes).  This
// kernel reads Q_W once, as int8, with 16-byte loads, U K-steps ahead of the
// MMAs, and multiplies on the integer mma.sync path (m16n8k32, s8 x s8 ->
// s32, exact).  The K range of a 32-column block is split across the CTAs of
// a thread-block cluster (1, 2, 4 or 8 of them): each CTA reduces its 4 warps
// in shared memory, and the cluster's first CTA adds the others' partials
// through distributed shared memory (integer adds: exact, deterministic) and
// applies the epilogue.  No global atomics and nothing to zero beforehand.
//
// Operand fragments.  For one 64-wide K step, lane (g = lane/4, t = lane%4)
// loads 16 consecutive bytes k0 + 16t .. k0 + 16t + 15 of a weight row and of
// the activation rows g and g + 8.  The two m16n8k32 MMAs of the step take
// bytes [8s, 8s + 8) of those (s = 0, 1): the MMA's K positions 4t..4t+3 and
// 16+4t..16+4t+3 map to the same real k for A and for B, so the products are
// the right ones (a sum over k does not depend on the order of k).
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
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

// kExt: the epilogue honours the bias / bf16 fields of EpilogueArgs.
template <int MT, int U, bool kExt>
__global__ void __launch_bounds__(kSkinnyWarps * 32) gemm_skinny_kernel(const GemmSkinnyArgs p) {
  __shared__ int32_t red[MT * 16][kSkinnyCols];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int cs = p.splits;             // CTAs of the cluster (K slices of the block)
  const int split = blockIdx.x % cs;   // = rank in the cluster
  const int n0 = (blockIdx.x / cs) * kSkinnyCols;
  const int k_begin = split * p.k_per_split;
  const int k_end = min(p.K, k_begin + p.k_per_split);

  for (int i = threadIdx.x; i < MT * 16 * kSkinnyCols; i += blockDim.x)
    (&red[0][0])[i] = 0;
  // The weight does not come from the previous kernel: start its slice on its
  // way into L2 while that kernel finishes (a prefetch returns nothing to the
  // SM; L2 is the point of coherence).  32 rows x (k_end - k_begin) bytes,
  // one 128-byte line per prefetch.
  {
    const int lines = (k_end - k_begin) / 128;
    for (int i = threadIdx.x; i < kSkinnyCols * lines; i += blockDim.x) {
      const int n = n0 + i / lines;
      if (n < p.N) {
        const int8_t* line = p.QW + static_cast<int64_t>(n) * p.K + k_begin + (i % lines) * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
      }
    }
  }
  // Launched with programmatic dependent launch: the codes come from the
  // previous kernel.
  grid_dep_wait();
  grid_dep_launch();

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
  constexpr int kStep = kSkinnyWarps * 64;  // K per iteration of the CTA
  for (int k = k_begin + warp * 64; k < k_end; k += kStep * U) {
    uint4 bq[U][4];
    uint4 aq[U][MT][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = k + u * kStep;
      const bool in = kk < k_end;
#pragma unroll
      for (int j = 0; j < 4; ++j) bq[u][j] = (in && wok[j]) ? ldg_stream(wrow[j] + kk) : zero;
#pragma unroll
      for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          aq[u][a][h] = (in && xok[a][h]) ? *reinterpret_cast<const uint4*>(xrow[a][h] + kk) : zero;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mma_s8_16832(acc[a][j], aq[u][a][0].x, aq[u][a][1].x, aq[u][a][0].y, aq[u][a][1].y,
                       bq[u][j].x, bq[u][j].y);
          mma_s8_16832(acc[a][j], aq[u][a][0].z, aq[u][a][1].z, aq[u][a][0].w, aq[u][a][1].w,
                       bq[u][j].z, bq[u][j].w);
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
  if (cs > 1) {
    // Every CTA of the cluster reaches both barriers unconditionally (the
    // kernel has no other waits): the first makes every CTA's red[] visible
    // to the cluster, the second keeps the others' shared memory alive until
    // the first CTA has read it.
    cluster_sync_all();
    if (split == 0) {
      for (int i = threadIdx.x; i < p.M * kSkinnyCols; i += blockDim.x) {
        int32_t* mine = &red[0][0] + (i / kSkinnyCols) * kSkinnyCols + (i % kSkinnyCols);
        int32_t v = *mine;
        for (int q = 1; q < cs; ++q) v += ld_cluster_s32(map_to_cta(mine, static_cast<uint32_t>(q)));
        *mine = v;
      }
    }
    cluster_sync_all();
    if (split != 0) return;
  } else {
    __syncthreads();
  }
  for (int i = threadIdx.x; i < p.M * (kSkinnyCols / 8); i += blockDim.x) {
    const int m = i / (kSkinnyCols / 8);
    const int c = 8 * (i % (kSkinnyCols / 8));
    int32_t s8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) s8[e] = red[m][c + e];
    epilogue_store<8, true, kExt>(p.ep, p.N, m, n0 + c, s8);
  }
}

int skinny_cluster_size(int64_t N, int64_t K, int sms) {
  const int64_t nblk = (N + kSkinnyCols - 1) / kSkinnyCols;
  int cs = 1;
  // Enough CTAs to stream the weight (about two per SM), slices of >= 256 K.
  while (cs < 8 && nblk * cs < 2 * static_cast<int64_t>(sms) && K / (2 * cs) >= 256 &&
         (K / (2 * cs)) % 256 == 0)
    cs *= 2;
  return cs;
}

template <int MT, int U, bool kExt>
static cudaError_t launch_skinny(const GemmSkinnyArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((a.N + kSkinnyCols - 1) / kSkinnyCols) * a.splits);
  cfg.blockDim = dim3(kSkinnyWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(a.splits);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<MT, U, kExt>, a);
}

cudaError_t launch_gemm_skinny(const GemmSkinnyArgs& a, cudaStream_t stream) {
  if (a.splits != 1 && a.splits != 2 && a.splits != 4 && a.splits != 8) return cudaErrorInvalidValue;
  const bool ext = a.ep.bias != nullptr || a.ep.out_bf16 != 0 || a.ep.lora_bf16 != 0;
  switch ((a.M + 15) / 16) {
    case 1: return ext ? launch_skinny<1, 4, true>(a, stream) : launch_skinny<1, 4, false>(a, stream);
    case 2: return ext ? launch_skinny<2, 2, true>(a, stream) : launch_skinny<2, 2, false>(a, stream);
    case 3: return ext ? launch_skinny<3, 1, true>(a, stream) : launch_skinny<3, 1, false>(a, stream);
    case 4: return ext ? launch_skinny<4, 1, true>(a, stream) : launch_skinny<4, 1, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace convrot
