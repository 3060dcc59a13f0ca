// LoRA down-projection T = X lora_down^T for the unmerged LoRA term of the
// page "[PR #249] Add an mps backend: weight-only INT8 and W4A8/W6A8 linears
// for Apple GPUs" (section "What": lora_down [R, K], lora_up [N, R],
// lora_scale), applied to the unrotated activation X.
//
// fp16 (or bf16) operands, fp32 accumulation on the mma.sync m16n8k16 path.  A warp
// owns 16 rows of X and every LoRA rank (up to kLoraMaxR / 8 n8 tiles) over
// one K slice; slices are summed into the zeroed T with fp32 atomics.  The
// operands of U consecutive 32-wide K steps are loaded before their MMAs, so
// each warp keeps U steps of loads in flight (the kernel streams X from HBM
// and is otherwise latency-bound).
//
// Fragment mapping for one 32-wide K step: lane (g = lane/4, t = lane%4)
// loads 8 consecutive fp16 k0 + 8t .. k0 + 8t + 7 of X rows g, g + 8 and of
// lora_down row g of each n8 tile; MMA s (0, 1) takes elements [4s, 4s + 4):
// the MMA K positions (2t, 2t+1) and (2t+8, 2t+9) map to the same real k for
// A and B, which is all a sum over k needs.
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace convrot {

// kBf16: bf16 operands (X and lora_down), otherwise fp16.
template <bool kBf16>
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (kBf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

constexpr int kLoraWarps = 4;

template <int NT, int U, bool kBf16>
__global__ void __launch_bounds__(kLoraWarps * 32) lora_down_kernel(const LoraDownArgs p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  grid_dep_wait();  // launched with programmatic dependent launch
  grid_dep_launch();
  const int m_base = (blockIdx.x * kLoraWarps + warp) * 16;
  if (m_base >= p.M) return;
  const int k_begin = blockIdx.y * p.k_per_split;
  const int k_end = min(p.K, k_begin + p.k_per_split);

  const uint16_t* xr[2];
  bool xok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = m_base + g + 8 * h;
    xok[h] = m < p.M;
    xr[h] = p.X + static_cast<int64_t>(xok[h] ? m : 0) * p.K + 8 * t;
  }
  // lora_down row 8j + g of n8 tile j starts at d_base + j * d_step.
  const uint16_t* d_base = p.down + static_cast<int64_t>(g) * p.K + 8 * t;
  const int64_t d_step = 8 * static_cast<int64_t>(p.K);
  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;

  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int k = k_begin; k < k_end; k += 32 * U) {
    uint4 x0[U], x1[U], d[U][NT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = k + 32 * u;
      const bool in = kk < k_end;
      x0[u] = (in && xok[0]) ? __ldg(reinterpret_cast<const uint4*>(xr[0] + kk)) : zero;
      x1[u] = (in && xok[1]) ? __ldg(reinterpret_cast<const uint4*>(xr[1] + kk)) : zero;
#pragma unroll
      for (int j = 0; j < NT; ++j)
        d[u][j] = (in && 8 * j + g < p.R)
                      ? __ldg(reinterpret_cast<const uint4*>(d_base + j * d_step + kk))
                      : zero;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        mma_f16_16816<kBf16>(acc[j], x0[u].x, x1[u].x, x0[u].y, x1[u].y, d[u][j].x, d[u][j].y);
        mma_f16_16816<kBf16>(acc[j], x0[u].z, x1[u].z, x0[u].w, x1[u].w, d[u][j].z, d[u][j].w);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c = 8 * j + 2 * t;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = m_base + g + 8 * h;
      if (m < p.M) {
        if (c < p.R) atomicAdd(&p.T[static_cast<int64_t>(m) * p.R + c], acc[j][2 * h]);
        if (c + 1 < p.R) atomicAdd(&p.T[static_cast<int64_t>(m) * p.R + c + 1], acc[j][2 * h + 1]);
      }
    }
  }
}

cudaError_t launch_lora_down(const LoraDownArgs& a, cudaStream_t stream) {
  const dim3 grid((a.M + 16 * kLoraWarps - 1) / (16 * kLoraWarps), a.splits);
  const int nt = (a.R + 7) / 8;
  void (*kernel)(const LoraDownArgs);
  // U keeps the operand registers per step group near 100.
  const bool b = a.bf16 != 0;
  if (nt <= 2)
    kernel = b ? lora_down_kernel<2, 8, true> : lora_down_kernel<2, 8, false>;
  else if (nt <= 4)
    kernel = b ? lora_down_kernel<4, 4, true> : lora_down_kernel<4, 4, false>;
  else if (nt <= 8)
    kernel = b ? lora_down_kernel<8, 2, true> : lora_down_kernel<8, 2, false>;
  else if (nt <= 16)
    kernel = b ? lora_down_kernel<16, 1, true> : lora_down_kernel<16, 1, false>;
  else
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kLoraWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace convrot
