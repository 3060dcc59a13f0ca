// Throughput ceilings of the two exact int8 product engines on this GPU.
//
// The layer's product A = Q_X Q_W^T (page "INT8ConvRot GEMM vs fp16 on M1 Max
// with Metal, MPSMatrix, and MLX", section "What changed in the
// computation") runs on one of two tensor-core paths, because sm_103a has no
// integer tcgen05 MMA:
//   * mma.sync m16n8k32 s8 x s8 -> s32 (the legacy warp-level path; the
//     small-M engine), and
//   * tcgen05.mma kind::f16 on operands that hold the int8 values exactly
//     (the large-M engines).
// These kernels measure what each path can do when nothing else limits it:
// operands already in registers (mma.sync) or in shared memory (tcgen05),
// no loads, no epilogue.  The benchmark reports the GEMM's fraction of these
// next to its fraction of the measured dense bf16 peak.  Two more warp-level
// engines serve the small-M paths: the 4-way int8 dot product (dp4a, the
// one-kernel layer at M <= 2) and mma.sync m16n8k16 f16 -> f32 on operands
// that hold the int8 values exactly (the small-M GEMM at M >= 3).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace convrot {
namespace {

constexpr int kS8Warps = 8;       // warps per CTA
constexpr int kS8Chains = 8;      // independent accumulators per warp
constexpr int kS8CtasPerSm = 4;
constexpr double kS8OpsPerMma = 2.0 * 16 * 8 * 32;

// Written only to keep the probe's accumulators live.
__device__ int g_peak_sink;

// Back-to-back m16n8k32 s8 MMAs from registers.  The operands come from the
// thread index, so the compiler cannot fold them; the accumulators are
// written out so that nothing is dead.
__global__ void __launch_bounds__(kS8Warps * 32) peak_mma_s8_kernel(int64_t reps) {
  const uint32_t t = threadIdx.x;
  const uint32_t a0 = t * 0x01010101u, a1 = a0 ^ 0x5a5a5a5au, a2 = a0 + 0x03030303u,
                 a3 = a0 ^ 0x0f0f0f0fu;
  const uint32_t b0 = a0 + 0x11111111u, b1 = a0 ^ 0x33333333u;
  int d[kS8Chains][4];
#pragma unroll
  for (int c = 0; c < kS8Chains; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[c][i] = 0;
  for (int64_t r = 0; r < reps; ++r) {
#pragma unroll
    for (int c = 0; c < kS8Chains; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
          "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
          : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int c = 0; c < kS8Chains; ++c) s += d[c][0] ^ d[c][1] ^ d[c][2] ^ d[c][3];
  if (s == 0x7fffffff) g_peak_sink = s;
}

// Back-to-back m16n8k16 f16 x f16 -> f32 MMAs from registers (fp16 bit
// patterns kept finite and small), the small-M GEMM's engine.
constexpr double kF16OpsPerMma = 2.0 * 16 * 8 * 16;
__global__ void __launch_bounds__(kS8Warps * 32) peak_mma_f16_kernel(int64_t reps) {
  const uint32_t t = threadIdx.x;
  const uint32_t a0 = (t * 0x00010001u) & 0x3bff3bffu, a1 = (a0 ^ 0x00110011u) & 0x3bff3bffu,
                 a2 = (a0 + 0x00030003u) & 0x3bff3bffu, a3 = (a0 ^ 0x000f000fu) & 0x3bff3bffu;
  const uint32_t b0 = (a0 + 0x01110111u) & 0x3bff3bffu, b1 = (a0 ^ 0x00330033u) & 0x3bff3bffu;
  float d[kS8Chains][4];
#pragma unroll
  for (int c = 0; c < kS8Chains; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[c][i] = 0.0f;
  for (int64_t r = 0; r < reps; ++r) {
#pragma unroll
    for (int c = 0; c < kS8Chains; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
          "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
          : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kS8Chains; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
  if (s == 1234.5f) g_peak_sink = 1;
}

// Back-to-back dp4a (4 int8 products into an int32 each), 8 chains of 4 per
// thread, the one-kernel small-M layer's engine.
constexpr int kDp4aPerStep = kS8Chains * 4;
__global__ void __launch_bounds__(kS8Warps * 32) peak_dp4a_kernel(int64_t reps) {
  const int t = static_cast<int>(threadIdx.x);
  const int a = t * 0x01010101, b = a ^ 0x5a5a5a5a;
  int d[kDp4aPerStep];
#pragma unroll
  for (int i = 0; i < kDp4aPerStep; ++i) d[i] = i;
  for (int64_t r = 0; r < reps; ++r) {
#pragma unroll
    for (int i = 0; i < kDp4aPerStep; ++i) d[i] = __dp4a(a + i, b, d[i]);
  }
  int s = 0;
#pragma unroll
  for (int i = 0; i < kDp4aPerStep; ++i) s ^= d[i];
  if (s == 0x7fffffff) g_peak_sink = s;
}

// tcgen05.mma kind::f16, M = 128, N = 256, K = 16 per instruction, issued
// back to back by one thread on one shared-memory stage (zeros) into one
// tensor-memory accumulator: the 1-SM tensor pipe's own rate.
constexpr int kTcN = 256;
constexpr uint32_t kTcABytes = 128 * 128;  // 128 rows x 64 fp16
constexpr uint32_t kTcBBytes = kTcN * 128;
constexpr size_t kTcSmem = 1024 + kTcABytes + kTcBBytes + 64;
constexpr double kTcOpsPerMma = 2.0 * 128 * kTcN * 16;

__global__ void __launch_bounds__(128, 1) peak_tcgen05_kernel(int64_t reps, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kTcABytes;
  uint64_t* done = reinterpret_cast<uint64_t*>(sB + kTcBBytes);
  uint32_t* slot = reinterpret_cast<uint32_t*>(done + 1);
  for (uint32_t i = threadIdx.x * 16; i < kTcABytes + kTcBBytes; i += 128 * 16)
    *reinterpret_cast<uint4*>(base + i) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();  // the zeros are read by the tensor cores
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(slot, kTcN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 32) {
    constexpr uint32_t idesc = idesc_f16_f32(128, kTcN);
    const uint32_t a = smem_u32(sA), b = smem_u32(sB);
    for (int64_t r = 0; r < reps; ++r) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc_mma_f16(tmem, smem_desc_k128(a + kk * 32), smem_desc_k128(b + kk * 32), idesc,
                   (r > 0 || kk > 0) ? 1u : 0u);
    }
    tc_commit(done);
    mbar_wait(done, 0, err, DEVERR_TIMEOUT_DRAIN);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTcN);
}

}  // namespace

cudaError_t launch_peak_engine(int engine, int64_t reps, int sms, int* err, double* ops,
                               cudaStream_t st) {
  if (engine == 0) {
    const int grid = sms * kS8CtasPerSm;
    peak_mma_s8_kernel<<<grid, kS8Warps * 32, 0, st>>>(reps);
    *ops = kS8OpsPerMma * kS8Chains * kS8Warps * static_cast<double>(grid) *
           static_cast<double>(reps);
    return cudaGetLastError();
  }
  if (engine == 2 || engine == 3) {
    const int grid = sms * kS8CtasPerSm;
    const double threads = static_cast<double>(grid) * kS8Warps * 32;
    if (engine == 2) {
      peak_mma_f16_kernel<<<grid, kS8Warps * 32, 0, st>>>(reps);
      *ops = kF16OpsPerMma * kS8Chains * kS8Warps * static_cast<double>(grid) *
             static_cast<double>(reps);
    } else {
      peak_dp4a_kernel<<<grid, kS8Warps * 32, 0, st>>>(reps);
      *ops = 8.0 * kDp4aPerStep * threads * static_cast<double>(reps);  // 4 multiply-adds each
    }
    return cudaGetLastError();
  }
  const cudaError_t e = cudaFuncSetAttribute(
      peak_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kTcSmem));
  if (e != cudaSuccess) return e;
  peak_tcgen05_kernel<<<sms, 128, kTcSmem, st>>>(reps, err);
  *ops = kTcOpsPerMma * 4 * static_cast<double>(sms) * static_cast<double>(reps);
  return cudaGetLastError();
}

}  // namespace convrot
