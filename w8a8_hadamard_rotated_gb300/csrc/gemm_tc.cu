// Exact int8 x int8 -> int32 GEMM on the sm_103a tensor cores (tcgen05).
//
// Page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX",
// section "What changed in the computation": A = Q_X Q_W^T accumulated in
// int32, then Y = A (.) s_X s_W^T.
//
// sm_103a has no integer tcgen05 MMA (ptxas rejects .kind::i8 for this
// target), so the product runs on .kind::f16 with exact operands:
//   * every int8 value is exact in fp16 and every product (|p| <= 2^14) is
//     exact in fp32;
//   * the fp32 accumulator in tensor memory is drained every 1024 K (16 K
//     blocks of 64): a chunk sum is an integer of magnitude <= 1024 * 2^14 =
//     2^24, which fp32 holds exactly;
//   * each drained chunk is converted with round-to-nearest (a no-op on an
//     exact integer) and added into int32 registers, so A is exact for any K.
// Two accumulator buffers in tensor memory alternate between chunks, so the
// MMAs of chunk c+1 run while the epilogue warps drain chunk c.
//
// CTA layout (320 threads, 1 CTA per SM):
//   warp 0      TMA producer: A (128 x 64) and B (BN x 64) fp16 tiles into a
//               STAGES-deep ring of 128-byte-swizzled shared-memory buffers.
//   warp 1      tensor-memory allocator and MMA issuer (one lane): 4 MMAs of
//               128 x BN x 16 per K block, commits free the ring slots.
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4).. (its hardware
//               quadrant) and column half (w-2)/4 of the tile; keeps BN/2
//               int32 sums per thread; writes Y (or A) at the end.
// Split-K (gridDim.z > 1): each split adds its exact int32 partial into a
// zeroed workspace with atomics (integer adds commute, so the result is
// deterministic); the last split to arrive at a tile writes the output.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace convrot {

constexpr int kBM = 128;
constexpr int kBK = 64;            // fp16 elements per K block (128 bytes: one swizzle row)
constexpr int kChunkKB = 16;       // K blocks per exact fp32 chunk (1024 K)
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;

template <int BN>
struct TcCfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;       // two accumulators
  static constexpr int kEpiCols = BN / 2;                 // sums per epilogue thread
  static constexpr int kStoreCols = kEpiCols >= 128 ? 8 : 16;  // columns per store group
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes + 256;
};

template <int BN, bool kLora>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const GemmTcArgs p) {
  using C = TcCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;                                     // kStages x 16 KB
  uint8_t* sB = base + C::kStages * C::kABytes;           // kStages x BN*128 B
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* accf = empty + C::kStages;  // [2]
  uint64_t* acce = accf + 2;            // [2]
  uint64_t* done = acce + 2;            // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* is_last = reinterpret_cast<int*>(tmem_slot + 1);
  int* abort_flag = is_last + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * kBM;
  const int split = blockIdx.z;
  const int nkb_total = p.K / kBK;
  const int kb_begin = split * p.kb_per_split;
  const int kb_end = min(nkb_total, kb_begin + p.kb_per_split);
  const int nkb = max(0, kb_end - kb_begin);
  const int nchunks = (nkb + kChunkKB - 1) / kChunkKB;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], kEpiWarps);
    }
    mbar_init(done, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, p.err, DEVERR_TIMEOUT_EMPTY)) break;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        const int kx = (kb_begin + i) * kBK;
        tma_load_2d(sA + s * C::kABytes, &tm_a, &full[s], kx, m0);
        tma_load_2d(sB + s * C::kBBytes, &tm_b, &full[s], kx, n0);
        issued = i + 1;
      }
      // Leave no copy in flight: wait (bounded) for the last load of every
      // slot.  On the normal path the MMA issuer consumed them all already.
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
      bool ok = true;
      int i = 0;
      for (int c = 0; c < nchunks && ok; ++c) {
        const int a = c & 1;
        if (!mbar_wait(&acce[a], ((c >> 1) & 1) ^ 1, p.err, DEVERR_TIMEOUT_ACC_EMPTY)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + a * BN;
        const int kend = min(nkb, (c + 1) * kChunkKB);
        for (; i < kend; ++i) {
          const int s = i % C::kStages;
          if (!mbar_wait(&full[s], (i / C::kStages) & 1, p.err, DEVERR_TIMEOUT_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + s * C::kABytes);
          const uint32_t b_addr = smem_u32(sB + s * C::kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc_flag = (i > c * kChunkKB || kk > 0) ? 1u : 0u;
            tc_mma_f16(d_tmem, smem_desc_k128(a_addr + kk * 32), smem_desc_k128(b_addr + kk * 32),
                       idesc, acc_flag);
          }
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&accf[a]);
      }
      // Every MMA issued so far must be complete before the accumulators are
      // freed.
      tc_commit(done);
      mbar_wait(done, 0, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int kHalf = C::kEpiCols;
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    int32_t sum[kHalf];
#pragma unroll
    for (int i = 0; i < kHalf; ++i) sum[i] = 0;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int a = c & 1;
      if (!mbar_wait(&accf[a], (c >> 1) & 1, p.err, DEVERR_TIMEOUT_ACC_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t0 = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + a * BN + half * kHalf;
#pragma unroll
      for (int j = 0; j < kHalf / 16; ++j) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(t0 + j * 16, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) sum[j * 16 + e] += __float2int_rn(__uint_as_float(r[e]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[a]);
    }
    // Every epilogue warp must agree on success before touching the outputs.
    if (!ok && lane == 0) *abort_flag = 1;
    named_barrier_sync(1, kEpiWarps * 32);
    if (*reinterpret_cast<volatile int*>(abort_flag) == 0) {
      const int64_t m = static_cast<int64_t>(m0) + quad * 32 + lane;
      const int nb = n0 + half * kHalf;
      const bool row_ok = m < p.M;
      if (p.splits > 1) {
        // Add this split's exact partial; the last split to arrive finishes.
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < kHalf; ++i)
            if (nb + i < p.N) atomicAdd(&p.acc[m * p.N + nb + i], sum[i]);
        }
        __threadfence();
        named_barrier_sync(1, kEpiWarps * 32);
        if (ew == 0 && lane == 0) {
          const int prev = atomicAdd(&p.counters[blockIdx.y * gridDim.x + blockIdx.x], 1);
          *is_last = (prev == p.splits - 1) ? 1 : 0;
        }
        named_barrier_sync(1, kEpiWarps * 32);
        const bool last = *reinterpret_cast<volatile int*>(is_last) != 0;
        if (last) {
          __threadfence();
#pragma unroll
          for (int i = 0; i < kHalf; ++i)
            sum[i] = (row_ok && nb + i < p.N) ? __ldcg(&p.acc[m * p.N + nb + i]) : 0;
        }
        if (!last) goto epilogue_done;
      }
      if (row_ok) {
        constexpr int G = C::kStoreCols;
#pragma unroll
        for (int j = 0; j < kHalf / G; ++j) {
          int32_t sg[G];
#pragma unroll
          for (int e = 0; e < G; ++e) sg[e] = sum[j * G + e];
          epilogue_store<G, kLora>(p.ep, p.N, m, nb + j * G, sg);
        }
      }
    }
  epilogue_done:;
  }

  // All roles meet here; the epilogue then writes the outputs.
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace convrot

namespace convrot {

size_t gemm_tc_smem_bytes(int bn) { return bn == 256 ? TcCfg<256>::kSmem : TcCfg<128>::kSmem; }

template <int BN, bool kLora>
static cudaError_t launch_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const GemmTcArgs& a,
                             cudaStream_t stream) {
  const dim3 grid((a.N + BN - 1) / BN, (a.M + kBM - 1) / kBM, a.splits);
  const size_t smem = TcCfg<BN>::kSmem;
  cudaFuncSetAttribute(gemm_tc_kernel<BN, kLora>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(smem));
  gemm_tc_kernel<BN, kLora><<<grid, kThreads, smem, stream>>>(tm_a, tm_b, a);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const GemmTcArgs& a,
                           int bn, cudaStream_t stream) {
  const bool lora = a.ep.mode == kOutF16 && a.ep.R > 0;
  if (bn == 256)
    return lora ? launch_tc<256, true>(tm_a, tm_b, a, stream)
                : launch_tc<256, false>(tm_a, tm_b, a, stream);
  return lora ? launch_tc<128, true>(tm_a, tm_b, a, stream)
              : launch_tc<128, false>(tm_a, tm_b, a, stream);
}

}  // namespace convrot
