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
//
// Persistent kernel: one CTA per SM walks a static schedule of work units
// (output tile 128 x BN, and K split when there are too few tiles).  Two
// accumulators in tensor memory alternate between consecutive chunks, across
// tiles too, so the MMAs of the next chunk -- or of the next tile -- run while
// the epilogue warps drain the previous one and write its outputs.
//
// CTA layout (320 threads, 1 CTA per SM), BN = 64, 128 or 256:
//   warp 0      TMA producer: A (128 x 64) and B (BN x 64) fp16 tiles into a
//               STAGES-deep ring of 128-byte-swizzled shared-memory buffers.
//   warp 1      tensor-memory allocator and MMA issuer (one lane): 4 MMAs of
//               128 x BN x 16 per K block, commits free the ring slots.
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4).. (its hardware
//               quadrant) and column half (w-2)/4 of the tile; keeps BN/2
//               int32 sums per thread.  The tile's scales are staged in
//               shared memory; Y is written as 128 x 64 fp16 boxes, staged
//               128-byte swizzled in a buffer per column half and stored with
//               TMA (the store of one box overlaps the next box's math).
// Split-K units add their exact int32 partial into a zeroed workspace with
// atomics (integer adds commute: deterministic); the last split of a tile to
// arrive writes the output.
// Launched with programmatic dependent launch: set-up (barriers, TMEM,
// descriptor prefetch) overlaps the previous kernel's tail; the first global
// access waits for that kernel's results.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace convrot {

constexpr int kBM = 128;
constexpr int kBK = 64;            // fp16 elements per K block (128 bytes: one swizzle row)
constexpr int kChunkKB = 16;       // 64-wide K blocks per exact fp32 chunk (1024 K)
constexpr int kPrefetchKB = 16;    // weight K blocks brought into L2 before the dependency wait
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr uint32_t kYBoxBytes = kBM * 64 * 2;  // one 128 x 64 fp16 store box (16 KB)

// Named barriers (0 is __syncthreads).
constexpr int kBarEpi = 1;    // all epilogue warps
constexpr int kBarHalf0 = 2;  // epilogue warps of column half 0 (+1 for half 1)

// A ring stage holds KSUB consecutive 64-wide K blocks of A and B.  Every
// stage costs one full/empty hand-off between the TMA producer and the MMA
// issuer, which takes a few hundred cycles; only 256-wide MMAs hide it, so
// narrower tiles move 128 K per stage (8 MMAs per hand-off).
template <int BN>
struct TcCfg {
  static constexpr int kSub = (BN == 256) ? 1 : 2;              // 64-wide K blocks per stage
  static constexpr uint32_t kABox = kBM * kBK * 2;              // 16 KB
  static constexpr uint32_t kBBox = BN * kBK * 2;
  static constexpr uint32_t kABytes = kSub * kABox;
  static constexpr uint32_t kBBytes = kSub * kBBox;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (BN == 256) ? 4 : (BN == 128 ? 3 : 4);
  static constexpr int kChunkStages = kChunkKB / kSub;  // stages per exact fp32 chunk
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  static constexpr int kEpiCols = BN / 2;        // sums per epilogue thread
  static constexpr int kStoreCols = kEpiCols >= 128 ? 8 : 16;  // direct-store group
  // Shared memory: ring | Y staging (2 x 16 KB) | scales | barriers.
  static constexpr uint32_t kRingBytes = kStages * kStageBytes;
  static constexpr uint32_t kStagingOff = kRingBytes;
  static constexpr uint32_t kScaleOff = kStagingOff + 2 * kYBoxBytes;  // sW[BN], sX[128]
  static constexpr uint32_t kBarOff = kScaleOff + (BN + kBM) * 4;
  static constexpr size_t kSmem = 1024 + kBarOff + 256;
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct Unit {
  int m0, n0, split, tile;
};

__device__ __forceinline__ Unit unit_of(int u, int tiles_m, int splits, int bn) {
  Unit r;
  r.split = u % splits;
  const int tile = u / splits;
  r.tile = tile;
  r.m0 = (tile % tiles_m) * kBM;  // M fastest: concurrent tiles share weight tiles
  r.n0 = (tile / tiles_m) * bn;
  return r;
}

template <int BN, bool kLora>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_y, const GemmTcArgs p) {
  using C = TcCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;                                     // kStages x kSub x 16 KB
  uint8_t* sB = base + C::kStages * C::kABytes;           // kStages x kSub x BN*128 B
  uint8_t* staging = base + C::kStagingOff;               // 2 x 16 KB
  float* sw_s = reinterpret_cast<float*>(base + C::kScaleOff);  // [BN]
  float* sx_s = sw_s + BN;                                       // [128]
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  uint64_t* accf = empty + C::kStages;  // [2]
  uint64_t* acce = accf + 2;            // [2]
  uint64_t* done = acce + 2;            // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* is_last = reinterpret_cast<int*>(tmem_slot + 1);
  int* abort_flag = is_last + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + kBM - 1) / kBM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int units = tiles_m * tiles_n * p.splits;
  const int nkb_total = p.K / kBK;  // 64-wide K blocks (a multiple of 4)

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    if (p.tma_store) tma_prefetch_desc(&tm_y);
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

  // The weight does not depend on the previous kernel: while that kernel
  // finishes, bring the first weight tiles of this CTA's first unit into L2.
  if (warp == 0 && lane == 0 && blockIdx.x < units) {
    const Unit w = unit_of(blockIdx.x, tiles_m, p.splits, BN);
    const int kb0 = w.split * p.kb_per_split;
    const int kb1 = min(nkb_total, min(kb0 + p.kb_per_split, kb0 + kPrefetchKB));
    for (int kb = kb0; kb < kb1; ++kb) tma_prefetch_l2_2d(&tm_b, kb * kBK, w.n0);
  }

  // Everything above touched only this CTA's own resources and the weight.
  // From here on the kernel reads what the previous kernel on the stream
  // wrote.
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;  // K blocks issued by this CTA so far (ring position)
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(u, tiles_m, p.splits, BN);
        const int kb0 = w.split * p.kb_per_split;
        const int kb1 = min(nkb_total, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; kb += C::kSub, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&empty[s], ((it / C::kStages) & 1) ^ 1, p.err, DEVERR_TIMEOUT_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
          for (int q = 0; q < C::kSub; ++q) {
            tma_load_2d(sA + s * C::kABytes + q * C::kABox, &tm_a, &full[s], (kb + q) * kBK, w.m0);
            tma_load_2d(sB + s * C::kBBytes + q * C::kBBox, &tm_b, &full[s], (kb + q) * kBK, w.n0);
          }
        }
      }
      // Leave no copy in flight: wait (bounded) for the last load of every
      // slot.  On the normal path the MMA issuer consumed them all already.
      for (int i = max(0, it - C::kStages); i < it; ++i)
        mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBM, BN);
      bool ok = true;
      int it = 0;  // K blocks consumed (ring position)
      int gc = 0;  // chunks issued (accumulator buffer = gc & 1)
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(u, tiles_m, p.splits, BN);
        const int kb0 = w.split * p.kb_per_split;
        const int nkb = max(0, min(nkb_total, kb0 + p.kb_per_split) - kb0);
        const int nst = nkb / C::kSub;  // stages of this unit
        for (int c0 = 0; c0 < nst && ok; c0 += C::kChunkStages, ++gc) {
          const int a = gc & 1;
          if (!mbar_wait(&acce[a], ((gc >> 1) & 1) ^ 1, p.err, DEVERR_TIMEOUT_ACC_EMPTY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + a * BN;
          const int c1 = min(nst, c0 + C::kChunkStages);
          for (int i = c0; i < c1; ++i, ++it) {
            const int s = it % C::kStages;
            if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err, DEVERR_TIMEOUT_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + s * C::kABytes);
            const uint32_t b_addr = smem_u32(sB + s * C::kBBytes);
#pragma unroll
            for (int q = 0; q < C::kSub; ++q) {
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint32_t acc_flag = (i > c0 || q > 0 || kk > 0) ? 1u : 0u;
                tc_mma_f16(d_tmem, smem_desc_k128(a_addr + q * C::kABox + kk * 32),
                           smem_desc_k128(b_addr + q * C::kBBox + kk * 32), idesc, acc_flag);
              }
            }
            tc_commit(&empty[s]);
          }
          if (ok) tc_commit(&accf[a]);
        }
      }
      // Every MMA issued so far must be complete before the accumulators are
      // freed.
      tc_commit(done);
      mbar_wait(done, 0, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int kHalf = C::kEpiCols;
    const int et = threadIdx.x - 64;  // 0..255
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int row = quad * 32 + lane;  // row within the tile
    // The thread that issues this half's TMA stores (BN = 64: one for both).
    const bool issuer = (BN == 64) ? (et == 0) : ((ew & 3) == 0 && lane == 0);
    int gc = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = unit_of(u, tiles_m, p.splits, BN);
      const int kb0 = w.split * p.kb_per_split;
      const int nkb = max(0, min(nkb_total, kb0 + p.kb_per_split) - kb0);
      int32_t sum[kHalf];
#pragma unroll
      for (int i = 0; i < kHalf; ++i) sum[i] = 0;
      // This unit's scales, loaded now so their latency hides behind the MMAs;
      // they go to shared memory once the previous unit's readers are done.
      float sw_reg = 0.0f, sx_reg = 0.0f;
      if (p.tma_store) {
        if (et < BN && w.n0 + et < p.N) sw_reg = p.ep.sW[w.n0 + et];
        if (et < kBM && w.m0 + et < p.M) sx_reg = p.ep.sX[w.m0 + et];
      }
      for (int c0 = 0; c0 < nkb / C::kSub; c0 += C::kChunkStages, ++gc) {
        const int a = gc & 1;
        if (*reinterpret_cast<volatile int*>(abort_flag) == 0) {
          // One lane per warp polls the barrier; the others block in the
          // shuffle instead of spinning on shared memory next to the MMAs.
          int got = 1;
          if (lane == 0) got = mbar_wait(&accf[a], (gc >> 1) & 1, p.err, DEVERR_TIMEOUT_ACC_FULL);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            *abort_flag = 1;
          } else {
            tc_fence_after();
            const uint32_t t0 =
                tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + a * BN + half * kHalf;
#pragma unroll
            for (int j = 0; j < kHalf / 16; ++j) {
              uint32_t r[16];
              tmem_ld_32x32b_x16(t0 + j * 16, r);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) sum[j * 16 + e] += __float2int_rn(__uint_as_float(r[e]));
            }
            tc_fence_before();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[a]);
      }

      // The whole epilogue group agrees on what to do with this unit.
      named_barrier_sync(kBarEpi, kEpiThreads);
      const bool aborted = *reinterpret_cast<volatile int*>(abort_flag) != 0;
      const int64_t m = static_cast<int64_t>(w.m0) + row;
      const int nb = w.n0 + half * kHalf;
      const bool row_ok = m < p.M;
      bool write = !aborted;
      if (!aborted && p.splits > 1) {
        // Add this split's exact partial; the last split to arrive finishes.
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < kHalf; ++i)
            if (nb + i < p.N) atomicAdd(&p.acc[m * p.N + nb + i], sum[i]);
        }
        __threadfence();
        named_barrier_sync(kBarEpi, kEpiThreads);
        if (et == 0) {
          const int prev = atomicAdd(&p.counters[w.tile], 1);
          *is_last = (prev == p.splits - 1) ? 1 : 0;
        }
        named_barrier_sync(kBarEpi, kEpiThreads);
        write = *reinterpret_cast<volatile int*>(is_last) != 0;
        if (write) {
          __threadfence();
#pragma unroll
          for (int i = 0; i < kHalf; ++i)
            sum[i] = (row_ok && nb + i < p.N) ? __ldcg(&p.acc[m * p.N + nb + i]) : 0;
        }
      }
      if (write && p.tma_store) {
        // Scales of this tile into shared memory (the previous unit's readers
        // are past the barrier above).
        if (et < BN) sw_s[et] = sw_reg;
        if (et < kBM) sx_s[et] = sx_reg;
        named_barrier_sync(kBarEpi, kEpiThreads);
        const float sx = sx_s[row];
        // Boxes of 64 columns; half h owns boxes [h*kHalf/64, (h+1)*kHalf/64)
        // (BN = 64: both halves share box 0).
        constexpr int kBoxes = (kHalf >= 64) ? kHalf / 64 : 1;
        constexpr int kBoxCols = (kHalf >= 64) ? 64 : kHalf;
        uint8_t* buf = staging + ((BN == 64) ? 0 : half * kYBoxBytes);
        const int bar = (BN == 64) ? kBarEpi : kBarHalf0 + half;
        const int bar_n = (BN == 64) ? kEpiThreads : kEpiThreads / 2;
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) {
          // The buffer is free once its previous store has read it.
          if (issuer) tma_store_wait_read();
          named_barrier_sync(bar, bar_n);
#pragma unroll
          for (int g = 0; g < kBoxCols / 16; ++g) {
            const int cl = b * 64 + g * 16;  // column within this half
            float y[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              y[e] = (static_cast<float>(sum[cl + e]) * sx) * sw_s[half * kHalf + cl + e];
            if (kLora && p.ep.R > 0 && row_ok) {
              int32_t zero16[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) zero16[e] = 0;
              float l[16];
              EpilogueArgs lo = p.ep;
              lo.lora_scale = p.ep.lora_scale;
              // epilogue_values with zero sums yields only the LoRA term.
              epilogue_values<16, kLora>(lo, p.N, m, nb + cl, zero16, l);
#pragma unroll
              for (int e = 0; e < 16; ++e) y[e] += l[e];
            }
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
              // column within the box: BN = 64 puts both halves in one box
              const int col = ((BN == 64) ? half * kHalf : 0) + g * 16 + h8 * 8;
              const int chunk = col >> 3;
              uint4 o;
              o.x = pack_half2(y[h8 * 8 + 0], y[h8 * 8 + 1]);
              o.y = pack_half2(y[h8 * 8 + 2], y[h8 * 8 + 3]);
              o.z = pack_half2(y[h8 * 8 + 4], y[h8 * 8 + 5]);
              o.w = pack_half2(y[h8 * 8 + 6], y[h8 * 8 + 7]);
              *reinterpret_cast<uint4*>(buf + row * 128 + ((chunk ^ (row & 7)) << 4)) = o;
            }
          }
          fence_proxy_async_smem();
          named_barrier_sync(bar, bar_n);
          if (issuer) {
            const int x = (BN == 64) ? w.n0 : w.n0 + half * kHalf + b * 64;
            if (x < p.N) tma_store_2d(&tm_y, buf, x, w.m0);
            tma_store_commit();
          }
        }
      } else if (write && row_ok) {
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
    // Shared memory must outlive the stores' reads of it; the writes
    // themselves complete with the grid.
    if (issuer) tma_store_wait_read();
  }

  // All roles meet here before the tensor memory is released.
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

size_t gemm_tc_smem_bytes(int bn) {
  return bn == 256 ? TcCfg<256>::kSmem : (bn == 128 ? TcCfg<128>::kSmem : TcCfg<64>::kSmem);
}

template <int BN, bool kLora>
static cudaError_t launch_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                             const CUtensorMap& tm_y, const GemmTcArgs& a, int grid,
                             cudaStream_t stream) {
  const size_t smem = TcCfg<BN>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, kLora>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, kLora>, tm_a, tm_b, tm_y, a);
}

cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_y,
                           const GemmTcArgs& a, int bn, int grid, cudaStream_t stream) {
  const bool lora = a.ep.mode == kOutF16 && a.ep.R > 0;
  switch (bn) {
    case 256:
      return lora ? launch_tc<256, true>(tm_a, tm_b, tm_y, a, grid, stream)
                  : launch_tc<256, false>(tm_a, tm_b, tm_y, a, grid, stream);
    case 128:
      return lora ? launch_tc<128, true>(tm_a, tm_b, tm_y, a, grid, stream)
                  : launch_tc<128, false>(tm_a, tm_b, tm_y, a, grid, stream);
    case 64:
      return lora ? launch_tc<64, true>(tm_a, tm_b, tm_y, a, grid, stream)
                  : launch_tc<64, false>(tm_a, tm_b, tm_y, a, grid, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace convrot
