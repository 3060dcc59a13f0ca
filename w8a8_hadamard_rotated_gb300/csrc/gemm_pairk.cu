// Exact int8 GEMM with the K range split across the two CTAs of a cluster and
// a streaming exchange of the two fp32 partials (sm_103a).
//
// Page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX",
// section "What changed in the computation": A = Q_X Q_W^T accumulated in
// int32, then Y = A (.) s_X s_W^T (fp32 ((float)A * s_X) * s_W, one rounding
// to fp16).
//
// The product runs on tcgen05 kind::f16 with operands that hold the int8
// codes exactly (sm_103a has no integer tcgen05 MMA).  Each CTA of a 2-CTA
// cluster computes one 128 x BN output tile over one half of K.  A half is
// at most 1024 K (K <= 2048), so its fp32 accumulator in tensor memory holds
// the exact integer partial P_c (|P_c| <= 1024 * 2^14 = 2^24), and the fp32
// sum P_0 + P_1 rounds the exact A once: it is (float)A, bit for bit what the
// single-CTA kernels produce.
//
// Why this shape: 128 x 256 MMAs keep the tensor pipe busier than 128 x 128
// ones (each instruction covers twice the hand-off cost), and at M = 1024,
// N = 2048 the 64 such tiles fill 128 SMs only with K split in two.
//
// Exchange.  CTA c finalizes columns [c * BN/2, (c + 1) * BN/2) of the tile.
// Each of its 8 epilogue warps -- TMEM lane quadrant q, column group g --
//   1. reads its 32 rows x BN/4 columns of the partner's half from tensor
//      memory, stages them in shared memory (padded rows: no bank
//      conflicts) and pushes them with one bulk copy (distributed shared
//      memory) into the partner's matching receive block, completing on the
//      partner's per-block mbarrier;
//   2. waits for the partner's block of its own columns and streams them,
//      16 columns at a time, from tensor memory: fp32 add, scale, fp16,
//      staged 128-byte swizzled, then one TMA store per 64-column box.
// Nothing is kept in registers across the exchange.  A CTA pushes into the
// partner's ring only after the partner's MMAs are done ("ring free", a
// remote arrival), and leaves only after the partner has consumed its block
// ("read") and made its own remote arrivals.  Every wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace convrot {
namespace {

constexpr int kPkBM = 128;
constexpr int kPkEpiWarps = 8;
constexpr int kPkThreads = 64 + 32 * kPkEpiWarps;

__host__ __device__ constexpr uint32_t pk_align1024(uint32_t v) { return (v + 1023u) & ~1023u; }

template <int BN>
struct PkCfg {
  static constexpr int kStageK = (BN == 256) ? 64 : 128;  // K per ring stage
  static constexpr int kSub = kStageK / 64;                // 64-wide TMA boxes per stage
  static constexpr uint32_t kABox = kPkBM * 128;           // 128 rows x 64 fp16
  static constexpr uint32_t kBBox = BN * 128;
  static constexpr uint32_t kABytes = kSub * kABox;
  static constexpr uint32_t kBBytes = kSub * kBBox;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (BN == 256) ? 4 : 3;
  static constexpr uint32_t kRingBytes = kStages * kStageBytes;
  static constexpr int kOwn = BN / 2;       // columns this CTA finalizes
  static constexpr int kSubCols = kOwn / 2;  // columns of one epilogue warp
  static constexpr uint32_t kBlkRow = kSubCols * 4 + 16;  // padded fp32 row
  static constexpr uint32_t kBlkBytes = 32 * kBlkRow;     // one warp's block
  // Inside the ring once the MMAs are done: 8 receive blocks, 8 send blocks,
  // then the fp16 Y boxes (128 rows x 64 columns, 128-byte swizzled).
  static constexpr uint32_t kRecvOff = 0;
  static constexpr uint32_t kSendOff = 8 * kBlkBytes;
  static constexpr uint32_t kYOff = pk_align1024(kSendOff + 8 * kBlkBytes);
  static constexpr int kYBoxes = kOwn / 64;
  static constexpr uint32_t kYBytes = kYBoxes * kPkBM * 128;
  static_assert(kYOff + kYBytes <= kRingBytes, "exchange buffers fit the ring");
  static_assert(kBlkBytes % 16 == 0 && kSendOff % 16 == 0, "bulk copy alignment");
  static constexpr uint32_t kScaleOff = kRingBytes;  // s_W of the own columns
  static constexpr uint32_t kBarOff = kScaleOff + kOwn * 4;
  static constexpr size_t kSmem = 1024 + kBarOff + 256;
  static_assert(kSmem <= 232448, "shared memory budget");
};

// Barriers: full[kStages], empty[kStages], accf, done, recv[8], peer_free,
// peer_read; then the tensor-memory slot.
template <int BN>
__global__ void __launch_bounds__(kPkThreads, 1)
    gemm_pairk_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_y, const GemmTcArgs p) {
  using C = PkCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::kStages * C::kABytes;
  float* sw_s = reinterpret_cast<float*>(base + C::kScaleOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  uint64_t* accf = empty + C::kStages;
  uint64_t* done = accf + 1;
  uint64_t* recv = done + 1;          // [8]
  uint64_t* peer_free = recv + 8;     // the partner's MMAs are done (its ring is free)
  uint64_t* peer_read = peer_free + 1;  // the partner consumed this CTA's blocks (8 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(peer_read + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t c = cluster_ctarank();  // this CTA's K half
  const uint32_t peer = c ^ 1u;
  const int tiles_m = (p.M + kPkBM - 1) / kPkBM;
  const int tile = static_cast<int>(blockIdx.x >> 1);
  const int m0 = (tile % tiles_m) * kPkBM;
  const int n0 = (tile / tiles_m) * BN;
  const int kb_half = p.K / 128;  // 64-wide K blocks per half
  const int kb0 = static_cast<int>(c) * kb_half;
  const int nst = kb_half / C::kSub;  // ring stages of this CTA
  const int own0 = static_cast<int>(c) * C::kOwn;  // first column this CTA finalizes

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_y);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(done, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&recv[i], 1);
    mbar_init(peer_free, 1);
    mbar_init(peer_read, kPkEpiWarps);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The partner may arrive on this CTA's barriers only once they exist.
  cluster_sync_all();

  // The weight does not depend on the previous kernel.  With weight_early
  // (the previous launch is this library's rotate + quantize kernel, which
  // signals its dependents only after its own dependency wait), the first
  // ring stages are armed and their weight boxes loaded now, one stage per
  // epilogue warp.
  const int pre = p.weight_early ? min(C::kStages, nst) : 0;
  if (warp >= 2 && lane == 0 && warp - 2 < pre) {
    const int i = warp - 2;
    mbar_arrive_expect_tx(&full[i], C::kStageBytes);
#pragma unroll
    for (int q = 0; q < C::kSub; ++q)
      tma_load_2d(sB + i * C::kBBytes + q * C::kBBox, &tm_b, &full[i],
                  (kb0 + i * C::kSub + q) * 64, n0);
  }
  // Without early loads, the first weight blocks go into L2 instead.  (With
  // them, no further prefetch: the eight CTAs that share a weight panel
  // would each prefetch it, and those requests delay the first activation
  // loads -- measured +0.8 us per layer.)
  if (!p.weight_early && warp == 0 && lane == 0) {
    for (int kb = kb0; kb < min(kb0 + kb_half, kb0 + 4 * C::kSub); ++kb)
      tma_prefetch_l2_2d(&tm_b, kb * 64, n0);
  }

  // From here on the kernel reads what the previous kernel wrote.
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      for (; it < nst; ++it) {
        const int s = it % C::kStages;
        const int kb = kb0 + it * C::kSub;
        if (it < pre) {
#pragma unroll
          for (int q = 0; q < C::kSub; ++q)
            tma_load_2d(sA + s * C::kABytes + q * C::kABox, &tm_a, &full[s], (kb + q) * 64, m0);
          continue;
        }
        if (!mbar_wait(&empty[s], ((it / C::kStages) & 1) ^ 1, p.err, DEVERR_TIMEOUT_EMPTY)) break;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
        for (int q = 0; q < C::kSub; ++q) {
          tma_load_2d(sA + s * C::kABytes + q * C::kABox, &tm_a, &full[s], (kb + q) * 64, m0);
          tma_load_2d(sB + s * C::kBBytes + q * C::kBBox, &tm_b, &full[s], (kb + q) * 64, n0);
        }
      }
      // Leave no copy in flight (on the normal path the MMAs consumed all).
      const int armed = max(it, pre);
      for (int i = max(0, armed - C::kStages); i < armed; ++i)
        mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kPkBM, BN);
      bool ok = true;
      for (int it = 0; it < nst; ++it) {
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
          for (int kk = 0; kk < 4; ++kk) {
            tc_mma_f16(tmem_base, smem_desc_k128(a_addr + q * C::kABox + kk * 32),
                       smem_desc_k128(b_addr + q * C::kBBox + kk * 32), idesc,
                       (it > 0 || q > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc_commit(&empty[s]);
      }
      if (ok) tc_commit(accf);
      // Every MMA issued must be complete before the tensor memory is freed.
      tc_commit(done);
      mbar_wait(done, 0, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;  // 0..255
    const int q = warp & 3;           // TMEM lane quadrant
    const int g = (warp - 2) >> 2;    // column group
    const int blk = q * 2 + g;        // exchange block of this warp
    const int row = q * 32 + lane;    // row within the tile
    // The partner's block for this warp's columns: expected bytes, armed now.
    if (lane == 0) mbar_arrive_expect_tx(&recv[blk], C::kBlkBytes);
    // Scales while the MMAs run.
    if (et < C::kOwn) sw_s[et] = (n0 + own0 + et < p.N) ? p.ep.sW[n0 + own0 + et] : 0.0f;
    const float sx = (m0 + row < p.M) ? __ldcg(&p.ep.sX[m0 + row]) : 0.0f;

    int got = 1;
    if (lane == 0) got = mbar_wait(accf, 0, p.err, DEVERR_TIMEOUT_ACC_FULL);
    got = __shfl_sync(0xffffffffu, got, 0);
    tc_fence_after();
    // This CTA's MMAs are done: its ring may take the partner's blocks.
    if (got && et == 0) mbar_arrive_remote(map_to_cta(peer_free, peer));

    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // 1. The partner's columns of this warp -> send block -> partner.
    if (got) {
      const int pcol = static_cast<int>(peer) * C::kOwn + g * C::kSubCols;
      uint8_t* dst = base + C::kSendOff + blk * C::kBlkBytes + lane * C::kBlkRow;
#pragma unroll
      for (int j = 0; j < C::kSubCols / 32; ++j) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_lane + pcol + j * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<uint4*>(dst + (j * 32 + e) * 4) = make_uint4(r[e], r[e + 1], r[e + 2], r[e + 3]);
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0 && got) {
      if (mbar_wait_cluster(peer_free, 0, p.err, DEVERR_TIMEOUT_CLUSTER))
        bulk_copy_to_cta(map_to_cta(base + C::kRecvOff + blk * C::kBlkBytes, peer),
                         base + C::kSendOff + blk * C::kBlkBytes, C::kBlkBytes,
                         map_to_cta(&recv[blk], peer));
      else
        got = 0;
    }
    got = __shfl_sync(0xffffffffu, got, 0);

    // 2. This warp's own columns: partner's partial + own, scaled, fp16.
    named_barrier_sync(1, 32 * kPkEpiWarps);  // s_W staged
    int in = 0;
    if (lane == 0 && got) in = mbar_wait_cluster(&recv[blk], 0, p.err, DEVERR_TIMEOUT_CLUSTER);
    in = __shfl_sync(0xffffffffu, in, 0);
    if (in) {
      const int ocol = own0 + g * C::kSubCols;   // tile column of this warp's first value
      const int lcol = g * C::kSubCols;          // the same within the own half
      const uint8_t* src = base + C::kRecvOff + blk * C::kBlkBytes + lane * C::kBlkRow;
#pragma unroll
      for (int j = 0; j < C::kSubCols / 16; ++j) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(t_lane + ocol + j * 16, r);
        tmem_wait_ld();
        float y[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + (j * 16 + e) * 4);
          const float4 w4 = *reinterpret_cast<const float4*>(sw_s + lcol + j * 16 + e);
          // (float)A = fl(P_c + P_peer): both exact integers of at most 2^24.
          y[e + 0] = (__uint_as_float(r[e + 0]) + __uint_as_float(v.x)) * sx * w4.x;
          y[e + 1] = (__uint_as_float(r[e + 1]) + __uint_as_float(v.y)) * sx * w4.y;
          y[e + 2] = (__uint_as_float(r[e + 2]) + __uint_as_float(v.z)) * sx * w4.z;
          y[e + 3] = (__uint_as_float(r[e + 3]) + __uint_as_float(v.w)) * sx * w4.w;
        }
        // Box (64 columns) and 16-byte chunks of these 16 columns.
        const int bc = lcol + j * 16;
        uint8_t* box = base + C::kYOff + (bc / 64) * (kPkBM * 128);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int chunk = ((bc % 64) >> 3) + h;
          uint4 o;
          o.x = pack_half2(y[h * 8 + 0], y[h * 8 + 1]);
          o.y = pack_half2(y[h * 8 + 2], y[h * 8 + 3]);
          o.z = pack_half2(y[h * 8 + 4], y[h * 8 + 5]);
          o.w = pack_half2(y[h * 8 + 6], y[h * 8 + 7]);
          *reinterpret_cast<uint4*>(box + row * 128 + ((chunk ^ (row & 7)) << 4)) = o;
        }
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    // The partner's block has been consumed: the copy that filled it is done
    // reading the partner's staging.
    if (lane == 0 && in) mbar_arrive_remote(map_to_cta(peer_read, peer));
    // A box is written by the warps of its column group (BN = 256: one box
    // per group) or by all eight (BN = 128: one box).
    const bool wrote = !named_barrier_or(2, 32 * kPkEpiWarps, !in);
    if (wrote) {
      const bool issuer = lane == 0 && (C::kYBoxes == 2 ? q == 0 : warp == 2);
      if (issuer) {
        const int b = (C::kYBoxes == 2) ? g : 0;
        const int x = n0 + own0 + b * 64;
        if (x < p.N && m0 < p.M) tma_store_2d(&tm_y, base + C::kYOff + b * (kPkBM * 128), x, m0);
        tma_store_commit();
        tma_store_wait_read();
      }
    }
  }

  // Before this CTA's shared memory goes away, the partner's remote arrivals
  // on it must have landed; the copies into it completed on recv[] above.
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 64) {
    mbar_wait_cluster(peer_free, 0, p.err, DEVERR_TIMEOUT_CLUSTER);
    mbar_wait_cluster(peer_read, 0, p.err, DEVERR_TIMEOUT_CLUSTER);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, BN);
  }
}

template <int BN>
cudaError_t launch_pk(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_y,
                      const GemmTcArgs& a, cudaStream_t stream) {
  using C = PkCfg<BN>;
  auto fn = gemm_pairk_kernel<BN>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmem));
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + kPkBM - 1) / kPkBM) * ((a.N + BN - 1) / BN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * tiles);
  cfg.blockDim = dim3(kPkThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, tm_a, tm_b, tm_y, a);
}

}  // namespace

cudaError_t launch_gemm_pairk(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                              const CUtensorMap& tm_y, const GemmTcArgs& a, int bn,
                              cudaStream_t stream) {
  if (a.K % 256 != 0 || a.K > 2048 || a.tma_store != 1 || a.ep.mode != kOutF16 || a.ep.R != 0 ||
      a.ep.bias != nullptr || a.ep.out_bf16 != 0)
    return cudaErrorInvalidValue;
  switch (bn) {
    case 256: return launch_pk<256>(tm_a, tm_b, tm_y, a, stream);
    case 128: return launch_pk<128>(tm_a, tm_b, tm_y, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace convrot
