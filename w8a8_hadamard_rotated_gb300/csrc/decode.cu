// The whole small-M layer (M <= 16) in one kernel: rotate + quantize + exact
// int8 product + scale restore (page "INT8ConvRot GEMM vs fp16 on M1 Max with
// Metal, MPSMatrix, and MLX", section "What changed in the computation":
// X_rot = X H, s_X = max|X_rot| / 127 per row, Q_X = round(X_rot / s_X),
// A = Q_X Q_W^T, Y = A (.) s_X s_W^T).
//
// At M <= 16 a layer is a stream over the int8 weight.  Done as two kernels
// (rotate + quantize, then a small-M GEMM) it pays two kernel boundaries and
// a hand-off through global memory; and a weight stream through 16-byte
// register loads is capped by the misses one SM can keep in flight (a
// fraction of HBM's rate).  Here one launch does the layer and the weight
// moves by bulk asynchronous copies:
//   * A CTA owns 32 output columns and one K slice (a multiple of 256, at
//     most 4096); the slices of a column block are the CTAs of one
//     thread-block cluster.  Four compute warps and one copy warp.
//   * The copy warp moves the CTA's 32 weight rows of the slice into shared
//     memory, one bulk copy per row on one mbarrier.  With `weights_early`
//     it does so before the dependency wait: a layer's weight is not written
//     by the kernel ahead of it, so the stream overlaps that kernel's tail
//     and the launch gap instead of following them.  Without it the copies
//     follow the wait (an L2 prefetch of the slice goes ahead of it).
//   * After the wait every compute warp takes its (row, 256-group) items of
//     X -- up to 4 per warp straight from global memory, more from a tile
//     that the copy warp brings into shared memory ahead of the weight --
//     rotates them (3 butterfly stages in registers, 5 across lanes; lane
//     l holds elements 8l..8l+7) and keeps each row's max |x_rot| over the
//     slice.  Up to 4 items per warp stay in registers for the quantize step;
//     more are transformed again.
//   * The CTAs of the cluster push their row maxima to each other in
//     distributed shared memory (one barrier); every CTA then has the whole
//     row's max, the same s_X and the same 127 / max, and quantizes its slice
//     into int8 codes in shared memory (one fused multiply-add against a
//     magic constant, the prologue's rounding).
//   * The product once the weight has landed, on 4-way int8 dot products
//     (dp4a, exact in int32): lane c owns output column n0 + c, warp w a
//     quarter of the slice; the code bytes are read by all lanes at once
//     (one broadcast).  At M <= 16 this beats the tensor path available to
//     int8 here (mma.sync m16n8k32 pads the M rows to 16 and runs at the
//     legacy rate).  Partial sums are added over the warps in shared memory
//     and over the cluster by integer atomic adds into rank 0 (exact, so the
//     result does not depend on their order); rank 0 restores the scales
//     ((float)A * s_X) * s_W -> fp16.
// No workspace, no global scratch.  fp16 X and Y, no LoRA, no bias (other
// calls take the two-kernel path).  The codes, scales and Y are bit for bit
// those of the two-kernel path.
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "fwht.cuh"
#include "kernels.h"

namespace convrot {
namespace {

constexpr int kDecWarps = 4;        // compute warps; warp 4 copies the weight
constexpr int kDecThreads = (kDecWarps + 1) * 32;
constexpr int kDecCols = 32;        // output columns per CTA (4 n8 tiles)
constexpr int kDecHold = 4;         // (row, group) items a warp keeps in registers
constexpr int kDecMaxSlice = kDecodeMaxSlice;

// Row pitch of the weight tile in shared memory: the 16-byte pad puts the
// rows that 8 lanes read at the same K on different banks.
__host__ __device__ constexpr int dec_stride(int slice) { return slice + 16; }
// Dynamic shared memory: codes [M][slice] int8 | weight [32][stride] int8 |
// X [M][slice] fp16 | red [16][32] int32 | rmax_in [8][16] int32 | two
// mbarriers (weight, X).
__host__ __device__ constexpr size_t dec_smem(int M, int slice) {
  return static_cast<size_t>(M) * slice + static_cast<size_t>(32) * dec_stride(slice) +
         static_cast<size_t>(2) * M * slice + 16 * kDecCols * 4 + 8 * 16 * 4 + 16;
}

// Global -> this CTA's shared memory, completing as transaction bytes on
// `bar` (both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Barrier 1 among the compute warps only (the copy warp may still be
// issuing).
__device__ __forceinline__ void compute_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
}

__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int32_t v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_cluster_add_s32(uint32_t addr, int32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.s32 [%0], %1;" ::"r"(addr), "r"(v)
               : "memory");
}

// NB (1, 2 or 4) of this warp's (row, 256-group) items at once, it0 + 4j
// (j < NB; four compute warps take turns), from
// the X tile in shared memory (row pitch xstride halves): their butterfly
// stages interleaved so that the cross-lane steps of one item overlap the
// others' (each item alone is a chain of dependent shuffles).  An item past
// `items` (it0 itself may be, when a row has fewer items than there are
// warps) is computed on item 0's data and not used, so that every load stays
// inside X's M rows.
template <int NB>
__device__ __forceinline__ void fwht_items(const uint16_t* xs, int xstride, int groups, int items,
                                           int it0, int lane, uint32_t sbits, float (&v)[4][8]) {
  uint4 raw[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    int it = it0 + kDecWarps * j;
    it = it < items ? it : 0;
    raw[j] = *reinterpret_cast<const uint4*>(xs + (it / groups) * xstride + (it % groups) * 256 +
                                             lane * 8);
  }
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw[j]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h2[e]);
      v[j][2 * e] = f.x;
      v[j][2 * e + 1] = f.y;
    }
    apply_signs<8>(v[j], sbits);
    fwht_regs<8>(v[j]);
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1)
#pragma unroll
    for (int j = 0; j < NB; ++j) fwht_xlane<8>(v[j], lane, m);
}

// max |v| of each of the NB items over the warp, into its row's slot
// (fp32 bit patterns of non-negative values order like ints).
template <int NB>
__device__ __forceinline__ void row_max_items(const float (&v)[4][8], int groups, int items, int it0,
                                              int lane, int* rmax) {
  float a[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    a[j] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a[j] = fmaxf(a[j], fabsf(v[j][i]));
  }
#pragma unroll
  for (int s = 1; s < 32; s <<= 1)
#pragma unroll
    for (int j = 0; j < NB; ++j) a[j] = fmaxf(a[j], __shfl_xor_sync(0xffffffffu, a[j], s));
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (it0 + kDecWarps * j < items) atomicMax(&rmax[(it0 + kDecWarps * j) / groups], __float_as_int(a[j]));
}

__device__ __forceinline__ void quantize_store(const float (&v)[8], float inv, int8_t* dst) {
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = round_magic(v[i], inv);
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(codes_s8x4(r[0], r[1], r[2], r[3]), codes_s8x4(r[4], r[5], r[6], r[7]));
}

// MR rows of codes [MR][slice] against one weight row (this lane's column):
// warp w takes bytes [w q, (w + 1) q) of the slice (q = slice / 4, a
// multiple of 64), 16 * U at a time with U independent sums per row; the
// sums are added into red[m][column] (red points at the column).
template <int MR>
__device__ __forceinline__ void dot_rows(const int8_t* codes, const int8_t* wrow, int slice,
                                         int warp, int32_t* red) {
  constexpr int U = MR <= 2 ? 4 : (MR <= 4 ? 2 : 1);
  int32_t acc[MR][U];
#pragma unroll
  for (int m = 0; m < MR; ++m)
#pragma unroll
    for (int u = 0; u < U; ++u) acc[m][u] = 0;
  const int q = slice / kDecWarps;
  for (int k = warp * q; k < (warp + 1) * q; k += 16 * U) {
    int4 b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) b[u] = *reinterpret_cast<const int4*>(wrow + k + 16 * u);
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int4 a = *reinterpret_cast<const int4*>(codes + m * slice + k + 16 * u);
        acc[m][u] = __dp4a(a.x, b[u].x, acc[m][u]);
        acc[m][u] = __dp4a(a.y, b[u].y, acc[m][u]);
        acc[m][u] = __dp4a(a.z, b[u].z, acc[m][u]);
        acc[m][u] = __dp4a(a.w, b[u].w, acc[m][u]);
      }
  }
  // Over U and the warps (integer adds: exact in any order).
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    int32_t t = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) t += acc[m][u];
    atomicAdd(&red[m * kDecCols], t);
  }
}

template <int kMaxM>
__global__ void __launch_bounds__(kDecThreads) decode_layer_kernel(const __grid_constant__ DecodeArgs p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ int rmax_loc[16];
  __shared__ float inv_s[16];
  __shared__ float sx_s[16];
  const int slice = p.k_per_split;
  const int stride = dec_stride(slice);
  int8_t* codes = reinterpret_cast<int8_t*>(dsm);
  int8_t* wq = codes + p.M * slice;
  uint16_t* xs = reinterpret_cast<uint16_t*>(wq + 32 * stride);
  int32_t* red = reinterpret_cast<int32_t*>(xs + p.M * slice);
  int32_t* rmax_in = red + 16 * kDecCols;
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(rmax_in + 8 * 16);
  uint64_t* bar_x = bar_w + 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cs = p.splits;
  const uint32_t rank = cluster_ctarank();  // = this CTA's K slice
  const int n0 = static_cast<int>(blockIdx.x / cs) * kDecCols;
  const int rows = min(kDecCols, p.N - n0);  // weight rows this CTA holds
  const int k_begin = static_cast<int>(rank) * slice;
  const int groups = slice / 256;  // 256-groups of the slice
  const int8_t* wsrc = p.QW + static_cast<int64_t>(n0) * p.K + k_begin;
  // One slice per row: the CTA's own max is the row's.  Otherwise the
  // slices' maxima are exchanged in the cluster.  (Each CTA rotating the
  // whole rows instead measured slower even at a few 256-groups per row.)
  const bool local_max = cs == 1;

  for (int i = threadIdx.x; i < 16 * kDecCols; i += blockDim.x) red[i] = 0;
  if (threadIdx.x < 16) rmax_loc[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_x, 1);
    fence_mbarrier_init();
  }
  // First half of the cluster barrier after which other CTAs' shared memory
  // may be written: every CTA has started, and rank 0's red[] is zero.
  if (cs > 1) cluster_arrive_release();
  if (warp == kDecWarps) {
    // L2 prefetches ahead of the wait (they return nothing to the SM, so the
    // previous kernel's writes to X are still what the loads below see).
    if (lane < p.M) {
      bulk_prefetch_l2(p.X + static_cast<int64_t>(lane) * p.K + k_begin,
                       static_cast<uint32_t>(slice) * 2);
    }
    if (!p.weights_early && lane < rows)
      bulk_prefetch_l2(wsrc + static_cast<int64_t>(lane) * p.K, slice);
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // The copy warp: the X tile (lane m: row m of the slice, after the
    // dependency wait) and the weight (lane r: row n0 + r of the slice,
    // before the wait with `weights_early`, else after the X tile).
    // Items held in registers read X straight from global memory (a few
    // loads per lane); otherwise X comes as a tile.
    const bool x_tile = p.M * (slice / 256) > kDecWarps * kDecHold;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_w, rows * slice);
      mbar_arrive_expect_tx(bar_x, x_tile ? p.M * slice * 2 : 0);
    }
    __syncwarp();
    if (p.weights_early && lane < rows)
      bulk_load(wq + lane * stride, wsrc + static_cast<int64_t>(lane) * p.K, slice, bar_w);
    grid_dep_wait();
    if (x_tile && lane < p.M)
      bulk_load(xs + lane * slice, p.X + static_cast<int64_t>(lane) * p.K + k_begin, slice * 2, bar_x);
    // It takes part in the cluster barriers and nothing else; its arrival at
    // the row-max barrier goes ahead of the weight copies, which may wait for
    // room in the copy engine.
    if (cs > 1) {
      cluster_wait_acquire();
      cluster_arrive_release();
    }
    if (!p.weights_early && lane < rows)
      bulk_load(wq + lane * stride, wsrc + static_cast<int64_t>(lane) * p.K, slice, bar_w);
    grid_dep_launch();
    if (cs > 1) {
      cluster_wait_acquire();
      cluster_arrive_release();
      if (rank == 0) cluster_wait_acquire();
    }
    return;
  }

  grid_dep_wait();  // s_W is read below (X comes through the copy warp)
  grid_dep_launch();
  // A copy that has not landed must not outlive the CTA: a wait that ran out
  // is taken once more (its own limit) before going on.
  if (!mbar_wait(bar_x, 0, p.err, DEVERR_TIMEOUT_FULL))
    mbar_wait(bar_x, 0, p.err, DEVERR_TIMEOUT_DRAIN);

  // 1. Row maxima.  (The parameter is __grid_constant__: the indexed read of
  // its sign words stays in parameter space.)
  const uint32_t sbits = (p.sign[lane >> 2] >> ((lane & 3) * 8)) & 0xffu;
  const int items = p.M * groups;
  const bool hold = items <= kDecWarps * kDecHold;  // one batch per warp
  float v[kDecHold][8];
  if (hold) {
    // As many items per warp as there are (1, 2 or 4 at a time).
    const int nb = (items + kDecWarps - 1) / kDecWarps;
    if (nb == 1) {
      fwht_items<1>(p.X + k_begin, p.K, groups, items, warp, lane, sbits, v);
      row_max_items<1>(v, groups, items, warp, lane, rmax_loc);
    } else if (nb == 2) {
      fwht_items<2>(p.X + k_begin, p.K, groups, items, warp, lane, sbits, v);
      row_max_items<2>(v, groups, items, warp, lane, rmax_loc);
    } else {
      fwht_items<4>(p.X + k_begin, p.K, groups, items, warp, lane, sbits, v);
      row_max_items<4>(v, groups, items, warp, lane, rmax_loc);
    }
  } else {
    for (int it0 = warp; it0 < items; it0 += kDecWarps * kDecHold) {
      float w[kDecHold][8];
      fwht_items<4>(xs, slice, groups, items, it0, lane, sbits, w);
      row_max_items<4>(w, groups, items, it0, lane, rmax_loc);
    }
  }
  compute_sync();
  if (!local_max) {
    // 2. The slices' maxima: each CTA writes its own into slot `rank` of
    // every CTA of the cluster, then one barrier publishes them.
    cluster_wait_acquire();  // every CTA has started
    if (threadIdx.x < cs * 16) {
      const int q = threadIdx.x >> 4, m = threadIdx.x & 15;
      if (m < p.M)
        st_cluster_s32(map_to_cta(&rmax_in[rank * 16 + m], static_cast<uint32_t>(q)), rmax_loc[m]);
    }
    cluster_sync_all();
  }
  if (threadIdx.x < p.M) {
    int a = rmax_loc[threadIdx.x];
    if (!local_max)
      for (int q = 0; q < cs; ++q) a = max(a, rmax_in[q * 16 + threadIdx.x]);
    const float amax = __int_as_float(a);
    sx_s[threadIdx.x] = (amax * 0.0625f) / 127.0f;  // x 1/16 is exact
    inv_s[threadIdx.x] = amax > 0.0f ? 127.0f / amax : 0.0f;
  }
  compute_sync();

  // 3. Quantize the slice into codes[m][k].
  if (hold) {
#pragma unroll
    for (int i = 0; i < kDecHold; ++i) {
      const int it = warp + kDecWarps * i;
      if (it < items) {
        const int m = it / groups;
        quantize_store(v[i], inv_s[m], codes + m * slice + (it % groups) * 256 + lane * 8);
      }
    }
  } else {
    for (int it0 = warp; it0 < items; it0 += kDecWarps * kDecHold) {
      float w[kDecHold][8];
      fwht_items<4>(xs, slice, groups, items, it0, lane, sbits, w);
#pragma unroll
      for (int j = 0; j < kDecHold; ++j) {
        const int it = it0 + kDecWarps * j;
        if (it < items) {
          const int m = it / groups;
          quantize_store(w[j], inv_s[m], codes + m * slice + (it % groups) * 256 + lane * 8);
        }
      }
    }
  }
  compute_sync();

  // 4. The product (lane c: weight row n0 + c).
  if (!mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_FULL))
    mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_DRAIN);
  const int8_t* wrow = wq + lane * stride;
  if (kMaxM <= 4) {
    switch (p.M) {
      case 1: dot_rows<1>(codes, wrow, slice, warp, red + lane); break;
      case 2: dot_rows<2>(codes, wrow, slice, warp, red + lane); break;
      case 3: dot_rows<3>(codes, wrow, slice, warp, red + lane); break;
      default: dot_rows<4>(codes, wrow, slice, warp, red + lane); break;
    }
  } else {
    switch (p.M) {
      case 5: dot_rows<5>(codes, wrow, slice, warp, red + lane); break;
      case 6: dot_rows<6>(codes, wrow, slice, warp, red + lane); break;
      case 7: dot_rows<7>(codes, wrow, slice, warp, red + lane); break;
      case 8: dot_rows<8>(codes, wrow, slice, warp, red + lane); break;
      case 9: dot_rows<9>(codes, wrow, slice, warp, red + lane); break;
      case 10: dot_rows<10>(codes, wrow, slice, warp, red + lane); break;
      case 11: dot_rows<11>(codes, wrow, slice, warp, red + lane); break;
      case 12: dot_rows<12>(codes, wrow, slice, warp, red + lane); break;
      case 13: dot_rows<13>(codes, wrow, slice, warp, red + lane); break;
      case 14: dot_rows<14>(codes, wrow, slice, warp, red + lane); break;
      case 15: dot_rows<15>(codes, wrow, slice, warp, red + lane); break;
      default: dot_rows<16>(codes, wrow, slice, warp, red + lane); break;
    }
  }
  compute_sync();
  if (cs > 1) {
    // Over the cluster: ranks > 0 add their sums into rank 0's red[] (zeroed
    // before the first barrier, which they have waited for), arrive
    // (releasing their adds) and leave; rank 0 waits for them.
    if (rank != 0)
      for (int i = threadIdx.x; i < p.M * kDecCols; i += kDecWarps * 32)
        red_cluster_add_s32(map_to_cta(&red[i], 0), red[i]);
    cluster_arrive_release();
    if (rank != 0) return;
    cluster_wait_acquire();
  }
  // Scale restore ((float)A * s_X) * s_W, fp16 out.
  for (int i = threadIdx.x; i < p.M * kDecCols; i += kDecWarps * 32) {
    const int m = i / kDecCols, c = i % kDecCols;
    const int n = n0 + c;
    if (n < p.N) {
      const float y = (static_cast<float>(red[i]) * sx_s[m]) * p.sW[n];
      p.Y[static_cast<int64_t>(m) * p.N + n] = __half_as_ushort(__float2half_rn(y));
    }
  }
}


// ---------------------------------------------------------------------------
// The same layer with the product on the fp16 warp MMA (mma.sync m16n8k16,
// fp32 accumulation), for M from 3 to 16.  Here the legacy fp16 MMA runs at
// four times the int8 MMA's and dp4a's rate; its operands hold the int8
// values exactly (the weight widened in registers, the codes written as fp16
// by the quantize step), each product is exact, and an fp32 sum of at most
// 1024 of them (|sum| <= 2^24) is exact, so the sums are moved to int32
// every 1024 K and the result is the integer product, bit for bit.
//   * A CTA owns 128 weight rows (output columns) and a K slice of at most
//     1024: four times fewer CTAs repeat the rotation than with 32 columns.
//   * Warp w owns weight rows 32w .. 32w + 31 (two m16 tiles) over the whole
//     slice and all M rows (one or two n8 tiles), so no sums are shared
//     inside the CTA.
//   * K order inside each 64-byte step: lane t of a quad reads bytes
//     16t .. 16t + 15 of its weight rows and the fp16 codes of the same K
//     positions; k16 sub-block s takes the lane's bytes 4s .. 4s + 3 as the
//     MMA's K indices 2t, 2t+1, 2t+8, 2t+9 on both operands (any K order
//     shared by the operands gives the same sum).
// ---------------------------------------------------------------------------
constexpr int kDmRows = 128;
constexpr int kDmMaxSlice = 1024;

// Weight row pitch (bytes): the 64-byte pad puts the two rows a quarter-warp
// reads on different banks.  Code row pitch (halves): the 8-half pad does
// the same for the codes.
__host__ __device__ constexpr int dm_wstride(int slice) { return slice + 64; }
__host__ __device__ constexpr int dm_cstride(int slice) { return slice + 8; }
// Dynamic shared memory: weight [128][wstride] int8 | X, then codes [16]
// [cstride] fp16 | red [16][128] int32 | rmax_in [8][16] int32 | two
// mbarriers (weight, X).
__host__ __device__ constexpr size_t dm_smem(int slice) {
  return static_cast<size_t>(kDmRows) * dm_wstride(slice) +
         static_cast<size_t>(16) * dm_cstride(slice) * 2 + 16 * kDmRows * 4 + 8 * 16 * 4 + 16;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four int8 values (one word) -> two fp16 pairs (bytes 0,1 and 2,3), exact:
// 0x64 above the biased byte is the fp16 1024 + (v + 128); minus 1152 is v.
__device__ __forceinline__ void widen_i8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t y = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(y, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(y, 0x64646464u, 0x4342);
  const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), k1152);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), k1152);
  lo = *reinterpret_cast<const uint32_t*>(&rl);
  hi = *reinterpret_cast<const uint32_t*>(&rh);
}

__device__ __forceinline__ void quantize_store_f16(const float (&v)[8], float inv, uint16_t* dst) {
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = round_magic(v[i], inv);
  *reinterpret_cast<uint4*>(dst) = make_uint4(codes_f16x2(r[0], r[1]), codes_f16x2(r[2], r[3]),
                                              codes_f16x2(r[4], r[5]), codes_f16x2(r[6], r[7]));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// kNT: n8 tiles of M rows (1: M <= 8, 2: M <= 16).
template <int kNT>
__global__ void __launch_bounds__(kDecThreads) decode_mma_kernel(const __grid_constant__ DecodeArgs p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ int rmax_loc[16];
  __shared__ float inv_s[16];
  __shared__ float sx_s[16];
  const int slice = p.k_per_split;
  const int wstride = dm_wstride(slice);
  const int cstride = dm_cstride(slice);
  int8_t* wq = reinterpret_cast<int8_t*>(dsm);
  // The X tile arrives in the code rows (same pitch); the quantize step
  // writes each item's codes over its X.
  uint16_t* codes = reinterpret_cast<uint16_t*>(wq + kDmRows * wstride);
  uint16_t* xs = codes;
  int32_t* red = reinterpret_cast<int32_t*>(codes + 16 * cstride);
  int32_t* rmax_in = red + 16 * kDmRows;
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(rmax_in + 8 * 16);
  uint64_t* bar_x = bar_w + 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cs = p.splits;
  const uint32_t rank = cluster_ctarank();  // = this CTA's K slice
  const int n0 = static_cast<int>(blockIdx.x / cs) * kDmRows;
  const int rows = min(kDmRows, p.N - n0);  // weight rows this CTA holds
  const int k_begin = static_cast<int>(rank) * slice;
  const int groups = slice / 256;
  const int8_t* wsrc = p.QW + static_cast<int64_t>(n0) * p.K + k_begin;
  const bool local_max = cs == 1;

  for (int i = threadIdx.x; i < 16 * kDmRows; i += blockDim.x) red[i] = 0;
  if (threadIdx.x < 16) rmax_loc[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_x, 1);
    fence_mbarrier_init();
  }
  // First half of the cluster barrier after which other CTAs' shared memory
  // may be written: every CTA has started, and rank 0's red[] is zero.
  if (cs > 1) cluster_arrive_release();
  if (warp == kDecWarps) {
    // L2 prefetches ahead of the wait (they return nothing to the SM).
    if (lane < p.M)
      bulk_prefetch_l2(p.X + static_cast<int64_t>(lane) * p.K + k_begin,
                       static_cast<uint32_t>(slice) * 2);
    if (!p.weights_early)
      for (int r = lane; r < rows; r += 32) bulk_prefetch_l2(wsrc + static_cast<int64_t>(r) * p.K, slice);
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // The copy warp: the X tile (lane m: row m of the slice, after the
    // dependency wait) and the weight (lane l: rows l, l + 32, l + 64, l + 96
    // of the slice, before the wait with `weights_early`, else after the X
    // tile).
    // Items held in registers read X straight from global memory (a few
    // loads per lane); otherwise X comes as a tile.
    const bool x_tile = p.M * (slice / 256) > kDecWarps * kDecHold;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_w, rows * slice);
      mbar_arrive_expect_tx(bar_x, x_tile ? p.M * slice * 2 : 0);
    }
    __syncwarp();
    if (p.weights_early)
      for (int r = lane; r < rows; r += 32)
        bulk_load(wq + r * wstride, wsrc + static_cast<int64_t>(r) * p.K, slice, bar_w);
    grid_dep_wait();
    if (x_tile && lane < p.M)
      bulk_load(xs + lane * cstride, p.X + static_cast<int64_t>(lane) * p.K + k_begin, slice * 2,
                bar_x);
    // Its arrival at the row-max barrier goes ahead of the weight copies,
    // which may wait for room in the copy engine.
    if (cs > 1) {
      cluster_wait_acquire();
      cluster_arrive_release();
    }
    if (!p.weights_early)
      for (int r = lane; r < rows; r += 32)
        bulk_load(wq + r * wstride, wsrc + static_cast<int64_t>(r) * p.K, slice, bar_w);
    grid_dep_launch();
    if (cs > 1) {
      cluster_wait_acquire();
      cluster_arrive_release();
      if (rank == 0) cluster_wait_acquire();
    }
    return;
  }

  grid_dep_wait();  // s_W is read below (X comes through the copy warp)
  grid_dep_launch();
  // A copy that has not landed must not outlive the CTA: a wait that ran out
  // is taken once more (its own limit) before going on.
  if (!mbar_wait(bar_x, 0, p.err, DEVERR_TIMEOUT_FULL))
    mbar_wait(bar_x, 0, p.err, DEVERR_TIMEOUT_DRAIN);

  // 1. Row maxima over the slice (as in decode_layer_kernel).
  const uint32_t sbits = (p.sign[lane >> 2] >> ((lane & 3) * 8)) & 0xffu;
  const int items = p.M * groups;
  const bool hold = items <= kDecWarps * kDecHold;  // one batch per warp
  float v[kDecHold][8];
  if (hold) {
    // As many items per warp as there are (1, 2 or 4 at a time).
    const int nb = (items + kDecWarps - 1) / kDecWarps;
    if (nb == 1) {
      fwht_items<1>(p.X + k_begin, p.K, groups, items, warp, lane, sbits, v);
      row_max_items<1>(v, groups, items, warp, lane, rmax_loc);
    } else if (nb == 2) {
      fwht_items<2>(p.X + k_begin, p.K, groups, items, warp, lane, sbits, v);
      row_max_items<2>(v, groups, items, warp, lane, rmax_loc);
    } else {
      fwht_items<4>(p.X + k_begin, p.K, groups, items, warp, lane, sbits, v);
      row_max_items<4>(v, groups, items, warp, lane, rmax_loc);
    }
  } else {
    for (int it0 = warp; it0 < items; it0 += kDecWarps * kDecHold) {
      float w[kDecHold][8];
      fwht_items<4>(xs, cstride, groups, items, it0, lane, sbits, w);
      row_max_items<4>(w, groups, items, it0, lane, rmax_loc);
    }
  }
  compute_sync();
  if (!local_max) {
    // 2. The slices' maxima, pushed to every CTA of the cluster.
    cluster_wait_acquire();  // every CTA has started
    if (threadIdx.x < cs * 16) {
      const int q = threadIdx.x >> 4, m = threadIdx.x & 15;
      if (m < p.M)
        st_cluster_s32(map_to_cta(&rmax_in[rank * 16 + m], static_cast<uint32_t>(q)), rmax_loc[m]);
    }
    cluster_sync_all();
  }
  if (threadIdx.x < p.M) {
    int a = rmax_loc[threadIdx.x];
    if (!local_max)
      for (int q = 0; q < cs; ++q) a = max(a, rmax_in[q * 16 + threadIdx.x]);
    const float amax = __int_as_float(a);
    sx_s[threadIdx.x] = (amax * 0.0625f) / 127.0f;  // x 1/16 is exact
    inv_s[threadIdx.x] = amax > 0.0f ? 127.0f / amax : 0.0f;
  }
  compute_sync();

  // 3. Quantize into the fp16 code image codes[m][k].  Rows M .. 8 kNT - 1
  // are never written: they reach only output rows that are dropped.
  if (hold) {
#pragma unroll
    for (int i = 0; i < kDecHold; ++i) {
      const int it = warp + kDecWarps * i;
      if (it < items) {
        const int m = it / groups;
        quantize_store_f16(v[i], inv_s[m], codes + m * cstride + (it % groups) * 256 + lane * 8);
      }
    }
  } else {
    // In place: a batch reads its items' X before writing their codes over
    // them, and no other item reads them.
    for (int it0 = warp; it0 < items; it0 += kDecWarps * kDecHold) {
      float w[kDecHold][8];
      fwht_items<4>(xs, cstride, groups, items, it0, lane, sbits, w);
#pragma unroll
      for (int j = 0; j < kDecHold; ++j) {
        const int it = it0 + kDecWarps * j;
        if (it < items) {
          const int m = it / groups;
          quantize_store_f16(w[j], inv_s[m], codes + m * cstride + (it % groups) * 256 + lane * 8);
        }
      }
    }
  }
  compute_sync();

  // 4. The product.
  if (!mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_FULL))
    mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_DRAIN);
  const int g = lane >> 2, t = lane & 3;
  float acc[2][kNT][4];
  int32_t tot[2][kNT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f, tot[mt][nt][e] = 0;
  const int8_t* wrow = wq + (32 * warp + g) * wstride + 16 * t;
  const uint16_t* crow = codes + g * cstride + 16 * t;
  for (int k = 0; k < slice; k += 64) {
    uint4 wa[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      wa[mt][0] = *reinterpret_cast<const uint4*>(wrow + (16 * mt) * wstride + k);
      wa[mt][1] = *reinterpret_cast<const uint4*>(wrow + (16 * mt + 8) * wstride + k);
    }
    uint4 cb[kNT][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      cb[nt][0] = *reinterpret_cast<const uint4*>(crow + 8 * nt * cstride + k);
      cb[nt][1] = *reinterpret_cast<const uint4*>(crow + 8 * nt * cstride + k + 8);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t a0, a1, a2, a3;
        widen_i8x4(word_of(wa[mt][0], s), a0, a2);  // row g: K 2t, 2t+1 | 2t+8, 2t+9
        widen_i8x4(word_of(wa[mt][1], s), a1, a3);  // row g + 8
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          mma_f16(acc[mt][nt], a0, a1, a2, a3, word_of(cb[nt][s >> 1], (s & 1) * 2),
                  word_of(cb[nt][s >> 1], (s & 1) * 2 + 1));
      }
    }
    if (((k + 64) & 1023) == 0 || k + 64 == slice) {
      // At most 1024 K since the last move: each sum is an exact integer.
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            tot[mt][nt][e] += static_cast<int32_t>(acc[mt][nt][e]);
            acc[mt][nt][e] = 0.0f;
          }
    }
  }
  // D[row][m]: rows 32w + 16mt + g (+8), m = 8nt + 2t (+1).
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = 32 * warp + 16 * mt + g + (e >= 2 ? 8 : 0);
        const int m = 8 * nt + 2 * t + (e & 1);
        if (m < p.M) atomicAdd(&red[m * kDmRows + r], tot[mt][nt][e]);
      }
  compute_sync();
  if (cs > 1) {
    if (rank != 0)
      for (int i = threadIdx.x; i < p.M * kDmRows; i += kDecWarps * 32)
        red_cluster_add_s32(map_to_cta(&red[i], 0), red[i]);
    cluster_arrive_release();
    if (rank != 0) return;
    cluster_wait_acquire();
  }
  // Scale restore ((float)A * s_X) * s_W, fp16 out.
  for (int i = threadIdx.x; i < p.M * kDmRows; i += kDecWarps * 32) {
    const int m = i / kDmRows, r = i % kDmRows;
    const int n = n0 + r;
    if (n < p.N) {
      const float y = (static_cast<float>(red[i]) * sx_s[m]) * p.sW[n];
      p.Y[static_cast<int64_t>(m) * p.N + n] = __half_as_ushort(__float2half_rn(y));
    }
  }
}


// ---------------------------------------------------------------------------
// The small-M GEMM of the two-kernel path on the same skeleton: 32 output
// columns per CTA, the prologue's int8 codes Q_X and the weight slice by bulk
// copies, the product on the fp16 warp MMA with both operands widened in
// registers (exact: int8 values, each warp's fp32 sum over at most 1024 K is
// an exact integer), the cluster's K slices summed into rank 0 as int32, the
// plain fp16 epilogue.  Warp w takes the K quarter [w q, (w + 1) q) of the
// slice for all 32 weight rows (two m16 tiles) and all M rows (one or two
// n8 tiles); the K order inside each 64-byte step is decode_mma_kernel's.
// ---------------------------------------------------------------------------
// Row pitch of both tiles: the 64-byte pad puts the two rows a quarter-warp
// reads on different banks.
__host__ __device__ constexpr int sg_stride(int slice) { return slice + 64; }
// Dynamic shared memory: weight [32][stride] int8 | codes [16][stride] int8 |
// red [16][32] int32 | two mbarriers.
__host__ __device__ constexpr size_t sg_smem(int slice) {
  return static_cast<size_t>(48) * sg_stride(slice) + 16 * kDecCols * 4 + 16;
}

template <int kNT>
__global__ void __launch_bounds__(kDecThreads) skinny_f16_kernel(const __grid_constant__ SkinnyF16Args p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  const int slice = p.k_per_split;
  const int stride = sg_stride(slice);
  int8_t* wq = reinterpret_cast<int8_t*>(dsm);
  int8_t* cq = wq + 32 * stride;
  int32_t* red = reinterpret_cast<int32_t*>(cq + 16 * stride);
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(red + 16 * kDecCols);
  uint64_t* bar_x = bar_w + 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cs = p.splits;
  const uint32_t rank = cluster_ctarank();  // = this CTA's K slice
  const int n0 = static_cast<int>(blockIdx.x / cs) * kDecCols;
  const int rows = min(kDecCols, p.N - n0);
  const int k_begin = static_cast<int>(rank) * slice;
  const int8_t* wsrc = p.QW + static_cast<int64_t>(n0) * p.K + k_begin;

  for (int i = threadIdx.x; i < 16 * kDecCols; i += blockDim.x) red[i] = 0;
  if (threadIdx.x == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_x, 1);
    fence_mbarrier_init();
  }
  // First half of the cluster barrier after which rank 0's red[] may be
  // added into: every CTA has started, and red[] is zero.
  if (cs > 1) cluster_arrive_release();
  if (warp == kDecWarps && !p.weights_early && lane < rows)
    bulk_prefetch_l2(wsrc + static_cast<int64_t>(lane) * p.K, slice);
  __syncthreads();

  if (warp == kDecWarps) {
    // The copy warp: the codes (lane m: row m of the slice, after the
    // dependency wait) and the weight (lane r: row n0 + r, before the wait
    // with `weights_early`, else after the codes).
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_w, rows * slice);
      mbar_arrive_expect_tx(bar_x, p.M * slice);
    }
    __syncwarp();
    if (p.weights_early && lane < rows)
      bulk_load(wq + lane * stride, wsrc + static_cast<int64_t>(lane) * p.K, slice, bar_w);
    grid_dep_wait();
    if (lane < p.M)
      bulk_load(cq + lane * stride, p.QX + static_cast<int64_t>(lane) * p.K + k_begin, slice, bar_x);
    if (!p.weights_early && lane < rows)
      bulk_load(wq + lane * stride, wsrc + static_cast<int64_t>(lane) * p.K, slice, bar_w);
    grid_dep_launch();
    if (cs > 1) {
      cluster_wait_acquire();
      cluster_arrive_release();
      if (rank == 0) cluster_wait_acquire();
    }
    return;
  }

  grid_dep_wait();  // s_X and s_W are read below (the codes come through the copy warp)
  grid_dep_launch();
  // A copy that has not landed must not outlive the CTA: a wait that ran out
  // is taken once more (its own limit) before going on.
  if (!mbar_wait(bar_x, 0, p.err, DEVERR_TIMEOUT_FULL))
    mbar_wait(bar_x, 0, p.err, DEVERR_TIMEOUT_DRAIN);
  if (!mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_FULL))
    mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_DRAIN);

  // The product.  Code rows M .. 8 kNT - 1 hold stale bytes: they reach only
  // output rows that are dropped.
  const int g = lane >> 2, t = lane & 3;
  float acc[2][kNT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f;
  const int q = slice / kDecWarps;  // a multiple of 64, at most 1024
  const int8_t* wrow = wq + g * stride + 16 * t;
  const int8_t* crow = cq + g * stride + 16 * t;
  for (int k = warp * q; k < (warp + 1) * q; k += 64) {
    uint4 wa[2][2], cb[kNT];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      wa[mt][0] = *reinterpret_cast<const uint4*>(wrow + (16 * mt) * stride + k);
      wa[mt][1] = *reinterpret_cast<const uint4*>(wrow + (16 * mt + 8) * stride + k);
    }
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) cb[nt] = *reinterpret_cast<const uint4*>(crow + 8 * nt * stride + k);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t b0[kNT], b1[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) widen_i8x4(word_of(cb[nt], s), b0[nt], b1[nt]);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t a0, a1, a2, a3;
        widen_i8x4(word_of(wa[mt][0], s), a0, a2);  // row g: K 2t, 2t+1 | 2t+8, 2t+9
        widen_i8x4(word_of(wa[mt][1], s), a1, a3);  // row g + 8
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) mma_f16(acc[mt][nt], a0, a1, a2, a3, b0[nt], b1[nt]);
      }
    }
  }
  // D[weight row][m]: rows 16mt + g (+8), m = 8nt + 2t (+1); over the warps
  // as exact int32 adds.
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 16 * mt + g + (e >= 2 ? 8 : 0);
        const int m = 8 * nt + 2 * t + (e & 1);
        if (m < p.M) atomicAdd(&red[m * kDecCols + c], static_cast<int32_t>(acc[mt][nt][e]));
      }
  compute_sync();
  if (cs > 1) {
    cluster_wait_acquire();  // every CTA has started; rank 0's red[] is zero
    if (rank != 0)
      for (int i = threadIdx.x; i < p.M * kDecCols; i += kDecWarps * 32)
        red_cluster_add_s32(map_to_cta(&red[i], 0), red[i]);
    cluster_arrive_release();
    if (rank != 0) return;
    cluster_wait_acquire();
  }
  for (int i = threadIdx.x; i < p.M * kDecCols; i += kDecWarps * 32) {
    const int m = i / kDecCols, c = i % kDecCols;
    const int n = n0 + c;
    if (n < p.N) {
      const float y = (static_cast<float>(red[i]) * p.sX[m]) * p.sW[n];
      p.Y[static_cast<int64_t>(m) * p.N + n] = __half_as_ushort(__float2half_rn(y));
    }
  }
}


// ---------------------------------------------------------------------------
// The one-kernel layer with the rotation shared by column blocks, for M up to
// 16: a cluster is `cs` K slices x `cn` column blocks of 32 outputs (rank r:
// slice r % cs, block r / cs).  Each CTA rotates only 1 / cn of its slice's
// 256-groups (its items stay in registers), the row maxima of all the
// cluster's CTAs are exchanged, and each CTA writes its share of the int8
// codes into the code tile of every CTA on the same slice (distributed
// shared memory), so every CTA holds the slice's codes after one rotation
// per cluster instead of one per column block.  The weight arrives by bulk
// copies (before the dependency wait with `weights_early`), the product is
// skinny_f16_kernel's (fp16 warp MMA on widened int8 values, exact), the
// slices' sums meet as int32 in the slice-0 CTA of each block, which
// restores the scales.  Four cluster barrier phases: A (every CTA started;
// red[] zeroed), B (row maxima), C (codes), D (sums).
// ---------------------------------------------------------------------------
__host__ __device__ constexpr size_t ds_smem(int slice) {
  return static_cast<size_t>(48) * sg_stride(slice) + 16 * kDecCols * 4 + 8 * 16 * 4 + 16;
}

__device__ __forceinline__ void st_cluster_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

template <int kNT>
__global__ void __launch_bounds__(kDecThreads) decode_shared_kernel(const __grid_constant__ DecodeArgs p,
                                                                   int cn) {
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ int rmax_loc[16];
  __shared__ float inv_s[16];
  __shared__ float sx_s[16];
  const int slice = p.k_per_split;
  const int stride = sg_stride(slice);
  int8_t* wq = reinterpret_cast<int8_t*>(dsm);
  int8_t* cq = wq + 32 * stride;
  int32_t* red = reinterpret_cast<int32_t*>(cq + 16 * stride);
  int32_t* rmax_in = red + 16 * kDecCols;
  uint64_t* bar_w = reinterpret_cast<uint64_t*>(rmax_in + 8 * 16);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cs = p.splits;
  const int csize = cs * cn;
  const uint32_t rank = cluster_ctarank();
  const int sidx = static_cast<int>(rank) % cs;  // K slice
  const int bidx = static_cast<int>(rank) / cs;  // column block within the cluster
  const int n0 = (static_cast<int>(blockIdx.x) / csize * cn + bidx) * kDecCols;
  const int rows = max(0, min(kDecCols, p.N - n0));
  const int k_begin = sidx * slice;
  const int share = (slice / 256) / cn;  // 256-groups this CTA rotates
  const int g0 = bidx * share;           // its first group within the slice
  const int8_t* wsrc = p.QW + static_cast<int64_t>(max(n0, 0)) * p.K + k_begin;

  for (int i = threadIdx.x; i < 16 * kDecCols; i += blockDim.x) red[i] = 0;
  if (threadIdx.x < 16) rmax_loc[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    mbar_init(bar_w, 1);
    fence_mbarrier_init();
  }
  cluster_arrive_release();  // A
  if (warp == kDecWarps && !p.weights_early && lane < rows)
    bulk_prefetch_l2(wsrc + static_cast<int64_t>(lane) * p.K, slice);
  __syncthreads();

  if (warp == kDecWarps) {
    if (lane == 0) mbar_arrive_expect_tx(bar_w, rows * slice);
    __syncwarp();
    if (p.weights_early && lane < rows)
      bulk_load(wq + lane * stride, wsrc + static_cast<int64_t>(lane) * p.K, slice, bar_w);
    grid_dep_wait();
    cluster_wait_acquire();   // A
    cluster_arrive_release();  // B, ahead of the weight copies (they may wait for the copy engine)
    if (!p.weights_early && lane < rows)
      bulk_load(wq + lane * stride, wsrc + static_cast<int64_t>(lane) * p.K, slice, bar_w);
    grid_dep_launch();
    cluster_wait_acquire();  // B
    cluster_sync_all();      // C
    cluster_arrive_release();  // D
    if (sidx == 0) cluster_wait_acquire();
    return;
  }

  grid_dep_wait();  // X may come from the previous kernel
  grid_dep_launch();

  // 1. This CTA's share of the rows' groups: rotate, keep, row maxima.
  const uint32_t sbits = (p.sign[lane >> 2] >> ((lane & 3) * 8)) & 0xffu;
  const int items = p.M * share;  // at most 16 (the host's choice of cn)
  const uint16_t* xs = p.X + k_begin + g0 * 256;
  float v[kDecHold][8];
  const int nb = (items + kDecWarps - 1) / kDecWarps;
  if (nb == 1) {
    fwht_items<1>(xs, p.K, share, items, warp, lane, sbits, v);
    row_max_items<1>(v, share, items, warp, lane, rmax_loc);
  } else if (nb == 2) {
    fwht_items<2>(xs, p.K, share, items, warp, lane, sbits, v);
    row_max_items<2>(v, share, items, warp, lane, rmax_loc);
  } else {
    fwht_items<4>(xs, p.K, share, items, warp, lane, sbits, v);
    row_max_items<4>(v, share, items, warp, lane, rmax_loc);
  }
  compute_sync();
  // 2. Every CTA's maxima into slot `rank` of every CTA of the cluster.
  cluster_wait_acquire();  // A: every CTA has started
  if (threadIdx.x < csize * 16) {
    const int q = threadIdx.x >> 4, m = threadIdx.x & 15;
    if (m < p.M)
      st_cluster_s32(map_to_cta(&rmax_in[rank * 16 + m], static_cast<uint32_t>(q)), rmax_loc[m]);
  }
  cluster_sync_all();  // B
  if (threadIdx.x < p.M) {
    int a = 0;
    for (int q = 0; q < csize; ++q) a = max(a, rmax_in[q * 16 + threadIdx.x]);
    const float amax = __int_as_float(a);
    sx_s[threadIdx.x] = (amax * 0.0625f) / 127.0f;  // x 1/16 is exact
    inv_s[threadIdx.x] = amax > 0.0f ? 127.0f / amax : 0.0f;
  }
  compute_sync();
  // 3. This share's codes into the code tile of every CTA on this slice.
#pragma unroll
  for (int i = 0; i < kDecHold; ++i) {
    const int it = warp + kDecWarps * i;
    if (it < items) {
      const int m = it / share;
      const float inv = inv_s[m];
      uint32_t r[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = round_magic(v[i][e], inv);
      const uint32_t lo = codes_s8x4(r[0], r[1], r[2], r[3]);
      const uint32_t hi = codes_s8x4(r[4], r[5], r[6], r[7]);
      int8_t* dst = cq + m * stride + (g0 + it % share) * 256 + lane * 8;
      for (int b = 0; b < cn; ++b)
        st_cluster_v2(map_to_cta(dst, static_cast<uint32_t>(b * cs + sidx)), lo, hi);
    }
  }
  cluster_sync_all();  // C: every CTA has the slice's codes

  // 4. The product (skinny_f16_kernel's).  Code rows M .. 8 kNT - 1 hold
  // stale bytes: they reach only output rows that are dropped.
  if (!mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_FULL))
    mbar_wait(bar_w, 0, p.err, DEVERR_TIMEOUT_DRAIN);
  const int g = lane >> 2, t = lane & 3;
  float acc[2][kNT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f;
  const int q = slice / kDecWarps;  // a multiple of 64, at most 1024
  const int8_t* wrow = wq + g * stride + 16 * t;
  const int8_t* crow = cq + g * stride + 16 * t;
  for (int k = warp * q; k < (warp + 1) * q; k += 64) {
    uint4 wa[2][2], cb[kNT];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      wa[mt][0] = *reinterpret_cast<const uint4*>(wrow + (16 * mt) * stride + k);
      wa[mt][1] = *reinterpret_cast<const uint4*>(wrow + (16 * mt + 8) * stride + k);
    }
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) cb[nt] = *reinterpret_cast<const uint4*>(crow + 8 * nt * stride + k);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t b0[kNT], b1[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) widen_i8x4(word_of(cb[nt], s), b0[nt], b1[nt]);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t a0, a1, a2, a3;
        widen_i8x4(word_of(wa[mt][0], s), a0, a2);
        widen_i8x4(word_of(wa[mt][1], s), a1, a3);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) mma_f16(acc[mt][nt], a0, a1, a2, a3, b0[nt], b1[nt]);
      }
    }
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 16 * mt + g + (e >= 2 ? 8 : 0);
        const int m = 8 * nt + 2 * t + (e & 1);
        if (m < p.M) atomicAdd(&red[m * kDecCols + c], static_cast<int32_t>(acc[mt][nt][e]));
      }
  compute_sync();
  // 5. The slices' sums into the block's slice-0 CTA (red[] zeroed before A).
  if (sidx != 0)
    for (int i = threadIdx.x; i < p.M * kDecCols; i += kDecWarps * 32)
      red_cluster_add_s32(map_to_cta(&red[i], static_cast<uint32_t>(bidx * cs)), red[i]);
  cluster_arrive_release();  // D
  if (sidx != 0) return;
  cluster_wait_acquire();
  for (int i = threadIdx.x; i < p.M * kDecCols; i += kDecWarps * 32) {
    const int m = i / kDecCols, c = i % kDecCols;
    const int n = n0 + c;
    if (n < p.N) {
      const float y = (static_cast<float>(red[i]) * sx_s[m]) * p.sW[n];
      p.Y[static_cast<int64_t>(m) * p.N + n] = __half_as_ushort(__float2half_rn(y));
    }
  }
}

}  // namespace

size_t decode_layer_smem(int M, int k_per_split) { return dec_smem(M, k_per_split); }

cudaError_t launch_decode_layer(const DecodeArgs& a, cudaStream_t stream) {
  if (a.M < 1 || a.M > kDecodeMaxM || a.k_per_split % 256 != 0 || a.k_per_split > kDecMaxSlice ||
      a.k_per_split * a.splits != a.K ||
      (a.splits != 1 && a.splits != 2 && a.splits != 4 && a.splits != 8))
    return cudaErrorInvalidValue;
  const size_t smem = dec_smem(a.M, a.k_per_split);
  if (smem > kDecodeMaxSmem) return cudaErrorInvalidValue;
  // One fixed limit (a captured launch must not depend on a size set last).
  auto kernel = a.M <= 4 ? decode_layer_kernel<4> : decode_layer_kernel<kDecodeMaxM>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDecodeMaxSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((a.N + kDecCols - 1) / kDecCols) * a.splits);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
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
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace convrot

namespace convrot {

size_t decode_mma_smem(int k_per_split) { return dm_smem(k_per_split); }

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t stream) {
  if (a.M < 1 || a.M > kDecodeMaxM || a.k_per_split % 256 != 0 || a.k_per_split > kDmMaxSlice ||
      a.k_per_split * a.splits != a.K ||
      (a.splits != 1 && a.splits != 2 && a.splits != 4 && a.splits != 8))
    return cudaErrorInvalidValue;
  static_assert(dm_smem(kDmMaxSlice) <= kDecodeMaxSmem, "shared memory limit");
  auto kernel = a.M <= 8 ? decode_mma_kernel<1> : decode_mma_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDecodeMaxSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((a.N + kDmRows - 1) / kDmRows) * a.splits);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = dm_smem(a.k_per_split);
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
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace convrot

namespace convrot {

size_t skinny_f16_smem(int k_per_split) { return sg_smem(k_per_split); }

cudaError_t launch_skinny_f16(const SkinnyF16Args& a, cudaStream_t stream) {
  if (a.M < 1 || a.M > kDecodeMaxM || a.k_per_split % 256 != 0 || a.k_per_split > 4096 ||
      a.k_per_split * a.splits != a.K ||
      (a.splits != 1 && a.splits != 2 && a.splits != 4 && a.splits != 8))
    return cudaErrorInvalidValue;
  static_assert(sg_smem(4096) <= kDecodeMaxSmem, "shared memory limit");
  auto kernel = a.M <= 8 ? skinny_f16_kernel<1> : skinny_f16_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDecodeMaxSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((a.N + kDecCols - 1) / kDecCols) * a.splits);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = sg_smem(a.k_per_split);
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
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace convrot

namespace convrot {

size_t decode_shared_smem(int k_per_split) { return ds_smem(k_per_split); }

cudaError_t launch_decode_shared(const DecodeArgs& a, int blocks, cudaStream_t stream) {
  const int groups = a.k_per_split / 256;
  if (a.M < 1 || a.M > kDecodeMaxM || a.k_per_split % 256 != 0 || a.k_per_split > 4096 ||
      a.k_per_split * a.splits != a.K ||
      (a.splits != 1 && a.splits != 2 && a.splits != 4 && a.splits != 8) ||
      (blocks != 2 && blocks != 4 && blocks != 8) || a.splits * blocks > 8 ||
      groups % blocks != 0 || a.M * (groups / blocks) > 4 * kDecHold)
    return cudaErrorInvalidValue;
  static_assert(ds_smem(4096) <= kDecodeMaxSmem, "shared memory limit");
  auto kernel = a.M <= 8 ? decode_shared_kernel<1> : decode_shared_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDecodeMaxSmem));
  if (e != cudaSuccess) return e;
  const int nblk = (a.N + kDecCols - 1) / kDecCols;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((nblk + blocks - 1) / blocks) * a.splits * blocks);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = ds_smem(a.k_per_split);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(a.splits * blocks);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a, blocks);
}

}  // namespace convrot
