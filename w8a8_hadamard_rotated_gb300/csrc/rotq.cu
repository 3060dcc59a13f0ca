// Rotate + quantize kernels of the INT8ConvRot layer (sm_103a).
//
// Page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix, and MLX",
// section "What changed in the computation":
//   X_rot = X H (H: Kronecker power of 4x4 Hadamards / 16, groups of 256 along
//   the last dimension), s_X[m] = max_k |X_rot[m,k]| / 127,
//   Q_X = round(X_rot / s_X) clamped to [-128, 127];
//   the weight gets the same treatment once, with W_rot = W H^T (= W H, H is
//   symmetric).
//
// H with the Sylvester 4x4 base is the normalized Walsh-Hadamard matrix, so
// x H is computed as a fast Walsh-Hadamard transform: 8 butterfly stages over
// the 256 entries of a group (a + b, a - b), then a factor 1/16.  The factor
// cancels in Q = round(x * 127 / amax) and is applied to the scale only
// (multiplying by 1/16 is exact).
//
// Kernels:
//   rotq_tile_kernel    per-call activation step for K <= 16384: TMA brings a
//                       tile of X into shared memory (128-byte swizzle), each
//                       lane owns 64 (or 32) consecutive values of a group
//                       (6 or 5 butterfly stages in registers, 2 or 3 across
//                       lanes with shuffles),
//                       the row max is reduced with shuffles (and shared memory
//                       when a row spans warps), and int8 (or the fp16 image of
//                       the int8 values) plus s_X are written in one pass; the
//                       fp16 image is written back into the tile in shared
//                       memory and leaves with one TMA store per tile.
//                       Persistent: each CTA loops over tiles with two buffers
//                       so the next tile's load overlaps this tile's math.
//   rotq_row_kernel     one CTA per row, two passes (row max, then quantize),
//                       fp32 or fp16 input, any K: weight prep and very wide K.
//   widen_i8_kernel     int8 -> fp16 copy (exact) for operand images.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "fwht.cuh"
#include "kernels.h"

namespace convrot {

__device__ __forceinline__ uint32_t pack2_f16(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack2_h(int a, int b) {
  const __half2 h = __floats2half2_rn(static_cast<float>(a), static_cast<float>(b));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// rotq_tile_kernel
// ---------------------------------------------------------------------------
// X is viewed as a 2-D tensor of 64-element "segments": [M*K/64, 64] fp16,
// which TMA copies into shared memory as 128-byte rows with the 128-byte
// swizzle (16-byte chunk c of row r lands at chunk c ^ (r % 8)).
//   VPL = 64: a lane owns one segment (64 consecutive values): 6 butterfly
//             stages in registers, 2 across the 4 lanes of a 256-group.
//   VPL = 32: two lanes share a segment (32 values each): 5 stages in
//             registers, 3 across the 8 lanes of a group.  Twice the warps
//             for the same data: lower latency on small problems.
// Either way a warp reads its rows without bank conflicts.  A tile is W warps'
// worth of segments.  The host uses this kernel only when K/VPL is a power of
// two and either a row fits in one warp (K <= 32 * VPL) or K/(32 * VPL)
// divides W (a row is whole warps of one CTA), so tiles never split a row.

constexpr int kTileMaxWarps = 8;
constexpr int64_t kL2PrefetchChunk = 32768;  // bytes per bulk L2 prefetch

// kInBf16: X holds bf16 values (otherwise fp16).
// kRotOnly (with kOutF16): write the rotated activation X H itself, rounded to
// fp16, instead of codes -- no row max, no scale (the weight-only W8A16
// comparator's prologue).
// kSigned: negate the inputs by the sign pattern of a non-Sylvester 4x4 base
// (RotqTileArgs::sign) before the transform.
template <bool kOutF16, int VPL, bool kInBf16 = false, bool kRotOnly = false,
          bool kSigned = false>
__global__ void __launch_bounds__(256) rotq_tile_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                        const __grid_constant__ CUtensorMap tm_q,
                                                        RotqTileArgs p) {
  constexpr int kLanesPerSeg = 64 / VPL;           // 1 or 2
  constexpr int kSegsPerWarp = 32 / kLanesPerSeg;  // 32 or 16
  constexpr int kChunks = VPL / 8;                 // 16-byte chunks per lane
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Two 1024-aligned buffers of (W * kSegsPerWarp) rows x 128 bytes, then barriers.
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int W = p.warps;
  const int segs_per_tile = W * kSegsPerWarp;
  const uint32_t buf_bytes = static_cast<uint32_t>(segs_per_tile) * 128u;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + 2 * buf_bytes);  // [2]
  float* red = reinterpret_cast<float*>(bar + 2);                       // [W]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t tiles = p.tiles;
  const int lanes_per_row = p.K / VPL;  // lanes covering one row of X

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_x);
    if (kOutF16) tma_prefetch_desc(&tm_q);
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbarrier_init();
    // Start pulling this CTA's first two tiles of X into L2 while the
    // previous kernel finishes.  A prefetch only moves lines into L2 (the
    // point of coherence) and returns nothing to the SM, so it is safe even
    // if the previous kernel is still writing X: the loads below, issued
    // after the dependency wait, see its writes.
    for (int b = 0; b < 2; ++b) {
      const int64_t t = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(b) * gridDim.x;
      if (t < p.tiles)
        tma_prefetch_l2_2d(&tm_x, 0, static_cast<int32_t>(t * p.warps * (32 / (64 / VPL))));
    }
    // This CTA's slice of the next GEMM's weight image, from HBM into L2
    // while the previous kernel finishes: the GEMM's first weight loads then
    // hit L2 instead of waiting on HBM.  (The weight is read-only here and a
    // prefetch returns nothing to the SM.)
    if (p.l2_pf_bytes > 0) {
      const int64_t per = ((p.l2_pf_bytes + gridDim.x - 1) / gridDim.x + 15) & ~int64_t{15};
      const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
      const int64_t b1 = min(p.l2_pf_bytes, b0 + per);
      const uint8_t* w = static_cast<const uint8_t*>(p.l2_pf);
      for (int64_t b = b0; b < b1; b += kL2PrefetchChunk)
        bulk_prefetch_l2(w + b, static_cast<uint32_t>(b1 - b < kL2PrefetchChunk ? b1 - b : kL2PrefetchChunk));
    }
  }
  __syncthreads();
  // Launched with programmatic dependent launch: wait for the previous
  // kernel on the stream (it may have written X, or still read the buffers
  // this kernel overwrites) before the first global access.
  grid_dep_wait();
  if (p.early_dependents) grid_dep_launch();

  int64_t tile = blockIdx.x;
  // Loads issued into / waited for in each buffer (thread 0's counts matter).
  int issued0 = 0, issued1 = 0, consumed0 = 0, consumed1 = 0;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      const int64_t t = tile + static_cast<int64_t>(b) * gridDim.x;
      if (t < tiles) {
        mbar_arrive_expect_tx(&bar[b], buf_bytes);
        tma_load_2d(base + b * buf_bytes, &tm_x, &bar[b], 0,
                    static_cast<int32_t>(t * segs_per_tile));
        if (b == 0) ++issued0; else ++issued1;
      }
    }
  }

  // Zero this CTA's share of the next GEMM's split-K accumulator while the
  // first tiles load (after the dependency wait: the previous GEMM may have
  // been reading it).
  if (p.zero_n16 > 0) {
    const int64_t per = (p.zero_n16 + gridDim.x - 1) / gridDim.x;
    const int64_t z0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t z1 = z0 + per < p.zero_n16 ? z0 + per : p.zero_n16;
    for (int64_t i = z0 + threadIdx.x; i < z1; i += blockDim.x) p.zero[i] = make_uint4(0, 0, 0, 0);
  }

  bool ok = true;
  for (int it = 0; tile < tiles; ++it, tile += gridDim.x) {
    const int b = it & 1;
    const uint32_t parity = (it >> 1) & 1;
    if (kOutF16 && threadIdx.x == 0 && it > 0) {
      // The previous tile's codes leave buffer b^1 by a TMA store; once the
      // store has read them, the buffer takes the tile after this one.
      const int64_t t2 = tile + static_cast<int64_t>(gridDim.x);
      if (t2 < tiles) {
        tma_store_wait_read();
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bar[b ^ 1], buf_bytes);
        tma_load_2d(base + (b ^ 1) * buf_bytes, &tm_x, &bar[b ^ 1], 0,
                    static_cast<int32_t>(t2 * segs_per_tile));
        if (b == 1) ++issued0; else ++issued1;
      }
    }
    if (!mbar_wait(&bar[b], parity, p.err, DEVERR_TIMEOUT_PROLOGUE)) {
      ok = false;
    }
    // Every thread decides to stop together: a timeout on any thread ends the
    // loop for the whole CTA.
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    if (b == 0) ++consumed0; else ++consumed1;

    // Segment (row of the swizzled buffer) and part of it owned by this lane.
    const int row_in_tile = warp * kSegsPerWarp + lane / kLanesPerSeg;
    const int part = lane % kLanesPerSeg;
    uint8_t* rowp = base + b * buf_bytes + row_in_tile * 128;
    float2 w[VPL / 2];
    load_swizzled_row2<VPL / 2, kInBf16>(rowp, row_in_tile, part * kChunks, w);
    if constexpr (kSigned) {
      // This lane's input signs: bits (s & 3) * 64 + part * VPL .. + VPL,
      // with s & 3 the segment's place in its 256-group.
      const int64_t s = tile * segs_per_tile + row_in_tile;
      const int b0 = static_cast<int>(s & 3) * 64 + part * VPL;
      uint64_t bits = p.sign[b0 >> 5];
      if constexpr (VPL == 64) bits |= static_cast<uint64_t>(p.sign[(b0 >> 5) + 1]) << 32;
      apply_signs2<VPL / 2>(w, bits);
    }
    if (!kOutF16) {
      __syncthreads();  // buffer b fully read by every lane
      if (threadIdx.x == 0) {
        const int64_t t2 = tile + 2 * static_cast<int64_t>(gridDim.x);
        if (t2 < tiles) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&bar[b], buf_bytes);
          tma_load_2d(base + b * buf_bytes, &tm_x, &bar[b], 0,
                      static_cast<int32_t>(t2 * segs_per_tile));
          if (b == 0) ++issued0; else ++issued1;
        }
      }
    }

    // Walsh-Hadamard transform of each 256-group: element bits below
    // log2(VPL) live in registers, the rest in the low lane bits.
    fwht_regs2<VPL / 2>(w);
#pragma unroll
    for (int mask = 1; mask < 256 / VPL; mask <<= 1) fwht_xlane2<VPL / 2>(w, lane, mask);

    // This lane's max |x| in four independent chains (max is exact and
    // ignores NaNs in any order: the same value as one chain, in a quarter of
    // the dependent steps).
    float am[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < VPL / 2; ++i) am[i & 3] = fmaxf(am[i & 3], fmaxf(fabsf(w[i].x), fabsf(w[i].y)));
    float amax = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));

    // Row max over the lanes that cover a row of X.
    if constexpr (kRotOnly) {
    } else if (lanes_per_row <= 32) {
      for (int m = 1; m < lanes_per_row; m <<= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    } else {
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      if (lane == 0) red[warp] = amax;
      __syncthreads();
      const int wpr = lanes_per_row / 32;
      const int w0 = (warp / wpr) * wpr;
      float a = 0.0f;
      for (int w = 0; w < wpr; ++w) a = fmaxf(a, red[w0 + w]);
      amax = a;
      __syncthreads();  // red[] may be rewritten by the next tile
    }

    // Global segment index, and the element offset of this lane's values.
    const int64_t seg = tile * segs_per_tile + row_in_tile;
    const bool valid = seg < p.segments;
    const int64_t elem = seg * 64 + part * VPL;
    const int64_t m = elem / p.K;
    if (!kRotOnly && valid && (elem % p.K) == 0) {
      // s_X = (amax / 16) / 127; x1/16 is exact.
      p.s_out[m] = (amax * 0.0625f) / 127.0f;
    }
    const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
    if constexpr (kOutF16) {
      // The codes replace this lane's inputs in the swizzled tile (each lane
      // rewrites exactly what it read), and the whole tile goes out with one
      // TMA store: full-line writes instead of a lane-strided pattern.
      const float2 inv2 = make_float2(inv, inv);
#pragma unroll
      for (int c = 0; c < VPL / 8; ++c) {
        const float2* s = w + c * 4;
        uint4 o;
        if constexpr (kRotOnly) {
          // X H = (butterfly sums) / 16: the factor is exact in fp32.
          o.x = pack2_f16(s[0].x * 0.0625f, s[0].y * 0.0625f);
          o.y = pack2_f16(s[1].x * 0.0625f, s[1].y * 0.0625f);
          o.z = pack2_f16(s[2].x * 0.0625f, s[2].y * 0.0625f);
          o.w = pack2_f16(s[3].x * 0.0625f, s[3].y * 0.0625f);
        } else {
          o.x = codes_f16x2_packed(s[0], inv2);
          o.y = codes_f16x2_packed(s[1], inv2);
          o.z = codes_f16x2_packed(s[2], inv2);
          o.w = codes_f16x2_packed(s[3], inv2);
        }
        const int phys = (part * kChunks + c) ^ (row_in_tile & 7);
        *reinterpret_cast<uint4*>(rowp + phys * 16) = o;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        // Rows past the end of the array are clipped by the tensor map.
        tma_store_2d(&tm_q, base + b * buf_bytes, 0, static_cast<int32_t>(tile * segs_per_tile));
        tma_store_commit();
      }
    } else if (valid) {
      {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<int8_t*>(p.q_out) + elem);
#pragma unroll
        for (int c = 0; c < VPL / 16; ++c) {
          const float* s = reinterpret_cast<const float*>(w + c * 8);
          uint4 o;
          o.x = codes_s8x4(round_magic(s[0], inv), round_magic(s[1], inv),
                           round_magic(s[2], inv), round_magic(s[3], inv));
          o.y = codes_s8x4(round_magic(s[4], inv), round_magic(s[5], inv),
                           round_magic(s[6], inv), round_magic(s[7], inv));
          o.z = codes_s8x4(round_magic(s[8], inv), round_magic(s[9], inv),
                           round_magic(s[10], inv), round_magic(s[11], inv));
          o.w = codes_s8x4(round_magic(s[12], inv), round_magic(s[13], inv),
                           round_magic(s[14], inv), round_magic(s[15], inv));
          dst[c] = o;
        }
      }
    }
  }

  if (threadIdx.x == 0) {
    // Shared memory must outlive the reads of the last stores.
    if (kOutF16) tma_store_wait_read();
    // Do not leave the CTA while a copy into shared memory may be in flight:
    // wait (bounded) for every load that was issued but not waited for.  On
    // the normal path every issued load was consumed and nothing waits.
    if (issued0 > consumed0)
      mbar_wait(&bar[0], static_cast<uint32_t>(issued0 - 1) & 1u, p.err, DEVERR_TIMEOUT_DRAIN);
    if (issued1 > consumed1)
      mbar_wait(&bar[1], static_cast<uint32_t>(issued1 - 1) & 1u, p.err, DEVERR_TIMEOUT_DRAIN);
  }
}

// ---------------------------------------------------------------------------
// rotq_row_kernel: one CTA (8 warps) per row; warp w handles groups w, w+8, ..
// Lane l holds elements 8l..8l+7 of the group: 3 butterfly stages in
// registers, 5 across lanes.  Pass 1 finds the row max, pass 2 recomputes the
// transform and quantizes.
// ---------------------------------------------------------------------------
template <typename InT>
__device__ __forceinline__ void load8(const InT* src, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<float>(const float* src, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 b = *reinterpret_cast<const float4*>(src + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* src, float (&v)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(src);
  const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {  // exact: a bf16 is the top half of an fp32
    v[2 * e] = __uint_as_float(u[e] << 16);
    v[2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
  }
}

template <>
__device__ __forceinline__ void load8<__half>(const __half* src, float (&v)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(src);
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(h2[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

// sbits: the input signs of this lane's 8 elements (0 for Sylvester's base).
template <typename InT>
__device__ __forceinline__ void group_fwht(const InT* grp, int lane, uint32_t sbits,
                                           float (&v)[8]) {
  load8<InT>(grp + lane * 8, v);
  apply_signs<8>(v, sbits);
  fwht_regs<8>(v);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) fwht_xlane<8>(v, lane, m);
}

template <typename InT>
__global__ void __launch_bounds__(256) rotq_row_kernel(RotqRowArgs p) {
  __shared__ float red[8];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int groups = p.K / 256;
  // Lane l holds elements 8l..8l+7 of a group: sign bits 8l..8l+7.
  const uint32_t sbits = (p.sign[lane >> 2] >> ((lane & 3) * 8)) & 0xffu;
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const InT* x = static_cast<const InT*>(p.in) + row * p.K;
    float amax = 0.0f;
    for (int g = warp; g < groups; g += 8) {
      float v[8];
      group_fwht<InT>(x + g * 256, lane, sbits, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();
    if (threadIdx.x == 0) p.s_out[row] = (amax * 0.0625f) / 127.0f;
    // An fp32 row whose rotated max is below 2^-100 is quantized after an
    // exact scaling by 2^64, so that 127 / amax stays finite.  (An fp16 row's
    // rotated max is at least its 2-norm, >= 2^-24, and never needs it.)
    const float pre = amax < 0x1p-100f ? 0x1p64f : 1.0f;
    const float inv = amax > 0.0f ? 127.0f / (amax * pre) : 0.0f;
    for (int g = warp; g < groups; g += 8) {
      float v[8];
      group_fwht<InT>(x + g * 256, lane, sbits, v);
      uint32_t r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) r[i] = round_magic(v[i] * pre, inv);
      const int64_t off = row * p.K + g * 256 + lane * 8;
      if (p.q_out) {
        uint2 o;
        o.x = codes_s8x4(r[0], r[1], r[2], r[3]);
        o.y = codes_s8x4(r[4], r[5], r[6], r[7]);
        *reinterpret_cast<uint2*>(p.q_out + off) = o;
      }
      if (p.img_out) {
        uint4 o;
        o.x = codes_f16x2(r[0], r[1]);
        o.y = codes_f16x2(r[2], r[3]);
        o.z = codes_f16x2(r[4], r[5]);
        o.w = codes_f16x2(r[6], r[7]);
        *reinterpret_cast<uint4*>(p.img_out + off) = o;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// widen_i8_kernel: out[i] = (fp16) in[i], 16 elements per thread per step.
// ---------------------------------------------------------------------------
__global__ void widen_i8_kernel(const int8_t* __restrict__ in, uint16_t* __restrict__ out,
                                int64_t n16) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 raw = reinterpret_cast<const uint4*>(in)[i];
    const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
    uint4 o0, o1;
    o0.x = pack2_h(b[0], b[1]);
    o0.y = pack2_h(b[2], b[3]);
    o0.z = pack2_h(b[4], b[5]);
    o0.w = pack2_h(b[6], b[7]);
    o1.x = pack2_h(b[8], b[9]);
    o1.y = pack2_h(b[10], b[11]);
    o1.z = pack2_h(b[12], b[13]);
    o1.w = pack2_h(b[14], b[15]);
    reinterpret_cast<uint4*>(out)[2 * i] = o0;
    reinterpret_cast<uint4*>(out)[2 * i + 1] = o1;
  }
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
size_t rotq_tile_smem_bytes(int warps, int vpl) {
  return 1024 + 2 * static_cast<size_t>(warps * (32 * vpl / 64) * 128) + 2 * sizeof(uint64_t) +
         kTileMaxWarps * sizeof(float);
}

// The tile kernels are launched with different shared-memory sizes (tile
// width, CTA cap).  Their dynamic shared-memory limit is set once to the
// device maximum, so that no launch -- nor a graph node captured earlier and
// relaunched by a tool -- depends on which size was set last.
static cudaError_t allow_max_smem(void (*kernel)(const CUtensorMap, const CUtensorMap,
                                                 RotqTileArgs),
                                  int* max_block) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(max_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, *max_block);
}

// Shared-memory request that lets at most `cap` CTAs of `kernel` reside on
// an SM: (cap + 1) CTAs must not fit, cap CTAs must.  Checked against the
// occupancy calculator once per (variant, warps, cap) and cached.
static std::atomic<int> g_cap_smem[16][2][kTileMaxWarps + 1][33];

static size_t capped_smem(void (*kernel)(const CUtensorMap, const CUtensorMap, RotqTileArgs),
                          int variant, int vpl, int warps, int cap, size_t need) {
  if (cap <= 0 || cap > 32 || warps > kTileMaxWarps) return need;
  std::atomic<int>& slot = g_cap_smem[variant][vpl == 64 ? 1 : 0][warps][cap];
  const int cached = slot.load(std::memory_order_relaxed);
  if (cached > 0) return std::max(need, static_cast<size_t>(cached));
  int dev = 0, per_sm = 0, reserved = 0, max_block = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
          cudaSuccess ||
      allow_max_smem(kernel, &max_block) != cudaSuccess)
    return need;
  size_t s = static_cast<size_t>(per_sm / (cap + 1) + 128 - reserved);
  s = (s + 127) / 128 * 128;
  s = std::max(s, need);
  // Grow in 1 KB steps while the occupancy calculator still fits more than
  // `cap` (allocation granularity); give up (the kernel's own need) if the
  // request would exceed what one CTA may have.
  for (int i = 0; i < 16; ++i) {
    if (s > static_cast<size_t>(max_block)) return need;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, 32 * warps, s) !=
        cudaSuccess)
      return need;
    if (blocks <= cap) {
      slot.store(static_cast<int>(s), std::memory_order_relaxed);
      return s;
    }
    s += 1024;
  }
  return need;
}

cudaError_t launch_rotq_tile(const CUtensorMap& tm_x, const CUtensorMap& tm_q,
                             const RotqTileArgs& a, bool out_f16, int grid, int max_per_sm,
                             cudaStream_t stream) {
  const dim3 block(32 * a.warps);
  void (*kernel)(const CUtensorMap, const CUtensorMap, RotqTileArgs);
  if (a.rot_only) {
    if (!out_f16) return cudaErrorInvalidValue;
    if (a.vpl == 32)
      kernel = a.in_bf16 ? rotq_tile_kernel<true, 32, true, true> : rotq_tile_kernel<true, 32, false, true>;
    else
      kernel = a.in_bf16 ? rotq_tile_kernel<true, 64, true, true> : rotq_tile_kernel<true, 64, false, true>;
  } else if (a.has_sign) {
    // A base other than Sylvester's that negates inputs: its own variants,
    // so that the default ones stay free of the sign step.
    if (a.vpl == 32) {
      kernel = a.in_bf16 ? (out_f16 ? rotq_tile_kernel<true, 32, true, false, true>
                                    : rotq_tile_kernel<false, 32, true, false, true>)
                         : (out_f16 ? rotq_tile_kernel<true, 32, false, false, true>
                                    : rotq_tile_kernel<false, 32, false, false, true>);
    } else {
      kernel = a.in_bf16 ? (out_f16 ? rotq_tile_kernel<true, 64, true, false, true>
                                    : rotq_tile_kernel<false, 64, true, false, true>)
                         : (out_f16 ? rotq_tile_kernel<true, 64, false, false, true>
                                    : rotq_tile_kernel<false, 64, false, false, true>);
    }
  } else if (a.in_bf16) {
    if (a.vpl == 32)
      kernel = out_f16 ? rotq_tile_kernel<true, 32, true> : rotq_tile_kernel<false, 32, true>;
    else
      kernel = out_f16 ? rotq_tile_kernel<true, 64, true> : rotq_tile_kernel<false, 64, true>;
  } else if (a.vpl == 32) {
    kernel = out_f16 ? rotq_tile_kernel<true, 32> : rotq_tile_kernel<false, 32>;
  } else {
    kernel = out_f16 ? rotq_tile_kernel<true, 64> : rotq_tile_kernel<false, 64>;
  }
  int max_block = 0;
  cudaError_t e = allow_max_smem(kernel, &max_block);
  if (e != cudaSuccess) return e;
  const size_t smem = capped_smem(kernel,
                                  (out_f16 ? 1 : 0) + (a.in_bf16 ? 2 : 0) + (a.rot_only ? 4 : 0) +
                                      (a.has_sign && !a.rot_only ? 8 : 0),
                                  a.vpl, a.warps,
                                  max_per_sm,
                                  rotq_tile_smem_bytes(a.warps, a.vpl));
  if (smem > static_cast<size_t>(max_block)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tm_x, tm_q, a);
}

cudaError_t launch_rotq_row(const RotqRowArgs& a, int in_type, int grid, cudaStream_t stream) {
  if (in_type == kRowInF32)
    rotq_row_kernel<float><<<grid, 256, 0, stream>>>(a);
  else if (in_type == kRowInBf16)
    rotq_row_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a);
  else
    rotq_row_kernel<__half><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_widen_i8(const int8_t* in, uint16_t* out, int64_t n, int grid,
                            cudaStream_t stream) {
  widen_i8_kernel<<<grid, 256, 0, stream>>>(in, out, n / 16);
  return cudaGetLastError();
}

}  // namespace convrot
