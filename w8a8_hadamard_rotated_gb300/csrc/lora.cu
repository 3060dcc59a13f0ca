// LoRA down-projection T = X lora_down^T for the unmerged LoRA term of the
// page "[PR #249] Add an mps backend: weight-only INT8 and W4A8/W6A8 linears
// for Apple GPUs" (section "What": lora_down [R, K], lora_up [N, R],
// lora_scale), applied to the unrotated activation X.
//
// fp16 (or bf16) operands, fp32 accumulation on the mma.sync m16n8k16 path.  A warp
// owns 16 rows of X and half of the LoRA ranks (every rank at R > 64) over
// one K slice.  The S slices of a block of 64 rows run on the S CTAs of a
// thread-block cluster (S = 1, 2, 4 or 8): each CTA leaves its partial in
// shared memory, and after a cluster barrier CTA r adds rows [r * 64/S,
// (r + 1) * 64/S) of the S partials in rank order through distributed shared
// memory and writes them to T.  The sum order is fixed, so T -- and the
// layer's Y -- is the same bits on every run; no atomics, nothing to zero.
// The operands of U consecutive 32-wide K steps are loaded before their MMAs,
// so each warp keeps U steps of loads in flight (the kernel streams X and is
// otherwise latency-bound).
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

// Dynamic shared memory of lora_down_kernel: the partial [64][8 NT] fp32.
// (Staging the CTA's lora_down slice there too measured slower: 47 us against
// 34 us at M = 4096, K = 8192, R = 32 -- its 75 KB per CTA halved the warps
// in flight, and the four warps' repeated slice reads hit L1 anyway.  So did
// a copy warp moving X and lora_down by bulk copies through a ring of 128-K
// stages: 53 us -- 100 KB per CTA, two waves of 512 CTAs, 768 copies of 256
// bytes per CTA, the lora_down slice copied again by every CTA.  A bulk L2
// prefetch of each warp's X rows before the dependency wait changed nothing
// (34.7 us): the kernel ran at ~0.6 instructions per cycle per SM, each
// warp's chain of loads and MMAs exposed, not waiting on DRAM.  Two warps
// per 16-row group, each with half of the ranks and 64 registers (twice the
// warps in flight, half the chain each): 34 -> ~21 us.)
__host__ __device__ constexpr size_t lora_down_smem(int nt) {
  return static_cast<size_t>(64) * 8 * nt * 4;
}

// H warps share each 16-row group, each taking NT / H of the n8 tiles of
// ranks (the group's X fragments are loaded by each of them; the second
// load hits L1): shorter chains of MMAs per warp and H times the warps.
template <int NT, int U, int H, bool kBf16>
__global__ void __launch_bounds__(kLoraWarps * H * 32, 4) lora_down_kernel(const LoraDownArgs p) {
  constexpr int NTW = NT / H;  // n8 tiles of ranks per warp
  extern __shared__ __align__(16) float part[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int rg = warp % kLoraWarps;  // 16-row group
  const int j0 = (warp / kLoraWarps) * NTW;  // first n8 tile of ranks
  const int m_base = (blockIdx.x * kLoraWarps + rg) * 16;
  const int k_begin = blockIdx.y * p.k_per_split;
  const int k_end = min(p.K, k_begin + p.k_per_split);
  grid_dep_wait();  // launched with programmatic dependent launch
  grid_dep_launch();

  const uint16_t* xr[2];
  bool xok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = m_base + g + 8 * h;
    xok[h] = m < p.M;
    xr[h] = p.X + static_cast<int64_t>(xok[h] ? m : 0) * p.K + 8 * t;
  }
  // lora_down row 8j + g of n8 tile j starts at d_base + j * d_step.
  const uint16_t* d_base = p.down + static_cast<int64_t>(8 * j0 + g) * p.K + 8 * t;
  const int64_t d_step = 8 * static_cast<int64_t>(p.K);

  float acc[NTW][4];
#pragma unroll
  for (int j = 0; j < NTW; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;

  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int k = k_begin; k < k_end; k += 32 * U) {
    uint4 x0[U], x1[U], d[U][NTW];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = k + 32 * u;
      const bool in = kk < k_end;
      x0[u] = (in && xok[0]) ? __ldg(reinterpret_cast<const uint4*>(xr[0] + kk)) : zero;
      x1[u] = (in && xok[1]) ? __ldg(reinterpret_cast<const uint4*>(xr[1] + kk)) : zero;
#pragma unroll
      for (int j = 0; j < NTW; ++j)
        d[u][j] = (in && 8 * (j0 + j) + g < p.R)
                      ? __ldg(reinterpret_cast<const uint4*>(d_base + j * d_step + kk))
                      : zero;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int j = 0; j < NTW; ++j) {
        mma_f16_16816<kBf16>(acc[j], x0[u].x, x1[u].x, x0[u].y, x1[u].y, d[u][j].x, d[u][j].y);
        mma_f16_16816<kBf16>(acc[j], x0[u].z, x1[u].z, x0[u].w, x1[u].w, d[u][j].z, d[u][j].w);
      }
    }
  }
  // This CTA's partial [64 rows][8 NT] into shared memory (fragment layout:
  // rows g and g + 8 of this warp's 16, columns 8j + 2t, + 1).
#pragma unroll
  for (int j = 0; j < NTW; ++j) {
    const int c = 8 * (j0 + j) + 2 * t;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rg * 16 + g + 8 * h;
      *reinterpret_cast<float2*>(&part[r * (8 * NT) + c]) = make_float2(acc[j][2 * h], acc[j][2 * h + 1]);
    }
  }
  // Every CTA of the cluster reaches this barrier (no early exit above for a
  // CTA whose rows lie past M: its partial is zeros).
  cluster_sync_all();
  const int S = static_cast<int>(gridDim.y);  // = the cluster size
  const uint32_t rank = cluster_ctarank();
  const int rows = 64 / S;                    // rows this CTA finalizes
  const int row0 = static_cast<int>(rank) * rows;
  const int cols = 8 * NT;
  for (int i = threadIdx.x; i < rows * cols; i += kLoraWarps * H * 32) {
    const int r = row0 + i / cols, c = i % cols;
    const int m = blockIdx.x * 64 + r;
    float v = 0.0f;
    for (int q = 0; q < S; ++q) {  // rank order: the same sum on every run
      const uint32_t a = map_to_cta(&part[r * cols + c], static_cast<uint32_t>(q));
      float f;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(f) : "r"(a) : "memory");
      v += f;
    }
    if (m < p.M && c < p.R) p.T[static_cast<int64_t>(m) * p.R + c] = v;
  }
  // No CTA leaves while its partial may still be read by another.
  cluster_sync_all();
}

// LoRA up-projection sums S[m, n] = sum_r T[m, r] * lora_up[n, r] in fp32
// (the epilogues add lora_scale * S before the single rounding of Y).  The
// ranks are taken in pairs by paired fp32 FMAs, pair 0 first:
//   acc = fma2((T[m, 2j], T[m, 2j+1]), (up[n, 2j], up[n, 2j+1]), acc),  S = acc.x + acc.y
// (ranks past R count as zeros).  A CTA covers 64 rows and up to 4 chunks of
// 64 columns: the rows' T is staged in shared memory once, each chunk's
// lora_up in turn (coalesced loads).  Each lane owns two columns of the
// chunk and each warp 8 rows.  lora_up is staged lane-major, the two
// columns' values of two rank pairs side by side, so that a lane reads them
// with one 16-byte load and the 8 lanes of a load phase hit distinct banks;
// the rows' T values are 16-byte broadcasts.  A warp's 64 sums of a row
// leave as one coalesced 256-byte store.  It serves R not a multiple of 8
// (lora_up_mma_kernel below takes the rest): at M = 4096, N = 2048, R = 32
// this form took 26 us, bound by instruction issue and the FMA pipe (neither
// the chunking nor the conflict-free staging changed that).
constexpr int kLoraUpRows = 64;
constexpr int kLoraUpCols = 64;
constexpr int kLoraUpChunks = 4;

// Row stride of the T tile (floats): 16-byte aligned rows.
__host__ __device__ constexpr int lora_t_stride(int R) { return ((R + 31) & ~31) + 4; }
// Lane stride of the lora_up tile (floats): pairs of ranks x 2 columns,
// + 4 so that consecutive lanes' 16-byte reads fall on different banks.
__host__ __device__ constexpr int lora_u_stride(int R) { return 2 * ((R + 31) & ~31) + 4; }
__host__ __device__ constexpr size_t lora_up_smem(int R) {
  return (static_cast<size_t>(kLoraUpRows) * lora_t_stride(R) +
          static_cast<size_t>(kLoraUpCols / 2) * lora_u_stride(R)) * 4;
}

template <bool kBf16>
__device__ __forceinline__ float2 lora_w2(uint32_t w) {
  return kBf16 ? make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u))
               : __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <bool kBf16>
__global__ void __launch_bounds__(256, 3) lora_up_kernel(const LoraUpArgs p) {
  extern __shared__ __align__(16) float sm[];
  const int Rp = (p.R + 31) & ~31;  // ranks in whole chunks of 32
  const int ts = lora_t_stride(p.R);
  const int us = lora_u_stride(p.R);
  float* t_s = sm;                     // [64 rows][ts]: T of this CTA's rows
  float* u_s = sm + kLoraUpRows * ts;  // [32 lanes][us]: (pair j, column 2l / 2l+1) at 4j + 2c
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * kLoraUpRows;
  grid_dep_wait();  // T comes from the previous kernel on the stream
  grid_dep_launch();
  if (p.R % 8 == 0) {
    // R a multiple of 8: T in 16-byte loads, two passes of four per thread
    // (64 rows x 128 ranks / 4 / 256), each pass's loads issued before any
    // is used.
    const int tq = p.R / 4;
    for (int pass = 0; pass < 2; ++pass) {
      float4 tv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = threadIdx.x + (pass * 4 + k) * 256;
        const int r = i / tq, c = (i % tq) * 4;
        tv[k] = (i < kLoraUpRows * tq && m0 + r < p.M)
                    ? __ldg(reinterpret_cast<const float4*>(p.T + static_cast<int64_t>(m0 + r) * p.R + c))
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = threadIdx.x + (pass * 4 + k) * 256;
        if (i < kLoraUpRows * tq) {
          const int r = i / tq, c = (i % tq) * 4;
          *reinterpret_cast<float4*>(t_s + r * ts + c) = tv[k];
        }
      }
    }
  } else {
    for (int i = threadIdx.x; i < kLoraUpRows * p.R; i += 256) {
      const int r = i / p.R, c = i % p.R;
      t_s[r * ts + c] = m0 + r < p.M ? p.T[static_cast<int64_t>(m0 + r) * p.R + c] : 0.0f;
    }
  }
  // Ranks R .. Rp - 1 of both tiles are zero (the chunks' staging below
  // writes ranks < R only).
  for (int i = threadIdx.x; i < kLoraUpRows * (Rp - p.R); i += 256) {
    const int c = i / (Rp - p.R), r = p.R + i % (Rp - p.R);
    t_s[c * ts + r] = 0.0f;
    u_s[(c >> 1) * us + (r >> 1) * 4 + (c & 1) * 2 + (r & 1)] = 0.0f;
  }
  const float* up_l = u_s + lane * us;
  const float* tp = t_s + (warp * 8) * ts;
  for (int chunk = 0; chunk < kLoraUpChunks; ++chunk) {
    const int n0 = (blockIdx.x * kLoraUpChunks + chunk) * kLoraUpCols;
    if (n0 >= p.N) break;  // the same for the whole CTA
    if (chunk > 0) __syncthreads();  // the previous chunk's readers are done with u_s
    if (p.R % 8 == 0) {
      // Up to 64 columns x 128 ranks / 8 = 1024 16-byte loads: four per
      // thread, each 8 ranks of one column, stored as 4 rank pairs.
      const int uq = p.R / 8;
      uint4 uv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = threadIdx.x + k * 256;
        const int c = i / uq, r = (i % uq) * 8;
        uv[k] = (i < kLoraUpCols * uq && n0 + c < p.N)
                    ? __ldg(reinterpret_cast<const uint4*>(p.up + static_cast<int64_t>(n0 + c) * p.R + r))
                    : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = threadIdx.x + k * 256;
        if (i < kLoraUpCols * uq) {
          const int c = i / uq, r = (i % uq) * 8;
          float* d = u_s + (c >> 1) * us + (r >> 1) * 4 + (c & 1) * 2;
          *reinterpret_cast<float2*>(d) = lora_w2<kBf16>(uv[k].x);
          *reinterpret_cast<float2*>(d + 4) = lora_w2<kBf16>(uv[k].y);
          *reinterpret_cast<float2*>(d + 8) = lora_w2<kBf16>(uv[k].z);
          *reinterpret_cast<float2*>(d + 12) = lora_w2<kBf16>(uv[k].w);
        }
      }
    } else {
      for (int i = threadIdx.x; i < kLoraUpCols * p.R; i += 256) {
        const int c = i / p.R, r = i % p.R;
        float v = 0.0f;
        if (n0 + c < p.N) {
          const uint16_t h = p.up[static_cast<int64_t>(n0 + c) * p.R + r];
          v = kBf16 ? __uint_as_float(static_cast<uint32_t>(h) << 16)
                    : __half2float(*reinterpret_cast<const __half*>(&h));
        }
        u_s[(c >> 1) * us + (r >> 1) * 4 + (c & 1) * 2 + (r & 1)] = v;
      }
    }
    __syncthreads();
    // Two rank pairs per step: the lane's lora_up values of both pairs for
    // its two columns (two 16-byte reads) and the 8 rows' T values of the
    // four ranks (16-byte broadcasts).  Each output's sum runs over the rank
    // pairs (2j, 2j+1) in j order.
    float2 acc[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = make_float2(0.0f, 0.0f);
#pragma unroll 1
    for (int r = 0; r < Rp; r += 4) {
      const float4 ua = *reinterpret_cast<const float4*>(up_l + (r >> 1) * 4);
      const float4 ub = *reinterpret_cast<const float4*>(up_l + (r >> 1) * 4 + 4);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 t4 = *reinterpret_cast<const float4*>(tp + i * ts + r);
        acc[i][0] = __ffma2_rn(make_float2(t4.x, t4.y), make_float2(ua.x, ua.y), acc[i][0]);
        acc[i][1] = __ffma2_rn(make_float2(t4.x, t4.y), make_float2(ua.z, ua.w), acc[i][1]);
        acc[i][0] = __ffma2_rn(make_float2(t4.z, t4.w), make_float2(ub.x, ub.y), acc[i][0]);
        acc[i][1] = __ffma2_rn(make_float2(t4.z, t4.w), make_float2(ub.z, ub.w), acc[i][1]);
      }
    }
    const int n = n0 + 2 * lane;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int m = m0 + warp * 8 + i;
      if (m >= p.M) continue;
      float* dst = p.S + static_cast<int64_t>(m) * p.N + n;
      const float2 v = make_float2(acc[i][0].x + acc[i][0].y, acc[i][1].x + acc[i][1].y);
      if (n + 1 < p.N && (p.N & 1) == 0)
        *reinterpret_cast<float2*>(dst) = v;  // 8-byte aligned: N and n even
      else {
        if (n < p.N) dst[0] = v.x;
        if (n + 1 < p.N) dst[1] = v.y;
      }
    }
  }
}


// The same sums on the tensor cores, for R a multiple of 8: T = T_hi + T_lo
// with T_hi = tf32(T) and T_lo = tf32(T - T_hi) (T - T_hi is exact in fp32),
// lora_up exact in tf32 (an fp16 or bf16 value has at most 10 fraction
// bits), so each product of mma.sync m16n8k8 tf32 is exact and
// S = sum_r T_hi up + T_lo up with fp32 accumulation differs from the exact
// sum by at most ~2^-22 sum_r |T up| plus the accumulation roundings.  The
// MMAs' order of summation is fixed by the hardware, so S is the same bits
// on every run.
//   A CTA of 4 warps covers 64 rows and up to 4 chunks of 64 columns; warp
// w owns rows 16w .. 16w + 15.  Each chunk's lora_up slice is staged once in
// shared memory as fp32 (row n: its R ranks, pitch Rp + 2 floats: the 16
// lanes of an 8-byte load phase hit distinct banks).  Rank order inside an
// MMA: the 32 ranks of block b go to 4 k-steps; lane t of a quad holds ranks
// 32b + 8t .. 32b + 8t + 7 of its rows of T, and k-step s takes ranks
// 32b + 8t + 2s, + 1 of T and of lora_up as the MMA's k = t and t + 4 (any
// order shared by the two operands gives the same products).
constexpr int kLoraMmaWarps = 4;
constexpr int kLoraMmaRows = 16 * kLoraMmaWarps;

__host__ __device__ constexpr int lora_mma_u_stride(int R) { return ((R + 31) & ~31) + 2; }
__host__ __device__ constexpr size_t lora_mma_smem(int R) {
  return static_cast<size_t>(kLoraUpCols) * lora_mma_u_stride(R) * 4;
}

__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool kBf16>
__global__ void __launch_bounds__(kLoraMmaWarps * 32) lora_up_mma_kernel(const LoraUpArgs p) {
  constexpr int kThreads = kLoraMmaWarps * 32;
  extern __shared__ __align__(16) float us_[];
  const int Rp = (p.R + 31) & ~31;
  const int us = lora_mma_u_stride(p.R);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int m_lo = blockIdx.y * kLoraMmaRows + warp * 16 + g;  // rows m_lo, m_lo + 8
  grid_dep_wait();  // T comes from the previous kernel on the stream
  grid_dep_launch();
  // Ranks R .. Rp - 1 of the staged slice are zero (staging writes ranks < R).
  for (int i = threadIdx.x; i < kLoraUpCols * (Rp - p.R); i += kThreads) {
    const int c = i / (Rp - p.R), r = p.R + i % (Rp - p.R);
    us_[c * us + r] = 0.0f;
  }
  const float* trow[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = m_lo + 8 * h;
    trow[h] = m < p.M ? p.T + static_cast<int64_t>(m) * p.R : nullptr;
  }
  const int uq = p.R / 8;  // 16-byte loads per lora_up row
  for (int chunk = 0; chunk < kLoraUpChunks; ++chunk) {
    const int n0 = (blockIdx.x * kLoraUpChunks + chunk) * kLoraUpCols;
    if (n0 >= p.N) break;  // the same for the whole CTA
    if (chunk > 0) __syncthreads();  // the previous chunk's readers are done
    // Stage lora_up[n0 .. n0 + 63][0 .. R) as fp32: at most 64 x 16 16-byte
    // loads, in two passes of four per thread.
    for (int pass = 0; pass < 2; ++pass) {
      uint4 uv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = threadIdx.x + (pass * 4 + k) * kThreads;
        const int c = i / uq, r = (i % uq) * 8;
        uv[k] = (i < kLoraUpCols * uq && n0 + c < p.N)
                    ? __ldg(reinterpret_cast<const uint4*>(p.up + static_cast<int64_t>(n0 + c) * p.R + r))
                    : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = threadIdx.x + (pass * 4 + k) * kThreads;
        if (i < kLoraUpCols * uq) {
          const int c = i / uq, r = (i % uq) * 8;
          float2* d = reinterpret_cast<float2*>(us_ + c * us + r);
          d[0] = lora_w2<kBf16>(uv[k].x);
          d[1] = lora_w2<kBf16>(uv[k].y);
          d[2] = lora_w2<kBf16>(uv[k].z);
          d[3] = lora_w2<kBf16>(uv[k].w);
        }
      }
    }
    __syncthreads();
    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;
    for (int b = 0; b < Rp; b += 32) {
      const int r0 = b + 8 * t;  // this lane's 8 ranks
      // T of rows m_lo and m_lo + 8 at ranks r0 .. r0 + 7 (zeros past R or M).
      float x[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 v0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), v1 = v0;
        if (trow[h] && r0 < p.R) {
          v0 = __ldg(reinterpret_cast<const float4*>(trow[h] + r0));
          v1 = __ldg(reinterpret_cast<const float4*>(trow[h] + r0 + 4));
        }
        x[h][0] = v0.x; x[h][1] = v0.y; x[h][2] = v0.z; x[h][3] = v0.w;
        x[h][4] = v1.x; x[h][5] = v1.y; x[h][6] = v1.z; x[h][7] = v1.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // hi and lo tf32 parts of the k-step's A fragment: rows g / g + 8 at
        // MMA k = t (rank r0 + 2k) and k = t + 4 (rank r0 + 2k + 1).
        uint32_t ah[4], al[4];
        const float xa[4] = {x[0][2 * k], x[1][2 * k], x[0][2 * k + 1], x[1][2 * k + 1]};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ah[e] = tf32_rna(xa[e]);
          al[e] = tf32_rna(xa[e] - __uint_as_float(ah[e]));
        }
        const float* u = us_ + g * us + r0 + 2 * k;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 w = *reinterpret_cast<const float2*>(u + 8 * j * us);
          const uint32_t b0 = __float_as_uint(w.x), b1 = __float_as_uint(w.y);
          mma_tf32_1688(acc[j], ah[0], ah[1], ah[2], ah[3], b0, b1);
          mma_tf32_1688(acc[j], al[0], al[1], al[2], al[3], b0, b1);
        }
      }
    }
    // S rows m_lo, m_lo + 8, columns n0 + 8j + 2t, + 1.
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + 8 * j + 2 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = m_lo + 8 * h;
        if (m >= p.M) continue;
        float* dst = p.S + static_cast<int64_t>(m) * p.N + n;
        if (n + 1 < p.N && (p.N & 1) == 0) {
          *reinterpret_cast<float2*>(dst) = make_float2(acc[j][2 * h], acc[j][2 * h + 1]);
        } else {
          if (n < p.N) dst[0] = acc[j][2 * h];
          if (n + 1 < p.N) dst[1] = acc[j][2 * h + 1];
        }
      }
    }
  }
}

cudaError_t launch_lora_up(const LoraUpArgs& a, cudaStream_t stream) {
  if (a.R <= 0 || a.R > kLoraMaxR) return cudaErrorInvalidValue;
  if (a.R % 8 == 0) {
    cudaLaunchConfig_t cfg = {};
    constexpr int kCtaCols = kLoraUpCols * kLoraUpChunks;
    cfg.gridDim = dim3((a.N + kCtaCols - 1) / kCtaCols, (a.M + kLoraMmaRows - 1) / kLoraMmaRows);
    cfg.blockDim = dim3(kLoraMmaWarps * 32);
    cfg.dynamicSmemBytes = lora_mma_smem(a.R);
    const int max_smem = static_cast<int>(lora_mma_smem(kLoraMaxR));
    cudaError_t e = cudaFuncSetAttribute(lora_up_mma_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(lora_up_mma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               max_smem);
    if (e != cudaSuccess) return e;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return a.bf16 ? cudaLaunchKernelEx(&cfg, lora_up_mma_kernel<true>, a)
                  : cudaLaunchKernelEx(&cfg, lora_up_mma_kernel<false>, a);
  }
  cudaLaunchConfig_t cfg = {};
  constexpr int kCtaCols = kLoraUpCols * kLoraUpChunks;
  cfg.gridDim = dim3((a.N + kCtaCols - 1) / kCtaCols, (a.M + kLoraUpRows - 1) / kLoraUpRows);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = lora_up_smem(a.R);
  // One fixed limit for the largest R (a captured launch must not depend on a
  // size set last).
  const int max_smem = static_cast<int>(lora_up_smem(kLoraMaxR));
  cudaError_t e = cudaFuncSetAttribute(lora_up_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(lora_up_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.bf16 ? cudaLaunchKernelEx(&cfg, lora_up_kernel<true>, a)
                : cudaLaunchKernelEx(&cfg, lora_up_kernel<false>, a);
}

template <int NT, int U, int H, bool kBf16>
static cudaError_t lora_down_launch(const LoraDownArgs& a, cudaStream_t stream) {
  auto kernel = lora_down_kernel<NT, U, H, kBf16>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.M + 16 * kLoraWarps - 1) / (16 * kLoraWarps), a.splits);
  cfg.blockDim = dim3(kLoraWarps * H * 32);
  cfg.dynamicSmemBytes = lora_down_smem(NT);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = static_cast<unsigned>(a.splits);
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

cudaError_t launch_lora_down(const LoraDownArgs& a, cudaStream_t stream) {
  if (a.splits != 1 && a.splits != 2 && a.splits != 4 && a.splits != 8) return cudaErrorInvalidValue;
  if (a.k_per_split % 32 != 0) return cudaErrorInvalidValue;
  const int nt = (a.R + 7) / 8;
  // U keeps the operand registers per step group near 100.
  const bool b = a.bf16 != 0;
  if (nt <= 2) return b ? lora_down_launch<2, 2, 2, true>(a, stream) : lora_down_launch<2, 2, 2, false>(a, stream);
  if (nt <= 4) return b ? lora_down_launch<4, 2, 2, true>(a, stream) : lora_down_launch<4, 2, 2, false>(a, stream);
  if (nt <= 8) return b ? lora_down_launch<8, 1, 2, true>(a, stream) : lora_down_launch<8, 1, 2, false>(a, stream);
  if (nt <= 16) return b ? lora_down_launch<16, 1, 1, true>(a, stream) : lora_down_launch<16, 1, 1, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace convrot
