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
// Split-K units (kSplit) add their exact int32 partial into a zeroed
// workspace accumulator: 32-column boxes staged in shared memory and pushed
// with TMA bulk reduce-adds (per-element atomics only when Y leaves by plain
// stores).  Integer adds commute, so the sum is deterministic; the last split
// of a tile to arrive (an arrival counter) loads the sum back and writes the
// output.
// Pair variant (kPair): the two halves of K of one tile run on the two CTAs
// of a thread-block cluster, one tile per CTA.  After the drain each CTA
// stages the int32 sums of the other CTA's column half in its own (now idle)
// ring, pushes them with one bulk copy into the other CTA's ring (distributed
// shared memory, completing on that CTA's mbarrier), and finalizes its own
// column half with the partial it receives: wide tiles (whose MMAs keep the
// tensor pipe busy) without too few tiles, and no atomics.
// Launched with programmatic dependent launch: set-up (barriers, TMEM,
// descriptor prefetch) overlaps the previous kernel's tail; the first global
// access waits for that kernel's results.
//
// Fused variant (the whole layer in one launch, no LoRA): one CTA per SM, all
// co-resident (cooperative launch).  Each CTA first rotates and quantizes a
// contiguous share of the rows of X -- 256 segments of 64 values per pass,
// brought by TMA into the idle ring, one segment per epilogue thread: 6
// butterfly stages in registers, 2 across the 4 lanes of a 256-group, the row
// max by shuffles (and shared memory when a row spans warps) -- and writes
// the fp16 code image and s_X to the workspace, where they stay in L2.  The
// CTAs then meet at a grid barrier (an arrival counter, below) and run
// the GEMM above on the codes.  This removes the second launch, its
// dependency hand-off and the uneven tail of a separate prologue grid.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "fwht.cuh"
#include "kernels.h"

namespace convrot {

constexpr int kBM = 128;
constexpr int kBK = 64;            // fp16 elements per K block (128 bytes: one swizzle row)
constexpr int kChunkKB = 16;       // 64-wide K blocks per exact fp32 chunk (1024 K)
constexpr int kPrefetchKB = 16;    // weight K blocks brought into L2 before the dependency wait
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kIssuerWarp1 = 2 + kEpiWarps;  // the second MMA issuer (narrow tiles)
constexpr uint32_t kYBoxBytes = kBM * 64 * 2;  // one 128 x 64 fp16 store box (16 KB)

// Named barriers (0 is __syncthreads).
constexpr int kBarEpi = 1;    // all epilogue warps
constexpr int kBarHalf0 = 2;  // epilogue warps of column half 0 (+1 for half 1)
constexpr uint32_t kSendOff = 96 * 1024;  // pair: staged partial, inside the idle ring

// A ring stage holds KSUB consecutive 64-wide K blocks of A and B.  Every
// stage costs one full/empty hand-off between the TMA producer and the MMA
// issuer, which takes a few hundred cycles; only 256-wide MMAs hide it, so
// narrower tiles move 128 K per stage (8 MMAs per hand-off).
// Narrow tiles (BN <= 128) have two MMA-issuing threads in different warps.
// A 128-wide MMA keeps the tensor pipe busy for about as long as one thread
// needs to issue it, so any other work of the issuing thread (barrier waits,
// commits) shows as idle tensor cycles; a second issuer taking every other
// ring stage, into its own TMEM accumulator, hides it (measured: 63 % -> 100 %
// of the MMA rate for 128-K stages of 128-wide MMAs).  The epilogue adds the
// two accumulators: each holds at most half a 1024-K chunk, |.| <= 2^23, so
// their fp32 sum is exact.
// kTwoSmCfg: the MMAs span the two CTAs of a pair (256 x BN per MMA, each CTA
// holding its 128 rows of A and half of B's BN rows, 24 or 32 KB per stage).
template <int BN, bool kLoraCfg = false, bool kTwoSmCfg = false>
struct TcCfg {
  static constexpr int kIssuers = (BN <= 128) ? 2 : 1;
  static constexpr int kThreads = 64 + kEpiThreads + 32 * (kIssuers - 1);
  // 64-wide K blocks per stage: one, except for narrow tiles with a single
  // issuer (not built now), where two per stage halve the hand-offs.
  static constexpr int kSub = (BN == 256 || kIssuers == 2) ? 1 : 2;
  static constexpr uint32_t kABox = kBM * kBK * 2;              // 16 KB
  static constexpr uint32_t kBBox = (kTwoSmCfg ? BN / 2 : BN) * kBK * 2;
  static constexpr uint32_t kABytes = kSub * kABox;
  static constexpr uint32_t kBBytes = kSub * kBBox;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kTwoSmCfg ? (BN == 256 ? 6 : 8) : ((BN == 256) ? 4 : (BN == 128 ? 6 : 8));
  static constexpr int kChunkStages = kChunkKB / kSub;  // stages per exact fp32 chunk
  // Two chunk buffers x issuers accumulators of BN columns.
  static constexpr uint32_t kTmemCols = 2 * kIssuers * BN;
  static_assert(kTmemCols <= 512, "tensor memory");
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

// 16 columns of a chunk's accumulator for this thread's TMEM lane: with two
// issuers, the sum of their accumulators (BN columns apart; exact in fp32).
template <int kIssuers, int BN>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld_32x32b_x16(taddr, r);
  if constexpr (kIssuers == 2) {
    uint32_t r2[16];
    tmem_ld_32x32b_x16(taddr + BN, r2);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
  } else {
    tmem_wait_ld();
  }
}

// ------------------------------------------------------------ fused prologue
// Grid barrier of the fused kernel, with its state in the workspace:
//   sync[0] B  value of the arrival counter when this call started
//   sync[1] V  mix64(B) while the state is valid
//   sync[2] C  arrival counter
//   sync[3] W  (tag << 24 | count), used only to rebuild the state
// Fast path (V == mix64(B)): a CTA arrives with one atomicAdd on C and waits
// until C - B reaches the grid size; CTA 0 then advances B and V (every CTA
// read them before arriving, so the next call is the first to see them).  A
// zero-filled area is valid (mix64(0) = 0).  Anything else -- an
// uninitialized workspace, or one left by a call that timed out -- takes the
// rebuild path once: arrivals by compare-and-swap on W with a tag hashed from
// (B, V), which counts afresh whatever W held before (a stale word matches
// the 40-bit tag only by hash collision), after which CTA 0 writes the
// valid zero state.  The rebuild path serializes its compare-and-swaps (tens
// of microseconds); the fast path costs one atomic per CTA.
constexpr int kCountBits = 24;

// splitmix64 output function (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014); maps 0 to 0.
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Arrives (if `arrive`) and, if `wait`, waits for every CTA of the grid.  One
// thread per CTA; B and V are sync[0] and sync[1] as read at the start of the
// call.  Returns false on a timeout (after marking the state invalid).
static __device__ bool fused_grid_barrier(unsigned long long* sync, uint64_t B, uint64_t V, bool arrive,
                                   bool wait, int* err) {
  const uint64_t G = gridDim.x;
  const bool fast = V == mix64(B);
  const long long t0 = clock64();
  bool ok = true;
  if (fast) {
    if (arrive) {
      __threadfence();  // this CTA's codes and scales before its arrival
      atomicAdd(&sync[2], 1ull);
    }
    if (wait) {
      while (ld_relaxed_gpu(&sync[2]) - B < G) {
        if (clock64() - t0 > kWaitBudgetCycles) {
          ok = false;
          break;
        }
      }
    }
  } else {
    const uint64_t tag = mix64(B ^ mix64(V ^ 0x9e3779b97f4a7c15ull)) >> kCountBits;
    const uint64_t target = (tag << kCountBits) | G;
    if (arrive) {
      __threadfence();
      uint64_t old = *reinterpret_cast<volatile unsigned long long*>(&sync[3]);
      while (true) {
        const uint64_t want = ((old >> kCountBits) == tag) ? old + 1 : ((tag << kCountBits) | 1u);
        const uint64_t prev = atomicCAS(&sync[3], old, want);
        if (prev == old) break;
        old = prev;
        if (clock64() - t0 > kWaitBudgetCycles) {
          ok = false;
          break;
        }
      }
    }
    if (ok && wait) {
      while (ld_relaxed_gpu(&sync[3]) != target) {
        if (clock64() - t0 > kWaitBudgetCycles) {
          ok = false;
          break;
        }
      }
    }
  }
  if (!ok) {
    record_error(err, DEVERR_TIMEOUT_GRID);
    // Invalid, and different on every timeout, so the next call rebuilds
    // with a tag no earlier call used.
    sync[1] = mix64(B) ^ (1ull | (static_cast<uint64_t>(clock64()) << 1));
    return false;
  }
  if (wait) {
    __threadfence();
    fence_proxy_async_global();  // the codes are read next by TMA (async proxy)
    if (blockIdx.x == 0) {
      if (fast) {
        sync[0] = B + G;
        sync[1] = mix64(B + G);
      } else {
        sync[2] = 0;
        sync[0] = 0;
        sync[1] = 0;
      }
    }
  }
  return true;
}

// Rows [r0, r0 + nrows) of X are CTA b's share (of G CTAs).
__device__ __forceinline__ void fused_rows(int M, int G, int b, int& r0, int& nrows) {
  const int base_rows = M / G, extra = M % G;
  r0 = b * base_rows + min(b, extra);
  nrows = base_rows + (b < extra ? 1 : 0);
}

// Rotate + quantize of this CTA's share of the rows of X, by the 256
// epilogue threads (et = 0..255).  Pass buffers: two 32 KB halves of `xbuf`;
// `red` holds 8 floats.  Returns false if a wait timed out (the CTA then
// does not arrive at the grid barrier).
// The codes go back into the pass buffer in place (each thread rewrites the
// 128 bytes it read) and leave by TMA stores: one 256-segment box (tm_qs)
// for a pass of whole rows of this CTA, else one box per row (tm_qr, K/64
// segments), or -- when a row is shorter than the 1024-byte swizzle atom
// (K = 256) -- plain stores from the registers.
static __device__ bool fused_rotq_rows(const CUtensorMap* tm_x, const CUtensorMap* tm_qs,
                                const CUtensorMap* tm_qr, const GemmTcArgs& p, uint8_t* xbuf,
                                uint64_t* xbar, float* red, int et) {
  constexpr uint32_t kPassBytes = kEpiThreads * 128;  // 256 segments of 64 fp16
  const int ew = et >> 5;
  const int lane = et & 31;
  const int spr = p.K >> 6;           // segments per row: power of two, 4..256
  const int rpp = kEpiThreads / spr;  // rows per pass
  int r0, nrows;
  fused_rows(p.M, gridDim.x, blockIdx.x, r0, nrows);
  const int passes = (nrows + rpp - 1) / rpp;
  int issued[2] = {0, 0}, consumed[2] = {0, 0};  // thread et == 0's bookkeeping
  if (et == 0) {
    for (int q = 0; q < 2 && q < passes; ++q) {
      mbar_arrive_expect_tx(&xbar[q], kPassBytes);
      tma_load_2d(xbuf + q * kPassBytes, tm_x, &xbar[q], 0, (r0 + q * rpp) * spr);
      ++issued[q];
    }
  }
  bool ok = true;
  for (int i = 0; i < passes; ++i) {
    const int q = i & 1;
    if (et == 0 && i > 0 && i + 1 < passes) {
      // Buffer q^1 held pass i-1, whose codes are leaving by TMA store: once
      // the store has read them it takes pass i+1.
      tma_store_wait_read();
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&xbar[q ^ 1], kPassBytes);
      tma_load_2d(xbuf + (q ^ 1) * kPassBytes, tm_x, &xbar[q ^ 1], 0, (r0 + (i + 1) * rpp) * spr);
      ++issued[q ^ 1];
    }
    int got = 1;
    if (lane == 0) got = mbar_wait(&xbar[q], (i >> 1) & 1, p.err, DEVERR_TIMEOUT_PROLOGUE);
    got = __shfl_sync(0xffffffffu, got, 0);
    if (named_barrier_or(kBarEpi, kEpiThreads, !got)) {
      ok = false;
      break;
    }
    if (et == 0) ++consumed[q];
    uint8_t* rowp = xbuf + q * kPassBytes + et * 128;
    float v[64];
    load_swizzled_row<64>(rowp, et, 0, v);
    // Walsh-Hadamard transform of the 256-group: 6 stages over this thread's
    // 64 values, 2 over the 4 lanes holding the group.
    fwht_regs<64>(v);
    fwht_xlane<64>(v, lane, 1);
    fwht_xlane<64>(v, lane, 2);
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 64; ++e) amax = fmaxf(amax, fabsf(v[e]));
    if (spr <= 32) {
      for (int m = 1; m < spr; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    } else {
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      if (lane == 0) red[ew] = amax;
      named_barrier_sync(kBarEpi, kEpiThreads);
      const int wpr = spr >> 5;
      const int w0 = (ew / wpr) * wpr;
      float a = 0.0f;
      for (int w = 0; w < wpr; ++w) a = fmaxf(a, red[w0 + w]);
      amax = a;
      named_barrier_sync(kBarEpi, kEpiThreads);  // red[] is rewritten next pass
    }
    const int rows_here = min(rpp, nrows - i * rpp);  // rows of this CTA in the pass
    const bool by_tma = rows_here == rpp || spr >= 8;
    const int rr = i * rpp + et / spr;  // row within this CTA's share
    const int64_t m = r0 + rr;
    const int seg = et & (spr - 1);
    const float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
    if (rr < nrows && seg == 0) p.sx_out[m] = (amax * 0.0625f) / 127.0f;  // x 1/16 is exact
    uint4* dst = reinterpret_cast<uint4*>(p.qx_out + m * p.K + seg * 64);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float* w8 = v + c * 8;
      uint4 o;
      o.x = codes_f16x2(round_magic(w8[0], inv), round_magic(w8[1], inv));
      o.y = codes_f16x2(round_magic(w8[2], inv), round_magic(w8[3], inv));
      o.z = codes_f16x2(round_magic(w8[4], inv), round_magic(w8[5], inv));
      o.w = codes_f16x2(round_magic(w8[6], inv), round_magic(w8[7], inv));
      if (by_tma)
        *reinterpret_cast<uint4*>(rowp + ((c ^ (et & 7)) << 4)) = o;
      else if (rr < nrows)
        dst[c] = o;
    }
    if (by_tma) {
      fence_proxy_async_smem();
      named_barrier_sync(kBarEpi, kEpiThreads);
      if (et == 0) {
        uint8_t* buf = xbuf + q * kPassBytes;
        const int y = (r0 + i * rpp) * spr;
        if (rows_here == rpp) {
          tma_store_2d(tm_qs, buf, 0, y);
        } else {
          for (int r = 0; r < rows_here; ++r) tma_store_2d(tm_qr, buf + r * spr * 128, 0, y + r * spr);
        }
        tma_store_commit();
      }
    }
  }
  if (et == 0) {
    // Every code of this CTA written (not only read out of shared memory)
    // before the CTA arrives at the grid barrier.
    tma_store_wait_all();
    fence_proxy_async_global();
    // Leave no copy in flight (only after a timeout is anything outstanding).
    for (int q = 0; q < 2; ++q)
      if (issued[q] > consumed[q])
        mbar_wait(&xbar[q], static_cast<uint32_t>(issued[q] - 1) & 1u, p.err, DEVERR_TIMEOUT_DRAIN);
  }
  named_barrier_sync(kBarEpi, kEpiThreads);  // all codes of this CTA written
  return ok;
}

// Unit u: output tile (tile rows bm: 128, or 256 for a CTA pair's MMAs) and
// K split.
__device__ __forceinline__ Unit unit_of(int u, int tiles_m, int splits, int bn, int bm = kBM) {
  Unit r;
  r.split = u % splits;
  const int tile = u / splits;
  r.tile = tile;
  r.m0 = (tile % tiles_m) * bm;  // M fastest: concurrent tiles share weight tiles
  r.n0 = (tile / tiles_m) * bn;
  return r;
}

// kTwoSm: each unit is a 256 x BN tile computed by the two CTAs of a cluster
// with CTA-pair MMAs (.cta_group::2).  CTA rank c holds rows 128c.. of A and
// of the output and rows BN/2 * c.. of the B tile.  The even CTA ("leader")
// issues the MMAs; its full[] barriers take both CTAs' copies (the leader
// arms each stage for both CTAs' bytes, the odd CTA's copies complete on the
// leader's barrier).  The leader's commits reach both CTAs (multicast): the
// ring slots, the accumulators and the final drain, so each producer reloads
// its own slot as soon as the tensor cores are done with it.  A thread-to-
// thread hand-off per stage was measured to serialize the ring: a cluster-
// scope release arrival waits for the issuing warp's copies in flight.  The
// odd CTA's epilogue frees an accumulator by a remote arrival on the
// leader's barrier.
// kSplit: the variant that may split K (splits > 1, not the CTA pair); the
// others carry no split-K epilogue code (its registers cost the plain tiles).
// kExt: the variant whose epilogue adds a bias and writes bf16 Y or reads a
// bf16 LoRA up weight (EpilogueArgs); the plain ones stay fp16-only code.
template <int BN, bool kLora, bool kFused, bool kPair, bool kTwoSm = false, bool kSplit = false,
          bool kExt = false>
__global__ void __launch_bounds__(TcCfg<BN, kLora, kTwoSm>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_qs,
                   const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_y,
                   const GemmTcArgs p) {
  static_assert(!(kFused && kLora), "the fused kernel has no LoRA term");
  static_assert(!kPair || (!kFused && !kLora && BN >= 128), "pair variant: plain, wide tiles");
  static_assert(!kTwoSm || (!kFused && !kPair && BN >= 128), "pair MMAs: unfused, unsplit tiles");
  using C = TcCfg<BN, kLora, kTwoSm>;
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
  uint64_t* xbar = done + 1;            // [2] fused prologue passes / split-K reloads
  uint64_t* pair_bar = xbar + 2;  // [3] pair: partner's ring free, data in, partner read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pair_bar + 3);
  int* is_last = reinterpret_cast<int*>(tmem_slot + 1);
  int* abort_flag = is_last + 1;
  int* run_flag = abort_flag + 1;
  int* pair_sent = run_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kUnitM = kTwoSm ? 2 * kBM : kBM;  // output rows per unit
  const int tiles_m = (p.M + kUnitM - 1) / kUnitM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int units = tiles_m * tiles_n * p.splits;
  const int nkb_total = p.K / kBK;  // 64-wide K blocks (a multiple of 4)
  // Pair MMAs: units are dealt to clusters; this CTA's rows and B rows within
  // a unit.
  const uint32_t crank = kTwoSm ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int u_first = kTwoSm ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int u_step = kTwoSm ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int m_off = static_cast<int>(crank) * kBM;
  const int nb_off = static_cast<int>(crank) * (BN / 2);

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    if (p.tma_store) tma_prefetch_desc(&tm_y);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], C::kIssuers);  // one commit per issuer
      // Pair MMAs: both CTAs' epilogue warps free the leader's accumulator.
      mbar_init(&acce[a], kTwoSm ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(done, C::kIssuers);
    // xbar: the fused prologue's passes, or split K's reloads of the sum.
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    if (kFused) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_qs);
      tma_prefetch_desc(&tm_qr);
    } else if (p.splits > 1 && p.acc_tma) {
      tma_prefetch_desc(&tm_x);
    }
    if (kPair) {
      mbar_init(&pair_bar[0], 1);  // the partner's ring is free (its remote arrival)
      mbar_init(&pair_bar[1], 1);  // the partner's partial is in (local arm + copy bytes)
      mbar_init(&pair_bar[2], 1);  // the partner has read this CTA's staged partial
    }
    fence_mbarrier_init();
  }
  if (warp == 1) {
    if constexpr (kTwoSm) {
      tmem_alloc_pair(tmem_slot, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::kTmemCols);
      tmem_relinquish();
    }
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *pair_sent = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The partner may arrive on this CTA's barriers only once they exist.
  if (kPair || kTwoSm) cluster_sync_all();

  // The weight does not depend on the previous kernel: while that kernel
  // finishes, bring the first weight tiles of this CTA's first unit into L2.
  // With weight_early (the previous launch is this library's rotate +
  // quantize kernel, which signals its dependents only after its own
  // dependency wait, so whatever wrote the weight has completed), the first
  // ring stages are armed and their weight halves loaded right away; the
  // producer adds their A halves after the wait.
  // The early loads are issued by an epilogue thread (idle until the first
  // accumulator), so that the producer reaches the dependency wait at once:
  // the first TMA operations of a CTA take ~0.1 us each to issue, and the
  // CTAs of this kernel usually start after the previous kernel's last CTA
  // left their SM, i.e. right at the release.  Without early loads, an L2
  // prefetch of the first weight tiles is issued instead.
  int pre_b = 0;  // ring stages whose B half is issued early (producer and loaders)
  const bool loader = warp >= 2 && warp < 2 + kEpiWarps && lane == 0;  // stage (warp - 2)
  if (u_first < units && (threadIdx.x == 0 || loader)) {
    const Unit w = unit_of(u_first, tiles_m, p.splits, BN, kUnitM);
    const int kb0 = w.split * p.kb_per_split;
    const int kend = min(nkb_total, kb0 + p.kb_per_split);
    if (!kFused && !kTwoSm && p.weight_early) {
      pre_b = min(C::kStages, (kend - kb0 + C::kSub - 1) / C::kSub);
      // Epilogue warp e loads stages e, e + 8, ... (one TMA issue chain per
      // warp: the issues run in parallel).
      if (loader) {
        for (int i = warp - 2; i < pre_b; i += kEpiWarps) {
          mbar_arrive_expect_tx(&full[i], C::kStageBytes);
#pragma unroll
          for (int q = 0; q < C::kSub; ++q)
            tma_load_2d(sB + i * C::kBBytes + q * C::kBBox, &tm_b, &full[i],
                        (kb0 + i * C::kSub + q) * kBK, w.n0);
        }
      }
    } else if (threadIdx.x == 0) {
      const int kb1 = min(kend, kb0 + kPrefetchKB);
      for (int kb = kb0; kb < kb1; ++kb) tma_prefetch_l2_2d(&tm_b, kb * kBK, w.n0 + nb_off);
    }
  }
  if (kFused && threadIdx.x == 64) {
    // This CTA's rows of X, into L2 (a prefetch returns nothing to the SM and
    // L2 is the point of coherence: safe before the dependency wait).
    int r0, nrows;
    fused_rows(p.M, gridDim.x, blockIdx.x, r0, nrows);
    const int spr = p.K >> 6;
    const int rpp = kEpiThreads / spr;
    for (int r = 0; r < nrows && r < 8 * rpp; r += rpp) tma_prefetch_l2_2d(&tm_x, 0, (r0 + r) * spr);
  }

  // Everything above touched only this CTA's own resources and the weight.
  // From here on the kernel reads what the previous kernel on the stream
  // wrote.
  grid_dep_wait();
  grid_dep_launch();

  bool run = true;
  if constexpr (kFused) {
    // ---------------------------------------------------- rotate + quantize
    // The ring is idle until the GEMM starts: its first 64 KB (inside the A
    // half of the ring) hold the passes.  Meanwhile the producer loads the B
    // (weight) half of the first stages, which does not depend on X.
    if (warp == 0 && lane == 0 && blockIdx.x < units) {
      const Unit w = unit_of(blockIdx.x, tiles_m, p.splits, BN);
      const int kb0 = w.split * p.kb_per_split;
      const int kb1 = min(nkb_total, kb0 + p.kb_per_split);
      for (int kb = kb0; kb < kb1 && pre_b < C::kStages; kb += C::kSub, ++pre_b) {
        mbar_arrive_expect_tx(&full[pre_b], C::kStageBytes);
#pragma unroll
        for (int q = 0; q < C::kSub; ++q)
          tma_load_2d(sB + pre_b * C::kBBytes + q * C::kBBox, &tm_b, &full[pre_b],
                      (kb + q) * kBK, w.n0);
      }
    }
    static_assert(2 * kEpiThreads * 128 <= C::kStages * C::kABytes, "passes fit the A half");
    if (warp >= 2 && warp < kIssuerWarp1) {
      const int et = threadIdx.x - 64;
      uint64_t sb = 0, sv = 0;
      if (et == 0) {
        sb = *reinterpret_cast<volatile unsigned long long*>(&p.sync[0]);
        sv = *reinterpret_cast<volatile unsigned long long*>(&p.sync[1]);
      }
      const bool ok = fused_rotq_rows(&tm_x, &tm_qs, &tm_qr, p, base, xbar, sx_s, et);
      if (et == 0) {
        // CTAs without a GEMM unit only contribute rows: they do not wait.
        const bool waits = blockIdx.x < units;
        const bool through = fused_grid_barrier(p.sync, sb, sv, ok, ok && waits, p.err);
        *run_flag = (through && waits) ? 1 : 0;
      }
    }
    __syncthreads();
    run = *reinterpret_cast<volatile int*>(run_flag) != 0;
    if (run && warp == 0 && lane == 0) {
      // The pass buffers were read through the generic proxy; the ring loads
      // below write them through the async proxy.
      fence_proxy_async_smem();
      fence_proxy_async_global();
    }
  }

  if (!run) {
    // A CTA without GEMM work, or a failed grid barrier.  Stages armed before
    // the barrier still expect their A half: load it (any codes will do) so
    // that no copy is left in flight, and wait for them.
    if (warp == 0 && lane == 0 && pre_b > 0) {
      const Unit w = unit_of(blockIdx.x, tiles_m, p.splits, BN);
      const int kb0 = w.split * p.kb_per_split;
      fence_proxy_async_smem();
      for (int i = 0; i < pre_b; ++i)
#pragma unroll
        for (int q = 0; q < C::kSub; ++q)
          tma_load_2d(sA + i * C::kABytes + q * C::kABox, &tm_a, &full[i],
                      (kb0 + i * C::kSub + q) * kBK, w.m0);
      for (int i = 0; i < pre_b; ++i) mbar_wait(&full[i], 0, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;  // K blocks issued by this CTA so far (ring position)
      bool ok = true;
      for (int u = u_first; u < units && ok; u += u_step) {
        const Unit w = unit_of(u, tiles_m, p.splits, BN, kUnitM);
        const int kb0 = w.split * p.kb_per_split;
        const int kb1 = min(nkb_total, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; kb += C::kSub, ++it) {
          const int s = it % C::kStages;
          if constexpr (kTwoSm) {
            if (leader) {
              if (!mbar_wait(&empty[s], ((it / C::kStages) & 1) ^ 1, p.err, DEVERR_TIMEOUT_EMPTY)) {
                ok = false;
                break;
              }
              // Both CTAs' bytes (the odd CTA's copies may land first: the
              // transaction count may go negative until this arrival).
              mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
#pragma unroll
              for (int q = 0; q < C::kSub; ++q) {
                tma_load_2d(sA + s * C::kABytes + q * C::kABox, &tm_a, &full[s], (kb + q) * kBK, w.m0);
                tma_load_2d(sB + s * C::kBBytes + q * C::kBBox, &tm_b, &full[s], (kb + q) * kBK, w.n0);
              }
            } else {
              // The leader's commits free this CTA's stage too (multicast).
              if (!mbar_wait(&empty[s], ((it / C::kStages) & 1) ^ 1, p.err, DEVERR_TIMEOUT_EMPTY)) {
                ok = false;
                break;
              }
              const uint32_t fb = map_to_cta(&full[s], 0);
#pragma unroll
              for (int q = 0; q < C::kSub; ++q) {
                tma_load_2d_peer_bar(sA + s * C::kABytes + q * C::kABox, &tm_a, fb, (kb + q) * kBK,
                                     w.m0 + m_off);
                tma_load_2d_peer_bar(sB + s * C::kBBytes + q * C::kBBox, &tm_b, fb, (kb + q) * kBK,
                                     w.n0 + nb_off);
              }
            }
            continue;
          }
          if (it < pre_b) {
            // Armed before the barrier with its B half already loading.
#pragma unroll
            for (int q = 0; q < C::kSub; ++q)
              tma_load_2d(sA + s * C::kABytes + q * C::kABox, &tm_a, &full[s], (kb + q) * kBK,
                          w.m0);
            continue;
          }
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
      // Pair MMAs: the leader's full[] barriers count the odd CTA's copies
      // too.  The odd CTA waits for the commit that consumed its last load
      // of every slot: then that load has landed (on an aborted run the
      // bounded wait outlasts any copy in flight).
      if (!kTwoSm || leader) {
        for (int i = max(0, it - C::kStages); i < it; ++i)
          mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1, p.err, DEVERR_TIMEOUT_DRAIN);
      } else {
        for (int i = max(0, it - C::kStages); i < it; ++i)
          mbar_wait(&empty[i % C::kStages], (i / C::kStages) & 1, p.err, DEVERR_TIMEOUT_DRAIN);
      }
    }
  } else if (warp == 1 || (C::kIssuers == 2 && warp == kIssuerWarp1)) {
    // ------------------------------------------------------------ MMA issuers
    if (kTwoSm && !leader) {
      // The odd CTA issues nothing; its tensor memory and shared memory stay
      // until the leader's last MMA (multicast commit) has completed.
      if (warp == 1 && lane == 0) mbar_wait_cluster(done, 0, p.err, DEVERR_TIMEOUT_DRAIN);
    } else if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kTwoSm ? 2 * kBM : kBM, BN);
      const int t = (warp == 1) ? 0 : 1;  // this issuer takes the stages it % kIssuers == t
      bool ok = true;
      int it = 0;  // ring stages consumed by both issuers so far (ring position)
      int gc = 0;  // chunks issued (accumulator buffer = gc & 1)
      for (int u = u_first; u < units && ok; u += u_step) {
        const Unit w = unit_of(u, tiles_m, p.splits, BN, kUnitM);
        const int kb0 = w.split * p.kb_per_split;
        const int nkb = max(0, min(nkb_total, kb0 + p.kb_per_split) - kb0);
        const int nst = nkb / C::kSub;  // stages of this unit
        for (int c0 = 0; c0 < nst && ok; c0 += C::kChunkStages, ++gc) {
          const int a = gc & 1;
          const bool freed =
              kTwoSm ? mbar_wait_cluster(&acce[a], ((gc >> 1) & 1) ^ 1, p.err, DEVERR_TIMEOUT_ACC_EMPTY)
                     : mbar_wait(&acce[a], ((gc >> 1) & 1) ^ 1, p.err, DEVERR_TIMEOUT_ACC_EMPTY);
          if (!freed) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (a * C::kIssuers + t) * BN;
          const int n = min(nst, c0 + C::kChunkStages) - c0;  // stages of this chunk
          // This issuer's stages of the chunk, and only those: ring stage
          // it + j for j = t, t + kIssuers, ... (a flat loop: walking the
          // other issuer's stages too measurably slows the issue rate).
          for (int j = (t - it % C::kIssuers + C::kIssuers) % C::kIssuers; j < n;
               j += C::kIssuers) {
            const int g = it + j;
            const int s = g % C::kStages;
            if (!mbar_wait(&full[s], (g / C::kStages) & 1, p.err, DEVERR_TIMEOUT_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + s * C::kABytes);
            const uint32_t b_addr = smem_u32(sB + s * C::kBBytes);
            const bool first = j < C::kIssuers;  // this issuer's first stage of the chunk
#pragma unroll
            for (int q = 0; q < C::kSub; ++q) {
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint32_t acc_flag = (!first || q > 0 || kk > 0) ? 1u : 0u;
                const uint64_t ad = smem_desc_k128(a_addr + q * C::kABox + kk * 32);
                const uint64_t bd = smem_desc_k128(b_addr + q * C::kBBox + kk * 32);
                if constexpr (kTwoSm)
                  tc_mma_f16_pair(d_tmem, ad, bd, idesc, acc_flag);
                else
                  tc_mma_f16(d_tmem, ad, bd, idesc, acc_flag);
              }
            }
            if constexpr (kTwoSm)
              tc_commit_pair_mc(&empty[s], 0x3);  // both CTAs' stage s is free
            else
              tc_commit(&empty[s]);
          }
          it += n;
          if (ok) {
            if constexpr (kTwoSm)
              tc_commit_pair_mc(&accf[a], 0x3);  // both CTAs' epilogues
            else
              tc_commit(&accf[a]);
          }
        }
      }
      // Every MMA issued so far must be complete before the accumulators are
      // freed.
      if constexpr (kTwoSm)
        tc_commit_pair_mc(done, 0x3);
      else
        tc_commit(done);
      mbar_wait(done, 0, p.err, DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp < kIssuerWarp1) {
    // ------------------------------------------------------------ epilogue
    constexpr int kHalf = C::kEpiCols;
    const int et = threadIdx.x - 64;  // 0..255
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int row = quad * 32 + lane;  // row within the tile
    // The thread that issues this half's TMA stores (BN = 64: one for both).
    const bool issuer = (BN == 64) ? (et == 0) : ((ew & 3) == 0 && lane == 0);
    // The bulk-copy issuer of this column half (split-K partial boxes).
    const bool issuer_h = (ew & 3) == 0 && lane == 0;
    uint32_t xuse = 0;  // split K: loads of this half's staging buffer so far
    int gc = 0;
    for (int u = u_first; u < units; u += u_step) {
      const Unit w = unit_of(u, tiles_m, p.splits, BN, kUnitM);
      const int m0c = w.m0 + m_off;  // this CTA's first output row
      const int kb0 = w.split * p.kb_per_split;
      const int nkb = max(0, min(nkb_total, kb0 + p.kb_per_split) - kb0);
      // sum[]: the int32 partial sums of this thread's row and columns, or --
      // once `as_float` -- the fp32 bit patterns of (float)A.  The float form
      // skips the float <-> int conversions (a slow pipe) on the exposed last
      // chunk: a chunk value is an exact integer with |c| <= 2^24, so with a
      // single chunk the accumulator already is (float)A; with more, the
      // earlier chunks are summed in int32 while the next chunk's MMAs run,
      // and if every partial S has |S| <= 2^24 it is converted to fp32
      // exactly, and fp32(S + c) rounds the exact integer S + c once, i.e.
      // equals (float)A.  Split and pair partials stay in int32.
      // `as_float` is uniform across each warp (the TMEM loads of the drain
      // are warp-collective): one row beyond 2^24 keeps its warp in int32.
      int32_t sum[kHalf];
#pragma unroll
      for (int i = 0; i < kHalf; ++i) sum[i] = 0;
      const int nchunks = (nkb / C::kSub + C::kChunkStages - 1) / C::kChunkStages;
      const bool float_ok = !kPair && p.splits == 1 && p.tma_store;
      // CTA-pair K split with one chunk per K half: each half's partial is an
      // exact integer of at most 2^24 in magnitude, i.e. an exact fp32, and
      // the fp32 sum of the two rounds the exact A once: (float)A.  Both CTAs
      // of the pair have the same number of chunks, so they agree.
      bool as_float = (float_ok || (kPair && p.tma_store)) && nchunks == 1;
      int ci = 0;
      // This unit's scales, loaded now so their latency hides behind the MMAs;
      // they go to shared memory once the previous unit's readers are done.
      float sw_reg = 0.0f, sx_reg = 0.0f;
      if (kPair) {
        // Own column half only: thread hi of the half loads column hi, and
        // every thread the scale of its own row.
        const int hi = (ew & 3) * 32 + lane;
        const int n = w.n0 + half * kHalf + hi;
        if (hi < kHalf && n < p.N) sw_reg = p.ep.sW[n];
        if (m0c + row < p.M) sx_reg = __ldcg(&p.ep.sX[m0c + row]);
      } else if (p.tma_store) {
        if (et < BN && w.n0 + et < p.N) sw_reg = p.ep.sW[w.n0 + et];
        // s_X may have been written by other CTAs of this grid (fused): read
        // it from L2, never from a stale L1 line.
        if (et < kBM && m0c + et < p.M) sx_reg = __ldcg(&p.ep.sX[m0c + et]);
      }
      const bool lora_fast = kLora && p.ep.R > 0 && p.tma_store;
      for (int c0 = 0; c0 < nkb / C::kSub; c0 += C::kChunkStages, ++gc, ++ci) {
        const int a = gc & 1;
        if (*reinterpret_cast<volatile int*>(abort_flag) == 0) {
          // One lane per warp polls the barrier; the others block in the
          // shuffle instead of spinning on shared memory next to the MMAs.
          int got = 1;
          if (lane == 0)
            got = kTwoSm ? mbar_wait_cluster(&accf[a], (gc >> 1) & 1, p.err, DEVERR_TIMEOUT_ACC_FULL)
                         : mbar_wait(&accf[a], (gc >> 1) & 1, p.err, DEVERR_TIMEOUT_ACC_FULL);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            *abort_flag = 1;
          } else {
            tc_fence_after();
            const uint32_t t0 = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                a * C::kIssuers * BN + half * kHalf;
            if (as_float) {
#pragma unroll
              for (int j = 0; j < kHalf / 16; ++j) {
                uint32_t r[16];
                tmem_ld_chunk<C::kIssuers, BN>(t0 + j * 16, r);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  sum[j * 16 + e] =
                      __float_as_int(__int_as_float(sum[j * 16 + e]) + __uint_as_float(r[e]));
              }
            } else {
#pragma unroll
              for (int j = 0; j < kHalf / 16; ++j) {
                uint32_t r[16];
                tmem_ld_chunk<C::kIssuers, BN>(t0 + j * 16, r);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  sum[j * 16 + e] += __float2int_rn(__uint_as_float(r[e]));
              }
            }
            tc_fence_before();
          }
        }
        __syncwarp();
        if (lane == 0) {
          if (kTwoSm && !leader)
            mbar_arrive_remote(map_to_cta(&acce[a], 0));  // the leader's accumulator barrier
          else
            mbar_arrive(&acce[a]);
        }
        if (float_ok && !as_float && ci == nchunks - 2) {
          // Before the last chunk: into fp32 if every partial is exact there.
          // Decided per WARP: the drain above is a warp-collective TMEM load
          // and must not run under a divergent branch.
          int mx = 0;
#pragma unroll
          for (int i = 0; i < kHalf; ++i) mx = max(mx, abs(sum[i]));
          if (__all_sync(0xffffffffu, mx <= (1 << 24))) {
#pragma unroll
            for (int i = 0; i < kHalf; ++i) sum[i] = __float_as_int(static_cast<float>(sum[i]));
            as_float = true;
          }
        }
      }

      // The whole epilogue group agrees on what to do with this unit.
      named_barrier_sync(kBarEpi, kEpiThreads);
      const bool aborted = *reinterpret_cast<volatile int*>(abort_flag) != 0;
      const int64_t m = static_cast<int64_t>(m0c) + row;
      const int nb = w.n0 + half * kHalf;
      const bool row_ok = m < p.M;
      bool write = !aborted;
      if constexpr (kPair) {
        // ------------------------------------------------ pair reduction
        const uint32_t c = cluster_ctarank();  // = this CTA's K half
        const uint32_t q = c ^ 1u;             // the partner
        constexpr uint32_t kRowBytes = kHalf * 4 + 16;  // padded: no bank conflicts
        constexpr uint32_t kBlockBytes = kBM * kRowBytes;
        static_assert(kSendOff + kBlockBytes <= C::kRingBytes, "pair buffers fit the ring");
        uint8_t* recv = base;             // the partner's partial of this CTA's half
        uint8_t* send = base + kSendOff;  // this CTA's partial of the partner's half
        const int hi = (ew & 3) * 32 + lane;  // thread index within its half
        if (!aborted && hi == 0) {
          if (half == static_cast<int>(c)) {
            // Expect the partner's block; then tell the partner that this
            // CTA's MMAs are done, so its ring may be written.
            mbar_arrive_expect_tx(&pair_bar[1], kBlockBytes);
            mbar_arrive_remote(map_to_cta(&pair_bar[0], q));
          }
        }
        int got = aborted ? 0 : 1;
        if (half != static_cast<int>(c)) {
          // This half belongs to the partner: each warp stages its 32 rows
          // and sends them with its own bulk copy (four copies in flight; the
          // partner's barrier expects the whole block).  The words are the
          // int32 partials, or their exact fp32 values (as_float).
          constexpr uint32_t kWarpBytes = 32 * kRowBytes;
          if (got) {
            uint8_t* dst = send + row * kRowBytes;
#pragma unroll
            for (int j = 0; j < kHalf; j += 4)
              *reinterpret_cast<uint4*>(dst + j * 4) =
                  make_uint4(static_cast<uint32_t>(sum[j]), static_cast<uint32_t>(sum[j + 1]),
                             static_cast<uint32_t>(sum[j + 2]), static_cast<uint32_t>(sum[j + 3]));
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0 && got) {
            if (mbar_wait_cluster(&pair_bar[0], 0, p.err, DEVERR_TIMEOUT_CLUSTER)) {
              bulk_copy_to_cta(map_to_cta(recv + quad * kWarpBytes, q), send + quad * kWarpBytes,
                               kWarpBytes, map_to_cta(&pair_bar[1], q));
              *pair_sent = 1;
            }
          }
          write = false;
        } else {
          // Own half: add the partner's partial of the same rows and columns.
          if (lane == 0 && got) got = mbar_wait_cluster(&pair_bar[1], 0, p.err, DEVERR_TIMEOUT_CLUSTER);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (got) {
            const uint8_t* src = recv + row * kRowBytes;
            if (as_float) {
#pragma unroll
              for (int j = 0; j < kHalf; j += 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + j * 4);
                sum[j] = __float_as_int(__int_as_float(sum[j]) + __uint_as_float(v.x));
                sum[j + 1] = __float_as_int(__int_as_float(sum[j + 1]) + __uint_as_float(v.y));
                sum[j + 2] = __float_as_int(__int_as_float(sum[j + 2]) + __uint_as_float(v.z));
                sum[j + 3] = __float_as_int(__int_as_float(sum[j + 3]) + __uint_as_float(v.w));
              }
            } else {
#pragma unroll
              for (int j = 0; j < kHalf; j += 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + j * 4);
                sum[j] += static_cast<int32_t>(v.x);
                sum[j + 1] += static_cast<int32_t>(v.y);
                sum[j + 2] += static_cast<int32_t>(v.z);
                sum[j + 3] += static_cast<int32_t>(v.w);
              }
            }
            // The copy that filled recv has finished reading the partner's
            // staging: let the partner go.
            if (hi == 0) mbar_arrive_remote(map_to_cta(&pair_bar[2], q));
          }
          write = got != 0;
        }
      }
      if constexpr (kSplit && !kPair) {
      if (!aborted && p.splits > 1 && p.acc_tma) {
        // Add this split's exact int32 partial into acc through L2: boxes of
        // 32 columns x 128 rows, staged 128-byte swizzled in this half's
        // buffer and pushed with TMA bulk reduce-adds; the last split to
        // arrive loads the sum back.
        constexpr int kRBoxes = (kHalf >= 32) ? kHalf / 32 : 1;
        uint8_t* rbuf = staging + half * kYBoxBytes;
        const int hb = kBarHalf0 + half;
        constexpr int hn = kEpiThreads / 2;
#pragma unroll
        for (int b = 0; b < kRBoxes; ++b) {
          if (issuer_h) tma_store_wait_read();  // the buffer's previous copy has read it
          named_barrier_sync(hb, hn);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int i = b * 32 + c * 4;
            *reinterpret_cast<uint4*>(rbuf + row * 128 + ((c ^ (row & 7)) << 4)) =
                make_uint4(static_cast<uint32_t>(sum[i]), static_cast<uint32_t>(sum[i + 1]),
                           static_cast<uint32_t>(sum[i + 2]), static_cast<uint32_t>(sum[i + 3]));
          }
          fence_proxy_async_smem();
          named_barrier_sync(hb, hn);
          if (issuer_h) {
            if (nb + b * 32 < p.N && m0c < p.M) tma_reduce_add_2d(&tm_x, rbuf, nb + b * 32, m0c);
            tma_store_commit();
          }
        }
        if (issuer_h) {
          // This half's adds have completed in global memory before the
          // split arrives.
          tma_store_wait_all();
          fence_proxy_async_global();
          __threadfence();
        }
        named_barrier_sync(kBarEpi, kEpiThreads);
        if (et == 0) {
          const int prev = atomicAdd(&p.counters[w.tile], 1);
          *is_last = (prev == p.splits - 1) ? 1 : 0;
        }
        named_barrier_sync(kBarEpi, kEpiThreads);
        write = *reinterpret_cast<volatile int*>(is_last) != 0;
        if (write) {
          __threadfence();
          fence_proxy_async_global();  // the sum is read by TMA (async proxy)
#pragma unroll
          for (int b = 0; b < kRBoxes; ++b) {
            if (issuer_h) {
              mbar_arrive_expect_tx(&xbar[half], kYBoxBytes);
              tma_load_2d(rbuf, &tm_x, &xbar[half], nb + b * 32, m0c);
            }
            int got = 1;
            if (lane == 0) got = mbar_wait(&xbar[half], xuse & 1, p.err, DEVERR_TIMEOUT_DRAIN);
            got = __shfl_sync(0xffffffffu, got, 0);
            ++xuse;
            if (!got) write = false;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v =
                  *reinterpret_cast<const uint4*>(rbuf + row * 128 + ((c ^ (row & 7)) << 4));
              const int i = b * 32 + c * 4;
              sum[i] = static_cast<int32_t>(v.x);
              sum[i + 1] = static_cast<int32_t>(v.y);
              sum[i + 2] = static_cast<int32_t>(v.z);
              sum[i + 3] = static_cast<int32_t>(v.w);
            }
            named_barrier_sync(hb, hn);  // read before the next box lands
          }
          // A timed-out load leaves its half unwritten; the error is recorded.
          write = named_barrier_or(kBarEpi, kEpiThreads, !write) ? false : write;
          // Leave the accumulator tile and its counter zero for the next
          // call on this workspace (16-byte stores: N is a multiple of 8).
          if (write && row_ok) {
            int4* dst = reinterpret_cast<int4*>(p.acc + m * p.N + nb);
#pragma unroll
            for (int c = 0; c < kHalf / 4; ++c)
              if (nb + 4 * c < p.N) dst[c] = make_int4(0, 0, 0, 0);
          }
          if (write && et == 0) p.counters[w.tile] = 0;
        }
      } else if (!aborted && p.splits > 1) {
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
          // Leave the accumulator tile and its counter zero for the next call.
#pragma unroll
          for (int i = 0; i < kHalf; ++i)
            if (row_ok && nb + i < p.N) p.acc[m * p.N + nb + i] = 0;
          if (et == 0) p.counters[w.tile] = 0;
        }
      }
      }  // kSplit
      if (write && p.tma_store) {
        float sx;
        if constexpr (kPair) {
          // Only this half's threads are here: half-local barrier.
          const int hi = (ew & 3) * 32 + lane;
          if (hi < kHalf) sw_s[half * kHalf + hi] = sw_reg;
          named_barrier_sync(kBarHalf0 + half, kEpiThreads / 2);
          sx = sx_reg;
        } else {
          // Scales of this tile into shared memory (the previous unit's
          // readers are past the barrier above).
          if (et < BN) sw_s[et] = sw_reg;
          if (et < kBM) sx_s[et] = sx_reg;
          named_barrier_sync(kBarEpi, kEpiThreads);
          sx = sx_s[row];
        }
        // Boxes of 64 columns; half h owns boxes [h*kHalf/64, (h+1)*kHalf/64)
        // (BN = 64: both halves share box 0).
        // LoRA: this thread's row of the precomputed sums S = T up^T.
        const float* srow = lora_fast ? p.ep.S + (static_cast<int64_t>(m0c) + row) * p.N : nullptr;
        if (!as_float) {
          // int32 sums (split, pair, or partials beyond 2^24): (float)A.
#pragma unroll
          for (int i = 0; i < kHalf; ++i) sum[i] = __float_as_int(static_cast<float>(sum[i]));
        }
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
            for (int e = 0; e < 16; ++e) {
              if constexpr (kExt)
                y[e] = scale_bias(__int_as_float(sum[cl + e]), sx, sw_s[half * kHalf + cl + e],
                                  p.ep.bias, nb + cl + e, p.N);
              else
                y[e] = (__int_as_float(sum[cl + e]) * sx) * sw_s[half * kHalf + cl + e];
            }
            if (lora_fast) {
              // + lora_scale * S[m, n] (columns past N read nothing; N is a
              // multiple of 8 here, so a float4 lies wholly inside or outside).
              if (row_ok) {
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                  const int n = nb + cl + e;
                  const float4 sv = (n < p.N) ? *reinterpret_cast<const float4*>(srow + n)
                                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                  y[e + 0] = y[e + 0] + p.ep.lora_scale * sv.x;
                  y[e + 1] = y[e + 1] + p.ep.lora_scale * sv.y;
                  y[e + 2] = y[e + 2] + p.ep.lora_scale * sv.z;
                  y[e + 3] = y[e + 3] + p.ep.lora_scale * sv.w;
                }
              }
            }
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
              // column within the box: BN = 64 puts both halves in one box
              const int col = ((BN == 64) ? half * kHalf : 0) + g * 16 + h8 * 8;
              const int chunk = col >> 3;
              uint4 o;
              const bool obf = kExt && p.ep.out_bf16 != 0;
              o.x = pack_out2(y[h8 * 8 + 0], y[h8 * 8 + 1], obf);
              o.y = pack_out2(y[h8 * 8 + 2], y[h8 * 8 + 3], obf);
              o.z = pack_out2(y[h8 * 8 + 4], y[h8 * 8 + 5], obf);
              o.w = pack_out2(y[h8 * 8 + 6], y[h8 * 8 + 7], obf);
              *reinterpret_cast<uint4*>(buf + row * 128 + ((chunk ^ (row & 7)) << 4)) = o;
            }
          }
          fence_proxy_async_smem();
          named_barrier_sync(bar, bar_n);
          if (issuer) {
            const int x = (BN == 64) ? w.n0 : w.n0 + half * kHalf + b * 64;
            // (A pair-MMA tile's odd half may lie wholly below row M.)
            if (x < p.N && m0c < p.M) tma_store_2d(&tm_y, buf, x, m0c);
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
          epilogue_store<G, kLora, kExt>(p.ep, p.N, m, nb + j * G, sg);
        }
      }
    }
    // Shared memory must outlive the stores' reads of it; the writes
    // themselves complete with the grid.
    if (issuer) tma_store_wait_read();
  }

  // Pair: before this CTA's shared memory goes away, the partner's remote
  // arrivals on it must have landed ("ring free" always; "read" once this CTA
  // sent its block, whose source the copy reads).  On the normal path both
  // have long arrived; nothing else of the partner reaches a CTA that did not
  // itself signal first.
  // All roles meet here before the tensor memory is released.
  __syncthreads();
  if (kPair && threadIdx.x == 64) {
    mbar_wait_cluster(&pair_bar[0], 0, p.err, DEVERR_TIMEOUT_CLUSTER);
    if (*reinterpret_cast<volatile int*>(pair_sent))
      mbar_wait_cluster(&pair_bar[2], 0, p.err, DEVERR_TIMEOUT_CLUSTER);
  }
  // Pair MMAs: neither CTA leaves (or frees tensor memory) while the other
  // may still arrive on its barriers or the leader's copies and MMAs touch
  // its shared memory: every role above ends after bounded waits, so both
  // CTAs reach this cluster barrier.
  if (kTwoSm) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kTwoSm)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, bool kLora, bool kFused, bool kPair = false, bool kTwoSm = false,
          bool kSplit = false, bool kExt = false>
static cudaError_t launch_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_qs,
                             const CUtensorMap& tm_qr, const CUtensorMap& tm_a,
                             const CUtensorMap& tm_b, const CUtensorMap& tm_y, const GemmTcArgs& a,
                             int grid, bool pdl, bool coop, cudaStream_t stream) {
  using C = TcCfg<BN, kLora, kTwoSm>;
  const size_t smem = C::kSmem;
  auto fn = gemm_tc_kernel<BN, kLora, kFused, kPair, kTwoSm, kSplit, kExt>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  int n = 0;
  if (kPair || kTwoSm) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (coop) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, fn, tm_x, tm_qs, tm_qr, tm_a, tm_b, tm_y, a);
}

// The launchers of one epilogue kind (kExt: bias / bf16 fields honoured).
// The extended kinds are instantiated in their own translation unit
// (gemm_tc_ext.cu includes this file with CONVROT_GEMM_EXT_TU defined) so
// that the two sets compile in parallel.
template <bool kExt>
static cudaError_t tc_launch(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                             const CUtensorMap& tm_y, const CUtensorMap& tm_acc,
                             const GemmTcArgs& a, int bn, int grid, cudaStream_t stream) {
  const bool lora = a.ep.mode == kOutF16 && a.ep.R > 0;
  // The unfused kernel reads its tm_x slot only as the split-K accumulator.
  const CUtensorMap& none = tm_acc;
  if (a.splits > 1) {
    switch (bn) {
      case 256:
        return lora ? launch_tc<256, true, false, false, false, true, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                    : launch_tc<256, false, false, false, false, true, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
      case 128:
        return lora ? launch_tc<128, true, false, false, false, true, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                    : launch_tc<128, false, false, false, false, true, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
      case 64:
        return lora ? launch_tc<64, true, false, false, false, true, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                    : launch_tc<64, false, false, false, false, true, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 256:
      return lora ? launch_tc<256, true, false, false, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                  : launch_tc<256, false, false, false, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
    case 128:
      return lora ? launch_tc<128, true, false, false, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                  : launch_tc<128, false, false, false, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
    case 64:
      return lora ? launch_tc<64, true, false, false, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                  : launch_tc<64, false, false, false, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

template <bool kExt>
static cudaError_t pair_launch(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                               const CUtensorMap& tm_y, const GemmTcArgs& a, int bn, int grid,
                               cudaStream_t stream) {
  const CUtensorMap& none = tm_a;
  switch (bn) {
    case 256: return launch_tc<256, false, false, true, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
    case 128: return launch_tc<128, false, false, true, false, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <bool kExt>
static cudaError_t pair_mma_launch(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                   const CUtensorMap& tm_y, const GemmTcArgs& a, int bn,
                                   int clusters, cudaStream_t stream) {
  const CUtensorMap& none = tm_a;
  const int grid = 2 * clusters;
  const bool lora = a.ep.mode == kOutF16 && a.ep.R > 0;
  switch (bn) {
    case 256:
      return lora ? launch_tc<256, true, false, false, true, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                  : launch_tc<256, false, false, false, true, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
    case 128:
      return lora ? launch_tc<128, true, false, false, true, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream)
                  : launch_tc<128, false, false, false, true, false, kExt>(none, none, none, tm_a, tm_b, tm_y, a, grid, true, false, stream);
    default: return cudaErrorInvalidValue;
  }
}

#ifdef CONVROT_GEMM_EXT_TU

cudaError_t launch_gemm_tc_ext(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                               const CUtensorMap& tm_y, const CUtensorMap& tm_acc,
                               const GemmTcArgs& a, int bn, int grid, cudaStream_t stream) {
  return tc_launch<true>(tm_a, tm_b, tm_y, tm_acc, a, bn, grid, stream);
}

cudaError_t launch_gemm_pair_ext(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                 const CUtensorMap& tm_y, const GemmTcArgs& a, int bn, int grid,
                                 cudaStream_t stream) {
  return pair_launch<true>(tm_a, tm_b, tm_y, a, bn, grid, stream);
}

cudaError_t launch_gemm_pair_mma_ext(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                     const CUtensorMap& tm_y, const GemmTcArgs& a, int bn,
                                     int clusters, cudaStream_t stream) {
  return pair_mma_launch<true>(tm_a, tm_b, tm_y, a, bn, clusters, stream);
}

#else

size_t gemm_tc_smem_bytes(int bn) {
  return bn == 256 ? TcCfg<256>::kSmem : (bn == 128 ? TcCfg<128>::kSmem : TcCfg<64>::kSmem);
}

static bool ext_epilogue(const GemmTcArgs& a) {
  return a.ep.bias != nullptr || a.ep.out_bf16 != 0 || a.ep.lora_bf16 != 0;
}

// Clusters of two CTAs of the pair-MMA kernel that can be resident at once.
template <int BN>
static int pair_mma_clusters() {
  using C = TcCfg<BN, false, true>;
  auto fn = gemm_tc_kernel<BN, false, false, false, true>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(C::kSmem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) return 0;
  return n;
}

int gemm_pair_mma_max_clusters(int bn) {
  switch (bn) {
    case 256: return pair_mma_clusters<256>();
    case 128: return pair_mma_clusters<128>();
    default: return 0;
  }
}

cudaError_t launch_gemm_pair_mma(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                 const CUtensorMap& tm_y, const GemmTcArgs& a, int bn,
                                 int clusters, cudaStream_t stream) {
  if (ext_epilogue(a)) return launch_gemm_pair_mma_ext(tm_a, tm_b, tm_y, a, bn, clusters, stream);
  return pair_mma_launch<false>(tm_a, tm_b, tm_y, a, bn, clusters, stream);
}

cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_y,
                           const CUtensorMap& tm_acc, const GemmTcArgs& a, int bn, int grid,
                           cudaStream_t stream) {
  if (ext_epilogue(a)) return launch_gemm_tc_ext(tm_a, tm_b, tm_y, tm_acc, a, bn, grid, stream);
  return tc_launch<false>(tm_a, tm_b, tm_y, tm_acc, a, bn, grid, stream);
}

cudaError_t launch_gemm_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                             const CUtensorMap& tm_y, const GemmTcArgs& a, int bn, int grid,
                             cudaStream_t stream) {
  if (ext_epilogue(a)) return launch_gemm_pair_ext(tm_a, tm_b, tm_y, a, bn, grid, stream);
  return pair_launch<false>(tm_a, tm_b, tm_y, a, bn, grid, stream);
}

// The single-kernel engine takes plain fp16 epilogues only.
cudaError_t launch_gemm_fused(const CUtensorMap& tm_x, const CUtensorMap& tm_qs,
                              const CUtensorMap& tm_qr, const CUtensorMap& tm_a,
                              const CUtensorMap& tm_b, const CUtensorMap& tm_y,
                              const GemmTcArgs& a, int bn, int grid, int mode,
                              cudaStream_t stream) {
  if (ext_epilogue(a)) return cudaErrorInvalidValue;
  const bool pdl = mode == 0;
  switch (bn) {
    case 256: return launch_tc<256, false, true, false, false, true>(tm_x, tm_qs, tm_qr, tm_a, tm_b, tm_y, a, grid, pdl, true, stream);
    case 128: return launch_tc<128, false, true, false, false, true>(tm_x, tm_qs, tm_qr, tm_a, tm_b, tm_y, a, grid, pdl, true, stream);
    case 64: return launch_tc<64, false, true, false, false, true>(tm_x, tm_qs, tm_qr, tm_a, tm_b, tm_y, a, grid, pdl, true, stream);
    default: return cudaErrorInvalidValue;
  }
}

#endif  // CONVROT_GEMM_EXT_TU

}  // namespace convrot
