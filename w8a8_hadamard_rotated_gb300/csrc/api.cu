// Host side of the INT8ConvRot C ABI (include/convrot.h): argument checks,
// device checks, workspace carving, engine choice by shape, TMA descriptor
// encoding and kernel launches.  Everything here is enqueued on the caller's
// stream; nothing allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <utility>

#include "../../include/convrot.h"
#include "kernels.h"

namespace convrot {
namespace {

// Device error flag: a kernel that gives up on a bounded wait records a code
// here (first writer wins); convrot_check_device_error() reads and clears it.
__device__ int g_device_error;

constexpr int64_t kGroup = 256;
constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;
constexpr int kSplitTileLimit = 1024;  // split-K only when there are fewer 128x128 tiles
constexpr int kSkinnyAutoMaxM = 16;    // auto path: skinny kernel for M <= this
// Weight images up to this size are brought into L2 by the rotate + quantize
// kernel ahead of the GEMM.  Measured per layer at M=1024: 0.1-0.3 us faster for
// 1-4 MB images, no change at 8 MB, 1-2 us slower at 32 MB (the prefetch then
// competes with the activation reads for HBM).
constexpr size_t kL2WeightPrefetchMax = size_t{8} << 20;

struct DeviceInfo {
  bool init = false;
  bool supported = false;
  int sms = 0;
  int* err = nullptr;
  // Launch mode of the fused kernel, settled by its first launch outside a
  // stream capture: -1 unknown, 0 cooperative + programmatic dependent
  // launch, 1 cooperative only, 2 unavailable (two-kernel path).
  int fused_mode = -1;
  // Resident 2-CTA clusters of the pair-MMA GEMM for tile widths 128 and
  // 256 (-1: not queried yet, 0: unavailable).
  // (A cache filled on first use: mutable through const references.)
  mutable int pair_mma_clusters[2] = {-1, -1};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Test hook: forced tile width / split count for the tensor-core GEMM (0 = auto).
int g_force_bn = 0;
int g_force_splits = 0;
// Test hook (convrot_set_split_mode): 0 automatic, 1 never the CTA-pair
// split, 2 the CTA-pair split wherever it applies.
int g_split_mode = 0;
// Test hook (convrot_set_pair_mma): 0 automatic, 1 never the pair-MMA GEMM,
// 2 the pair-MMA GEMM wherever it applies.
int g_pair_mma_mode = 0;
// 1 selects the single-kernel layer (convrot_set_fused).  Off by default:
// on GB300 its grid barrier and the reload of the codes after it cost more
// than the launch hand-off it removes (the two-kernel engine is faster on
// every measured shape).
int g_fused_enabled = 0;
// Small-M engine: 0 auto, 1 two kernels, 2 the one-launch layer in its
// 32-column dp4a form at every M <= 16, 3 the one-launch layer in its
// 128-row fp16-MMA form at every M <= 16, 4 the one-launch layer with the
// rotation shared by the column blocks of a cluster wherever it applies
// (auto elsewhere).
int g_small_m_mode = 0;
// The two-kernel path's small-M GEMM: 0 auto, 1 the mma.sync s8 kernel with
// register loads, 2 the fp16-MMA kernel with bulk copies (where it applies).
int g_skinny_engine = 0;
// 1 (default): the one-launch layer copies its weight before the dependency
// wait (no kernel of this library that writes int8 data lets the next
// kernel start before it finishes).
int g_small_m_weights_early = 1;
// Auto mode takes the one-launch layer up to this M.
constexpr int64_t kDecodeAutoMaxM = 2;

// The 4x4 Hadamard base B of H = B (x) B (x) B (x) B / 16
// (convrot_set_hadamard_base; Sylvester's by default).  A symmetric 4x4
// Hadamard matrix factors as B = D1 H4 R, with D1 a diagonal of signs, H4
// Sylvester's matrix and R a signed permutation, so H = D H_S R4 with
// D = D1 (x) D1 (x) D1 (x) D1, H_S the Sylvester H and R4 = R (x) R (x) R (x) R.
// The kernels negate the inputs by D and run the Sylvester transform; R4
// (a signed permutation of the rotated columns, the same for X and W) is not
// applied: quantization commutes with it and the product Q_X Q_W^T does not
// see it, so Y is that of base B, with the codes in the library's order.
struct HadamardBase {
  bool sylvester = true;    // B is Sylvester's matrix itself
  uint32_t sign[8] = {};    // bit k: D[k] = -1 (k = 0..255)
  bool any_sign() const {
    for (uint32_t w : sign)
      if (w) return true;
    return false;
  }
};
HadamardBase g_base;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

convrot_status current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CONVROT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CONVROT_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return CONVROT_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
    if (d.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return CONVROT_ERR_CUDA;
      d.err = static_cast<int*>(p);
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
          return CONVROT_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
    d.init = true;
  }
  if (!d.supported) return CONVROT_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return CONVROT_OK;
}

// 2-D fp16 tensor map over a row-major [rows, cols] array, box [box_rows, 64],
// 128-byte swizzle, zero fill outside the array.
convrot_status make_map_f16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                            uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONVROT_OK : CONVROT_ERR_CUDA;
}

// 2-D int32 tensor map over a row-major [rows, cols] array, box [128, 32]
// (128 bytes wide: the 128-byte swizzle span), zero fill outside the array.
convrot_status make_map_s32(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void*>(ptr), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONVROT_OK : CONVROT_ERR_CUDA;
}

convrot_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA; }

bool valid_k(int64_t K) { return K > 0 && K % kGroup == 0 && K <= CONVROT_MAX_K; }
// M and N travel to the kernels as int (element offsets are 64-bit there).
bool valid_dim(int64_t v) { return v >= 0 && v <= CONVROT_MAX_DIM; }

// ---------------------------------------------------------------- planning
struct TcPlan {
  int bn = 256;
  int splits = 1;
  int kb_per_split = 0;
  bool pair = false;  // K split in two across a 2-CTA cluster (one tile per CTA)
  bool pair_mma = false;  // 256 x bn tiles on CTA-pair MMAs (.cta_group::2)
  int clusters = 0;       // pair_mma: persistent 2-CTA clusters
  bool stream = false;    // K halves on a 2-CTA cluster, streaming exchange (gemm_pairk.cu)
};

bool tc_may_split(int64_t M, int64_t N) { return cdiv(M, 128) * cdiv(N, 128) < kSplitTileLimit; }

// Picks the tile width and K split for the persistent GEMM.  Model: the
// units (tiles x splits) are dealt round-robin to one CTA per SM; the busiest
// CTA runs ceil(units / SMs) main loops back to back (tensor cycles per K
// block, narrower tiles a little less efficient) while its epilogues overlap
// the next unit's MMAs, plus one fixed cost (set-up, pipeline fill, the last
// epilogue); split-K adds the cost of its int32 atomics, which serialize in L2.
//
// The pair option (allow_pair: fp16 output through TMA stores, no LoRA) runs
// the two K halves of each tile on the two CTAs of a cluster, one tile per
// CTA, in ceil(tiles * 2 / SMs) waves; each CTA finalizes half the tile's
// columns after a shared-memory exchange.
//
// The pair-MMA option (pair_clusters given: fp16 output through TMA stores,
// LoRA allowed; pair_clusters[i] resident clusters for bn = 128, 256) runs
// 256 x bn tiles on the two CTAs of a cluster with
// MMAs that span both SMs, in ceil(tiles / clusters) waves.  Per SM the main
// loop runs at the 1-SM rate of the same width (each SM still reads its A
// rows and both halves of B from shared memory per MMA), but the operands
// come from L2 once per 256 rows instead of once per 128.  So every option's
// time is max(main loops, operand bytes / L2 bandwidth) plus its fixed
// costs: large layers are bound by L2 (measured: 4096^3 with 1-SM tiles
// streams ~10 TB/s of operands and takes 1.7x the pair-MMA time), small ones
// by the tensor pipe and the fixed costs, where 1-SM tiles win (the pair
// adds ~1 us of cluster hand-offs).  Auto mode considers 256-wide pair tiles
// only: at 128 wide the pair never measured faster than 1-SM tiles.
TcPlan plan_tc(int64_t M, int64_t N, int64_t K, int sms, bool allow_pair, int max_bn = 256,
               const int* pair_clusters = nullptr, bool tma_split = false,
               bool allow_stream = false) {
  const int64_t nkb = K / 64;
  TcPlan best;
  double best_cost = 1e300;
  // Streaming CTA-pair split (allow_stream: fp16 output through TMA stores,
  // no LoRA, no bias; K <= 2048 so that each half is one exact fp32 chunk):
  // one 128 x bn tile per 2-CTA cluster, not persistent, so every wave pays
  // the fixed costs: the first stage, the exchange of the partner's fp32
  // half (32 or 64 KB) through distributed shared memory and the epilogue.
  // Those per-wave costs are set against the other engines' models on the
  // measured layers (M = 1024: N = 256, K = 2048 in 8.26 us against 9.31 us
  // for the int32 pair split; N = K = 2048 in 12.8 us against 11.5 us for
  // 1-SM 128-wide tiles; N = 2048, K = 1024 in 9.7 us against 7.85 us).
  if (allow_stream && K <= 2048 && (g_split_mode == 0 || g_split_mode == 3) &&
      g_pair_mma_mode != 2 && (!g_force_splits || g_force_splits == 2)) {
    for (int bn : {256, 128}) {
      if (g_force_bn && bn != g_force_bn) continue;
      const int64_t units = cdiv(M, 128) * cdiv(N, bn) * 2;
      const int64_t waves = cdiv(units, sms);
      const double loop = (nkb / 2) * (bn == 256 ? 620.0 : 435.0);
      const double cost = waves * (loop + (bn == 256 ? 13500.0 : 5700.0));
      if (g_split_mode == 3 || cost < best_cost - 1e-9) {
        best_cost = g_split_mode == 3 ? -1.0 : cost;
        best = TcPlan{};
        best.bn = bn;
        best.splits = 2;
        best.kb_per_split = static_cast<int>(nkb / 2);
        best.stream = true;
      }
    }
    if (g_split_mode == 3 && best.stream) return best;
  }
  // Measured main-loop cycles per 64-wide K block by tile width.
  auto kb_cycles = [](int bn) { return bn == 256 ? 600.0 : (bn == 128 ? 435.0 : 410.0); };
  // The same for pair-MMA tiles (per SM: each holds 128 x bn of the output).
  auto kb_cycles_pair = [](int bn) { return bn == 256 ? 615.0 : 435.0; };
  // Operand bytes (fp16 images) from L2 to the SMs per cycle: ~14 TB/s
  // measured across the GEMM shapes at ~1.9 GHz.
  auto l2_cycles = [](double bytes) { return bytes / 7370.0; };
  if (pair_clusters && g_pair_mma_mode != 1 && g_split_mode != 2 &&
      (!g_force_splits || g_force_splits == 1)) {
    for (int bn : {256, 128}) {
      if (g_force_bn && bn != g_force_bn) continue;
      if (bn == 128 && g_pair_mma_mode != 2) continue;
      const int clusters_max = pair_clusters[bn == 256 ? 1 : 0];
      if (clusters_max <= 0) continue;
      const int64_t units = cdiv(M, 256) * cdiv(N, bn);
      const int64_t clusters = std::min<int64_t>(units, clusters_max);
      const int64_t waves = cdiv(units, clusters);
      const double loops = waves * (nkb * kb_cycles_pair(bn) + 400.0);
      const double cost = std::max(loops, l2_cycles(static_cast<double>(units) * (256 + bn) * K * 2)) +
                          2500.0 + 16.0 * bn + 2000.0;
      if (g_pair_mma_mode == 2 || cost < best_cost - 1e-9) {
        best_cost = g_pair_mma_mode == 2 ? -1.0 : cost;
        best.bn = bn;
        best.splits = 1;
        best.kb_per_split = static_cast<int>(nkb);
        best.pair = false;
        best.pair_mma = true;
        best.stream = false;
        best.clusters = static_cast<int>(clusters);
      }
    }
    if (g_pair_mma_mode == 2 && best.pair_mma) return best;
  }
  if (allow_pair && g_split_mode != 1 && nkb % 8 == 0 && (!g_force_splits || g_force_splits == 2)) {
    for (int bn : {256, 128}) {
      if (g_force_bn && bn != g_force_bn) continue;
      const int64_t units = cdiv(M, 128) * cdiv(N, bn) * 2;
      const int64_t waves = cdiv(units, sms);
      // Exchange (stage, bulk copy of the partial, wait, add): measured ~3 us
      // for 256-wide tiles, ~1.5 us for 128-wide.
      const double exchange = bn == 256 ? 6000.0 : 3000.0;
      const double loops = waves * ((nkb / 2) * kb_cycles(bn) + 400.0);
      const double cost =
          std::max(loops, l2_cycles(static_cast<double>(units) * (128 + bn) * (K / 2) * 2)) +
          2500.0 + 16.0 * bn + exchange;
      if (g_split_mode == 2 || cost < best_cost - 1e-9) {
        best_cost = g_split_mode == 2 ? -1.0 : cost;
        best.bn = bn;
        best.splits = 2;
        best.kb_per_split = static_cast<int>(nkb / 2);
        best.pair = true;
        best.pair_mma = false;
        best.stream = false;
      }
      if (g_split_mode == 2) return best;
    }
  }
  for (int bn : {256, 128, 64}) {
    if (g_force_bn && bn != g_force_bn) continue;
    if (bn > max_bn && !(g_force_bn == bn)) continue;
    const int64_t tiles = cdiv(M, 128) * cdiv(N, bn);
    const int64_t max_s = tc_may_split(M, N) ? std::min<int64_t>(16, nkb) : 1;
    for (int64_t s = 1; s <= max_s; ++s) {
      if (g_force_splits && s != g_force_splits && g_force_splits <= max_s) continue;
      // Split boundaries fall on multiples of 256 K (whole ring stages).
      const int64_t kbps = cdiv(cdiv(nkb, s), 4) * 4;
      const int64_t s_eff = cdiv(nkb, kbps);
      if (s_eff != s) continue;
      const int64_t per_cta = cdiv(tiles * s_eff, sms);
      const double unit = kbps * kb_cycles(bn) + 400.0;
      const double fixed = 2500.0 + 16.0 * bn;
      // tma_split: each split pushes its 128 x bn int32 partial into L2 with
      // TMA bulk reduce-adds and the last one reloads the sum.  The adds are
      // a shared resource: measured ~1.7 TB/s for the whole GPU (16.8 MB of
      // partials cost ~11 us at M=1024 N=2048 K=2048, 2 splits of 256-wide
      // tiles), i.e. ~880 bytes per cycle, plus ~2.3 us of hand-off (the
      // counter, the last split's reload, the prologue's zeroing).  Measured:
      // M=128 N=2048 K=8192 in 4 splits of 64-wide tiles 20.9 us (the CTA-pair
      // split 26.9 us); M=1024 N=256 K=2048 the CTA-pair split stays ahead
      // (9.7 us against 10.0).  Otherwise one int32 atomic per
      // element, a lane per row (32 cache lines per warp instruction):
      // measured ~4.5x the cost of a coalesced stream (M=128, N=2048,
      // K=8192, 4 splits: ~30 us).
      const double atomics =
          s_eff <= 1 ? 0.0
          : tma_split ? 4500.0 + static_cast<double>(tiles * s_eff) * 128 * bn * 4 / 880.0
                      : 3000.0 + static_cast<double>(s_eff) * M * N / (0.16 * sms);
      const double operands = static_cast<double>(tiles) * (128 + bn) * K * 2;
      const double cost = std::max(per_cta * unit, l2_cycles(operands)) + fixed + atomics;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best.bn = bn;
        best.splits = static_cast<int>(s_eff);
        best.kb_per_split = static_cast<int>(kbps);
        best.pair = false;
        best.pair_mma = false;
        best.stream = false;
      }
    }
  }
  if (best.kb_per_split == 0) {  // forced values that do not fit: plain tiles
    best.pair = false;
    best.pair_mma = false;
    best.stream = false;
    best.bn = g_force_bn ? g_force_bn : 256;
    best.splits = 1;
    best.kb_per_split = static_cast<int>(nkb);
  }
  return best;
}

bool use_skinny(int64_t M, int path) {
  if (path == CONVROT_PATH_SKINNY) return true;
  if (path == CONVROT_PATH_TCGEN05) return false;
  return M <= kSkinnyAutoMaxM;
}

// ---------------------------------------------------------------- workspace
struct LinearLayout {
  size_t sync = 0;
  size_t qx = 0, sx = 0, t = 0, s = 0, wimg = 0, acc = 0, cnt = 0, total = 0;
};

LinearLayout linear_layout(int64_t M, int64_t N, int64_t K, int64_t R, bool with_img, bool skinny) {
  LinearLayout L;
  size_t off = 0;
  // Fixed place at the start: the fused kernel's grid-barrier state, carried
  // from call to call.
  L.sync = off;
  off += kAlign;
  L.qx = off;
  off += align_up(static_cast<size_t>(M) * K * (skinny ? 1 : 2));
  L.sx = off;
  off += align_up(static_cast<size_t>(M) * 4);
  L.t = off;
  if (R > 0) off += align_up(static_cast<size_t>(M) * R * 4);
  // LoRA sums S = T lora_up^T, fp32 [M, N] (written by the GEMM stage).
  L.s = off;
  if (R > 0) off += align_up(static_cast<size_t>(M) * N * 4);
  L.wimg = off;
  if (!skinny && !with_img) off += align_up(static_cast<size_t>(N) * K * 2);
  L.acc = off;
  if (skinny || tc_may_split(M, N)) off += align_up(static_cast<size_t>(M) * N * 4);
  L.cnt = off;
  // Split-K tile counters (tiles as narrow as 64 columns), then the
  // small-M engine's 32-column blocks.
  off += align_up(static_cast<size_t>(cdiv(M, 128) * cdiv(N, 64) + cdiv(N, 32)) * 4);
  L.total = off;
  return L;
}

LinearLayout linear_layout_max(int64_t M, int64_t N, int64_t K, int64_t R, bool with_img) {
  // Large enough for either engine (the choice depends on M only).
  const LinearLayout a = linear_layout(M, N, K, R, with_img, use_skinny(M, CONVROT_PATH_AUTO));
  return a;
}

struct GemmLayout {
  size_t a_img = 0, b_img = 0, acc = 0, cnt = 0, total = 0;
};

GemmLayout gemm_layout(int64_t M, int64_t N, int64_t K, bool skinny) {
  GemmLayout L;
  size_t off = 0;
  if (!skinny) {
    L.a_img = off;
    off += align_up(static_cast<size_t>(M) * K * 2);
    L.b_img = off;
    off += align_up(static_cast<size_t>(N) * K * 2);
  }
  L.acc = off;
  if (skinny || tc_may_split(M, N)) off += align_up(static_cast<size_t>(M) * N * 4);
  L.cnt = off;
  // Split-K tile counters (tiles as narrow as 64 columns), then the
  // small-M engine's 32-column blocks.
  off += align_up(static_cast<size_t>(cdiv(M, 128) * cdiv(N, 64) + cdiv(N, 32)) * 4);
  L.total = off;
  return L;
}

uint8_t* at(void* ws, size_t off) { return static_cast<uint8_t*>(ws) + off; }

// ---------------------------------------------------------------- launches
// zero / zero_bytes (a multiple of 16): a range the tile kernel also sets to
// zero (the next GEMM's split-K accumulator); *zeroed tells whether it did.
// in_bf16: X holds bf16 values (otherwise fp16).
// l2_pf / l2_pf_bytes: the next GEMM's weight image, which the tile kernel
// brings into L2 before its dependency wait (ignored by the row kernel).
convrot_status run_rotq(const DeviceInfo& d, const uint16_t* X, int64_t M, int64_t K, void* q_out,
                        bool out_f16, float* s_out, cudaStream_t st, void* zero = nullptr,
                        size_t zero_bytes = 0, bool* zeroed = nullptr, bool in_bf16 = false,
                        bool rot_only = false, const void* l2_pf = nullptr,
                        size_t l2_pf_bytes = 0, bool early_dependents = true) {
  if (zeroed) *zeroed = false;
  const int64_t lpr = K / 64;
  const bool pow2 = (lpr & (lpr - 1)) == 0;
  if (pow2 && K <= 16384) {
    // 64 values per lane (one shuffle stage fewer than 32); 32 with 4-warp
    // tiles (twice the threads) only when there is less than half a warp's
    // worth of segments per SM.  Tiles of 64 values per lane are as small as
    // a row allows (one warp for K <= 2048): fine-grained tiles keep the SMs
    // evenly loaded when the previous kernel's tail leaves some SMs free
    // earlier than others (measured 3 % faster layers at K = 256..2048 than
    // 4-warp tiles).  Rows of up to 1024 values take 32 values per lane in
    // one-warp tiles: twice the CTAs, each half the work (measured at M=1024:
    // K=256 1.89 us against 2.22 us, K=1024 2.50 us against 2.69 us; at
    // K=8192 the same choice was slower, 9.24 us against 8.21 us).
    const int64_t segments = M * K / 64;
    const bool small = segments < static_cast<int64_t>(d.sms) * 16 && K <= 8192;
    const int vpl = (small || K <= 1024) ? 32 : 64;
    const int64_t warps_per_row = std::max<int64_t>(1, K / (32 * vpl));
    const int warps = static_cast<int>(std::max<int64_t>(small ? 4 : 1, warps_per_row));
    RotqTileArgs a;
    a.segments = segments;
    a.tiles = cdiv(segments, static_cast<int64_t>(warps) * 32 * vpl / 64);
    a.K = static_cast<int>(K);
    a.warps = warps;
    a.vpl = vpl;
    a.q_out = q_out;
    a.s_out = s_out;
    a.err = d.err;
    a.in_bf16 = in_bf16 ? 1 : 0;
    a.rot_only = rot_only ? 1 : 0;
    a.zero = static_cast<uint4*>(zero);
    a.zero_n16 = zero ? static_cast<int64_t>(zero_bytes / 16) : 0;
    a.l2_pf = l2_pf;
    a.l2_pf_bytes = l2_pf ? static_cast<int64_t>(l2_pf_bytes) : 0;
    a.early_dependents = early_dependents ? 1 : 0;
    std::memcpy(a.sign, g_base.sign, sizeof(a.sign));
    a.has_sign = g_base.any_sign() ? 1 : 0;
    if (zeroed) *zeroed = zero != nullptr;
    CUtensorMap map, qmap;
    const uint32_t box = static_cast<uint32_t>(warps * 32 * vpl / 64);
    convrot_status s = make_map_f16(&map, X, static_cast<uint64_t>(segments), 64, box);
    if (s != CONVROT_OK) return s;
    qmap = map;  // not read by the int8 variant
    if (out_f16) {
      s = make_map_f16(&qmap, q_out, static_cast<uint64_t>(segments), 64, box);
      if (s != CONVROT_OK) return s;
    }
    // Up to 8 CTAs per SM for the short rows (one tile each at the sweep's
    // sizes); 4 with a two-tile persistent loop for the long ones (measured
    // best at K = 8192).
    const int per_sm = K <= 2048 ? 8 : 4;
    const int grid = static_cast<int>(std::min<int64_t>(a.tiles, static_cast<int64_t>(d.sms) * per_sm));
    // At most ceil(grid / SMs) CTAs per SM: one even wave, however many SMs
    // the previous kernel still holds when the first CTAs start.
    const int cap = static_cast<int>(cdiv(grid, d.sms));
    return from_cuda(launch_rotq_tile(map, qmap, a, out_f16, grid, cap, st));
  }
  if (rot_only) return CONVROT_ERR_INVALID_ARG;  // the row kernel writes codes only
  if (zero) {
    if (cudaMemsetAsync(zero, 0, zero_bytes, st) != cudaSuccess) return CONVROT_ERR_CUDA;
    if (zeroed) *zeroed = true;
  }
  RotqRowArgs a;
  a.in = X;
  a.rows = M;
  a.K = static_cast<int>(K);
  a.q_out = out_f16 ? nullptr : static_cast<int8_t*>(q_out);
  a.img_out = out_f16 ? static_cast<uint16_t*>(q_out) : nullptr;
  a.s_out = s_out;
  std::memcpy(a.sign, g_base.sign, sizeof(a.sign));
  const int grid = static_cast<int>(std::min<int64_t>(M, static_cast<int64_t>(d.sms) * 8));
  return from_cuda(launch_rotq_row(a, in_bf16 ? kRowInBf16 : kRowInF16, grid, st));
}

convrot_status run_widen(const DeviceInfo& d, const int8_t* in, uint16_t* out, int64_t n,
                         cudaStream_t st) {
  const int64_t n16 = n / 16;  // n is a multiple of 256
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(n16, 256), d.sms * 8)));
  return from_cuda(launch_widen_i8(in, out, n, grid, st));
}

// Resident clusters of the pair-MMA kernel, queried once per device.
void pair_mma_query(const DeviceInfo& d) {
  for (int i = 0; i < 2; ++i) {
    if (d.pair_mma_clusters[i] >= 0) continue;
    std::lock_guard<std::mutex> lock(g_mu);
    d.pair_mma_clusters[i] = gemm_pair_mma_max_clusters(i == 0 ? 128 : 256);
  }
}

// The tensor-core plan for a GEMM with fp16 output Y (or int32/other output
// when !f16_out) and R LoRA ranks; have_acc: a split-K accumulator exists.
// plain_out: fp16 Y without a bias (the streaming pair split's epilogue).
TcPlan gemm_tc_plan(const DeviceInfo& d, int64_t M, int64_t N, int64_t K, bool tma_store, int64_t R,
                    bool have_acc, bool plain_out = false) {
  // The CTA-pair K splits (exchange of int32 or fp32 partials) take no LoRA
  // term; the pair-MMA tiles do (their epilogue is the 1-SM tiles').
  const bool plain = tma_store && R == 0;
  if (tma_store) pair_mma_query(d);
  TcPlan plan = plan_tc(M, N, K, d.sms, plain, 256,
                        tma_store ? d.pair_mma_clusters : nullptr, tma_store, plain && plain_out);
  if (plan.splits > 1 && !plan.pair && !plan.stream && !have_acc)
    plan = TcPlan{plan.bn, 1, static_cast<int>(K / 64)};
  return plan;
}

// Whether the plan adds split partials in the workspace accumulator (which
// must then be zero, with its tile counters, when the GEMM starts).
bool plan_uses_acc(const TcPlan& p) { return p.splits > 1 && !p.pair && !p.pair_mma && !p.stream; }

bool tma_store_ok(const EpilogueArgs& ep, int64_t N) {
  return ep.mode == kOutF16 && (N % 8) == 0 && aligned16(ep.Y);
}

// Runs A = Q_X Q_W^T on the tensor cores from fp16 operand images and applies
// the epilogue `ep`.  acc_zeroed: the previous launch (this call's prologue)
// zeroed the accumulator and its counters.
convrot_status run_gemm_tc(const DeviceInfo& d, const uint16_t* a_img, const uint16_t* b_img,
                           int64_t M, int64_t N, int64_t K, const EpilogueArgs& ep, int32_t* acc,
                           int* cnt, cudaStream_t st, bool weight_early = false,
                           bool acc_zeroed = false) {
  const bool tma_store = tma_store_ok(ep, N);
  const bool plain_out = ep.mode == kOutF16 && !ep.bias && !ep.out_bf16 && !ep.lora_bf16;
  const TcPlan plan = gemm_tc_plan(d, M, N, K, tma_store, ep.R, acc != nullptr, plain_out);
  CUtensorMap ma, mb, my;
  memset(&my, 0, sizeof(my));
  convrot_status s = make_map_f16(&ma, a_img, M, K, 128);
  if (s != CONVROT_OK) return s;
  // Pair-MMA tiles: each CTA loads half of the tile's B rows.
  s = make_map_f16(&mb, b_img, N, K, static_cast<uint32_t>(plan.pair_mma ? plan.bn / 2 : plan.bn));
  if (s != CONVROT_OK) return s;
  // fp16 Y goes out through TMA stores when its rows are 16-byte multiples.
  if (tma_store) {
    s = make_map_f16(&my, ep.Y, M, N, 128);
    if (s != CONVROT_OK) return s;
  }
  GemmTcArgs g;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.splits = plan.splits;
  g.kb_per_split = plan.kb_per_split;
  g.acc = acc;
  g.counters = cnt;
  g.tma_store = tma_store ? 1 : 0;
  g.ep = ep;
  g.err = d.err;
  g.weight_early = weight_early ? 1 : 0;
  // Split partials go through L2 with TMA bulk reduce-adds where the output
  // also leaves by TMA (rows of 16-byte multiples); per-element atomics
  // otherwise.
  const bool uses_acc = plan_uses_acc(plan);
  g.acc_tma = (uses_acc && tma_store) ? 1 : 0;
  CUtensorMap macc = ma;  // read only as the split-K accumulator
  if (g.acc_tma) {
    s = make_map_s32(&macc, acc, M, N);
    if (s != CONVROT_OK) return s;
  }
  if (plan.pair_mma)
    return from_cuda(launch_gemm_pair_mma(ma, mb, my, g, plan.bn, plan.clusters, st));
  if (plan.stream) return from_cuda(launch_gemm_pairk(ma, mb, my, g, plan.bn, st));
  const int64_t units = cdiv(M, 128) * cdiv(N, plan.bn) * plan.splits;
  if (plan.pair)  // one tile half per CTA: the grid is every unit
    return from_cuda(launch_gemm_pair(ma, mb, my, g, plan.bn, static_cast<int>(units), st));
  if (uses_acc && !acc_zeroed) {
    if (cudaMemsetAsync(acc, 0, static_cast<size_t>(M) * N * 4, st) != cudaSuccess ||
        cudaMemsetAsync(cnt, 0, static_cast<size_t>(cdiv(M, 128) * cdiv(N, plan.bn)) * 4, st) !=
            cudaSuccess)
      return CONVROT_ERR_CUDA;
  }
  const int grid = static_cast<int>(std::min<int64_t>(units, d.sms));
  return from_cuda(launch_gemm_tc(ma, mb, my, macc, g, plan.bn, grid, st));
}

bool fused_eligible(const DeviceInfo& d, int64_t K, int64_t R, bool skinny, cudaStream_t st) {
  const int64_t spr = K / 64;
  if (!g_fused_enabled || skinny || R > 0 || K < 256 || K > kFusedMaxK || (spr & (spr - 1)) != 0)
    return false;
  if (g_base.any_sign()) return false;  // its rotation is Sylvester's only
  if (d.fused_mode == 2) return false;
  if (d.fused_mode < 0) {
    // The launch mode is settled outside a capture only (a launch refused
    // inside a capture would invalidate it).
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
      return false;
  }
  return true;
}

// The whole layer in one launch: rotate + quantize, grid barrier, GEMM.
convrot_status run_fused(DeviceInfo& d, const LinearLayout& L, const uint16_t* X, int64_t M,
                         int64_t K, const uint16_t* wimg, int64_t N, const EpilogueArgs& ep,
                         void* workspace, cudaStream_t st) {
  uint16_t* qx = reinterpret_cast<uint16_t*>(at(workspace, L.qx));
  int32_t* acc = tc_may_split(M, N) ? reinterpret_cast<int32_t*>(at(workspace, L.acc)) : nullptr;
  int* cnt = reinterpret_cast<int*>(at(workspace, L.cnt));
  TcPlan plan = plan_tc(M, N, K, d.sms, false);
  if (plan.splits > 1 && !acc) plan = TcPlan{plan.bn, 1, static_cast<int>(K / 64)};
  CUtensorMap mx, mqs, mqr, ma, mb, my;
  memset(&my, 0, sizeof(my));
  const uint64_t segments = static_cast<uint64_t>(M * K / 64);
  convrot_status s = make_map_f16(&mx, X, segments, 64, 256);
  if (s != CONVROT_OK) return s;
  s = make_map_f16(&mqs, qx, segments, 64, 256);
  if (s != CONVROT_OK) return s;
  s = make_map_f16(&mqr, qx, segments, 64, static_cast<uint32_t>(K / 64));
  if (s != CONVROT_OK) return s;
  s = make_map_f16(&ma, qx, M, K, 128);
  if (s != CONVROT_OK) return s;
  s = make_map_f16(&mb, wimg, N, K, static_cast<uint32_t>(plan.bn));
  if (s != CONVROT_OK) return s;
  const bool tma_store = (N % 8) == 0 && aligned16(ep.Y);
  if (tma_store) {
    s = make_map_f16(&my, ep.Y, M, N, 128);
    if (s != CONVROT_OK) return s;
  }
  GemmTcArgs g;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.splits = plan.splits;
  g.kb_per_split = plan.kb_per_split;
  g.acc = acc;
  g.counters = cnt;
  g.tma_store = tma_store ? 1 : 0;
  g.ep = ep;
  g.err = d.err;
  g.weight_early = 0;
  g.acc_tma = 0;
  g.qx_out = qx;
  g.sx_out = reinterpret_cast<float*>(at(workspace, L.sx));
  g.sync = reinterpret_cast<unsigned long long*>(at(workspace, L.sync));
  if (plan.splits > 1) {
    if (cudaMemsetAsync(acc, 0, static_cast<size_t>(M) * N * 4, st) != cudaSuccess ||
        cudaMemsetAsync(cnt, 0, static_cast<size_t>(cdiv(M, 128) * cdiv(N, plan.bn)) * 4, st) !=
            cudaSuccess)
      return CONVROT_ERR_CUDA;
  }
  // One CTA per SM (each takes most of an SM's shared memory), all resident.
  const int grid = d.sms;
  if (d.fused_mode >= 0) return from_cuda(launch_gemm_fused(mx, mqs, mqr, ma, mb, my, g, plan.bn, grid,
                                                            d.fused_mode, st));
  for (int mode = 0; mode < 2; ++mode) {
    if (launch_gemm_fused(mx, mqs, mqr, ma, mb, my, g, plan.bn, grid, mode, st) == cudaSuccess) {
      d.fused_mode = mode;
      return CONVROT_OK;
    }
    (void)cudaGetLastError();  // a refused launch leaves nothing behind
  }
  d.fused_mode = 2;
  return CONVROT_ERR_UNSUPPORTED_DEVICE;  // caller falls back to two kernels
}

convrot_status run_gemm_skinny(const DeviceInfo& d, const int8_t* qx, const int8_t* qw, int64_t M,
                               int64_t N, int64_t K, const EpilogueArgs& ep, cudaStream_t st) {
  GemmSkinnyArgs g;
  g.QX = qx;
  g.QW = qw;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.splits = skinny_cluster_size(N, K, d.sms);
  g.k_per_split = static_cast<int>(K / g.splits);
  g.ep = ep;
  return from_cuda(launch_gemm_skinny(g, st));
}

// K slices per cluster of the small-M kernels that stream a 32-column
// weight slice into shared memory: the fewest that give 1.5 CTAs per SM with
// slices of at most 2048 (a longer slice leaves one CTA per SM, whose steps
// no other CTA overlaps).  Clusters are kept as small as that allows: a
// layer in clusters of two measured ~1.4 us slower than the same layer
// unsplit (M = 1, 8192x2048, one-kernel layer: 6.4 against 5.0 us).
int stream_splits(int64_t N, int64_t K, int sms) {
  const int64_t nblk = (N + 31) / 32;
  int splits = 1;
  while (splits < 8 && (K / splits > 2048 || nblk * splits * 2 < 3 * static_cast<int64_t>(sms)) &&
         (K / (2 * splits)) % 256 == 0)
    splits *= 2;
  return splits;
}

// K slices per cluster of the one-launch small-M layer.  A cluster costs a
// row-max exchange and a reduction; it pays for more CTAs streaming the
// weight and for less rotation per CTA.
// dp4a form (32 columns per CTA): at M = 1 one slice of up to 4096 where
// the column blocks alone give 0.8 CTAs per SM; otherwise at M <= 2
// stream_splits (each warp then holds at most 4 (row, group) items in
// registers at slices of 2048); above,
// the small-M GEMM's split raised until a slice is at most 1024 long (at
// M = 3 and slices of 2048 the rotation would go through an X tile: 10.3
// against 8.0 us).
// 0: no split gives a slice the form takes.
int decode_splits(int64_t M, int64_t N, int64_t K, int sms) {
  int splits = 1;
  if (M == 1 && K <= kDecodeMaxSlice && (N + 31) / 32 * 5 >= 4 * static_cast<int64_t>(sms)) {
    // One slice of up to 4096 where that still gives 0.8 CTAs per SM: no
    // cluster (M = 1, 16 layers in a graph: 4096x4096 5.6 against 6.4 us in
    // clusters of two, 14336x4096 16.4 against 17.7).  Slices of 4096 in
    // clusters measured slower than of 2048 (2048x8192: 6.6 against 6.4).
    splits = 1;
  } else if (M <= 2) {
    splits = stream_splits(N, K, sms);
  } else {
    splits = skinny_cluster_size(N, K, sms);
    while (K / splits > 1024 && splits < 8 && (K / (2 * splits)) % 256 == 0) splits *= 2;
  }
  return K / splits <= kDecodeMaxSlice &&
                 decode_layer_smem(static_cast<int>(M), static_cast<int>(K / splits)) <= kDecodeMaxSmem
             ? splits
             : 0;
}

// K slices of the two-kernel path's fp16-MMA small-M GEMM (skinny_f16_kernel)
// for a plain fp16 epilogue under the engine settings; 0: the mma.sync s8
// kernel runs instead (below M = 3, where the MMA pads most of its 8 rows,
// or slices over 4096, or the hook).
int skinny_f16_splits(int64_t M, int64_t N, int64_t K, int sms) {
  if (g_skinny_engine == 1 || (g_skinny_engine != 2 && M < 3)) return 0;
  const int splits = stream_splits(N, K, sms);
  return K / splits <= kDecodeMaxSlice ? splits : 0;
}

// fp16-MMA form (128 rows per CTA): the fewest slices of at most 1024 that
// give a CTA per SM.
int decode_mma_splits(int64_t N, int64_t K, int sms) {
  const int64_t nblk = (N + 127) / 128;
  int splits = 1;
  while (splits < 8 && (K / splits > 1024 || nblk * splits < sms) && (K / (2 * splits)) % 256 == 0)
    splits *= 2;
  return K / splits <= 1024 ? splits : 0;
}

struct LinearIO {
  bool x_bf16 = false;  // X (and the LoRA weights) hold bf16
  bool y_bf16 = false;  // Y is bf16
  const float* bias = nullptr;
};

// The one-launch layer's form and K slices if convrot_linear_ex takes it for
// these sizes and dtypes under the engine settings; splits 0 otherwise.
struct SmallMPlan {
  bool mma = false;  // the 128-row fp16-MMA form (else the 32-column dp4a form)
  int blocks = 0;    // > 0: the shared-rotation form, column blocks per cluster
  int splits = 0;
};

// Shared-rotation form: the K slices that give about two CTAs per SM (the
// nearest fewer, then more, where those do not fit), then the fewest column
// blocks per cluster (2, 4 or 8; slices x blocks <= 8) that divide the
// slice's 256-groups and leave each CTA at most 16 (row, group) items to
// rotate.  {0, 0}: the form does not apply.
std::pair<int, int> decode_shared_shape(int64_t M, int64_t N, int64_t K, int sms) {
  if (K % 256 != 0) return {0, 0};
  const int64_t nblk = (N + 31) / 32;
  int first = 1;
  while (first < 8 && nblk * first < 2 * static_cast<int64_t>(sms)) first *= 2;
  int order[4], n = 0;
  for (int cs = first; cs >= 1; cs /= 2) order[n++] = cs;
  for (int cs = 2 * first; cs <= 8; cs *= 2) order[n++] = cs;
  for (int i = 0; i < n; ++i) {
    const int cs = order[i];
    if (K % (256 * cs) != 0 || K / cs > kDecodeMaxSlice) continue;
    const int64_t groups = K / cs / 256;
    for (int blocks = 2; blocks <= 8 && cs * blocks <= 8; blocks *= 2)
      if (groups % blocks == 0 && M * (groups / blocks) <= 16 && nblk >= blocks) return {cs, blocks};
  }
  return {0, 0};
}

SmallMPlan small_m_plan(int64_t M, int64_t N, int64_t K, int64_t R, const LinearIO& io, int sms) {
  SmallMPlan pl;
  if (!use_skinny(M, CONVROT_PATH_AUTO) || io.x_bf16 || io.y_bf16 || io.bias || R != 0) return pl;
  if (g_small_m_mode == 1) return pl;
  // Auto: the dp4a form at M <= 2, where it measured faster than the two
  // kernels (8192x2048, 16 layers in a graph: M = 1 5.0 against 7.5 us;
  // M = 2 6.3 against 7.5).  From M = 3 the two-kernel path with the
  // fp16-MMA GEMM is faster (M = 3: 7.6 against 8.0; M = 16, 2048x2048: 6.2
  // against 8.5): the one-kernel layer repeats the rotation in every
  // 32-column block.  The fp16-MMA form of the one-kernel layer measured
  // slower than both (one CTA per SM, clusters of up to eight that do not
  // all fit at once), and so did the form that shares the rotation in a
  // cluster (M = 16, 8192x2048: 10.9-11.2 against 8.4 us).
  if (g_small_m_mode == 4) {
    const auto sh = decode_shared_shape(M, N, K, sms);
    if (sh.first > 0) {
      pl.splits = sh.first;
      pl.blocks = sh.second;
      return pl;
    }
  }
  if ((g_small_m_mode == 0 || g_small_m_mode == 4) && M > kDecodeAutoMaxM) return pl;
  pl.mma = g_small_m_mode == 3;
  pl.splits = pl.mma ? decode_mma_splits(N, K, sms) : decode_splits(M, N, K, sms);
  return pl;
}

convrot_status run_decode(const DeviceInfo& d, const uint16_t* X, int64_t M, int64_t K,
                          const int8_t* Q_W, const float* s_W, int64_t N, uint16_t* Y,
                          const SmallMPlan& pl, cudaStream_t st) {
  const int splits = pl.splits;
  DecodeArgs a;
  a.X = X;
  a.QW = Q_W;
  a.sW = s_W;
  a.Y = Y;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.err = d.err;
  a.splits = splits;
  a.k_per_split = static_cast<int>(K / splits);
  a.weights_early = g_small_m_weights_early;
  std::memcpy(a.sign, g_base.sign, sizeof(a.sign));
  if (pl.blocks > 0) return from_cuda(launch_decode_shared(a, pl.blocks, st));
  return from_cuda(pl.mma ? launch_decode_mma(a, st) : launch_decode_layer(a, st));
}

convrot_status run_lora_down(const DeviceInfo& d, const uint16_t* X, const uint16_t* down, float* T,
                             int64_t M, int64_t K, int64_t R, cudaStream_t st, bool bf16 = false) {
  LoraDownArgs a;
  a.X = X;
  a.down = down;
  a.T = T;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.R = static_cast<int>(R);
  a.bf16 = bf16 ? 1 : 0;
  // The kernel streams X and is latency-bound: split K (1, 2, 4 or 8 slices,
  // the CTAs of one cluster) until there are about 8 CTAs (32 warps) of work
  // per SM.  Each slice is a multiple of 32 K (K is a multiple of 256).
  const int64_t ctas_m = cdiv(M, 64);
  int s = 1;
  while (s < 8 && ctas_m * s < 8 * static_cast<int64_t>(d.sms)) s *= 2;
  a.splits = s;
  a.k_per_split = static_cast<int>(K / s);
  return from_cuda(launch_lora_down(a, st));
}

}  // namespace
}  // namespace convrot

using namespace convrot;

extern "C" {

const char* convrot_status_string(int status) {
  switch (status) {
    case CONVROT_OK: return "ok";
    case CONVROT_ERR_INVALID_ARG: return "invalid argument";
    case CONVROT_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case CONVROT_ERR_CUDA: return "CUDA error";
    case CONVROT_ERR_TIMEOUT: return "device wait timed out";
    case CONVROT_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int convrot_version(void) { return 100; }

size_t convrot_weight_image_bytes(int64_t N, int64_t K) {
  if (N < 0 || K < 0) return 0;
  return static_cast<size_t>(N) * static_cast<size_t>(K) * 2;
}

size_t convrot_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t R,
                                      int with_weight_image) {
  if (M <= 0 || N <= 0 || !valid_dim(M) || !valid_dim(N) || !valid_k(K) || R < 0) return 0;
  return linear_layout_max(M, N, K, R, with_weight_image != 0).total;
}

size_t convrot_linear_host_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t R,
                                           int with_weight_image) {
  if (M <= 0 || N <= 0 || !valid_k(K) || R < 0) return 0;
  return convrot_linear_workspace_bytes(M, N, K, R, with_weight_image) +
         align_up(static_cast<size_t>(M) * K * 2) + align_up(static_cast<size_t>(M) * N * 2);
}

size_t convrot_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int path) {
  if (M <= 0 || N <= 0 || !valid_dim(M) || !valid_dim(N) || !valid_k(K)) return 0;
  return gemm_layout(M, N, K, use_skinny(M, path) && M <= kSkinnyMaxM).total;
}

convrot_status convrot_prepare_weight(const float* W, int64_t N, int64_t K, int8_t* Q_W, float* s_W,
                                      uint16_t* W_img, void* stream) {
  if (!valid_dim(N) || !valid_k(K) || !W || !Q_W || !s_W) return CONVROT_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(Q_W) || !aligned16(W_img)) return CONVROT_ERR_INVALID_ARG;
  if (N == 0) return CONVROT_OK;
  DeviceInfo* d = nullptr;
  const convrot_status s = current_device(&d);
  if (s != CONVROT_OK) return s;
  RotqRowArgs a;
  a.in = W;
  a.rows = N;
  a.K = static_cast<int>(K);
  a.q_out = Q_W;
  a.img_out = W_img;
  a.s_out = s_W;
  std::memcpy(a.sign, g_base.sign, sizeof(a.sign));
  const int grid = static_cast<int>(std::min<int64_t>(N, static_cast<int64_t>(d->sms) * 8));
  return from_cuda(launch_rotq_row(a, kRowInF32, grid, static_cast<cudaStream_t>(stream)));
}

convrot_status convrot_rotate_quantize(const uint16_t* X, int64_t M, int64_t K, int8_t* Q_X,
                                       float* s_X, void* stream) {
  if (!valid_dim(M) || !valid_k(K) || !X || !Q_X || !s_X) return CONVROT_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q_X)) return CONVROT_ERR_INVALID_ARG;
  if (M == 0) return CONVROT_OK;
  DeviceInfo* d = nullptr;
  const convrot_status s = current_device(&d);
  if (s != CONVROT_OK) return s;
  // Its codes may be the next call's weight, which the one-kernel small-M
  // layer copies before its dependency wait: the next kernel starts only
  // when this one has finished.
  return run_rotq(*d, X, M, K, Q_X, false, s_X, static_cast<cudaStream_t>(stream), nullptr, 0,
                  nullptr, false, false, nullptr, 0, false);
}

convrot_status convrot_rotate(const uint16_t* X, int64_t M, int64_t K, uint16_t* X_rot,
                              void* stream) {
  // The tile kernel's shapes only: K / 64 a power of two, K <= 16384; and
  // Sylvester's base only (another base's X H has its columns in B's order,
  // which the library's kernels do not produce).
  const int64_t spr = K / 64;
  if (!valid_dim(M) || !valid_k(K) || K > 16384 || (spr & (spr - 1)) != 0 || !X || !X_rot ||
      !g_base.sylvester)
    return CONVROT_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(X_rot)) return CONVROT_ERR_INVALID_ARG;
  if (M == 0) return CONVROT_OK;
  DeviceInfo* d = nullptr;
  const convrot_status s = current_device(&d);
  if (s != CONVROT_OK) return s;
  return run_rotq(*d, X, M, K, X_rot, true, nullptr, static_cast<cudaStream_t>(stream), nullptr, 0,
                  nullptr, false, true);
}

// Data types and bias of one convrot_linear call (convrot_linear_ex).
static convrot_status linear_checks(const uint16_t* X, int64_t M, int64_t K, const int8_t* Q_W,
                                    const float* s_W, const uint16_t* W_img, int64_t N,
                                    const uint16_t* lora_down, const uint16_t* lora_up, int64_t R,
                                    const uint16_t* Y, bool need_x, bool need_w) {
  if (!valid_dim(M) || !valid_dim(N) || !valid_k(K)) return CONVROT_ERR_INVALID_ARG;
  if ((need_x && !X) || (need_w && (!Q_W || !s_W || !Y))) return CONVROT_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q_W) || !aligned16(W_img) || !aligned16(Y))
    return CONVROT_ERR_INVALID_ARG;
  if (R < 0 || R > kLoraMaxR) return CONVROT_ERR_INVALID_ARG;
  if (R > 0 && need_x && (!lora_down || !aligned16(lora_down))) return CONVROT_ERR_INVALID_ARG;
  if (R > 0 && need_w && (!lora_up || !aligned16(lora_up))) return CONVROT_ERR_INVALID_ARG;
  return CONVROT_OK;
}

// The workspace range the prologue zeroes for a GEMM that adds split
// partials in the accumulator (its tile counters included); tma_store: the
// GEMM's Y leaves through TMA stores (-1: not known yet, either way).
static void linear_zero_range(const DeviceInfo& d, const LinearLayout& L, bool skinny, int64_t M,
                              int64_t N, int64_t K, int64_t R, int tma_store, void* workspace,
                              void** zero, size_t* zero_bytes) {
  *zero = nullptr;
  *zero_bytes = 0;
  if (skinny || !tc_may_split(M, N)) return;
  const bool uses =
      (tma_store != 0 && plan_uses_acc(gemm_tc_plan(d, M, N, K, true, R, true))) ||
      (tma_store != 1 && plan_uses_acc(gemm_tc_plan(d, M, N, K, false, R, true)));
  if (!uses) return;
  *zero = at(workspace, L.acc);
  *zero_bytes = L.total - L.acc;
}

// w_img / w_bytes: the weight image the GEMM step reads next (nullptr when
// unknown), prefetched into L2 by the rotate + quantize kernel when it is at
// most kL2WeightPrefetchMax bytes.
static convrot_status linear_prologue(const DeviceInfo& d, const LinearLayout& L, bool skinny,
                                      const uint16_t* X, int64_t M, int64_t K,
                                      const uint16_t* lora_down, int64_t R, void* workspace,
                                      cudaStream_t st, void* zero = nullptr,
                                      size_t zero_bytes = 0, bool* zeroed = nullptr,
                                      const LinearIO& io = LinearIO(),
                                      const void* w_img = nullptr, size_t w_bytes = 0) {
  float* sx = reinterpret_cast<float*>(at(workspace, L.sx));
  const bool pf = w_img && !skinny && w_bytes <= kL2WeightPrefetchMax;
  convrot_status s = run_rotq(d, X, M, K, at(workspace, L.qx), !skinny, sx, st, zero, zero_bytes,
                              zeroed, io.x_bf16, false, pf ? w_img : nullptr, pf ? w_bytes : 0);
  if (s != CONVROT_OK || R == 0) return s;
  return run_lora_down(d, X, lora_down, reinterpret_cast<float*>(at(workspace, L.t)), M, K, R, st,
                       io.x_bf16);
}

// after_prologue: launched right after this call's own rotate + quantize
// (convrot_linear).  Then, or with LoRA (the LoRA up kernel runs right before
// the GEMM), the launch before the GEMM is one of this library's kernels that
// writes no weight and signals its dependents only after its own dependency
// wait, so with a caller-provided weight image the GEMM may load the weight
// before its dependency wait (GemmTcArgs::weight_early).
static convrot_status linear_gemm(const DeviceInfo& d, const LinearLayout& L, bool skinny,
                                  int64_t M, int64_t K, const int8_t* Q_W, const float* s_W,
                                  const uint16_t* W_img, int64_t N, const uint16_t* lora_up,
                                  int64_t R, float lora_scale, uint16_t* Y, void* workspace,
                                  cudaStream_t st, bool after_prologue = false,
                                  bool acc_zeroed = false, const LinearIO& io = LinearIO()) {
  EpilogueArgs ep;
  ep.mode = kOutF16;
  ep.bias = io.bias;
  ep.out_bf16 = io.y_bf16 ? 1 : 0;
  ep.lora_bf16 = io.x_bf16 ? 1 : 0;
  ep.Y = Y;
  ep.A = nullptr;
  ep.sX = reinterpret_cast<const float*>(at(workspace, L.sx));
  ep.sW = s_W;
  ep.T = R > 0 ? reinterpret_cast<const float*>(at(workspace, L.t)) : nullptr;
  ep.up = lora_up;
  ep.S = R > 0 ? reinterpret_cast<const float*>(at(workspace, L.s)) : nullptr;
  ep.R = static_cast<int>(R);
  ep.lora_scale = lora_scale;
  if (R > 0) {
    // The LoRA sums S = T lora_up^T for the epilogue (T from the prologue).
    LoraUpArgs la;
    la.T = ep.T;
    la.up = lora_up;
    la.S = reinterpret_cast<float*>(at(workspace, L.s));
    la.M = static_cast<int>(M);
    la.N = static_cast<int>(N);
    la.R = static_cast<int>(R);
    la.bf16 = io.x_bf16 ? 1 : 0;
    if (launch_lora_up(la, st) != cudaSuccess) return CONVROT_ERR_CUDA;
  }
  int32_t* acc = reinterpret_cast<int32_t*>(at(workspace, L.acc));
  int* cnt = reinterpret_cast<int*>(at(workspace, L.cnt));
  if (skinny) {
    // A plain fp16 epilogue at M >= 3 (below, the MMA pads most of its 8
    // rows): the kernel with bulk copies and the fp16 warp MMA.
    const bool plain = !io.bias && !io.y_bf16 && R == 0;
    const int f16_splits = plain ? skinny_f16_splits(M, N, K, d.sms) : 0;
    if (f16_splits > 0) {
      SkinnyF16Args a;
      a.QX = reinterpret_cast<const int8_t*>(at(workspace, L.qx));
      a.QW = Q_W;
      a.sX = ep.sX;
      a.sW = s_W;
      a.Y = Y;
      a.err = d.err;
      a.M = static_cast<int>(M);
      a.N = static_cast<int>(N);
      a.K = static_cast<int>(K);
      a.splits = f16_splits;
      a.k_per_split = static_cast<int>(K / f16_splits);
      // Right after this library's own prologue kernel (which writes only the
      // workspace) the weight may be copied before the dependency wait.
      a.weights_early = (after_prologue && g_small_m_weights_early) ? 1 : 0;
      return from_cuda(launch_skinny_f16(a, st));
    }
    return run_gemm_skinny(d, reinterpret_cast<const int8_t*>(at(workspace, L.qx)), Q_W, M, N, K,
                           ep, st);
  }
  const uint16_t* wimg = W_img;
  if (!wimg) {
    uint16_t* w = reinterpret_cast<uint16_t*>(at(workspace, L.wimg));
    const convrot_status s = run_widen(d, Q_W, w, N * K, st);
    if (s != CONVROT_OK) return s;
    wimg = w;
  }
  return run_gemm_tc(d, reinterpret_cast<const uint16_t*>(at(workspace, L.qx)), wimg, M, N, K, ep,
                     tc_may_split(M, N) ? acc : nullptr, cnt, st,
                     (after_prologue || R > 0) && W_img != nullptr, acc_zeroed);
}

static convrot_status linear_setup(int64_t M, int64_t N, int64_t K, int64_t R, bool with_img,
                                   void* workspace, size_t workspace_bytes, LinearLayout* L,
                                   bool* skinny, DeviceInfo** d) {
  *skinny = use_skinny(M, CONVROT_PATH_AUTO);
  *L = linear_layout(M, N, K, R, with_img, *skinny);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < L->total)
    return CONVROT_ERR_WORKSPACE;
  return current_device(d);
}

convrot_status convrot_linear(const uint16_t* X, int64_t M, int64_t K, const int8_t* Q_W,
                              const float* s_W, const uint16_t* W_img, int64_t N,
                              const uint16_t* lora_down, const uint16_t* lora_up, int64_t R,
                              float lora_scale, uint16_t* Y, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return convrot_linear_ex(X, CONVROT_DTYPE_F16, M, K, Q_W, s_W, W_img, N, nullptr, lora_down,
                           lora_up, R, lora_scale, Y, CONVROT_DTYPE_F16, workspace,
                           workspace_bytes, stream);
}

convrot_status convrot_linear_ex(const void* X_, int x_dtype, int64_t M, int64_t K,
                                 const int8_t* Q_W, const float* s_W, const uint16_t* W_img,
                                 int64_t N, const float* bias, const void* lora_down_,
                                 const void* lora_up_, int64_t R, float lora_scale, void* Y_,
                                 int y_dtype, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if ((x_dtype != CONVROT_DTYPE_F16 && x_dtype != CONVROT_DTYPE_BF16) ||
      (y_dtype != CONVROT_DTYPE_F16 && y_dtype != CONVROT_DTYPE_BF16) ||
      (reinterpret_cast<uintptr_t>(bias) & 3u) != 0)
    return CONVROT_ERR_INVALID_ARG;
  const uint16_t* X = static_cast<const uint16_t*>(X_);
  const uint16_t* lora_down = static_cast<const uint16_t*>(lora_down_);
  const uint16_t* lora_up = static_cast<const uint16_t*>(lora_up_);
  uint16_t* Y = static_cast<uint16_t*>(Y_);
  LinearIO io;
  io.x_bf16 = x_dtype == CONVROT_DTYPE_BF16;
  io.y_bf16 = y_dtype == CONVROT_DTYPE_BF16;
  io.bias = bias;
  convrot_status s =
      linear_checks(X, M, K, Q_W, s_W, W_img, N, lora_down, lora_up, R, Y, true, true);
  if (s != CONVROT_OK) return s;
  if (M == 0 || N == 0) return CONVROT_OK;
  LinearLayout L;
  bool skinny = false;
  DeviceInfo* d = nullptr;
  s = linear_setup(M, N, K, R, W_img != nullptr, workspace, workspace_bytes, &L, &skinny, &d);
  if (s != CONVROT_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The single-kernel engine takes fp16 in and out without a bias.
  if (!io.x_bf16 && !io.y_bf16 && !io.bias && fused_eligible(*d, K, R, skinny, st)) {
    const uint16_t* wimg = W_img;
    if (!wimg) {
      uint16_t* w = reinterpret_cast<uint16_t*>(at(workspace, L.wimg));
      s = run_widen(*d, Q_W, w, N * K, st);
      if (s != CONVROT_OK) return s;
      wimg = w;
    }
    EpilogueArgs ep;
    ep.mode = kOutF16;
    ep.Y = Y;
    ep.A = nullptr;
    ep.sX = reinterpret_cast<const float*>(at(workspace, L.sx));
    ep.sW = s_W;
    ep.T = nullptr;
    ep.up = nullptr;
    ep.R = 0;
    ep.lora_scale = 0.0f;
    s = run_fused(*d, L, X, M, K, wimg, N, ep, workspace, st);
    if (s != CONVROT_ERR_UNSUPPORTED_DEVICE) return s;
  }
  // At small M (fp16 in and out, no bias, no LoRA) one kernel does the
  // layer; the workspace is not touched.
  const SmallMPlan pl = small_m_plan(M, N, K, R, io, d->sms);
  if (pl.splits > 0) return run_decode(*d, X, M, K, Q_W, s_W, N, Y, pl, st);
  // If the GEMM will add split partials in the workspace accumulator, the
  // prologue kernel zeroes it (and the tile counters) on the way: no memsets.
  void* zero = nullptr;
  size_t zero_bytes = 0;
  linear_zero_range(*d, L, skinny, M, N, K, R, ((N % 8) == 0 && aligned16(Y)) ? 1 : 0, workspace,
                    &zero, &zero_bytes);
  bool zeroed = false;
  s = linear_prologue(*d, L, skinny, X, M, K, lora_down, R, workspace, st, zero, zero_bytes,
                      &zeroed, io, W_img, static_cast<size_t>(N * K) * 2);
  if (s != CONVROT_OK) return s;
  return linear_gemm(*d, L, skinny, M, K, Q_W, s_W, W_img, N, lora_up, R, lora_scale, Y,
                     workspace, st, true, zeroed, io);
}

convrot_status convrot_linear_prologue(const uint16_t* X, int64_t M, int64_t K, int64_t N,
                                       const uint16_t* lora_down, int64_t R,
                                       int with_weight_image, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  convrot_status s = linear_checks(X, M, K, nullptr, nullptr, nullptr, N, lora_down, nullptr, R,
                                   nullptr, true, false);
  if (s != CONVROT_OK) return s;
  if (M == 0 || N == 0) return CONVROT_OK;
  LinearLayout L;
  bool skinny = false;
  DeviceInfo* d = nullptr;
  s = linear_setup(M, N, K, R, with_weight_image != 0, workspace, workspace_bytes, &L, &skinny, &d);
  if (s != CONVROT_OK) return s;
  // The GEMM step's output alignment is not known here: zero the split-K
  // accumulator if either plan adds partials in it.
  void* zero = nullptr;
  size_t zero_bytes = 0;
  linear_zero_range(*d, L, skinny, M, N, K, R, -1, workspace, &zero, &zero_bytes);
  return linear_prologue(*d, L, skinny, X, M, K, lora_down, R, workspace,
                         static_cast<cudaStream_t>(stream), zero, zero_bytes);
}

convrot_status convrot_linear_gemm(int64_t M, int64_t K, const int8_t* Q_W, const float* s_W,
                                   const uint16_t* W_img, int64_t N, const uint16_t* lora_up,
                                   int64_t R, float lora_scale, uint16_t* Y, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  convrot_status s = linear_checks(nullptr, M, K, Q_W, s_W, W_img, N, nullptr, lora_up, R, Y,
                                   false, true);
  if (s != CONVROT_OK) return s;
  if (M == 0 || N == 0) return CONVROT_OK;
  LinearLayout L;
  bool skinny = false;
  DeviceInfo* d = nullptr;
  s = linear_setup(M, N, K, R, W_img != nullptr, workspace, workspace_bytes, &L, &skinny, &d);
  if (s != CONVROT_OK) return s;
  // The accumulator is zero: the prologue step zeroed it, and every split
  // GEMM leaves its tiles zero again.
  return linear_gemm(*d, L, skinny, M, K, Q_W, s_W, W_img, N, lora_up, R, lora_scale, Y,
                     workspace, static_cast<cudaStream_t>(stream), false, true);
}

convrot_status convrot_linear_workspace_layout(int64_t M, int64_t N, int64_t K, int64_t R,
                                               int with_weight_image, int64_t* qx_offset,
                                               int* qx_format, int64_t* sx_offset) {
  if (M <= 0 || N <= 0 || !valid_dim(M) || !valid_dim(N) || !valid_k(K) || R < 0 ||
      R > kLoraMaxR || !qx_offset || !qx_format || !sx_offset)
    return CONVROT_ERR_INVALID_ARG;
  const bool skinny = use_skinny(M, CONVROT_PATH_AUTO);
  const LinearLayout L = linear_layout(M, N, K, R, with_weight_image != 0, skinny);
  *qx_offset = static_cast<int64_t>(L.qx);
  *qx_format = skinny ? CONVROT_CODES_I8 : CONVROT_CODES_F16;
  *sx_offset = static_cast<int64_t>(L.sx);
  return CONVROT_OK;
}

int convrot_linear_kernel_count(int64_t M, int64_t N, int64_t K, int64_t R, int with_weight_image) {
  if (M <= 0 || N <= 0 || !valid_dim(M) || !valid_dim(N) || !valid_k(K) || R < 0 ||
      R > kLoraMaxR)
    return -1;
  DeviceInfo* d = nullptr;
  if (current_device(&d) != CONVROT_OK) return -1;
  const LinearIO io;
  if (small_m_plan(M, N, K, R, io, d->sms).splits > 0) return 1;
  const bool skinny = use_skinny(M, CONVROT_PATH_AUTO);
  const int widen = (!skinny && !with_weight_image) ? 1 : 0;
  const int64_t spr = K / 64;
  if (g_fused_enabled && !skinny && R == 0 && K <= kFusedMaxK && (spr & (spr - 1)) == 0 &&
      !g_base.any_sign() && d->fused_mode != 2)
    return 1 + widen;
  return 2 + widen + (R > 0 ? 2 : 0);  // rotate+quantize, [LoRA down, LoRA up,] GEMM
}

convrot_status convrot_linear_host(const uint16_t* X_host, int64_t M, int64_t K, const int8_t* Q_W,
                                   const float* s_W, const uint16_t* W_img, int64_t N,
                                   const uint16_t* lora_down, const uint16_t* lora_up, int64_t R,
                                   float lora_scale, uint16_t* Y_host, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!valid_dim(M) || !valid_dim(N) || !valid_k(K) || !X_host || !Q_W || !s_W || !Y_host)
    return CONVROT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  const size_t need = convrot_linear_host_workspace_bytes(M, N, K, R, W_img != nullptr);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 || workspace_bytes < need)
    return CONVROT_ERR_WORKSPACE;
  const size_t inner = convrot_linear_workspace_bytes(M, N, K, R, W_img != nullptr);
  uint16_t* xd = reinterpret_cast<uint16_t*>(at(workspace, inner));
  uint16_t* yd = reinterpret_cast<uint16_t*>(at(workspace, inner + align_up(static_cast<size_t>(M) * K * 2)));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(xd, X_host, static_cast<size_t>(M) * K * 2, cudaMemcpyHostToDevice, st) !=
      cudaSuccess)
    return CONVROT_ERR_CUDA;
  const convrot_status s = convrot_linear(xd, M, K, Q_W, s_W, W_img, N, lora_down, lora_up, R,
                                          lora_scale, yd, workspace, inner, stream);
  if (s != CONVROT_OK) return s;
  if (cudaMemcpyAsync(Y_host, yd, static_cast<size_t>(M) * N * 2, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return CONVROT_ERR_CUDA;
  return CONVROT_OK;
}

convrot_status convrot_check_device_error(void* stream, int* detail) {
  DeviceInfo* d = nullptr;
  convrot_status s = current_device(&d);
  if (s != CONVROT_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CONVROT_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, d->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CONVROT_ERR_CUDA;
  if (code != 0 && cudaMemset(d->err, 0, sizeof(int)) != cudaSuccess) return CONVROT_ERR_CUDA;
  if (detail) *detail = code;
  return code ? CONVROT_ERR_TIMEOUT : CONVROT_OK;
}

static convrot_status gemm_entry(const int8_t* Q_X, const float* s_X, const int8_t* Q_W,
                                 const float* s_W, int64_t M, int64_t N, int64_t K, int32_t* A,
                                 uint16_t* Y, int path, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (!valid_dim(M) || !valid_dim(N) || !valid_k(K) || !Q_X || !Q_W) return CONVROT_ERR_INVALID_ARG;
  if (path < CONVROT_PATH_AUTO || path > CONVROT_PATH_SKINNY) return CONVROT_ERR_INVALID_ARG;
  if (!aligned16(Q_X) || !aligned16(Q_W) || !aligned16(A) || !aligned16(Y))
    return CONVROT_ERR_INVALID_ARG;
  const bool skinny = use_skinny(M, path);
  if (skinny && M > kSkinnyMaxM) return CONVROT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  const GemmLayout L = gemm_layout(M, N, K, skinny);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < L.total)
    return CONVROT_ERR_WORKSPACE;
  DeviceInfo* d = nullptr;
  convrot_status s = current_device(&d);
  if (s != CONVROT_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  EpilogueArgs ep;
  memset(&ep, 0, sizeof(ep));
  ep.mode = A ? kOutI32 : kOutF16;
  ep.A = A;
  ep.Y = Y;
  ep.sX = s_X;
  ep.sW = s_W;
  int32_t* acc = reinterpret_cast<int32_t*>(at(workspace, L.acc));
  int* cnt = reinterpret_cast<int*>(at(workspace, L.cnt));
  if (skinny) return run_gemm_skinny(*d, Q_X, Q_W, M, N, K, ep, st);
  uint16_t* a_img = reinterpret_cast<uint16_t*>(at(workspace, L.a_img));
  uint16_t* b_img = reinterpret_cast<uint16_t*>(at(workspace, L.b_img));
  s = run_widen(*d, Q_X, a_img, M * K, st);
  if (s != CONVROT_OK) return s;
  s = run_widen(*d, Q_W, b_img, N * K, st);
  if (s != CONVROT_OK) return s;
  return run_gemm_tc(*d, a_img, b_img, M, N, K, ep, tc_may_split(M, N) ? acc : nullptr, cnt, st);
}

convrot_status convrot_gemm_i32(const int8_t* Q_X, const int8_t* Q_W, int64_t M, int64_t N,
                                int64_t K, int32_t* A, int path, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (!A) return CONVROT_ERR_INVALID_ARG;
  return gemm_entry(Q_X, nullptr, Q_W, nullptr, M, N, K, A, nullptr, path, workspace,
                    workspace_bytes, stream);
}

convrot_status convrot_gemm_dequant(const int8_t* Q_X, const float* s_X, const int8_t* Q_W,
                                    const float* s_W, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                                    int path, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (!Y || !s_X || !s_W) return CONVROT_ERR_INVALID_ARG;
  return gemm_entry(Q_X, s_X, Q_W, s_W, M, N, K, nullptr, Y, path, workspace, workspace_bytes,
                    stream);
}

convrot_status convrot_selftest_wait_timeout(int64_t budget_cycles, void* stream) {
  if (budget_cycles <= 0 || budget_cycles > 2000000000LL) return CONVROT_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  const convrot_status s = current_device(&d);
  if (s != CONVROT_OK) return s;
  return from_cuda(
      launch_selftest_wait(d->err, budget_cycles, static_cast<cudaStream_t>(stream)));
}

convrot_status convrot_measure_engine_peak(int engine, int64_t reps, double* ops, float* ms,
                                           void* stream) {
  if ((engine != CONVROT_PEAK_MMA_S8 && engine != CONVROT_PEAK_TCGEN05_F16 &&
       engine != CONVROT_PEAK_MMA_F16 && engine != CONVROT_PEAK_DP4A) || reps <= 0 ||
      reps > (1LL << 24) || !ops || !ms)
    return CONVROT_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  const convrot_status s = current_device(&d);
  if (s != CONVROT_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess) return CONVROT_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return CONVROT_ERR_CUDA;
  }
  cudaError_t e = cudaEventRecord(e0, st);
  if (e == cudaSuccess)
    e = launch_peak_engine(engine == CONVROT_PEAK_MMA_S8       ? 0
                           : engine == CONVROT_PEAK_TCGEN05_F16 ? 1
                           : engine == CONVROT_PEAK_MMA_F16     ? 2
                                                                : 3,
                           reps, d->sms, d->err, ops, st);
  if (e == cudaSuccess) e = cudaEventRecord(e1, st);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return from_cuda(e);
}

convrot_status convrot_set_hadamard_base(const int8_t* base) {
  if (!base) {
    g_base = HadamardBase();
    return CONVROT_OK;
  }
  int b[4][4];
  for (int i = 0; i < 16; ++i) {
    if (base[i] != 1 && base[i] != -1) return CONVROT_ERR_INVALID_ARG;
    b[i / 4][i % 4] = base[i];
  }
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) {
      if (b[i][j] != b[j][i]) return CONVROT_ERR_INVALID_ARG;  // H is symmetric
      int dot = 0;
      for (int k = 0; k < 4; ++k) dot += b[i][k] * b[j][k];
      if (dot != (i == j ? 4 : 0)) return CONVROT_ERR_INVALID_ARG;  // not Hadamard
    }
  // Sylvester's H4[i][j] = (-1)^popcount(i & j).
  auto h4 = [](int i, int j) { return (__builtin_popcount(static_cast<unsigned>(i & j)) & 1) ? -1 : 1; };
  // B = D1 H4 R: B[i][j] = d1[i] H4[i][pi(j)] d2[j], found by search (eight
  // factorizations exist; the first in the order of d1's sign mask, so a
  // base that needs no input signs gets none).
  int d1_found = -1;
  for (int m1 = 0; m1 < 16 && d1_found < 0; ++m1) {
    int perm[4] = {0, 1, 2, 3};
    do {
      bool ok = true;
      for (int j = 0; j < 4 && ok; ++j) {
        // d2[j] is fixed by row 0; the other rows must agree.
        const int d2 = b[0][j] * ((m1 & 1) ? -1 : 1) * h4(0, perm[j]);
        for (int i = 0; i < 4 && ok; ++i)
          ok = b[i][j] == (((m1 >> i) & 1) ? -1 : 1) * h4(i, perm[j]) * d2;
      }
      if (ok) d1_found = m1;
    } while (d1_found < 0 && std::next_permutation(perm, perm + 4));
  }
  if (d1_found < 0) return CONVROT_ERR_INVALID_ARG;  // unreachable for a Hadamard B
  HadamardBase nb;
  nb.sylvester = true;
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) nb.sylvester = nb.sylvester && b[i][j] == h4(i, j);
  // D[k] = prod over the base-4 digits k_d of k of d1[k_d].
  for (int k = 0; k < 256; ++k) {
    int neg = 0;
    for (int d = 0; d < 4; ++d) neg ^= (d1_found >> ((k >> (2 * d)) & 3)) & 1;
    if (neg) nb.sign[k >> 5] |= 1u << (k & 31);
  }
  g_base = nb;
  return CONVROT_OK;
}

convrot_status convrot_set_split_mode(int mode) {
  if (mode < 0 || mode > 3) return CONVROT_ERR_INVALID_ARG;
  g_split_mode = mode;
  return CONVROT_OK;
}

convrot_status convrot_set_pair_mma(int mode) {
  if (mode < 0 || mode > 2) return CONVROT_ERR_INVALID_ARG;
  g_pair_mma_mode = mode;
  return CONVROT_OK;
}

convrot_status convrot_set_small_m_engine(int mode) {
  if (mode < 0 || mode > 4) return CONVROT_ERR_INVALID_ARG;
  g_small_m_mode = mode;
  return CONVROT_OK;
}

convrot_status convrot_set_skinny_engine(int mode) {
  if (mode < 0 || mode > 2) return CONVROT_ERR_INVALID_ARG;
  g_skinny_engine = mode;
  return CONVROT_OK;
}

convrot_status convrot_set_small_m_weights_early(int enable) {
  if (enable != 0 && enable != 1) return CONVROT_ERR_INVALID_ARG;
  g_small_m_weights_early = enable;
  return CONVROT_OK;
}

convrot_status convrot_set_fused(int enable) {
  if (enable != 0 && enable != 1) return CONVROT_ERR_INVALID_ARG;
  g_fused_enabled = enable;
  return CONVROT_OK;
}

convrot_status convrot_plan_gemm(int64_t M, int64_t N, int64_t K, int sms, int pair_clusters_128,
                                 int pair_clusters_256, int tma_store, int64_t R, int* bn,
                                 int* splits, int* engine) {
  if (M <= 0 || N <= 0 || !valid_k(K) || sms <= 0 || R < 0 || !bn || !splits || !engine)
    return CONVROT_ERR_INVALID_ARG;
  // The same choice as gemm_tc_plan, with the device's numbers given.
  const bool plain = tma_store != 0 && R == 0;
  const int clusters[2] = {pair_clusters_128, pair_clusters_256};
  const TcPlan p = plan_tc(M, N, K, sms, plain, 256, tma_store != 0 ? clusters : nullptr,
                           tma_store != 0, plain);
  *bn = p.bn;
  *splits = p.splits;
  *engine = p.stream     ? CONVROT_ENGINE_PAIR_STREAM
            : p.pair_mma ? CONVROT_ENGINE_PAIR_MMA
            : p.pair   ? CONVROT_ENGINE_PAIR_SPLIT
            : p.splits > 1 ? CONVROT_ENGINE_L2_SPLIT
                           : CONVROT_ENGINE_ONE_SM;
  return CONVROT_OK;
}

convrot_status convrot_plan_small_m(int64_t M, int64_t N, int64_t K, int sms, int* engine,
                                    int* splits, int* blocks) {
  if (M <= 0 || N <= 0 || !valid_dim(M) || !valid_dim(N) || !valid_k(K) || sms <= 0 || !engine ||
      !splits || !blocks)
    return CONVROT_ERR_INVALID_ARG;
  // The same choices as convrot_linear (fp16 X and Y, no bias, no LoRA),
  // with the device's SM count given.
  *blocks = 0;
  *splits = 0;
  if (!use_skinny(M, CONVROT_PATH_AUTO)) {
    *engine = CONVROT_SMALL_M_NONE;
    return CONVROT_OK;
  }
  const SmallMPlan pl = small_m_plan(M, N, K, 0, LinearIO(), sms);
  if (pl.splits > 0) {
    *engine = pl.blocks > 0 ? CONVROT_SMALL_M_ONE_SHARED
              : pl.mma      ? CONVROT_SMALL_M_ONE_MMA
                            : CONVROT_SMALL_M_ONE_DP4A;
    *splits = pl.splits;
    *blocks = pl.blocks;
    return CONVROT_OK;
  }
  const int f16 = skinny_f16_splits(M, N, K, sms);
  *engine = f16 > 0 ? CONVROT_SMALL_M_TWO_F16 : CONVROT_SMALL_M_TWO_S8;
  *splits = f16 > 0 ? f16 : skinny_cluster_size(N, K, sms);
  return CONVROT_OK;
}

convrot_status convrot_set_tile_override(int bn, int splits) {
  if ((bn != 0 && bn != 64 && bn != 128 && bn != 256) || splits < 0 || splits > 16)
    return CONVROT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_force_bn = bn;
  g_force_splits = splits;
  return CONVROT_OK;
}

}  // extern "C"

namespace convrot {
void hadamard_signs(uint32_t out[8]) { std::memcpy(out, g_base.sign, sizeof(g_base.sign)); }
}  // namespace convrot
