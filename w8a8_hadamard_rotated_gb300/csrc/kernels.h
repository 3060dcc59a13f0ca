// Internal interface between the host dispatch (api.cu) and the kernels of
// the INT8ConvRot library.  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace convrot {

// ---------------------------------------------------------------- rotate+quantize
struct RotqTileArgs {
  int64_t segments;  // M * K / 64
  int64_t tiles;     // ceil(segments / (warps * 32 * vpl / 64))
  int K;
  int warps;         // warps per CTA (1 to 8)
  int vpl;           // values per lane: 64 (a lane per 64-element segment) or 32
  void* q_out;       // int8 [M, K] or fp16 [M, K] (the int8 values widened)
  float* s_out;      // fp32 [M]
  int* err;
  // Optional: 16-byte words to set to zero after the dependency wait (the
  // next GEMM's split-K accumulator and tile counters); nullptr / 0 = none.
  uint4* zero;
  int64_t zero_n16;
  int in_bf16;       // 1: X holds bf16 values, 0: fp16
  int rot_only;      // 1 (with fp16 output): write X H rounded to fp16, no codes or scales
  // Optional: contiguous bytes (16-byte aligned, a multiple of 16) that the
  // CTAs bring into L2 before their dependency wait, a slice each: the next
  // GEMM's weight image.  nullptr / 0 = none.
  const void* l2_pf;
  int64_t l2_pf_bytes;
  // 1: let the next kernel on the stream start once every CTA is past its
  // dependency wait (programmatic dependent launch); 0: only when this one
  // has finished (its output may be read before the next kernel's wait).
  int early_dependents = 1;
  // Input signs of a non-Sylvester 4x4 Hadamard base (bit k of the 256:
  // negate element k of every 256-group before the transform); has_sign = 0
  // for Sylvester's base.
  uint32_t sign[8];
  int has_sign;
};

struct RotqRowArgs {
  const void* in;     // fp32, fp16 or bf16 [rows, K] (launch_rotq_row's in_type)
  int64_t rows;
  int K;
  int8_t* q_out;      // int8 [rows, K] or nullptr
  uint16_t* img_out;  // fp16 [rows, K] or nullptr
  float* s_out;       // fp32 [rows]
  uint32_t sign[8];   // input signs per 256-group, as in RotqTileArgs (all 0: none)
};

size_t rotq_tile_smem_bytes(int warps, int vpl);
// tm_q: the fp16 code image viewed like tm_x (out_f16 only; ignored otherwise).
// max_per_sm > 0: the shared-memory request is raised so that at most that
// many CTAs fit on an SM (the grid then spreads evenly even when it starts
// while the previous kernel still holds some SMs); 0: the kernel's own need.
cudaError_t launch_rotq_tile(const CUtensorMap& tm_x, const CUtensorMap& tm_q,
                             const RotqTileArgs& a, bool out_f16, int grid, int max_per_sm,
                             cudaStream_t stream);
enum : int { kRowInF16 = 0, kRowInF32 = 1, kRowInBf16 = 2 };
cudaError_t launch_rotq_row(const RotqRowArgs& a, int in_type, int grid, cudaStream_t stream);
cudaError_t launch_widen_i8(const int8_t* in, uint16_t* out, int64_t n, int grid,
                            cudaStream_t stream);

// ---------------------------------------------------------------- epilogue
// What a GEMM writes once it holds the exact int32 sums of a tile.
struct EpilogueArgs {
  int mode;              // kOutF16 (a 16-bit float Y: fp16, or bf16 with out_bf16) or kOutI32
  uint16_t* Y;           // fp16 or bf16 [M, N]  (kOutF16)
  int32_t* A;            // int32 [M, N] (kOutI32)
  const float* sX;       // fp32 [M]     (kOutF16)
  const float* sW;       // fp32 [N]     (kOutF16)
  const float* T;        // fp32 [M, R]  LoRA down-projection, or nullptr
  const uint16_t* up;    // fp16 or bf16 [N, R]  LoRA up weight, or nullptr
  // fp32 [M, N]: the LoRA sums sum_r T[m,r] up[n,r] (launch_lora_up), added as
  // lora_scale * S by the epilogues; present whenever R > 0.
  const float* S = nullptr;
  int R;
  float lora_scale;
  // y = ((float)A * s_X) * s_W, then + bias[n] (its own fp32 add), then
  // + the LoRA term, rounded once to fp16 or bf16.
  const float* bias = nullptr;  // fp32 [N], or nullptr
  int out_bf16 = 0;             // 1: Y is bf16 (round to nearest even)
  int lora_bf16 = 0;            // 1: `up` holds bf16
};
enum : int { kOutF16 = 0, kOutI32 = 1 };

// ---------------------------------------------------------------- tcgen05 GEMM
struct GemmTcArgs {
  int M, N, K;
  int splits;         // K split across gridDim.z
  int kb_per_split;   // 64-wide K blocks per split
  int32_t* acc;       // int32 [M, N] zeroed partial sums (splits > 1)
  int* counters;      // zeroed arrival counters, one per output tile (splits > 1)
  int tma_store;      // 1: fp16 Y written through the store tensor map tm_y
  EpilogueArgs ep;
  int* err;
  // Fused rotate + quantize (fused kernel only): the CTAs first turn X (read
  // through tm_x) into the fp16 code image qx_out [M, K] -- the A operand of
  // tm_a -- and s_X (ep.sX), then meet at a grid barrier in `sync`.
  uint16_t* qx_out;
  float* sx_out;
  unsigned long long* sync;  // grid-barrier state, 4 words kept from call to call
  // 1: the weight operand may be loaded before the dependency wait.  Set
  // only when the previous launch on the stream is this library's own
  // rotate + quantize kernel, which writes neither operand's weight and
  // signals its dependents only after its own dependency wait: so the
  // kernels before it, which might have written the weight, are complete
  // before this kernel can start.
  int weight_early;
  // Split K (splits > 1, not the CTA pair): 1 = each split adds its int32
  // partial into acc with TMA bulk reduce-adds through the int32 tensor map
  // passed in the tm_x slot (box 32 x 128, 128-byte swizzle), and the tile's
  // last split loads the sum back through it; 0 = per-element atomics.
  int acc_tma;
};

// Tile shape: BM = 128 rows of X, BN = 64, 128 or 256 columns of W, BK = 64.
// tm_y (fp16 Y, box 64 x 128, 128-byte swizzle) is used when a.tma_store.
// Persistent: `grid` CTAs walk the ceil(M/128) * ceil(N/BN) * splits units.
size_t gemm_tc_smem_bytes(int bn);
// tm_acc: the int32 [M, N] split-K accumulator (a.acc_tma), else ignored.
cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                           const CUtensorMap& tm_y, const CUtensorMap& tm_acc,
                           const GemmTcArgs& a, int bn, int grid, cudaStream_t stream);

// Pair variant: K split in two across the CTAs of 2-CTA clusters, one tile
// per CTA (grid = tiles * 2, a.splits = 2), reduced through distributed
// shared memory.  BN = 128 or 256, fp16 output through tm_y, no LoRA.
cudaError_t launch_gemm_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                             const CUtensorMap& tm_y, const GemmTcArgs& a, int bn, int grid,
                             cudaStream_t stream);

// CTA-pair K split with a streaming exchange: one 128 x bn tile (bn 128 or
// 256) per 2-CTA cluster, each CTA one half of K as a single exact fp32
// chunk (K <= 2048), the two fp32 partials added on the way out; fp16 Y
// through TMA stores (a.tma_store), no LoRA, no bias, fp16 output.  Grid =
// 2 * tiles (not persistent).
cudaError_t launch_gemm_pairk(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                              const CUtensorMap& tm_y, const GemmTcArgs& a, int bn,
                              cudaStream_t stream);

// Pair-MMA GEMM (.cta_group::2): 256 x bn tiles (bn 128 or 256), each on the
// two CTAs of a cluster; `clusters` persistent clusters (at most
// gemm_pair_mma_max_clusters(bn)).  No K split, no LoRA, fp16 output through
// TMA stores; tm_a box 128 rows, tm_b box bn/2 rows, tm_y box 128 rows.
cudaError_t launch_gemm_pair_mma(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                 const CUtensorMap& tm_y, const GemmTcArgs& a, int bn,
                                 int clusters, cudaStream_t stream);
// Clusters of the pair-MMA kernel that fit on the device at once (0 if the
// query fails).
int gemm_pair_mma_max_clusters(int bn);
// The same three launches for epilogues with a bias, bf16 Y or a bf16 LoRA
// up weight (EpilogueArgs); launch_gemm_tc / _pair / _pair_mma forward to
// them.  Instantiated in gemm_tc_ext.cu.
cudaError_t launch_gemm_tc_ext(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                               const CUtensorMap& tm_y, const CUtensorMap& tm_acc,
                               const GemmTcArgs& a, int bn, int grid, cudaStream_t stream);
cudaError_t launch_gemm_pair_ext(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                 const CUtensorMap& tm_y, const GemmTcArgs& a, int bn, int grid,
                                 cudaStream_t stream);
cudaError_t launch_gemm_pair_mma_ext(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                     const CUtensorMap& tm_y, const GemmTcArgs& a, int bn,
                                     int clusters, cudaStream_t stream);

// Self-test of the bounded waits: one CTA waits `budget` cycles on an
// mbarrier nothing arrives on, then records DEVERR_SELFTEST in `err`.
cudaError_t launch_selftest_wait(int* err, long long budget, cudaStream_t stream);

// Fused layer: rotate + quantize, grid barrier, GEMM + epilogue in one
// persistent kernel (no LoRA).  tm_x views X as [M*K/64, 64] fp16 segments
// with 256-row boxes; K is a power of two in [256, 16384]; `grid` CTAs (one
// per SM, all co-resident: cooperative launch) share the rows of X.
// `mode`: 0 = cooperative + programmatic dependent launch, 1 = cooperative only.
constexpr int kFusedMaxK = 16384;
// tm_qs / tm_qr view the code image qx_out like tm_x, with boxes of 256
// segments and of K/64 segments (one row).
cudaError_t launch_gemm_fused(const CUtensorMap& tm_x, const CUtensorMap& tm_qs,
                              const CUtensorMap& tm_qr, const CUtensorMap& tm_a,
                              const CUtensorMap& tm_b, const CUtensorMap& tm_y,
                              const GemmTcArgs& a, int bn, int grid, int mode,
                              cudaStream_t stream);

// ---------------------------------------------------------------- skinny GEMM
struct GemmSkinnyArgs {
  const int8_t* QX;   // int8 [M, K]
  const int8_t* QW;   // int8 [N, K]
  int M, N, K;
  int splits;         // K slices = CTAs per cluster: 1, 2, 4 or 8
  int k_per_split;    // K / splits, a multiple of 256
  EpilogueArgs ep;
};
constexpr int kSkinnyMaxM = 64;
// Cluster size (K slices per 32-column block) for an N x K weight.
int skinny_cluster_size(int64_t N, int64_t K, int sms);
cudaError_t launch_gemm_skinny(const GemmSkinnyArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- small-M layer
// The whole layer for M <= kDecodeMaxM in one launch (decode.cu): rotate +
// quantize of each CTA's K slice of the rows, row maxima combined across the
// cluster, the weight slice in shared memory by bulk copies, the exact
// product on mma.sync s8 and the scale restore.  fp16 X and Y, no LoRA, no
// bias; no workspace.
struct DecodeArgs {
  const uint16_t* X;  // fp16 [M, K]
  const int8_t* QW;   // int8 [N, K]
  const float* sW;    // fp32 [N]
  uint16_t* Y;        // fp16 [M, N]
  int* err;           // device error flag (bounded waits)
  int M, N, K;
  int splits;         // K slices = CTAs per cluster: 1, 2, 4 or 8
  int k_per_split;    // K / splits: a multiple of 256, at most kDecodeMaxSlice
  int weights_early;  // 1: copy the weight before the dependency wait
  uint32_t sign[8];   // input signs per 256-group (all 0: Sylvester's base)
};
constexpr int kDecodeMaxM = 16;
constexpr int kDecodeMaxSlice = 4096;
constexpr size_t kDecodeMaxSmem = 220 * 1024;  // under the per-CTA opt-in limit with the static part
size_t decode_layer_smem(int M, int k_per_split);
cudaError_t launch_decode_layer(const DecodeArgs& a, cudaStream_t stream);
// The same layer with 128 weight rows per CTA and the product on the fp16
// warp MMA (exact: int8 values, fp32 sums moved to int32 every 1024 K); K
// slices of at most 1024.
size_t decode_mma_smem(int k_per_split);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t stream);
// The two-kernel path's small-M GEMM on that skeleton (decode.cu): the
// prologue's int8 codes and s_X, the weight by bulk copies, 32 output columns
// per CTA, the product on the fp16 warp MMA, the plain fp16 epilogue (no
// bias, no LoRA, fp16 Y).
struct SkinnyF16Args {
  const int8_t* QX;   // int8 [M, K] (the prologue's codes)
  const int8_t* QW;   // int8 [N, K]
  const float* sX;    // fp32 [M]
  const float* sW;    // fp32 [N]
  uint16_t* Y;        // fp16 [M, N]
  int* err;
  int M, N, K;
  int splits;         // K slices = CTAs per cluster: 1, 2, 4 or 8
  int k_per_split;    // a multiple of 256, at most 4096
  int weights_early;  // 1: copy the weight before the dependency wait
};
size_t skinny_f16_smem(int k_per_split);
cudaError_t launch_skinny_f16(const SkinnyF16Args& a, cudaStream_t stream);
// The one-kernel layer with the rotation shared by `blocks` column blocks per
// cluster (2, 4 or 8; splits x blocks <= 8; each CTA's share of its slice's
// groups at most 16 items), the product on the fp16 warp MMA (decode.cu).
size_t decode_shared_smem(int k_per_split);
cudaError_t launch_decode_shared(const DecodeArgs& a, int blocks, cudaStream_t stream);

// ---------------------------------------------------------------- LoRA down
struct LoraDownArgs {
  const uint16_t* X;     // fp16 or bf16 [M, K]
  const uint16_t* down;  // same type [R, K]
  float* T;              // fp32 [M, R], written (no zeroing needed)
  int M, K, R;
  int splits;            // K slices = CTAs per cluster: 1, 2, 4 or 8
  int k_per_split;       // multiple of 32
  int bf16 = 0;          // 1: X and down hold bf16
};
constexpr int kLoraMaxR = 128;
cudaError_t launch_lora_down(const LoraDownArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- LoRA up
struct LoraUpArgs {
  const float* T;        // fp32 [M, R] (launch_lora_down)
  const uint16_t* up;    // fp16 or bf16 [N, R]
  float* S;              // fp32 [M, N]: sum_r T[m, r] up[n, r]
  int M, N, R;
  int bf16 = 0;          // 1: up holds bf16
};
cudaError_t launch_lora_up(const LoraUpArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- engine peaks
// Launches the throughput probe of one exact int8 product engine (0:
// mma.sync m16n8k32 s8, 1: tcgen05.mma kind::f16 M128 N256, 2: mma.sync
// m16n8k16 f16 -> f32, 3: dp4a) on `sms` SMs for `reps` repetitions; *ops
// receives the integer or floating-point operations the launch performs.
cudaError_t launch_peak_engine(int engine, int64_t reps, int sms, int* err, double* ops,
                               cudaStream_t st);

// The input signs (bit k: negate element k of every 256-group) of the 4x4
// Hadamard base set by convrot_set_hadamard_base; all zero for Sylvester's.
void hadamard_signs(uint32_t out[8]);

}  // namespace convrot
