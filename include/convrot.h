/*
 * convrot.h -- C ABI of the INT8ConvRot (W8A8, Hadamard-rotated) linear layer
 * for NVIDIA GB300 (sm_103a).
 *
 * The layer is defined on the page "INT8ConvRot GEMM vs fp16 on M1 Max with
 * Metal, MPSMatrix, and MLX", section "What changed in the computation":
 *
 *   H      = (4x4 Hadamard)^(x4) / 16, a symmetric 256x256 matrix with HH = I,
 *            applied to the last dimension in groups of 256;
 *   prep   : W_rot = W H^T,  s_W[n] = max_k |W_rot[n,k]| / 127,  Q_W = round(W_rot / s_W)
 *   call   : X_rot = X H,    s_X[m] = max_k |X_rot[m,k]| / 127,  Q_X = round(X_rot / s_X)
 *            A = Q_X Q_W^T (int32),  Y = A (.) s_X s_W^T
 *   rounded values are clamped to [-128, 127]; "round" is round-half-to-even.
 *
 * The optional unmerged LoRA term follows the page "[PR #249] Add an mps
 * backend: weight-only INT8 and W4A8/W6A8 linears for Apple GPUs", section
 * "What": lora_down [R, K], lora_up [N, R], lora_scale, applied to the
 * unrotated X:  Y += lora_scale * (X lora_down^T) lora_up^T.
 *
 * Conventions for every entry point below:
 *  - Pointers are DEVICE pointers unless the name says otherwise, owned and
 *    allocated by the caller.  The library never allocates device memory; the
 *    per-call scratch it needs is the caller's `workspace`.
 *  - Arrays are dense, row-major, with the last index contiguous.  Base
 *    addresses must be 16-byte aligned.
 *  - fp16 data is passed as uint16_t (IEEE binary16 bit patterns).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    are asynchronous on that stream: the return value reports argument and
 *    launch errors only.  A kernel that gives up on a bounded wait records a
 *    code that convrot_check_device_error() returns.
 *  - K must be a positive multiple of 256 (the Hadamard group size) and at
 *    most CONVROT_MAX_K; anything else is CONVROT_ERR_INVALID_ARG with nothing
 *    launched.  M = 0 or N = 0 is CONVROT_OK with nothing launched.  M and N
 *    are at most CONVROT_MAX_DIM (element counts such as M*N may exceed
 *    2^31); a larger M or N is CONVROT_ERR_INVALID_ARG.
 *  - Only compute capability 10.3 (sm_103a) devices are supported; any other
 *    device gives CONVROT_ERR_UNSUPPORTED_DEVICE.  There is no fallback path.
 *  - Argument checks happen before any CUDA call, so a rejected call touches
 *    no device state.
 */
#ifndef CONVROT_H
#define CONVROT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum convrot_status {
  CONVROT_OK = 0,
  CONVROT_ERR_INVALID_ARG = 1,        /* bad size, null or misaligned pointer */
  CONVROT_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not sm_103 */
  CONVROT_ERR_CUDA = 3,               /* a CUDA runtime/driver call failed */
  CONVROT_ERR_TIMEOUT = 4,            /* a kernel gave up on a bounded wait */
  CONVROT_ERR_WORKSPACE = 5           /* workspace missing or too small */
} convrot_status;

/* Largest K accepted (keeps |A| = |sum_k Q_X Q_W| below 2^31 for any int8). */
#define CONVROT_MAX_K 65536

/* Largest M (rows of X) and N (rows of the weight) accepted: 2^31 - 1. */
#define CONVROT_MAX_DIM 2147483647LL

/* GEMM engine selection for the entry points that take `path`. */
#define CONVROT_PATH_AUTO 0    /* the library picks by shape */
#define CONVROT_PATH_TCGEN05 1 /* tcgen05 tensor-core tiles (TMA + TMEM) */
#define CONVROT_PATH_SKINNY 2  /* int8 mma.sync split-K for small M */

/* Human-readable name of a status code (static string, never NULL). */
const char* convrot_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int convrot_version(void);

/*
 * Bytes of the optional fp16 operand image of a prepared weight: the int8
 * Q_W values widened to fp16 (exact), [N, K] row-major, 2*N*K bytes.  With
 * it, the tensor-core GEMM reads the weight directly; without it, each call
 * widens Q_W into the workspace first.
 */
size_t convrot_weight_image_bytes(int64_t N, int64_t K);

/*
 * Workspace bytes convrot_linear needs for this shape (R = LoRA rank, 0 for
 * none) when the weight image is supplied (`with_weight_image` != 0) or not.
 * The workspace holds the quantized activations, their scales, the LoRA
 * down-projection T [M, R] and the LoRA sums S = T lora_up^T [M, N] (fp32,
 * R > 0 only) and split-K partial sums; its contents need not be
 * initialized and are overwritten by every call.
 */
size_t convrot_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t R,
                                      int with_weight_image);

/*
 * One-time weight preparation (the page's "Once at model creation" step):
 *   W_rot = W H^T  (group-wise, groups of 256 along K),
 *   s_W[n] = max_k |W_rot[n,k]| / 127     (fp32),
 *   Q_W[n,k] = clamp(round_half_even(W_rot[n,k] / s_W[n]), -128, 127).
 * An all-zero row gives s_W = 0 and Q_W = 0.
 *   W      fp32 [N, K]   input (not modified)
 *   Q_W    int8 [N, K]   output
 *   s_W    fp32 [N]      output
 *   W_img  fp16 [N, K]   optional output (may be NULL): Q_W widened to fp16
 * The rotation runs in fp32 (a fast Walsh-Hadamard transform); a quantized
 * value may differ by one from an exact-arithmetic rounding only where the
 * exact value lies within ~1e-4 of a .5 tie.
 */
convrot_status convrot_prepare_weight(const float* W, int64_t N, int64_t K, int8_t* Q_W,
                                      float* s_W, uint16_t* W_img, void* stream);

/*
 * The per-call layer:
 *   X_rot = X H,  s_X = max|X_rot| / 127 per row,  Q_X = round(X_rot / s_X),
 *   A = Q_X Q_W^T (exact int32),
 *   Y = fp16( ((float)A * s_X[m]) * s_W[n]  +  lora_scale * sum_r T[m,r] * lora_up[n,r] ),
 *   T = X lora_down^T (fp32 accumulation, unrotated X), present only when R > 0;
 *   sum_r T[m,r] * lora_up[n,r] is accumulated in fp32 (two ranks per paired
 *   FMA) into the workspace by the GEMM stage and added, times lora_scale, in
 *   fp32 before the single rounding.  T's K slices are added in a fixed
 *   order, so with LoRA too Y is the same bits on every run.
 *   X          fp16 [M, K]
 *   Q_W, s_W   int8 [N, K], fp32 [N] from convrot_prepare_weight (or any int8 weight)
 *   W_img      fp16 [N, K] weight image or NULL
 *   lora_down  fp16 [R, K] or NULL (R = 0)
 *   lora_up    fp16 [N, R] or NULL (R = 0)
 *   Y          fp16 [M, N] output (fp16 overflow gives +-inf)
 *   workspace  at least convrot_linear_workspace_bytes(M, N, K, R, W_img != NULL)
 *              bytes, 256-byte aligned; must not overlap any other argument.
 * Calls that share a workspace must be ordered on one stream.
 *
 * Engines.  At small M (fp16 X and Y, no bias, R = 0) the whole layer is
 * ONE kernel by default (convrot_set_small_m_engine says which M and what the
 * other modes do).  Otherwise a rotate+quantize kernel is followed by the GEMM
 * kernel (exactly convrot_linear_prologue + convrot_linear_gemm below).  After
 * convrot_set_fused(1), calls with R = 0, M above the skinny range and K a
 * power of two in [256, 16384] run the whole layer as ONE persistent kernel
 * (one CTA per SM, cooperative launch): each CTA rotates and quantizes a
 * share of the rows of X, the CTAs meet at a grid barrier, then the same CTAs
 * run the tensor-core product on the codes.  Both engines give bit-identical
 * Y.
 * The first 256 bytes of the workspace carry the grid barrier's state from
 * one call to the next.  They need no initialization: a state that fails its
 * hash check (uninitialized memory, or a call that timed out) is rebuilt by
 * the next call, which then pays a slower barrier (tens of microseconds)
 * once.  Zero-filling them is always safe and starts in the valid state.
 * After CONVROT_ERR_TIMEOUT from convrot_check_device_error, treat the
 * workspace's other contents as undefined.
 */
convrot_status convrot_linear(const uint16_t* X, int64_t M, int64_t K, const int8_t* Q_W,
                              const float* s_W, const uint16_t* W_img, int64_t N,
                              const uint16_t* lora_down, const uint16_t* lora_up, int64_t R,
                              float lora_scale, uint16_t* Y, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * The rotated activation alone, X_rot = X H rounded to fp16 (X fp16 [M, K],
 * X_rot fp16 [M, K], both 16-byte aligned): the activation side of a
 * weight-only (W8A16) layer, which multiplies X_rot by the dequantized weight
 * in fp16.  Page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix,
 * and MLX", section "What changed in the computation" (X_rot = X H), and the
 * PR page's weight-only design ("the activation is rotated online").  Same
 * transform and fp32 butterflies as the quantizing prologue, without the
 * row max and codes.  K / 64 must be a power of two and K <= 16384 (other
 * shapes: CONVROT_ERR_INVALID_ARG).  Asynchronous on `stream`.
 */
convrot_status convrot_rotate(const uint16_t* X, int64_t M, int64_t K, uint16_t* X_rot,
                              void* stream);

/* Element types of convrot_linear_ex's activations, LoRA weights and output. */
#define CONVROT_DTYPE_F16 0
#define CONVROT_DTYPE_BF16 1

/*
 * convrot_linear with a choice of activation / output type and an optional
 * bias.  Page "[PR #249] Add an mps backend: weight-only INT8 and W4A8/W6A8
 * linears for Apple GPUs", section "Design": the epilogue adds the bias in
 * eager's order and writes bf16 as torch's cast does.
 *
 *   X        x_dtype [M, K] (fp16 or bf16; widened exactly to fp32 before the
 *            rotation).  lora_down [R, K] and lora_up [N, R] have the same
 *            type as X.
 *   bias     fp32 [N], 4-byte aligned, or NULL.
 *   Y        y_dtype [M, N]:
 *              y = fl(fl((float)A * s_X[m]) * s_W[n])   (the scale restore)
 *              y = fl(y + bias[n])                      (its own fp32 add)
 *              y = y + lora_scale * sum_r T[m,r] * lora_up[n,r]   (fp32)
 *            then one rounding to fp16 or bf16 (nearest even; overflow to
 *            +-inf).
 * Everything else is as convrot_linear (which is this call with fp16 in and
 * out and no bias).  The single-kernel engine (convrot_set_fused) applies to
 * fp16 in and out without a bias only; other calls run the two-kernel
 * engine.  Returns CONVROT_ERR_INVALID_ARG for another dtype value or a
 * misaligned bias.
 */
convrot_status convrot_linear_ex(const void* X, int x_dtype, int64_t M, int64_t K,
                                 const int8_t* Q_W, const float* s_W, const uint16_t* W_img,
                                 int64_t N, const float* bias, const void* lora_down,
                                 const void* lora_up, int64_t R, float lora_scale, void* Y,
                                 int y_dtype, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * convrot_linear in two stages, for callers that schedule or time them apart
 * (convrot_linear is exactly the prologue followed by the GEMM stage):
 *   convrot_linear_prologue  rotate + quantize X into the workspace (and the
 *                            LoRA down-projection T when R > 0);
 *   convrot_linear_gemm      the int8 product and the scale-restore/LoRA
 *                            epilogue from the workspace into Y.
 * Both take the same M, N, K, R, the same workspace and the same "weight image
 * supplied" choice, and must be ordered on one stream.  The GEMM stage may be
 * repeated after one prologue stage (the workspace then still holds the
 * codes); the workspace must not be written in between.  When the GEMM
 * splits K, its int32 partial sums meet in a workspace accumulator: the
 * prologue stage zeroes it, and every split GEMM leaves it zero again, so
 * neither stage needs a memset.
 */
convrot_status convrot_linear_prologue(const uint16_t* X, int64_t M, int64_t K, int64_t N,
                                       const uint16_t* lora_down, int64_t R,
                                       int with_weight_image, void* workspace,
                                       size_t workspace_bytes, void* stream);
convrot_status convrot_linear_gemm(int64_t M, int64_t K, const int8_t* Q_W, const float* s_W,
                                   const uint16_t* W_img, int64_t N, const uint16_t* lora_up,
                                   int64_t R, float lora_scale, uint16_t* Y, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * Parity and inspection only: where convrot_linear_prologue leaves the
 * activation codes and scales in a workspace of convrot_linear_workspace_bytes
 * (M, N, K, R, with_weight_image) bytes (page "INT8ConvRot GEMM vs fp16 on M1
 * Max with Metal, MPSMatrix, and MLX", section "What changed in the
 * computation": Q_X = round(X_rot / s_X), s_X = max|X_rot| / 127 per row).
 *   *qx_offset  byte offset of Q_X [M, K], row-major
 *   *qx_format  CONVROT_CODES_I8 (int8 codes, the small-M engine) or
 *               CONVROT_CODES_F16 (fp16 values that hold the int8 codes exactly:
 *               the tensor-core engines' operand image)
 *   *sx_offset  byte offset of s_X fp32 [M]
 * The contents are valid after a prologue stage on that workspace (or a
 * whole convrot_linear call, except one that runs the one-kernel small-M
 * layer, which leaves the workspace untouched), until the workspace is
 * written again.  Host-only:
 * no device work.  CONVROT_ERR_INVALID_ARG for sizes convrot_linear rejects
 * or null outputs.
 */
#define CONVROT_CODES_I8 0
#define CONVROT_CODES_F16 1
convrot_status convrot_linear_workspace_layout(int64_t M, int64_t N, int64_t K, int64_t R,
                                               int with_weight_image, int64_t* qx_offset,
                                               int* qx_format, int64_t* sx_offset);

/*
 * How many kernels one convrot_linear call (fp16 X and Y) with these sizes
 * launches on the current device under the current engine settings
 * (convrot_set_small_m_engine, convrot_set_fused): 1 for the one-kernel
 * small-M layer; otherwise rotate+quantize and the GEMM, plus the LoRA down-
 * and up-projections when R > 0, plus the weight widening when the call has
 * no weight image and uses a tensor-core engine.  Memsets are not counted.
 * Host-only.  -1 for sizes convrot_linear rejects or when the device query
 * fails.
 */
int convrot_linear_kernel_count(int64_t M, int64_t N, int64_t K, int64_t R, int with_weight_image);

/*
 * convrot_linear with the activation and the result in HOST memory: copies
 * X_host to the device (into `workspace`), runs the layer and copies Y back
 * to Y_host, all enqueued on `stream`.  X_host and Y_host should be pinned
 * (page-locked) for the copies to be asynchronous; Y_host is complete once
 * the stream is synchronized.  The workspace must hold
 * convrot_linear_host_workspace_bytes(M, N, K, R, W_img != NULL) bytes.
 */
size_t convrot_linear_host_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t R,
                                           int with_weight_image);
convrot_status convrot_linear_host(const uint16_t* X_host, int64_t M, int64_t K,
                                   const int8_t* Q_W, const float* s_W, const uint16_t* W_img,
                                   int64_t N, const uint16_t* lora_down,
                                   const uint16_t* lora_up, int64_t R, float lora_scale,
                                   uint16_t* Y_host, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * Synchronizes `stream`, then reads and clears the device error flag of the
 * current device.  CONVROT_ERR_TIMEOUT if a kernel gave up on a bounded wait
 * since the last check (its detail code is stored in *detail when detail is
 * not NULL), CONVROT_ERR_CUDA if the synchronization failed, else CONVROT_OK.
 */
convrot_status convrot_check_device_error(void* stream, int* detail);

/* Detail codes stored by convrot_check_device_error (the wait that ran out). */
#define CONVROT_DETAIL_MMA_WAIT_TILE 1      /* MMA issuer, for a loaded stage */
#define CONVROT_DETAIL_LOAD_WAIT_SLOT 2     /* TMA producer, for a free stage */
#define CONVROT_DETAIL_EPI_WAIT_ACC 3       /* epilogue, for a full accumulator */
#define CONVROT_DETAIL_MMA_WAIT_ACC 4       /* MMA issuer, for a drained accumulator */
#define CONVROT_DETAIL_ROTQ_WAIT_TILE 5     /* rotate+quantize, for its tile of X */
#define CONVROT_DETAIL_DRAIN 6              /* waiting for copies/MMAs on the way out */
#define CONVROT_DETAIL_GRID_BARRIER 7       /* single-kernel engine, for the other CTAs */
#define CONVROT_DETAIL_PAIR 8               /* CTA-pair split, for the partner CTA */
#define CONVROT_DETAIL_SELFTEST 9           /* convrot_selftest_wait_timeout */

/*
 * Failure-detection self-test: launches one CTA that waits on an mbarrier
 * nothing will ever arrive on, with a spin budget of `budget_cycles` SM clock
 * cycles (1 .. 2e9).  The wait gives up, records CONVROT_DETAIL_SELFTEST and
 * the kernel returns normally: nothing faults or hangs, and the context stays
 * usable.  The next convrot_check_device_error on that stream then returns
 * CONVROT_ERR_TIMEOUT with that detail.  This is the path every bounded wait
 * of the library takes when something it waits for never comes.
 * CONVROT_ERR_INVALID_ARG for a budget outside the range.
 */
convrot_status convrot_selftest_wait_timeout(int64_t budget_cycles, void* stream);

/* ------------------------------------------------------------------------
 * Entry points that expose one step of the path, for parity checks.
 * ------------------------------------------------------------------------ */

/*
 * The activation step alone ("Every time the linear layer is called, the
 * activations are rotated and quantized"): X fp16 [M, K] -> Q_X int8 [M, K],
 * s_X fp32 [M].  Same kernel and arithmetic as inside convrot_linear.
 */
convrot_status convrot_rotate_quantize(const uint16_t* X, int64_t M, int64_t K, int8_t* Q_X,
                                       float* s_X, void* stream);

/*
 * The integer product alone, A = Q_X Q_W^T (exact int32), with the given
 * GEMM engine.  Q_X int8 [M, K], Q_W int8 [N, K], A int32 [M, N].  The
 * workspace must hold convrot_gemm_workspace_bytes(M, N, K, path) bytes.
 */
size_t convrot_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int path);
convrot_status convrot_gemm_i32(const int8_t* Q_X, const int8_t* Q_W, int64_t M, int64_t N,
                                int64_t K, int32_t* A, int path, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * The product and the scale restore from given int8 operands and scales:
 * Y = fp16(((float)(Q_X Q_W^T) * s_X[m]) * s_W[n]).  Same workspace size as
 * convrot_gemm_i32.
 */
convrot_status convrot_gemm_dequant(const int8_t* Q_X, const float* s_X, const int8_t* Q_W,
                                    const float* s_W, int64_t M, int64_t N, int64_t K,
                                    uint16_t* Y, int path, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * The small-M layer for callers that cannot supply a workspace or allocate
 * device memory: plugin hosts that give a layer no scratch buffer, and
 * engines that forbid cudaMalloc once running (it can synchronize the device
 * and has no place in a fixed memory plan).  The pages have no counterpart to
 * this entry point; it exists for such callers only.
 *
 * Computes the same Y as convrot_linear without LoRA (X fp16 [M,K], Q_W int8
 * [N,K], s_W fp32 [N] -> Y fp16 [M,N]; the small-M engine) but takes its
 * scratch from a fixed array inside the library: CONVROT_NOALLOC_SCRATCH_BYTES
 * of device memory that every GPU which loads the library holds until the
 * process exits.  Limits: M <= CONVROT_NOALLOC_MAX_M (larger M returns
 * CONVROT_ERR_WORKSPACE with nothing launched).  One call uses M*K code bytes
 * and 4*M scale bytes of the array, each rounded up to 256: at most 1 MiB +
 * 512 bytes within these limits; a call that would not fit returns
 * CONVROT_ERR_WORKSPACE.  Calls no allocating routine (no cudaMalloc, no
 * cudaFree).
 *
 * The array is shared by every call on a device and keeps the previous call's
 * contents.  Nothing in it needs to start at zero, so no call clears it.
 * Calls that can overlap on the GPU -- on different streams without ordering
 * between them -- race on it.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture.
 */
#define CONVROT_NOALLOC_SCRATCH_BYTES (4u << 20)
#define CONVROT_NOALLOC_MAX_M 16
convrot_status convrot_linear_noalloc(const uint16_t* X, int64_t M, int64_t K, const int8_t* Q_W,
                                      const float* s_W, int64_t N, uint16_t* Y, void* stream);

/*
 * Measurement only: the throughput ceiling of one of the engines that
 * compute the exact product A = Q_X Q_W^T (page "INT8ConvRot GEMM vs fp16 on
 * M1 Max with Metal, MPSMatrix, and MLX", section "What changed in the
 * computation": int8 x int8 with int32 accumulation).  sm_103a has no integer
 * tcgen05 MMA, so the library computes that product with tcgen05.mma
 * kind::f16 on operands that hold the int8 values exactly
 * (CONVROT_PEAK_TCGEN05_F16, 128 x 256 x 16 MMAs, the large-M paths), with
 * mma.sync m16n8k16 f16 -> f32 on such operands (CONVROT_PEAK_MMA_F16, the
 * small-M GEMM at M >= 3), with 4-way int8 dot products (CONVROT_PEAK_DP4A,
 * the one-kernel small-M layer), or with mma.sync m16n8k32 s8 x s8 -> s32
 * (CONVROT_PEAK_MMA_S8, the small-M GEMM's other kernel).
 * Runs `reps` repetitions of back-to-back instructions on operands already in
 * registers or shared memory (no loads, no epilogue) on every SM, then
 * synchronizes `stream`.  *ops receives the integer or floating-point
 * operations performed (2 per multiply-add) and *ms the device time between
 * two events on `stream`.  reps must be in [1, 2^24]; an unknown engine or a
 * null output pointer is CONVROT_ERR_INVALID_ARG.
 */
#define CONVROT_PEAK_MMA_S8 0
#define CONVROT_PEAK_TCGEN05_F16 1
#define CONVROT_PEAK_MMA_F16 2
#define CONVROT_PEAK_DP4A 3
convrot_status convrot_measure_engine_peak(int engine, int64_t reps, double* ops, float* ms,
                                           void* stream);

/*
 * Engine choice for every later convrot_linear call in this process: enable
 * = 1 selects the single-kernel engine where it applies, 0 (the default) the
 * two-kernel engine.  Other values are rejected with CONVROT_ERR_INVALID_ARG.
 */
convrot_status convrot_set_fused(int enable);

/*
 * The engine of convrot_linear / convrot_linear_ex at M <= 16 with fp16 X
 * and Y, no bias and no LoRA, for every later call in this process.
 *   The one-kernel layer: each CTA of a thread-block cluster rotates and
 *     quantizes its K slice of the rows, the cluster combines the row maxima
 *     in distributed shared memory, and the same CTAs multiply by their
 *     weight slice and restore the scales; the workspace is not touched.  Two
 *     forms: 32 output columns per CTA with exact int8 dot products (dp4a),
 *     or 128 output columns per CTA with the fp16 warp MMA on exact int8
 *     values (fp32 sums moved to int32 every 1024 K).  The second repeats
 *     the rotation in four times fewer CTAs and runs the product at four
 *     times the rate, but holds one CTA per SM; it measured slower than the
 *     two-kernel path and is not chosen by default.  A third form shares
 *     the rotation among the column blocks of a cluster: a cluster of
 *     (K slices) x (2, 4 or 8 blocks of 32 columns), at most eight CTAs;
 *     each CTA rotates 1 / blocks of its slice's 256-groups (at most 16
 *     (row, group) items), the cluster exchanges row maxima, and each CTA
 *     writes its codes into the shared memory of every CTA on its slice;
 *     the product runs on the fp16 warp MMA.  It applies where the blocks
 *     divide the slice's groups with at most 16 items per CTA.
 *     See convrot_set_small_m_weights_early for when it reads Q_W.
 *   The two-kernel path: rotate + quantize into the workspace, then the
 *     small-M GEMM; every input is read after the dependency wait.
 *   mode 0 (the default): the dp4a form at M <= 2 where it takes K (slices
 *     of at most 4096 in eight); the two-kernel path otherwise.
 *   mode 1: the two-kernel path at every M.
 *   mode 2: the dp4a form at every M <= 16 (where it takes the sizes).
 *   mode 3: the MMA form at every M <= 16 (where it takes the sizes).
 *   mode 4: the shared-rotation form where it applies, mode 0 elsewhere.
 * Every mode gives the same bits.  Other values: CONVROT_ERR_INVALID_ARG.
 */
convrot_status convrot_set_small_m_engine(int mode);

/*
 * enable = 1 (the default): the one-kernel small-M layer copies its weight
 * slice into shared memory BEFORE it waits for the kernel ahead of it on the
 * stream (programmatic dependent launch), overlapping that kernel's tail and
 * the launch gap (about a microsecond a layer).  Q_W must then not be written
 * by that kernel if it lets dependents start before it finishes.  No kernel
 * of this library that writes int8 data does (convrot_prepare_weight,
 * convrot_rotate_quantize); a weight written by a copy, or by any kernel that
 * does not trigger dependent launch early, or separated from the call by an
 * event record, is safe.  X and s_W are always read after the wait.
 * enable = 0: every input is read after the wait.  Same bits either way.
 * Other values: CONVROT_ERR_INVALID_ARG.
 */
convrot_status convrot_set_small_m_weights_early(int enable);

/*
 * Testing hook: the GEMM of the two-kernel path at M <= 16, for every later
 * call in this process.  mode 0 (the default): at M >= 3 with fp16 Y, no
 * bias and no LoRA, a kernel that copies the prologue's codes and the weight
 * into shared memory by bulk copies and runs the product on the fp16 warp
 * MMA (the int8 values exact in fp16; each warp's fp32 sum over at most 1024
 * K an exact integer), 32 output columns per CTA and K slices across a
 * thread-block cluster, summed as int32; otherwise the mma.sync s8 kernel
 * with register loads.  mode 1: always the s8 kernel.  mode 2: the fp16-MMA
 * kernel wherever it applies.  Every mode gives the same bits.  Other
 * values: CONVROT_ERR_INVALID_ARG.
 */
convrot_status convrot_set_skinny_engine(int mode);

/*
 * Testing hook: how the tensor-core GEMM may split K, for every later call in
 * this process.  mode 0 (the default): chosen by shape; 1: never across a
 * CTA pair; 2: across a CTA pair wherever that applies (fp16 output in rows
 * of 16-byte multiples, no LoRA, K a multiple of 512); 3: the streaming
 * CTA-pair split wherever that applies (the same conditions, no bias, fp16
 * output, K <= 2048).  In the pair split the two halves of K of an output
 * tile run on the two CTAs of a thread-block cluster, which add their exact
 * partials through distributed shared memory; the streaming form moves each
 * half's fp32 partial (an exact integer of at most 2^24) straight from
 * tensor memory.  Other values: CONVROT_ERR_INVALID_ARG.
 */
convrot_status convrot_set_split_mode(int mode);

/*
 * Testing hook: whether the tensor-core GEMM may run its tiles on CTA-pair
 * MMAs, for every later call in this process.  mode 0 (the default): chosen
 * by shape; 1: never; 2: wherever that applies (fp16 output in rows of
 * 16-byte multiples, no K split; LoRA allowed).  A pair-MMA tile is 256 x 128 or
 * 256 x 256 outputs computed by the two CTAs of a thread-block cluster with
 * tcgen05 MMAs that span both SMs (.cta_group::2): each SM holds 128 rows of
 * the tile and loads half of its weight rows.  Results are bit-identical to
 * the one-SM tiles.  Other values: CONVROT_ERR_INVALID_ARG.
 */
convrot_status convrot_set_pair_mma(int mode);

/*
 * The 4x4 Hadamard base B of the rotation, for every later call in this
 * process (page "INT8ConvRot GEMM vs fp16 on M1 Max with Metal, MPSMatrix,
 * and MLX", section "What changed in the computation": H is the Kronecker
 * power of 4x4 Hadamard matrices over groups of 256, divided by 16, and
 * symmetric).  base: 16 int8 entries, row-major, each +1 or -1, symmetric,
 * with B B^T = 4 I; NULL restores the default, Sylvester's
 * [[1,1,1,1],[1,-1,1,-1],[1,1,-1,-1],[1,-1,-1,1]].  Anything else:
 * CONVROT_ERR_INVALID_ARG, with the base unchanged.  Host-only (no device
 * work); not synchronised with calls running on other threads.
 *
 * Such a B factors as D1 H4 R (D1 a diagonal of signs, H4 Sylvester's, R a
 * signed permutation).  The kernels negate the inputs by D1 (x) D1 (x) D1 (x)
 * D1 and run the Sylvester transform; the signed permutation R (x) R (x) R
 * (x) R of the rotated columns is left out.  Quantization commutes with it
 * and it is the same for X and W, so Y of convrot_linear (and of every entry
 * built on it) is exactly that of base B.  The codes written by
 * convrot_prepare_weight and convrot_rotate_quantize are therefore those of
 * base B with their columns in this library's order: weight codes made
 * elsewhere for a base other than Sylvester's must come from
 * convrot_prepare_weight.  convrot_rotate, whose output is X H itself, takes
 * Sylvester's base only (CONVROT_ERR_INVALID_ARG otherwise); the
 * single-kernel engine is not used with a sign-changing base.
 */
convrot_status convrot_set_hadamard_base(const int8_t* base);

/*
 * The tensor-core GEMM's plan for an M x N x K layer, computed on the host
 * from the numbers a device would give: sms streaming multiprocessors and
 * the resident 2-CTA clusters of the CTA-pair MMA tiles 128 and 256 wide
 * (0: that engine is unavailable).  tma_store: Y rows are 16-byte multiples
 * (fp16 output through TMA stores, taken as fp16 without a bias); R: LoRA
 * ranks.  Writes the tile width
 * (*bn: 64, 128 or 256 columns), the K split count (*splits, 1 = none) and
 * the engine (*engine, CONVROT_ENGINE_*).  The hooks
 * convrot_set_tile_override, convrot_set_split_mode and convrot_set_pair_mma
 * apply as in a real call.  No device work; CONVROT_ERR_INVALID_ARG on bad
 * sizes or null outputs.
 */
#define CONVROT_ENGINE_ONE_SM 0     /* 128 x bn tiles, one per CTA and SM */
#define CONVROT_ENGINE_PAIR_SPLIT 1 /* the two K halves of a tile on a 2-CTA cluster */
#define CONVROT_ENGINE_PAIR_MMA 2   /* 256 x bn tiles on tcgen05 .cta_group::2 MMAs */
#define CONVROT_ENGINE_L2_SPLIT 3   /* K splits added through L2 */
#define CONVROT_ENGINE_PAIR_STREAM 4 /* K halves on a 2-CTA cluster, streaming exchange */
convrot_status convrot_plan_gemm(int64_t M, int64_t N, int64_t K, int sms, int pair_clusters_128,
                                 int pair_clusters_256, int tma_store, int64_t R, int* bn,
                                 int* splits, int* engine);

/*
 * The small-M engine convrot_linear takes for an M x N x K layer with fp16 X
 * and Y, no bias and no LoRA, computed on the host from `sms` streaming
 * multiprocessors under the current engine settings
 * (convrot_set_small_m_engine, convrot_set_skinny_engine).  Writes the
 * engine (*engine, CONVROT_SMALL_M_*), its K slices per thread-block cluster
 * (*splits; 0 with CONVROT_SMALL_M_NONE) and, for the shared-rotation form,
 * the column blocks per cluster (*blocks, else 0).  No device work;
 * CONVROT_ERR_INVALID_ARG on bad sizes or null outputs.
 */
#define CONVROT_SMALL_M_NONE 0       /* M above the small-M range: the tensor-core GEMM */
#define CONVROT_SMALL_M_ONE_DP4A 1   /* one kernel, 32 columns per CTA, dp4a product */
#define CONVROT_SMALL_M_ONE_MMA 2    /* one kernel, 128 columns per CTA, fp16 warp MMA */
#define CONVROT_SMALL_M_ONE_SHARED 3 /* one kernel, the rotation shared by a cluster's column blocks */
#define CONVROT_SMALL_M_TWO_F16 4    /* rotate + quantize, then the fp16-MMA small-M GEMM */
#define CONVROT_SMALL_M_TWO_S8 5     /* rotate + quantize, then the mma.sync s8 small-M GEMM */
convrot_status convrot_plan_small_m(int64_t M, int64_t N, int64_t K, int sms, int* engine,
                                    int* splits, int* blocks);

/*
 * Testing hook: forces the tensor-core GEMM's tile width (64, 128 or 256
 * columns; 0 = automatic) and K split count (1..16; 0 = automatic) for every
 * later call in this process, so that tests can reach each code path on
 * small shapes.  A split count larger than the shape allows is ignored.
 */
convrot_status convrot_set_tile_override(int bn, int splits);

#ifdef __cplusplus
}
#endif

#endif /* CONVROT_H */
