// convrot_linear_noalloc: the small-M layer with library-owned scratch.
//
// The regular entry points take their scratch from a caller-provided
// workspace.  This one serves callers that cannot provide one and cannot
// allocate device memory themselves: plugin hosts that give a layer no
// scratch buffer, and engines that forbid cudaMalloc after start-up (it can
// synchronize the whole device, and a fixed memory plan has no room for it).
// Its scratch is a fixed, file-scope device array that every GPU which loads
// the library holds until the process exits.
//
// The scratch holds, for one call, the int8 activation codes Q_X [M, K] and
// the row scales s_X [M]: M*K + 4*M bytes, each part rounded up to 256.  The
// small-M product reduces its K slices inside each thread-block cluster
// (distributed shared memory), so nothing in the scratch needs to start at
// zero and no call clears it.  All calls on a device share the one array and
// it keeps the last call's contents: calls that can overlap on the GPU
// (different streams without ordering) race on it and give wrong results.
//
// Set-up: the first call on each device, with that device current, looks up
// the device address of the array with cudaGetSymbolAddress (in host code the
// array's name is only a host-side stand-in, not a device address) and caches
// it.  Make that first call before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/convrot.h"
#include "kernels.h"

namespace convrot {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[CONVROT_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;

struct NoallocDevice {
  bool init = false;
  bool supported = false;
  int sms = 0;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[kNoallocMaxDevices];

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

convrot_status noalloc_device(NoallocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CONVROT_ERR_CUDA;
  if (dev < 0 || dev >= kNoallocMaxDevices) return CONVROT_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocDevice& d = g_noalloc_dev[dev];
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
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return CONVROT_ERR_CUDA;
      d.scratch = static_cast<uint8_t*>(p);
    }
    d.init = true;
  }
  if (!d.supported) return CONVROT_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return CONVROT_OK;
}

struct NoallocLayout {
  size_t qx, sx, total;
};

// Codes, then scales.  With M <= CONVROT_NOALLOC_MAX_M and K <= CONVROT_MAX_K
// this is at most 1 MiB + 512 bytes; the capacity check in the entry point
// stays as a guard should either limit grow.
NoallocLayout noalloc_layout(int64_t M, int64_t K) {
  NoallocLayout L;
  size_t off = 0;
  L.qx = off;
  off += round256(static_cast<size_t>(M) * K);
  L.sx = off;
  off += round256(static_cast<size_t>(M) * 4);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace convrot

using namespace convrot;

extern "C" convrot_status convrot_linear_noalloc(const uint16_t* X, int64_t M, int64_t K,
                                                 const int8_t* Q_W, const float* s_W, int64_t N,
                                                 uint16_t* Y, void* stream) {
  if (M < 0 || N < 0 || N > CONVROT_MAX_DIM || K <= 0 || K % 256 != 0 || K > CONVROT_MAX_K)
    return CONVROT_ERR_INVALID_ARG;
  if (!X || !Q_W || !s_W || !Y) return CONVROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Q_W) |
       reinterpret_cast<uintptr_t>(Y)) & 15u)
    return CONVROT_ERR_INVALID_ARG;
  if (M > CONVROT_NOALLOC_MAX_M) return CONVROT_ERR_WORKSPACE;
  if (M == 0 || N == 0) return CONVROT_OK;
  const NoallocLayout L = noalloc_layout(M, K);
  if (L.total > CONVROT_NOALLOC_SCRATCH_BYTES) return CONVROT_ERR_WORKSPACE;
  NoallocDevice* d = nullptr;
  const convrot_status s = noalloc_device(&d);
  if (s != CONVROT_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int8_t* qx = reinterpret_cast<int8_t*>(d->scratch + L.qx);
  float* sx = reinterpret_cast<float*>(d->scratch + L.sx);

  // Rotate + quantize each row into the scratch codes and scales.
  RotqRowArgs r;
  r.in = X;
  r.rows = M;
  r.K = static_cast<int>(K);
  r.q_out = qx;
  r.img_out = nullptr;
  r.s_out = sx;
  hadamard_signs(r.sign);
  if (launch_rotq_row(r, kRowInF16, static_cast<int>(M), st) != cudaSuccess) return CONVROT_ERR_CUDA;

  // Skinny product and scale restore (K split across the CTAs of clusters,
  // reduced in shared memory: the scratch needs no zeroing).
  GemmSkinnyArgs g;
  g.QX = qx;
  g.QW = Q_W;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.splits = skinny_cluster_size(N, K, d->sms);
  g.k_per_split = static_cast<int>(K / g.splits);
  g.ep.mode = kOutF16;
  g.ep.Y = Y;
  g.ep.A = nullptr;
  g.ep.sX = sx;
  g.ep.sW = s_W;
  g.ep.T = nullptr;
  g.ep.up = nullptr;
  g.ep.R = 0;
  g.ep.lora_scale = 0.0f;
  return launch_gemm_skinny(g, st) == cudaSuccess ? CONVROT_OK : CONVROT_ERR_CUDA;
}
