// noalloc.cu -- m4q_mlp_noalloc: the gated MLP block of m4q_mlp for callers
// that cannot allocate device memory.
//
// Some callers of this library have no way to obtain a scratch buffer: an
// inference runtime that reserves all device memory up front and hands out
// no allocator to plug-ins, or a latency-critical loop that must not call
// cudaMalloc (which may synchronize the device).  m4q_mlp needs such a
// buffer for the fp16 intermediate H [M, F].  This entry point uses instead
// one fixed array that lives in the library's device code (kMaxH fp16
// elements, 2 MiB, held on every GPU that loads the library until the
// process exits), so the caller passes only inputs and the output.
//
// Set-up: the host cannot use the array's name as a device address.  The
// first call on each device checks that the device is an sm_103 part, looks
// the address up with cudaGetSymbolAddress, with that device current, and
// keeps it in a per-device table for the life of the process; later calls
// reuse it.  That first call should therefore be made before any stream
// capture on that device.  A cudaDeviceReset() destroys the array with the
// rest of the device's context and leaves the kept address stale, so a
// process that resets a device must not call this entry point on it again.
//
// Sharing: every call on a device writes the same array.  The gated
// projection overwrites all M * F elements of H before the down projection
// reads them (stream order), so nothing has to start at zero and no earlier
// call's contents can leak into a result; but two calls whose work overlaps
// on the GPU (different streams, no ordering between them) race on H.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/m4q.h"

namespace {

constexpr long long kMaxH = 1ll << 20;  // fp16 elements of the intermediate (2 MiB)
constexpr int kMaxDevices = 64;

static __device__ __align__(256) __half g_mlp_scratch[kMaxH];

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of g_mlp_scratch on the current device (looked up once).
// A device that is not sm_103 holds no image of this library's device code,
// so it is turned away before the lookup, with the status every other entry
// point returns for it.  A failed lookup leaves CUDA's last-error slot set;
// it is cleared here so that a later, unrelated launch check does not report
// it.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M4Q_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return M4Q_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return M4Q_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return M4Q_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mlp_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return M4Q_ERR_CUDA;
    }
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return M4Q_OK;
}

}  // namespace

extern "C" int m4q_mlp_noalloc(const void* X, const void* Wg, const void* Wu, const void* Wd,
                               int codec_gu, int codec_d, int64_t M, int64_t D, int64_t F, void* Y,
                               int act, m4q_stream_t stream) {
  if (M < 1 || F < 1) return M4Q_ERR_INVALID_ARG;
  if (M > kMaxH / F) return M4Q_ERR_SCRATCH_LIMIT;  // M * F > kMaxH, without overflow
  void* h = nullptr;
  const int rc = scratch_address(&h);
  if (rc != M4Q_OK) return rc;
  return m4q_mlp(X, Wg, Wu, Wd, codec_gu, codec_d, M, D, F, h, Y, act, stream);
}
