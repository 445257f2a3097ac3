// gemv.cu -- host launcher for the decode-sized (M <= 16) streaming kernels.
#include <atomic>

#include "gemv.cuh"
#include "launch.h"

namespace m4q {

template <int C, bool SWIGLU, int MT, bool WTMA>
cudaError_t launch_gemv_one(const ProjLaunch& L) {
  using Cfg = GemvCfg<C, SWIGLU>;
  auto kern = gemv_kernel<C, SWIGLU, MT, WTMA>;
  std::atomic<unsigned long long>& configured = attr_flag<std::integer_sequence<int, 2, C, SWIGLU, MT, WTMA>>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  GemvParams p;
  p.x = static_cast<const __half*>(L.x);
  p.w0 = static_cast<const uint8_t*>(L.w0);
  p.w1 = static_cast<const uint8_t*>(L.w1);
  p.y = static_cast<__half*>(L.y);
  p.M = L.M;
  p.N = L.N;
  p.K = L.K;
  p.row_bytes = L.row_bytes;
  p.kw = L.kw;
  p.nstages = L.nstages;
  p.status = L.status;
  p.limit_ns = L.limit_ns;
  const int rows_per_cta = 16 * (8 / L.kw);
  const unsigned grid = (unsigned)((L.N + rows_per_cta - 1) / rows_per_cta);
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream>>>(L.tm_w0, L.tm_w1, p);
  return cudaGetLastError();
}

template <int C, bool SWIGLU, bool WTMA>
cudaError_t launch_gemv_mt(const ProjLaunch& L) {
  return L.mt == 1 ? launch_gemv_one<C, SWIGLU, 1, WTMA>(L) : launch_gemv_one<C, SWIGLU, 2, WTMA>(L);
}

template <int C>
cudaError_t launch_gemv_codec(const ProjLaunch& L) {
  if (L.wtma) return L.swiglu ? launch_gemv_mt<C, true, true>(L) : launch_gemv_mt<C, false, true>(L);
  return L.swiglu ? launch_gemv_mt<C, true, false>(L) : launch_gemv_mt<C, false, false>(L);
}

cudaError_t launch_gemv(int codec, const ProjLaunch& L) {
  switch (codec) {
    case kQ4_0: return launch_gemv_codec<kQ4_0>(L);
    case kQ8_0: return launch_gemv_codec<kQ8_0>(L);
    default: return launch_gemv_codec<kQ2_0>(L);
  }
}

}  // namespace m4q
