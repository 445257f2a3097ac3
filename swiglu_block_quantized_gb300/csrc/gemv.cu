// gemv.cu -- host launcher for the decode-sized (M <= 16) streaming kernel.
#include <atomic>

#include "gemv.cuh"
#include "launch.h"

namespace m4q {

template <int C, bool SWIGLU, int MT, bool WTMA, bool XH>
cudaError_t launch_gemv_one(const ProjLaunch& L, GemvParams p) {
  using Cfg = GemvCfg<C, MT>;
  const int ring = Cfg::kRingBytes / (8 * p.pp);
  p.ring = ring < Cfg::kRingMax ? ring : Cfg::kRingMax;
  auto kern = gemv_kernel<C, SWIGLU, MT, WTMA, XH>;
  std::atomic<unsigned long long>& configured =
      attr_flag<std::integer_sequence<int, 2, C, SWIGLU, MT, WTMA, XH>>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const unsigned grid = (unsigned)(p.units < L.sms ? p.units : L.sms);
  return launch_proj(kern, grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream, 1u, p);
}

template <int C, bool SWIGLU, bool WTMA>
cudaError_t launch_gemv_mt(const ProjLaunch& L) {
  using Cfg = GemvCfg<C, 1>;   // stage sizes do not depend on MT
  GemvParams p;
  p.x = static_cast<const __half*>(L.x);
  p.w0 = static_cast<const uint8_t*>(L.w0);
  p.w1 = static_cast<const uint8_t*>(L.w1);
  p.y = static_cast<__half*>(L.y);
  p.M = L.M;
  p.N = L.N;
  p.K = L.K;
  p.row_bytes = L.row_bytes;
  // A row that fits one stage travels whole (row pairs are then contiguous);
  // longer rows in segments of kSBMax bytes.
  p.sb = (int)(L.row_bytes <= Cfg::kSBMax ? L.row_bytes : Cfg::kSBMax);
  p.nst = (int)((L.row_bytes + p.sb - 1) / p.sb);
  p.pp = 2 * p.sb + 16;
  p.units = (L.N + 15) / 16;
  p.act = L.act;
  p.head_dim = L.head_dim;
  p.status = L.status;
  p.limit_ns = L.limit_ns;
  // X fragments stay in registers when the row is exactly one full stage
  // (M <= 8; Q2_0 fragments are too large).
  if (L.mt == 2) return launch_gemv_one<C, SWIGLU, 2, WTMA, false>(L, p);
  if constexpr (C != kQ2_0) {
    if (L.row_bytes == Cfg::kSBMax) return launch_gemv_one<C, SWIGLU, 1, WTMA, true>(L, p);
  }
  return launch_gemv_one<C, SWIGLU, 1, WTMA, false>(L, p);
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
    case kMLX4: return launch_gemv_codec<kMLX4>(L);
    default: return launch_gemv_codec<kQ2_0>(L);
  }
}

}  // namespace m4q
