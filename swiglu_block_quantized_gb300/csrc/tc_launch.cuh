// tc_launch.cuh -- host launcher for the tcgen05 projection kernels of one
// codec (instantiated once per codec in tc_q*.cu so they compile in parallel).
#pragma once

#include <atomic>

#include "launch.h"
#include "tc_proj.cuh"
#include "tc_small.cuh"

namespace m4q {

// Largest K split, from `split` down by halves, whose clusters (one per
// output tile) can all be resident on the device at once; the occupancy
// answer is kept per kernel, device and cluster size.
template <typename Kern>
int fit_split(Kern kern, int split, long long tiles, unsigned threads, size_t smem, int dev,
              std::atomic<int> (&fit)[64][4]) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  while (split > 1) {
    const int lg = split == 2 ? 1 : (split == 4 ? 2 : 3);
    int known = fit[dev & 63][lg].load();
    if (known == 0) {
      cfg.gridDim = dim3((unsigned)(tiles * split), 1, 1);
      attr[0].val.clusterDim.x = (unsigned)split;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      known = 1 + n;
      fit[dev & 63][lg].store(known);
    }
    if ((long long)(known - 1) >= tiles) break;
    split /= 2;
  }
  return split;
}

template <int C, bool SWIGLU, int NX, bool WTMA, int ACT, int HD>
cudaError_t launch_tc_one(const ProjLaunch& L) {
  using Cfg = TcCfg<C, SWIGLU, NX, WTMA>;
  auto kern = tc_proj_kernel<C, SWIGLU, NX, WTMA, ACT, HD>;
  std::atomic<unsigned long long>& configured =
      attr_flag<std::integer_sequence<int, 1, C, SWIGLU, NX, WTMA, ACT, HD>>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  TcParams p;
  p.w0 = static_cast<const uint8_t*>(L.w0);
  p.w1 = static_cast<const uint8_t*>(L.w1);
  p.y = static_cast<__half*>(L.y);
  p.M = L.M;
  p.N = L.N;
  p.K = L.K;
  p.row_bytes = L.row_bytes;
  p.m_tiles = (L.M + NX - 1) / NX;
  p.tiles = p.m_tiles * ((L.N + Cfg::kOutRows - 1) / Cfg::kOutRows);
  p.status = L.status;
  p.limit_ns = L.limit_ns;
  p.split = 1;
  if constexpr (NX <= 128 && HD == 0 && WTMA) {   // the K-split epilogue exists for these
    if (L.split > 1) {
      static std::atomic<int> fit[64][4];
      p.split = fit_split(kern, L.split, p.tiles, Cfg::kThreads, Cfg::kSmemBytes, dev, fit);
    }
  }
  const int npk = (L.K + Cfg::S::KP - 1) / Cfg::S::KP;
  p.ks_per = (npk / p.split) * Cfg::S::SUB;   // the host picks splits that divide npk
  // Persistent CTAs, or (K split) one cluster of p.split CTAs per output tile.
  const unsigned grid = p.split == 1 ? (unsigned)(p.tiles < L.sms ? p.tiles : L.sms)
                                     : (unsigned)(p.tiles * p.split);
  return launch_proj(kern, grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream, (unsigned)p.split, L.tm_x, L.tm_w0,
                     L.tm_w1, L.tm_y, p);
}

template <int C, bool SWIGLU, bool WTMA, int ACT, int HD>
cudaError_t launch_tc_nx(const ProjLaunch& L) {
  switch (L.nx) {
    case 256: return launch_tc_one<C, SWIGLU, 256, WTMA, ACT, HD>(L);
    case 128: return launch_tc_one<C, SWIGLU, 128, WTMA, ACT, HD>(L);
    default: return launch_tc_one<C, SWIGLU, 64, WTMA, ACT, HD>(L);
  }
}

// GEMM: row-major Y or the direct-head layout for head dim 64 or 128.
template <int C, bool WTMA>
cudaError_t launch_tc_gemm(const ProjLaunch& L) {
  switch (L.head_dim) {
    case 64: return launch_tc_nx<C, false, WTMA, 0, 64>(L);
    case 128: return launch_tc_nx<C, false, WTMA, 0, 128>(L);
    default: return launch_tc_nx<C, false, WTMA, 0, 0>(L);
  }
}

// The gate activation is a template argument: the SiLU epilogue stays
// exactly as it is without the GELU code beside it.
template <int C, bool WTMA>
cudaError_t launch_tc_glu(const ProjLaunch& L) {
  return L.act ? launch_tc_nx<C, true, WTMA, 1, 0>(L) : launch_tc_nx<C, true, WTMA, 0, 0>(L);
}

// Small M (<= 128): activations as the A operand, decoded weights as B.
template <int C, bool SWIGLU, int ACT, int XR>
cudaError_t launch_tcs_one(const ProjLaunch& L) {
  using Cfg = TsCfg<C, SWIGLU, XR>;
  if constexpr (!Cfg::kFits) {
    return cudaErrorInvalidConfiguration;   // not dispatched here (see api.cu)
  } else {
  auto kern = tc_small_kernel<C, SWIGLU, ACT, XR>;
  std::atomic<unsigned long long>& configured =
      attr_flag<std::integer_sequence<int, 4, C, SWIGLU, ACT, XR>>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  TcParams p;
  p.w0 = static_cast<const uint8_t*>(L.w0);
  p.w1 = static_cast<const uint8_t*>(L.w1);
  p.y = static_cast<__half*>(L.y);
  p.M = L.M;
  p.N = L.N;
  p.K = L.K;
  p.row_bytes = L.row_bytes;
  p.m_tiles = 1;
  p.tiles = (L.N + Cfg::kOutRows - 1) / Cfg::kOutRows;
  p.status = L.status;
  p.limit_ns = L.limit_ns;
  const int npk = (L.K + Cfg::S::KP - 1) / Cfg::S::KP;
  p.split = 1;
  if (L.split > 1) {
    static std::atomic<int> fit[64][4];   // per device ordinal, per log2 split: 0 unknown, 1 + max clusters
    p.split = fit_split(kern, L.split, p.tiles, Cfg::kThreads, Cfg::kSmemBytes, dev, fit);
  }
  p.ks_per = (npk / p.split) * Cfg::S::SUB;   // the host picks splits that divide npk
  // Persistent CTAs, or (K split) one cluster of p.split CTAs per output tile.
  const unsigned grid = p.split == 1 ? (unsigned)(p.tiles < L.sms ? p.tiles : L.sms)
                                     : (unsigned)(p.tiles * p.split);
  return launch_proj(kern, grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream, (unsigned)p.split, L.tm_x, L.tm_w0,
                     L.tm_w1, L.tm_y, p);
  }
}

template <int C, int XR>
cudaError_t launch_tcs_xr(const ProjLaunch& L) {
  if (!L.swiglu) return launch_tcs_one<C, false, 0, XR>(L);
  return L.act ? launch_tcs_one<C, true, 1, XR>(L) : launch_tcs_one<C, true, 0, XR>(L);
}

// L.nx = X rows per stage (32, 64 or 128; the X tensor map's box height).
template <int C>
cudaError_t launch_tcs(const ProjLaunch& L) {
  if (L.nx == 32) return launch_tcs_xr<C, 32>(L);
  if (L.nx == 64) return launch_tcs_xr<C, 64>(L);
  return launch_tcs_xr<C, 128>(L);
}

template <int C>
cudaError_t launch_tc_impl(const ProjLaunch& L) {
  if (L.small) return launch_tcs<C>(L);
  if (L.wtma) {
    return L.swiglu ? launch_tc_glu<C, true>(L) : launch_tc_gemm<C, true>(L);
  }
  // Shapes whose packed rows are not 16-byte multiples: weights are read with
  // plain loads; one tile width suffices for this path.
  if (L.swiglu)
    return L.act ? launch_tc_one<C, true, 128, false, 1, 0>(L) : launch_tc_one<C, true, 128, false, 0, 0>(L);
  switch (L.head_dim) {
    case 64: return launch_tc_one<C, false, 128, false, 0, 64>(L);
    case 128: return launch_tc_one<C, false, 128, false, 0, 128>(L);
    default: return launch_tc_one<C, false, 128, false, 0, 0>(L);
  }
}

}  // namespace m4q
