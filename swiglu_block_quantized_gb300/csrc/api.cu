// api.cu -- the C ABI declared in include/m4q.h: argument checks, path
// selection (GEMV for M <= 16, tcgen05 otherwise), TMA descriptor encoding
// and kernel launch on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>

#include "../../include/m4q.h"
#include "launch.h"

namespace {

using m4q::ProjLaunch;

constexpr int kCodecs = 4;
constexpr int kBlock[kCodecs] = {32, 32, 128, 32};
constexpr int kBlockBytes[kCodecs] = {18, 34, 34, 20};
constexpr int kStageBytes[kCodecs] = {144, 272, 272, 160};    // bytes per packed stage

// Default limit of one device pipeline wait (ns); M4Q_WAIT_LIMIT_NS overrides.
unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* s = getenv("M4Q_WAIT_LIMIT_NS");
    unsigned long long x = s ? strtoull(s, nullptr, 10) : 0ull;
    return x ? x : 2000000000ull;
  }();
  return v;
}

// ------------------------------------------------------------ device facts

struct DevInfo {
  bool ok = false;
  bool sm103 = false;
  int sms = 0;
};

int current_device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return M4Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  DevInfo& d = cache[dev];
  if (!d.ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return M4Q_ERR_CUDA;
    d.sm103 = (major == 10 && minor == 3);
    d.sms = sms;
    d.ok = true;
  }
  *out = d;
  return M4Q_OK;
}

// ------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Cache of encoded tensor maps.  A map is a pure function of its
// description (element type, rank, base address, extents, pitches, box and
// swizzle), so a map found under an equal description is the one that
// encoding would produce, whatever happened to the memory in between; the
// cache holds no ownership of that memory.  Eager callers repeat the same
// few descriptions call after call (their weights and activation buffers),
// and a lookup costs far less than cuTensorMapEncodeTiled.  Direct-mapped,
// bounded, guarded by one mutex.
struct MapKey {
  uint32_t dt, rank, swz;
  uint64_t base;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  bool operator==(const MapKey& o) const {
    return dt == o.dt && rank == o.rank && swz == o.swz && base == o.base && dims[0] == o.dims[0] &&
           dims[1] == o.dims[1] && dims[2] == o.dims[2] && strides[0] == o.strides[0] &&
           strides[1] == o.strides[1] && box[0] == o.box[0] && box[1] == o.box[1] && box[2] == o.box[2];
  }
  uint64_t hash() const {
    uint64_t h = 0x9E3779B97F4A7C15ull;
    auto mix = [&h](uint64_t v) { h = (h ^ v) * 0xBF58476D1CE4E5B9ull; h ^= h >> 29; };
    mix(dt | ((uint64_t)rank << 8) | ((uint64_t)swz << 16));
    mix(base);
    for (int i = 0; i < 3; ++i) mix(dims[i]);
    for (int i = 0; i < 2; ++i) mix(strides[i]);
    mix(box[0] | ((uint64_t)box[1] << 20) | ((uint64_t)box[2] << 40));
    return h;
  }
};

struct MapSlot {
  bool used = false;
  MapKey key;
  CUtensorMap map;
};

constexpr int kMapSlots = 512;
std::mutex g_map_mu;
MapSlot g_maps[kMapSlots];

bool encode_cached(CUtensorMap* map, const MapKey& k, const cuuint32_t* estr, int rank) {
  const int slot = (int)(k.hash() % kMapSlots);
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_maps[slot].used && g_maps[slot].key == k) {
      *map = g_maps[slot].map;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {k.dims[0], k.dims[1], k.dims[2]};
  const cuuint64_t strides[2] = {k.strides[0], k.strides[1]};
  const cuuint32_t box[3] = {k.box[0], k.box[1], k.box[2]};
  if (fn(map, (CUtensorMapDataType)k.dt, rank, reinterpret_cast<void*>(k.base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, (CUtensorMapSwizzle)k.swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  g_maps[slot].used = true;
  g_maps[slot].key = k;
  g_maps[slot].map = *map;
  return true;
}

// 2-D map: inner extent `inner` elements, `outer` rows, row pitch in bytes.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz) {
  MapKey k{};
  k.dt = (uint32_t)dt;
  k.rank = 2;
  k.swz = (uint32_t)swz;
  k.base = reinterpret_cast<uint64_t>(base);
  k.dims[0] = inner;
  k.dims[1] = outer;
  k.strides[0] = pitch_bytes;
  k.box[0] = box_inner;
  k.box[1] = box_outer;
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_cached(map, k, estr, 2);
}

// Head-major Y [N / hd][M][hd] as a 3-D tensor (d, m, head), boxes of
// [128 / hd heads][32 m][hd] (one staged GEMM chunk of 128 outputs).
bool encode_heads(CUtensorMap* map, const void* base, uint64_t M, uint64_t N, uint32_t hd) {
  MapKey k{};
  k.dt = (uint32_t)CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  k.rank = 3;
  k.swz = (uint32_t)CU_TENSOR_MAP_SWIZZLE_NONE;
  k.base = reinterpret_cast<uint64_t>(base);
  k.dims[0] = hd;
  k.dims[1] = M;
  k.dims[2] = N / hd;
  k.strides[0] = (uint64_t)hd * 2;
  k.strides[1] = (uint64_t)M * hd * 2;
  k.box[0] = hd;
  k.box[1] = 32;
  k.box[2] = 128 / hd;
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_cached(map, k, estr, 3);
}

// ------------------------------------------------------------ validation

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool known_codec(int codec) { return codec >= 0 && codec < kCodecs; }

int check_shape(int codec, int64_t M, int64_t N, int64_t K) {
  if (!known_codec(codec)) return M4Q_ERR_UNSUPPORTED_CODEC;
  if (M < 1 || N < 1 || K < 1) return M4Q_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return M4Q_ERR_INVALID_ARG;
  if (K % kBlock[codec] != 0 || N % 8 != 0) return M4Q_ERR_BAD_SHAPE;
  return M4Q_OK;
}

// ------------------------------------------------------------ host pipeline

// Events of m4q_project_host: per device, recorded and waited in stream
// order, so one pool serves every call; calls enqueue one at a time.
constexpr int kHostChunks = 16;
constexpr int kMaxEventDevices = 64;
struct HostEvents {
  bool ready = false;
  cudaEvent_t e[2 * kHostChunks + 2];
};
HostEvents g_host_events[kMaxEventDevices];
std::mutex g_host_mu[kMaxEventDevices];

// ------------------------------------------------------------ dispatch

int project(const void* X, const void* W0, const void* W1, int codec, int64_t M, int64_t N,
            int64_t K, void* Y, int path, bool swiglu, int act, m4q_stream_t stream,
            int64_t head_dim = 0) {
  if (!X || !W0 || !Y || (swiglu && !W1)) return M4Q_ERR_INVALID_ARG;
  if (act != M4Q_ACT_SILU && act != M4Q_ACT_GELU) return M4Q_ERR_INVALID_ARG;
  if (head_dim != 0 && (swiglu || (head_dim != 64 && head_dim != 128))) return M4Q_ERR_INVALID_ARG;
  if (head_dim != 0 && N % head_dim != 0) return M4Q_ERR_BAD_SHAPE;
  int rc = check_shape(codec, M, N, K);
  if (rc != M4Q_OK) return rc;
  if (path < M4Q_PATH_AUTO || path > M4Q_PATH_TC) return M4Q_ERR_INVALID_ARG;
  if (path == M4Q_PATH_GEMV && M > 16) return M4Q_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W0) || !aligned16(Y) || (swiglu && !aligned16(W1)))
    return M4Q_ERR_MISALIGNED;
  DevInfo dev;
  rc = current_device_info(&dev);
  if (rc != M4Q_OK) return rc;
  if (!dev.sm103) return M4Q_ERR_UNSUPPORTED_DEVICE;

  ProjLaunch L{};
  L.x = X;
  L.w0 = W0;
  L.w1 = swiglu ? W1 : nullptr;
  L.y = Y;
  L.M = (int)M;
  L.N = (int)N;
  L.K = (int)K;
  L.row_bytes = (K / kBlock[codec]) * (long long)kBlockBytes[codec];
  L.swiglu = swiglu;
  L.act = act;
  L.head_dim = (int)head_dim;
  // Rows that are 16-byte multiples move by TMA.  For the 18- and 34-byte
  // blocks that makes K a multiple of the packed stage; for MLX4 (20-byte
  // blocks) a multiple of 128, and the TMA box of the last stage of a row
  // then reads past the row end, which it fills with zeros (zero scale and
  // bias: zero weights, multiplied by zero-filled X columns).
  L.wtma = (L.row_bytes % 16) == 0;
  L.status = m4q::status_words();
  if (!L.status) return M4Q_ERR_CUDA;
  L.limit_ns = wait_limit_ns();
  L.stream = reinterpret_cast<cudaStream_t>(stream);

  const bool gemv = (path == M4Q_PATH_GEMV) || (path == M4Q_PATH_AUTO && M <= 16);
  cudaError_t e;
  if (gemv) {
    L.mt = M <= 8 ? 1 : 2;
    L.sms = dev.sms;
    e = m4q::launch_gemv(codec, L);
  } else {
    // Output tiles along N (64 outputs per tile for the gated projections).
    const int64_t out_rows = swiglu ? 64 : 128;
    const int64_t ntiles = (N + out_rows - 1) / out_rows;
    // M <= 128 with TMA-able rows and row-major output: the small-M kernel
    // (one activation tile of 128 rows as the A operand).
    // (Not for a plain GEMM with 272-byte packed stages above M = 64: its
    // 128-row X stages and 128-output Y tile do not fit shared memory.)
    L.small = L.wtma && head_dim == 0 && M <= 128 && !(kStageBytes[codec] > 160 && !swiglu && M > 64);
    int nx = 64;
    L.split = 1;
    if (L.small) {
      nx = M <= 32 ? 32 : (M <= 64 ? 64 : 128);   // X rows per stage of the small-M kernel
      // Few output tiles leave most SMs idle: split K over a cluster of up
      // to 8 CTAs per tile, each CTA taking a whole number of packed
      // stages, as long as every cluster of the grid can be resident at
      // once (clusters must fit inside one GPC, so fewer clusters of 8 than
      // SMs / 8 fit the GPU).
      const int64_t tiles = (N + out_rows - 1) / out_rows;
      const int64_t npk = (K + 8 * kBlock[codec] - 1) / (8 * kBlock[codec]);   // packed stages
      L.split = 8;
      while (L.split > 1 && (npk % L.split != 0 || tiles * L.split > dev.sms)) L.split /= 2;
    } else if (!L.wtma) {
      nx = 128;
    } else {
      // Tile width and K split with the least estimated time.  The
      // persistent CTAs take ceil(tiles / SMs) tiles each; a tile costs its
      // 64-k sub-steps (divided by the split) times a width factor, since a
      // sub-step costs about the same at every width except 256, about 12%
      // more (measured on the 8B, 1B and Q2_0 shapes); a split adds its
      // cross-CTA reduction, about 2.5 sub-steps.  Ties go to the wider tile
      // (less decode per FLOP).  A split needs every cluster of the grid
      // resident at once: tiles * split <= SMs here, and the launcher halves
      // it further if clusters of that size do not all fit.
      const int64_t nks = (K + 63) / 64;
      const int64_t npk = (K + 8 * kBlock[codec] - 1) / (8 * kBlock[codec]);   // packed stages
      double best = 1e300;
      for (int w = 256; w >= 64; w /= 2) {
        const int64_t t = ((M + w - 1) / w) * ntiles;
        for (int sp = 1; sp <= 8; sp *= 2) {
          if (sp > 1 && (w > 128 || head_dim != 0 || npk % sp != 0 || t * sp > dev.sms)) continue;
          const double waves = (double)((t * sp + dev.sms - 1) / dev.sms);
          const double est = waves * (double)nks / sp * (w == 256 ? 1.12 : 1.0) + (sp > 1 ? 2.5 : 0.0);
          if (est < best - 1e-9) {
            best = est;
            nx = w;
            L.split = sp;
          }
        }
      }
    }
    L.nx = nx;
    L.sms = dev.sms;
    if (!encode_2d(&L.tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, K, M, K * 2, 64, nx,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return M4Q_ERR_CUDA;
    // Y boxes: GEMM stages [32 m][128 n] chunks per warpgroup; SwiGLU stores
    // one [nx/2 m][16 n] slab per epilogue warp.
    if (L.small) {
      // [128 m][64 n] boxes in the 128-byte swizzled layout
      if (!encode_2d(&L.tm_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Y, N, M, N * 2, 64, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return M4Q_ERR_CUDA;
    } else if (head_dim != 0) {
      if (!encode_heads(&L.tm_y, Y, M, N, (uint32_t)head_dim)) return M4Q_ERR_CUDA;
    } else if (!encode_2d(&L.tm_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Y, N, M, N * 2,
                          swiglu ? 16u : (uint32_t)out_rows, swiglu ? (uint32_t)(nx / 2) : 32u,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) {
      return M4Q_ERR_CUDA;
    }
    L.tm_w0 = L.tm_x;
    L.tm_w1 = L.tm_x;
    if (L.wtma) {
      const uint32_t box_rows = swiglu ? 64 : 128;
      if (!encode_2d(&L.tm_w0, CU_TENSOR_MAP_DATA_TYPE_UINT16, W0, L.row_bytes / 2, N,
                     L.row_bytes, kStageBytes[codec] / 2, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return M4Q_ERR_CUDA;
      if (swiglu && !encode_2d(&L.tm_w1, CU_TENSOR_MAP_DATA_TYPE_UINT16, W1, L.row_bytes / 2, N,
                               L.row_bytes, kStageBytes[codec] / 2, box_rows,
                               CU_TENSOR_MAP_SWIZZLE_NONE))
        return M4Q_ERR_CUDA;
    }
    switch (codec) {
      case M4Q_Q4_0: e = m4q::launch_tc_q4_0(L); break;
      case M4Q_Q8_0: e = m4q::launch_tc_q8_0(L); break;
      case M4Q_MLX4: e = m4q::launch_tc_mlx4(L); break;
      default: e = m4q::launch_tc_q2_0(L); break;
    }
  }
  return e == cudaSuccess ? M4Q_OK : M4Q_ERR_CUDA;
}

}  // namespace

extern "C" {

int m4q_gemm_ex(const void* X, const void* W, int codec, int64_t M, int64_t N, int64_t K, void* Y,
                int path, m4q_stream_t stream) {
  return project(X, W, nullptr, codec, M, N, K, Y, path, false, M4Q_ACT_SILU, stream);
}

int m4q_swiglu_ex(const void* X, const void* Wg, const void* Wu, int codec, int64_t M, int64_t N,
                  int64_t K, void* Y, int path, m4q_stream_t stream) {
  return project(X, Wg, Wu, codec, M, N, K, Y, path, true, M4Q_ACT_SILU, stream);
}

int m4q_gemm_heads(const void* X, const void* W, int codec, int64_t M, int64_t N, int64_t K,
                   int64_t head_dim, void* Y, m4q_stream_t stream) {
  if (head_dim == 0) return M4Q_ERR_INVALID_ARG;
  return project(X, W, nullptr, codec, M, N, K, Y, M4Q_PATH_AUTO, false, M4Q_ACT_SILU, stream, head_dim);
}

int m4q_glu_ex(const void* X, const void* Wg, const void* Wu, int codec, int64_t M, int64_t N,
               int64_t K, void* Y, int act, int path, m4q_stream_t stream) {
  return project(X, Wg, Wu, codec, M, N, K, Y, path, true, act, stream);
}

int m4q_geglu(const void* X, const void* Wg, const void* Wu, int codec, int64_t M, int64_t N,
              int64_t K, void* Y, m4q_stream_t stream) {
  return project(X, Wg, Wu, codec, M, N, K, Y, M4Q_PATH_AUTO, true, M4Q_ACT_GELU, stream);
}

int m4q_gemm(const void* X, const void* W, int codec, int64_t M, int64_t N, int64_t K, void* Y,
             m4q_stream_t stream) {
  return project(X, W, nullptr, codec, M, N, K, Y, M4Q_PATH_AUTO, false, M4Q_ACT_SILU, stream);
}

int m4q_swiglu(const void* X, const void* Wg, const void* Wu, int codec, int64_t M, int64_t N,
               int64_t K, void* Y, m4q_stream_t stream) {
  return project(X, Wg, Wu, codec, M, N, K, Y, M4Q_PATH_AUTO, true, M4Q_ACT_SILU, stream);
}

int m4q_mlp(const void* X, const void* Wg, const void* Wu, const void* Wd, int codec_gu,
            int codec_d, int64_t M, int64_t D, int64_t F, void* H, void* Y, int act,
            m4q_stream_t stream) {
  if (!H || !Wd) return M4Q_ERR_INVALID_ARG;
  // Validate both projections before enqueueing either.
  int rc = check_shape(codec_gu, M, F, D);
  if (rc != M4Q_OK) return rc;
  rc = check_shape(codec_d, M, D, F);
  if (rc != M4Q_OK) return rc;
  if (!aligned16(H) || !aligned16(Wd)) return M4Q_ERR_MISALIGNED;
  rc = project(X, Wg, Wu, codec_gu, M, F, D, H, M4Q_PATH_AUTO, true, act, stream);
  if (rc != M4Q_OK) return rc;
  return project(H, Wd, nullptr, codec_d, M, D, F, Y, M4Q_PATH_AUTO, false, M4Q_ACT_SILU, stream);
}

int m4q_project_host(const void* X_host, const void* W0, const void* W1, int codec, int act, int64_t M,
                     int64_t N, int64_t K, void* Y_host, void* X_dev, void* Y_dev, int64_t chunk_rows,
                     m4q_stream_t stream, m4q_stream_t h2d_stream, m4q_stream_t d2h_stream) {
  if (!X_host || !Y_host || !X_dev || !Y_dev || !W0 || chunk_rows < 0) return M4Q_ERR_INVALID_ARG;
  if (act != M4Q_ACT_SILU && act != M4Q_ACT_GELU) return M4Q_ERR_INVALID_ARG;
  int rc = check_shape(codec, M, N, K);
  if (rc != M4Q_OK) return rc;
  if (!aligned16(X_dev) || !aligned16(Y_dev) || !aligned16(W0) || (W1 && !aligned16(W1)))
    return M4Q_ERR_MISALIGNED;
  DevInfo dev;
  rc = current_device_info(&dev);
  if (rc != M4Q_OK) return rc;
  if (!dev.sm103) return M4Q_ERR_UNSUPPORTED_DEVICE;
  int64_t rows = chunk_rows ? chunk_rows : ((M + 3) / 4 + 127) / 128 * 128;
  if (rows > M) rows = M;
  const int64_t chunks = (M + rows - 1) / rows;
  if (chunks > kHostChunks) rows = (M + kHostChunks - 1) / kHostChunks;   // at most kHostChunks chunks
  int dev_id = 0;
  if (cudaGetDevice(&dev_id) != cudaSuccess || dev_id < 0 || dev_id >= kMaxEventDevices) return M4Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_host_mu[dev_id]);
  HostEvents& ev = g_host_events[dev_id];
  if (!ev.ready) {
    for (int i = 0; i < 2 * kHostChunks + 2; ++i)
      if (cudaEventCreateWithFlags(&ev.e[i], cudaEventDisableTiming) != cudaSuccess) {
        (void)cudaGetLastError();
        return M4Q_ERR_CUDA;
      }
    ev.ready = true;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t sin = reinterpret_cast<cudaStream_t>(h2d_stream);
  cudaStream_t sout = reinterpret_cast<cudaStream_t>(d2h_stream);
  auto fail = [] { return M4Q_ERR_CUDA; };
  // Both copy streams start after the work already on `stream`.
  if (cudaEventRecord(ev.e[0], s) != cudaSuccess || cudaStreamWaitEvent(sin, ev.e[0], 0) != cudaSuccess ||
      cudaStreamWaitEvent(sout, ev.e[0], 0) != cudaSuccess)
    return fail();
  const uint8_t* xh = static_cast<const uint8_t*>(X_host);
  uint8_t* yh = static_cast<uint8_t*>(Y_host);
  uint8_t* xd = static_cast<uint8_t*>(X_dev);
  uint8_t* yd = static_cast<uint8_t*>(Y_dev);
  int c = 0;
  for (int64_t r0 = 0; r0 < M; r0 += rows, ++c) {
    const int64_t n = (M - r0) < rows ? (M - r0) : rows;
    const size_t xoff = (size_t)(r0 * K * 2), yoff = (size_t)(r0 * N * 2);
    cudaEvent_t in = ev.e[1 + 2 * c], done = ev.e[2 + 2 * c];
    if (cudaMemcpyAsync(xd + xoff, xh + xoff, (size_t)(n * K * 2), cudaMemcpyHostToDevice, sin) != cudaSuccess ||
        cudaEventRecord(in, sin) != cudaSuccess || cudaStreamWaitEvent(s, in, 0) != cudaSuccess)
      return fail();
    rc = project(xd + xoff, W0, W1, codec, n, N, K, yd + yoff, M4Q_PATH_AUTO, W1 != nullptr, act, stream);
    if (rc != M4Q_OK) return rc;
    if (cudaEventRecord(done, s) != cudaSuccess || cudaStreamWaitEvent(sout, done, 0) != cudaSuccess ||
        cudaMemcpyAsync(yh + yoff, yd + yoff, (size_t)(n * N * 2), cudaMemcpyDeviceToHost, sout) != cudaSuccess)
      return fail();
  }
  cudaEvent_t last = ev.e[2 * kHostChunks + 1];
  if (cudaEventRecord(last, sout) != cudaSuccess || cudaStreamWaitEvent(s, last, 0) != cudaSuccess) return fail();
  return M4Q_OK;
}

size_t m4q_weight_bytes(int codec, int64_t N, int64_t K) {
  if (!known_codec(codec) || N < 0 || K < 0 || K % kBlock[codec] != 0) return 0;
  return (size_t)N * (size_t)(K / kBlock[codec]) * (size_t)kBlockBytes[codec];
}

int m4q_dequant(const void* W, int codec, int64_t N, int64_t K, void* Wf16, m4q_stream_t stream) {
  if (!W || !Wf16) return M4Q_ERR_INVALID_ARG;
  if (!known_codec(codec)) return M4Q_ERR_UNSUPPORTED_CODEC;
  if (N < 1 || K < 1 || N > INT32_MAX || K > INT32_MAX) return M4Q_ERR_INVALID_ARG;
  if (K % kBlock[codec] != 0) return M4Q_ERR_BAD_SHAPE;
  if (!aligned16(W) || !aligned16(Wf16)) return M4Q_ERR_MISALIGNED;
  DevInfo dev;
  int rc = current_device_info(&dev);
  if (rc != M4Q_OK) return rc;
  if (!dev.sm103) return M4Q_ERR_UNSUPPORTED_DEVICE;
  const long long row_bytes = (K / kBlock[codec]) * (long long)kBlockBytes[codec];
  return m4q::launch_dequant(codec, W, (int)N, (int)K, row_bytes, Wf16,
                             reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? M4Q_OK
             : M4Q_ERR_CUDA;
}

int m4q_mlx4_pack(const void* words, const void* scales, const void* biases, int64_t N, int64_t K,
                  void* W, m4q_stream_t stream) {
  if (!words || !scales || !biases || !W) return M4Q_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || N > INT32_MAX || K > INT32_MAX) return M4Q_ERR_INVALID_ARG;
  if (K % 32 != 0) return M4Q_ERR_BAD_SHAPE;
  if (!aligned16(words) || !aligned16(W) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(biases) & 1u))
    return M4Q_ERR_MISALIGNED;
  DevInfo dev;
  int rc = current_device_info(&dev);
  if (rc != M4Q_OK) return rc;
  if (!dev.sm103) return M4Q_ERR_UNSUPPORTED_DEVICE;
  return m4q::launch_mlx4_pack(words, scales, biases, (int)N, (int)K, W, dev.sms,
                               reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? M4Q_OK
             : M4Q_ERR_CUDA;
}

int m4q_repack(const void* W, int codec, int64_t N, int64_t K, void* Wplanar, m4q_stream_t stream) {
  if (!W || !Wplanar) return M4Q_ERR_INVALID_ARG;
  if (!known_codec(codec)) return M4Q_ERR_UNSUPPORTED_CODEC;
  if (N < 1 || K < 1 || N > INT32_MAX || K > INT32_MAX) return M4Q_ERR_INVALID_ARG;
  if (K % kBlock[codec] != 0) return M4Q_ERR_BAD_SHAPE;
  if (!aligned16(W) || !aligned16(Wplanar)) return M4Q_ERR_MISALIGNED;
  DevInfo dev;
  int rc = current_device_info(&dev);
  if (rc != M4Q_OK) return rc;
  if (!dev.sm103) return M4Q_ERR_UNSUPPORTED_DEVICE;
  const long long blocks = N * (K / kBlock[codec]);
  return m4q::launch_repack(codec, W, blocks, Wplanar, dev.sms, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? M4Q_OK
             : M4Q_ERR_CUDA;
}

// ------------------------------------------------------------ attention

}  // extern "C"

namespace {

// Key split of an attention call: CTAs = row tiles x KV heads; when that
// leaves the GPU under `per_sm` CTAs per SM (what the tiled kernel fits:
// two, for its registers or, decoding over an fp16 cache, its three-stage
// tile pipeline; three for the decode kernel over a Q8_0 cache), split the
// keys (tiles of 64) so the grid reaches about that, each split keeping at
// least two tiles.
struct AttnSplit {
  int rtiles, nsplit, tsplit;
  size_t ws_bytes;
};

AttnSplit attn_split(int64_t H, int64_t Hkv, int64_t M, int64_t T, int64_t D, int sms, int per_sm) {
  AttnSplit a;
  const int64_t R = M * (H / Hkv);
  a.rtiles = (int)((R + 63) / 64);
  const int64_t ctas = (int64_t)a.rtiles * Hkv;
  const int64_t ktiles = (T + 63) / 64;
  const int64_t target = (int64_t)per_sm * sms;
  int64_t ns = 1;
  if (ctas < target) {
    ns = (target + ctas - 1) / ctas;
    const int64_t most = ktiles / 2 > 1 ? ktiles / 2 : 1;
    if (ns > most) ns = most;
  }
  const int64_t per = (ktiles + ns - 1) / ns;     // key tiles per split
  a.tsplit = (int)(per * 64);
  a.nsplit = (int)((ktiles + per - 1) / per);
  a.ws_bytes = a.nsplit > 1 ? (size_t)a.nsplit * Hkv * a.rtiles * 64 * (size_t)(D * 4 + 8) : 0;
  return a;
}

// [heads][rows][D] fp16 as a 3-D tensor (d, row, head), boxes of
// [1][box_rows][64 d] with the 128-byte swizzle: the tcgen05 attention's Q,
// K and V tiles (rows past the extent read as zeros).
bool encode_kv(CUtensorMap* map, const void* base, uint64_t Hkv, uint64_t T, uint64_t D, uint32_t box_rows = 128) {
  MapKey k{};
  k.dt = (uint32_t)CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  k.rank = 3;
  k.swz = (uint32_t)CU_TENSOR_MAP_SWIZZLE_128B;
  k.base = reinterpret_cast<uint64_t>(base);
  k.dims[0] = D;
  k.dims[1] = T;
  k.dims[2] = Hkv;
  k.strides[0] = D * 2;
  k.strides[1] = T * D * 2;
  k.box[0] = 64;
  k.box[1] = box_rows;
  k.box[2] = 1;
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_cached(map, k, estr, 3);
}

// A Q8_0 cache can take the tcgen05 path after both caches are decoded to
// fp16 once (each key tile is read by every row tile of its KV head, so one
// decode replaces many): the staging needs 2 Hkv T D fp16 values.  False
// when the shape cannot take that path.
bool q8_staging_bytes(int64_t H, int64_t Hkv, int64_t M, int64_t T, int64_t D, size_t* bytes) {
  if (H < 1 || Hkv < 1 || M < 1 || T < 1 || H % Hkv != 0 || (D != 64 && D != 128)) return false;
  if (Hkv * T > INT32_MAX || M * (H / Hkv) > INT32_MAX) return false;
  m4q::AttnParams p{};
  p.H = (int)H;
  p.Hkv = (int)Hkv;
  p.G = (int)(H / Hkv);
  p.M = (int)M;
  p.D = (int)D;
  p.kv_row_bytes = 2 * D;
  if (!m4q::attention_tc_shape(p)) return false;
  *bytes = (size_t)2 * Hkv * T * D * 2;
  return true;
}

int check_attention(const void* Q, const void* K, const void* V, int kv_codec, int64_t H, int64_t Hkv,
                    int64_t M, int64_t T, int64_t D, int64_t q_offset, float scale, const void* O) {
  if (!Q || !K || !V || !O) return M4Q_ERR_INVALID_ARG;
  if (kv_codec != M4Q_KV_F16 && kv_codec != M4Q_Q8_0) return M4Q_ERR_UNSUPPORTED_CODEC;
  if (H < 1 || Hkv < 1 || M < 1 || T < 1 || q_offset < 0) return M4Q_ERR_INVALID_ARG;
  if (H > 65535 || M > INT32_MAX || T > INT32_MAX || q_offset > INT32_MAX || M * H > INT32_MAX)
    return M4Q_ERR_INVALID_ARG;
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return M4Q_ERR_INVALID_ARG;
  if (H % Hkv != 0 || (D != 64 && D != 128)) return M4Q_ERR_BAD_SHAPE;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return M4Q_ERR_MISALIGNED;
  return M4Q_OK;
}

}  // namespace

extern "C" {

size_t m4q_attention_workspace_bytes(int64_t H, int64_t Hkv, int64_t M, int64_t T, int64_t D) {
  if (H < 1 || Hkv < 1 || M < 1 || T < 1 || H % Hkv != 0 || (D != 64 && D != 128)) return 0;
  DevInfo dev;
  if (current_device_info(&dev) != M4Q_OK) return 0;
  // the larger of the two codecs' splits (a Q8_0 decode splits into more)
  return attn_split(H, Hkv, M, T, D, dev.sms, M * (H / Hkv) <= 16 ? 3 : 2).ws_bytes;
}

size_t m4q_attention_workspace(int kv_codec, int64_t H, int64_t Hkv, int64_t M, int64_t T, int64_t D) {
  // the path is chosen per call (the causal offset enters the estimate), so
  // the size covers both: the key split's results and a Q8_0 staging
  const size_t split = m4q_attention_workspace_bytes(H, Hkv, M, T, D);
  size_t stage = 0;
  if (kv_codec != M4Q_Q8_0 || !q8_staging_bytes(H, Hkv, M, T, D, &stage)) return split;
  return stage > split ? stage : split;
}

int m4q_attention(const void* Q, const void* K, const void* V, int kv_codec, int64_t H, int64_t Hkv,
                  int64_t M, int64_t T, int64_t D, int64_t q_offset, int causal, float scale, void* O,
                  void* workspace, size_t workspace_bytes, m4q_stream_t stream) {
  int rc = check_attention(Q, K, V, kv_codec, H, Hkv, M, T, D, q_offset, scale, O);
  if (rc != M4Q_OK) return rc;
  if (workspace && !aligned16(workspace)) return M4Q_ERR_MISALIGNED;
  DevInfo dev;
  rc = current_device_info(&dev);
  if (rc != M4Q_OK) return rc;
  if (!dev.sm103) return M4Q_ERR_UNSUPPORTED_DEVICE;
  AttnSplit a = attn_split(H, Hkv, M, T, D, dev.sms, (M * (H / Hkv) <= 16 && kv_codec == M4Q_Q8_0) ? 3 : 2);
  if (a.nsplit > 1 && (!workspace || workspace_bytes < a.ws_bytes)) {
    a.nsplit = 1;   // no room for partial results: one CTA walks all keys
    a.tsplit = (int)(((T + 63) / 64) * 64);
  }
  m4q::AttnParams p{};
  p.q = static_cast<const __half*>(Q);
  p.k = static_cast<const uint8_t*>(K);
  p.v = static_cast<const uint8_t*>(V);
  p.o = static_cast<__half*>(O);
  p.H = (int)H;
  p.Hkv = (int)Hkv;
  p.G = (int)(H / Hkv);
  p.M = (int)M;
  p.T = (int)T;
  p.D = (int)D;
  p.kv_row_bytes = kv_codec == M4Q_KV_F16 ? 2 * D : (D / 32) * 34;
  p.kv_vec16 = (T * p.kv_row_bytes) % 16 == 0;   // K and V are 16-byte aligned (checked above)
  p.q_offset = (int)q_offset;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.rtiles = a.rtiles;
  p.nsplit = a.nsplit;
  p.tsplit = a.tsplit;
  p.status = m4q::status_words();
  if (!p.status) return M4Q_ERR_CUDA;
  p.nsm = dev.sms;
  if (a.nsplit > 1) {
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                         (size_t)a.nsplit * Hkv * a.rtiles * 64 * D * 4);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  size_t stage = 0;
  m4q::AttnParams pf = p;   // the same call on an fp16 cache (the staged form)
  pf.kv_row_bytes = 2 * D;
  if (kv_codec == M4Q_Q8_0 && workspace && q8_staging_bytes(H, Hkv, M, T, D, &stage) && workspace_bytes >= stage &&
      m4q::attention_tc_applies(pf, true)) {
    // decode both caches to fp16 in the workspace, then the fp16 path
    __half* kf = static_cast<__half*>(workspace);
    __half* vf = kf + (size_t)Hkv * T * D;
    if (m4q::launch_kv_q8_stage(K, V, (long long)Hkv * T, (int)D, kf, vf, s) != cudaSuccess) return M4Q_ERR_CUDA;
    K = kf;
    V = vf;
    p.k = reinterpret_cast<const uint8_t*>(kf);
    p.v = reinterpret_cast<const uint8_t*>(vf);
    p.kv_row_bytes = 2 * D;
    p.kv_vec16 = true;
    kv_codec = M4Q_KV_F16;
  }
  if (kv_codec == M4Q_KV_F16 && m4q::attention_tc_applies(p, false)) {
    // Q [H][M][D] takes the same form as the caches, in boxes of the
    // 128 / G queries a CTA takes of each head
    CUtensorMap tm_q, tm_k, tm_v;
    if (!encode_kv(&tm_q, Q, H, M, D, (uint32_t)(128 / p.G)) || !encode_kv(&tm_k, K, Hkv, T, D) ||
        !encode_kv(&tm_v, V, Hkv, T, D))
      return M4Q_ERR_CUDA;
    return m4q::launch_attention_tc(p, tm_q, tm_k, tm_v, s) == cudaSuccess ? M4Q_OK : M4Q_ERR_CUDA;
  }
  return m4q::launch_attention(p, kv_codec == M4Q_Q8_0, s) == cudaSuccess ? M4Q_OK : M4Q_ERR_CUDA;
}

int m4q_check_finite(const void* x, int64_t n, m4q_stream_t stream) {
  if (!x || n < 0) return M4Q_ERR_INVALID_ARG;
  if (!aligned16(x)) return M4Q_ERR_MISALIGNED;
  uint32_t* words = m4q::status_words();
  if (!words) return M4Q_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (m4q::launch_finite_check(x, n, words + 1, s) != cudaSuccess) return M4Q_ERR_CUDA;
  uint32_t flag = 0;
  if (cudaMemcpyAsync(&flag, words + 1, sizeof(flag), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return M4Q_ERR_CUDA;
  return flag ? M4Q_ERR_NONFINITE : M4Q_OK;
}

int m4q_check_device_status(m4q_stream_t stream) {
  uint32_t* words = m4q::status_words();
  if (!words) return M4Q_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t st = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpy(&st, words, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return M4Q_ERR_CUDA;
  if (st) {
    if (cudaMemset(words, 0, sizeof(uint32_t)) != cudaSuccess) return M4Q_ERR_CUDA;
    return (st & m4q::kErrBoundsBit) ? M4Q_ERR_BOUNDS : M4Q_ERR_TIMEOUT;
  }
  return M4Q_OK;
}

int m4q_build_flags(void) {
#if M4Q_BOUNDS
  return M4Q_BUILD_BOUNDS;
#else
  return 0;
#endif
}

int m4q_bounds_site(m4q_stream_t stream) {
  uint32_t* words = m4q::status_words();
  if (!words) return M4Q_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t site = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpy(&site, words + 2, sizeof(site), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(words + 2, 0, sizeof(uint32_t)) != cudaSuccess)
    return M4Q_ERR_CUDA;
  return (int)site;
}

int m4q_selftest_wait_timeout(int64_t limit_ns, m4q_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000) return M4Q_ERR_INVALID_ARG;
  uint32_t* words = m4q::status_words();
  if (!words) return M4Q_ERR_CUDA;
  return m4q::launch_wait_selftest(words, (unsigned long long)limit_ns,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? M4Q_OK
             : M4Q_ERR_CUDA;
}

const char* m4q_status_string(int status) {
  switch (status) {
    case M4Q_OK: return "ok";
    case M4Q_ERR_INVALID_ARG: return "invalid argument";
    case M4Q_ERR_UNSUPPORTED_CODEC: return "unsupported codec";
    case M4Q_ERR_BAD_SHAPE: return "bad shape (K must be a multiple of the block, N of 8)";
    case M4Q_ERR_MISALIGNED: return "pointer not aligned (16 bytes; fp16 scale and bias arrays 2 bytes)";
    case M4Q_ERR_CUDA: return "CUDA error";
    case M4Q_ERR_NONFINITE: return "non-finite values found";
    case M4Q_ERR_TIMEOUT: return "a device pipeline wait gave up";
    case M4Q_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103";
    case M4Q_ERR_SCRATCH_LIMIT: return "M * F exceeds the fixed scratch of m4q_mlp_noalloc (1 << 20 fp16)";
    case M4Q_ERR_BOUNDS: return "an access was out of range (bounds-checked build)";
    default: return "unknown status";
  }
}

int m4q_version(void) { return 100; }

}  // extern "C"
