// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units.  No kernel code here.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>
#include <utility>

namespace m4q {

// One projection launch, already validated by the ABI layer.
struct ProjLaunch {
  const void* x;          // fp16 [M, K]
  const void* w0;         // packed weights (gate for SwiGLU)
  const void* w1;         // up weights (SwiGLU) or null
  void* y;                // fp16 [M, N]
  int M, N, K;
  long long row_bytes;
  bool swiglu;            // gated projection (gate and up weights)
  int act;                // gate activation: 0 SiLU, 1 GELU
  int head_dim;           // GEMM output: 0 row-major [M, N], else head-major [N / head_dim][M][head_dim]
  bool wtma;              // packed rows are 16-byte multiples: weights move by TMA (a
                          // last stage past the row end is zero-filled)
  uint32_t* status;       // device status word
  unsigned long long limit_ns;
  cudaStream_t stream;
  // tcgen05 path
  int nx;                 // activation rows per tile: 64, 128 or 256
  bool small;             // M <= 128 kernel (activations as the A operand, tc_small.cuh)
  int split;              // CTAs of a cluster splitting K for one tile (1, 2, 4, 8); the launcher
                          // lowers it until all clusters of the grid can be co-resident
  int sms;                // multiprocessors (persistent grid size, both paths)
  CUtensorMap tm_x, tm_w0, tm_w1, tm_y;
  // GEMV path
  int mt;                 // 1 (M <= 8) or 2 (M <= 16)
};

// Per-kernel, per-device "dynamic shared memory attribute set" flags.  An
// anonymous namespace gives them internal linkage, so two copies of the
// library loaded into one process never share them.
namespace {
template <typename Tag>
std::atomic<unsigned long long>& attr_flag() {
  static std::atomic<unsigned long long> f{0};
  return f;
}
}  // namespace

// Programmatic dependent launch of the projection kernels (on unless the
// environment sets M4Q_PDL=0): a kernel may be scheduled while the previous
// kernel of the stream finishes; it waits for that kernel (griddepcontrol)
// before its first global access.
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("M4Q_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

// Launch `kern` with the projection kernels' attributes: programmatic
// dependent launch, and a cluster of `cluster` CTAs along x when > 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_proj(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                        unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

cudaError_t launch_tc_q4_0(const ProjLaunch& L);
cudaError_t launch_tc_q8_0(const ProjLaunch& L);
cudaError_t launch_tc_q2_0(const ProjLaunch& L);
cudaError_t launch_tc_mlx4(const ProjLaunch& L);
cudaError_t launch_gemv(int codec, const ProjLaunch& L);

// attention.cu: attention of fp16 Q [H][M][D] over a KV cache [Hkv][T] of
// rows of D values (fp16, or Q8_0 blocks along D); O fp16 [M][H * D].
struct AttnParams {
  const __half* q;
  const uint8_t* k;
  const uint8_t* v;
  __half* o;
  float* ws_o;            // key splits: unnormalised O [nsplit][Hkv][rtiles * 64][D]
  float2* ws_ml;          // key splits: (max, sum) per row, same order
  int H, Hkv, G, M, T, D;
  long long kv_row_bytes; // bytes of one key row (2 D, or D / 32 * 34)
  int q_offset;           // causal: query i sees keys j <= q_offset + i
  int causal;
  float scale_log2;       // softmax scale * log2(e)
  int rtiles;             // ceil(M * G / 64) row tiles per KV head
  int nsplit, tsplit;     // key splits and keys per split (a multiple of 64)
  bool kv_vec16;          // every K/V tile start and T * kv_row_bytes are 16-byte aligned
  uint32_t* status;       // device status word (bounds-checked build)
  int nsm;                // SMs of the device (persistent grids)
};
cudaError_t launch_attention(const AttnParams& p, bool q8, cudaStream_t s);
// attention_tc.cu: the tcgen05 kernel for prefill-sized calls on an fp16 cache
// (tm_q: 3-D tensor map [H][M][D] of Q, boxes of [1][128 / G queries][64 d];
// tm_k, tm_v: [Hkv][T][D] of the caches, boxes of [1][128 keys][64 d]; all
// with the 128-byte swizzle)
bool attention_tc_shape(const AttnParams& p);                // the kernel takes the shape
bool attention_tc_applies(const AttnParams& p, bool q8);     // and is estimated faster than the split kernel
// Q8_0 caches K and V ([rows][D / 32 blocks]) decoded to fp16 kf, vf
// ([rows][D]), for the tensor-core path
cudaError_t launch_kv_q8_stage(const void* k, const void* v, long long rows, int D, void* kf, void* vf,
                               cudaStream_t s);
cudaError_t launch_attention_tc(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, cudaStream_t s);

// misc.cu
// Status bit of a failed bounds check (the kernels' kErrBounds), and the
// bounds-checked build switch (-DM4Q_BOUNDS=1).
constexpr uint32_t kErrBoundsBit = 4u;
#ifndef M4Q_BOUNDS
#define M4Q_BOUNDS 0
#endif
uint32_t* status_words();  // [0] wait/bounds status, [1] non-finite flag, [2] first bounds site; per current device
cudaError_t launch_dequant(int codec, const void* w, int N, int K, long long row_bytes, void* out,
                           cudaStream_t s);
cudaError_t launch_finite_check(const void* x, long long n, uint32_t* flag, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* status, unsigned long long limit_ns, cudaStream_t s);
cudaError_t launch_mlx4_pack(const void* words, const void* scales, const void* biases, int N, int K,
                             void* w, int sms, cudaStream_t s);
cudaError_t launch_repack(int codec, const void* w, long long blocks, void* out, int sms, cudaStream_t s);

}  // namespace m4q
