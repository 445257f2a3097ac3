// misc.cu -- device status word, the fp16 dequantization export, the
// non-finite tripwire and the bounded-wait self-test.
#include <mutex>

#include "codec.cuh"
#include "launch.h"

namespace m4q {

// [0]: bits set by kernels whose bounded waits gave up (or, in the
// bounds-checked build, whose bounds check failed); [1]: non-finite flag;
// [2]: site of the first failed bounds check (0: none); [3]: unused.
__device__ uint32_t g_status_words[4];

uint32_t* status_words() {
  static std::mutex mu;
  static uint32_t* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_words) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint32_t*>(p);
  }
  return addr[dev];
}

// ---------------------------------------------------------------- dequant

// One thread per (row n, 64-weight sub-step s): decode and write 64 (or, at
// an odd block count, 32) fp16 values.
template <int C>
__global__ void __launch_bounds__(256)
    dequant_kernel(const uint8_t* __restrict__ W, int N, int K, long long row_bytes,
                   __half* __restrict__ out) {
  using S = Stage<C>;
  const int nsub = (K + 63) / 64;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)N * nsub) return;
  const int n = (int)(idx / nsub), s = (int)(idx % nsub);
  const uint8_t* row = W + (long long)n * row_bytes;

  // Bytes of the blocks this sub-step needs, starting at word 0.
  constexpr int kBytes = (C == kQ2_0) ? S::BB : 2 * S::BB;
  const long long first = (C == kQ2_0) ? (long long)(s / 2) * S::BB : (long long)(2 * s) * S::BB;
  uint32_t w[(kBytes + 3) / 4 + 1];
#pragma unroll
  for (int i = 0; i < (kBytes + 3) / 4 + 1; ++i) {
    uint32_t lo = 0, hi = 0;
    const long long o = first + 4 * i;
    if (4 * i < kBytes && o < row_bytes) lo = __ldg(reinterpret_cast<const unsigned short*>(row + o));
    if (4 * i + 2 < kBytes && o + 2 < row_bytes)
      hi = __ldg(reinterpret_cast<const unsigned short*>(row + o + 2));
    w[i] = lo | (hi << 16);
  }
  uint32_t v[32];
  const DecK dk = make_deck();
  if (C == kQ2_0 && (s & 1)) decode_sub<C>(w, 1, v, dk);
  else decode_sub<C>(w, 0, v, dk);

  const int valid = (K - 64 * s) >= 64 ? 64 : (K - 64 * s);
  uint4* dst = reinterpret_cast<uint4*>(out + (long long)n * K + 64 * s);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (8 * i < valid) dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

cudaError_t launch_dequant(int codec, const void* w, int N, int K, long long row_bytes, void* out,
                           cudaStream_t s) {
  const long long threads = (long long)N * ((K + 63) / 64);
  if (threads == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  const auto* W = static_cast<const uint8_t*>(w);
  auto* O = static_cast<__half*>(out);
  switch (codec) {
    case kQ4_0: dequant_kernel<kQ4_0><<<blocks, 256, 0, s>>>(W, N, K, row_bytes, O); break;
    case kQ8_0: dequant_kernel<kQ8_0><<<blocks, 256, 0, s>>>(W, N, K, row_bytes, O); break;
    case kMLX4: dequant_kernel<kMLX4><<<blocks, 256, 0, s>>>(W, N, K, row_bytes, O); break;
    default: dequant_kernel<kQ2_0><<<blocks, 256, 0, s>>>(W, N, K, row_bytes, O); break;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- MLX4 pack

// MLX's planar arrays -> 20-byte MLX4 blocks.  In MLX's word order (code k of
// a row at bits 4 (k % 8) of word k / 8, little-endian) the 16 code bytes of a
// 32-weight group are exactly the 4 words of that group, so a block is the
// group's scale and bias followed by those words, copied unchanged.  One
// thread per block, grid-stride.
__global__ void __launch_bounds__(256)
    mlx4_pack_kernel(const uint4* __restrict__ words, const unsigned short* __restrict__ scales,
                     const unsigned short* __restrict__ biases, long long blocks,
                     uint32_t* __restrict__ out) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < blocks;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 q = __ldg(words + i);  // a row of K/8 words is K/32 groups of 4
    uint32_t* dst = out + 5 * i;       // 20-byte blocks, rows back to back
    dst[0] = (uint32_t)__ldg(scales + i) | ((uint32_t)__ldg(biases + i) << 16);
    dst[1] = q.x;
    dst[2] = q.y;
    dst[3] = q.z;
    dst[4] = q.w;
  }
}

// Grid of a grid-stride layout kernel: one thread per block, at most 16 CTAs
// of 256 threads per multiprocessor (a full SM's worth of resident threads
// is 8 such CTAs; twice that hides the tail).
long long layout_grid(long long blocks, int sms) {
  const long long grid = (blocks + 255) / 256;
  const long long cap = 16ll * (sms > 0 ? sms : 1);
  return grid < cap ? grid : cap;
}

cudaError_t launch_mlx4_pack(const void* words, const void* scales, const void* biases, int N, int K,
                             void* w, int sms, cudaStream_t s) {
  const long long blocks = (long long)N * (K / 32);
  const long long grid = layout_grid(blocks, sms);
  mlx4_pack_kernel<<<(unsigned)grid, 256, 0, s>>>(
      static_cast<const uint4*>(words), static_cast<const unsigned short*>(scales),
      static_cast<const unsigned short*>(biases), blocks, static_cast<uint32_t*>(w));
  return cudaGetLastError();
}

// ---------------------------------------------------------------- repack

// Blocks -> planes: the code bytes of every block in row-major block order,
// then the fp16 scales, then (MLX4) the fp16 biases.  One thread per block,
// grid-stride.  A block starts on an even byte, so it is read as 16-bit
// words; its CB code bytes (16 or 32) start on a 16-byte boundary of the
// codes plane and are written as 16-byte stores.
template <int C>
__global__ void __launch_bounds__(256)
    repack_kernel(const unsigned short* __restrict__ W, long long blocks, uint4* __restrict__ codes,
                  unsigned short* __restrict__ scales, unsigned short* __restrict__ biases) {
  constexpr int BB = CodecTraits<C>::BB;       // bytes per block (even)
  constexpr int HEAD = (C == kMLX4) ? 4 : 2;   // scale (and bias) bytes
  constexpr int CB = BB - HEAD;                // code bytes per block
  static_assert(BB % 2 == 0 && CB % 16 == 0, "block layout");
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < blocks;
       i += (long long)gridDim.x * blockDim.x) {
    const unsigned short* blk = W + i * (BB / 2);
    scales[i] = __ldg(blk);
    if (C == kMLX4) biases[i] = __ldg(blk + 1);
    uint32_t w[CB / 4];
#pragma unroll
    for (int j = 0; j < CB / 4; ++j)
      w[j] = (uint32_t)__ldg(blk + HEAD / 2 + 2 * j) | ((uint32_t)__ldg(blk + HEAD / 2 + 2 * j + 1) << 16);
    uint4* dst = codes + i * (CB / 16);
#pragma unroll
    for (int j = 0; j < CB / 16; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

template <int C>
cudaError_t launch_repack_c(const void* w, long long blocks, void* out, int sms, cudaStream_t s) {
  constexpr int CB = CodecTraits<C>::BB - ((C == kMLX4) ? 4 : 2);
  auto* base = static_cast<uint8_t*>(out);
  auto* scales = reinterpret_cast<unsigned short*>(base + blocks * CB);
  auto* biases = scales + blocks;  // written for MLX4 only
  const long long grid = layout_grid(blocks, sms);
  repack_kernel<C><<<(unsigned)grid, 256, 0, s>>>(static_cast<const unsigned short*>(w), blocks,
                                                    reinterpret_cast<uint4*>(base), scales, biases);
  return cudaGetLastError();
}

cudaError_t launch_repack(int codec, const void* w, long long blocks, void* out, int sms, cudaStream_t s) {
  if (blocks == 0) return cudaSuccess;
  switch (codec) {
    case kQ4_0: return launch_repack_c<kQ4_0>(w, blocks, out, sms, s);
    case kQ8_0: return launch_repack_c<kQ8_0>(w, blocks, out, sms, s);
    case kQ2_0: return launch_repack_c<kQ2_0>(w, blocks, out, sms, s);
    default: return launch_repack_c<kMLX4>(w, blocks, out, sms, s);
  }
}

// ---------------------------------------------------------------- finite check

__global__ void __launch_bounds__(256)
    finite_kernel(const unsigned short* __restrict__ x, long long n, uint32_t* flag) {
  bool bad = false;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    bad |= (x[i] & 0x7C00u) == 0x7C00u;  // exponent all ones: Inf or NaN
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(flag, 1u);
}

cudaError_t launch_finite_check(const void* x, long long n, uint32_t* flag, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  finite_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const unsigned short*>(x), n, flag);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- self-test

// One thread waits on a barrier that nothing completes; the bounded wait
// gives up after limit_ns, records the timeout and the kernel returns.
__global__ void wait_selftest_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl ctl{&abort_flag, status, limit_ns};
    (void)mbar_wait(&bar, 0, ctl);
  }
}

cudaError_t launch_wait_selftest(uint32_t* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace m4q
