// gemv.cuh -- weight-streaming kernel for decode-sized M (1 <= M <= 16):
// Y = X W^T and Y = SiLU(X Wg^T) x (X Wu^T).
//
// Pages: "Releases" v0.3.0 (M4QuantizedLinear dispatches M = 1 to a GEMV) and
// "v0.1 vs v0.2 comparison" 2.3 (register-level reductions).  At this M the
// packed weights are the whole memory traffic, so the kernel streams every
// weight byte exactly once with TMA and keeps all arithmetic in registers.
//
// Layout of the work: a CTA has 8 warps; warp w handles a 16-row weight tile
// (row tile w / KW of the CTA) over a contiguous range of packed stages
// (part w % KW of K).  Each warp owns a 2-deep shared-memory ring filled by
// TMA (one box = 16 rows x 8 blocks, per matrix).  The partial sums of the KW
// warps of a row tile are added in a fixed order through shared memory.
//
// Arithmetic: tensor-core mma.sync m16n8k16 with the weight tile as the A
// operand (16 rows x 16 k) and X^T as B (16 k x 8 activation rows; two n8
// tiles when M > 8), fp32 accumulation.  Weights are decoded exactly as on
// the tcgen05 path (codec.cuh): each is RNE((q - z) * d) in fp16.
//
// Inside a block the assignment of k positions to MMA slots is permuted
// (identically for W and X) so that every thread reads contiguous code
// bytes and contiguous X values; the sum over a block is unchanged.
#pragma once

#include "codec.cuh"

namespace m4q {

struct GemvParams {
  const __half* x;     // [M, K]
  const uint8_t* w0;   // [N, row_bytes] (gate for SwiGLU)
  const uint8_t* w1;   // up weights for SwiGLU
  __half* y;           // [M, N]
  int M, N, K;
  long long row_bytes;
  int kw;              // warps per row tile: 1, 2, 4 or 8
  int nstages;         // packed stages per row
  uint32_t* status;
  unsigned long long limit_ns;
};

template <int C, bool SWIGLU>
struct GemvCfg {
  using S = Stage<C>;
  static constexpr int kThreads = 256;
  static constexpr int kMats = SWIGLU ? 2 : 1;
  static constexpr int kRing = 2;
  static constexpr int kStageBytes = kMats * 16 * S::KPB;
  static constexpr int kRedFloats = 8 * 32 * 2 * 2 * 4;   // warps x lanes x mats x MT x 4
  static constexpr int kSmemBytes =
      8 * kRing * kStageBytes + kRedFloats * 4 + 8 * kRing * 8 + 256;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds_u16(const uint8_t* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}

__device__ __forceinline__ uint32_t spread16(uint32_t v) { return __byte_perm(v, 0u, 0x4140u); }

// X fragment loads for activation row m (zero when m >= M).
template <int BYTES>
__device__ __forceinline__ void ldx(uint32_t* dst, const __half* xrow, bool ok) {
  if constexpr (BYTES == 8) {
    uint2 v = ok ? __ldg(reinterpret_cast<const uint2*>(xrow)) : make_uint2(0, 0);
    dst[0] = v.x; dst[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < BYTES / 16; ++i) {
      uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(xrow) + i) : make_uint4(0, 0, 0, 0);
      dst[4 * i] = v.x; dst[4 * i + 1] = v.y; dst[4 * i + 2] = v.z; dst[4 * i + 3] = v.w;
    }
  }
}

// Accumulate block b of a stage.  `st` points at the stage in shared memory
// ([mat][16 rows][KPB]); g = lane / 4, t = lane % 4; kb = k of the block's
// first weight.
template <int C, bool SWIGLU, int MT>
__device__ __forceinline__ void gemv_block(const uint8_t* st, int b, int g, int t, int kb,
                                           const GemvParams& p, float (&acc)[2][2][4]) {
  using S = Stage<C>;
  constexpr int NM = SWIGLU ? 2 : 1;
  constexpr int BB = S::BB;

  // X fragments (shared by both matrices).
  uint32_t xf[MT][16];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = g + 8 * mt;
    const bool ok = m < p.M;
    const __half* xr = p.x + (size_t)(ok ? m : 0) * p.K + kb;
    if constexpr (C == kQ4_0) {
      ldx<8>(&xf[mt][0], xr + 4 * t, ok);
      ldx<8>(&xf[mt][2], xr + 16 + 4 * t, ok);
    } else if constexpr (C == kQ8_0) {
      ldx<16>(&xf[mt][0], xr + 8 * t, ok);
    } else {
      ldx<64>(&xf[mt][0], xr + 32 * t, ok);
    }
  }

#pragma unroll
  for (int mat = 0; mat < NM; ++mat) {
    const uint8_t* r0 = st + (mat * 16 + g) * S::KPB + b * BB;  // row g
    const uint8_t* r1 = r0 + 8 * S::KPB;                       // row g + 8
    const uint32_t d0 = dup_scale(lds_u16(r0)), d1 = dup_scale(lds_u16(r1));
    float(&a)[2][4] = acc[mat];

    if constexpr (C == kQ4_0) {
      const uint8_t* c0 = r0 + 2 + 4 * t;
      const uint8_t* c1 = r1 + 2 + 4 * t;
      uint32_t lo00, hi00, lo01, hi01, lo10, hi10, lo11, hi11;
      q4_pair(spread16(lds_u16(c0)), d0, lo00, hi00);
      q4_pair(spread16(lds_u16(c0 + 2)), d0, lo01, hi01);
      q4_pair(spread16(lds_u16(c1)), d1, lo10, hi10);
      q4_pair(spread16(lds_u16(c1 + 2)), d1, lo11, hi11);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mma_16816(a[mt], lo00, lo10, lo01, lo11, xf[mt][0], xf[mt][1]);
        mma_16816(a[mt], hi00, hi10, hi01, hi11, xf[mt][2], xf[mt][3]);
      }
    } else if constexpr (C == kQ8_0) {
      const uint8_t* c0 = r0 + 2 + 8 * t;
      const uint8_t* c1 = r1 + 2 + 8 * t;
      uint32_t w[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[0][i] = q8_pair(spread16(lds_u16(c0 + 2 * i)), d0);
        w[1][i] = q8_pair(spread16(lds_u16(c1 + 2 * i)), d1);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        mma_16816(a[mt], w[0][0], w[1][0], w[0][1], w[1][1], xf[mt][0], xf[mt][1]);
        mma_16816(a[mt], w[0][2], w[1][2], w[0][3], w[1][3], xf[mt][2], xf[mt][3]);
      }
    } else {
      const uint8_t* c0 = r0 + 2 + 8 * t;
      const uint8_t* c1 = r1 + 2 + 8 * t;
      uint32_t v0[4], v1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { v0[i] = lds_u16(c0 + 2 * i); v1[i] = lds_u16(c1 + 2 * i); }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t sel = (c & 1) ? 0x4141u : 0x4040u;  // byte c of the pair, replicated
        uint32_t a0, a1, a2, a3;
        q2_byte(__byte_perm(v0[c >> 1], 0u, sel), d0, a0, a2);
        q2_byte(__byte_perm(v1[c >> 1], 0u, sel), d1, a1, a3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          mma_16816(a[mt], a0, a1, a2, a3, xf[mt][2 * c], xf[mt][2 * c + 1]);
      }
    }
  }
}

template <int C, bool SWIGLU, int MT, bool WTMA>
__global__ void __launch_bounds__(256)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                const GemvParams p) {
  using Cfg = GemvCfg<C, SWIGLU>;
  using S = Stage<C>;
  constexpr int R = Cfg::kRing;
  constexpr int NM = Cfg::kMats;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * R * Cfg::kStageBytes;
  float* red = reinterpret_cast<float*>(smem + 8 * R * Cfg::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + Cfg::kRedFloats) + warp * R;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(
      reinterpret_cast<uint64_t*>(red + Cfg::kRedFloats) + 8 * R);

  const int kw = p.kw;
  const int rt = warp / kw, part = warp % kw;
  const int n_base = (blockIdx.x * (8 / kw) + rt) * 16;
  const int s_begin = (int)((long long)p.nstages * part / kw);
  const int s_end = (int)((long long)p.nstages * (part + 1) / kw);
  const int cnt = (n_base < p.N) ? s_end - s_begin : 0;  // tiles past N do nothing
  const int g = lane >> 2, t = lane & 3;

  if (threadIdx.x == 0) *abort_flag = 0;
  if (WTMA && lane == 0) {
    for (int i = 0; i < R; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};

  auto issue = [&](int i) {  // lane 0: load stage s_begin + i into slot i % R
    uint8_t* dst = ring + (i % R) * Cfg::kStageBytes;
    const int xc = (s_begin + i) * (S::KPB / 2);
    mbar_arrive_expect_tx(&full[i % R], Cfg::kStageBytes);
    tma_load_2d(dst, &tm_w0, &full[i % R], xc, n_base);
    if (SWIGLU) tma_load_2d(dst + 16 * S::KPB, &tm_w1, &full[i % R], xc, n_base);
  };

  float acc[2][2][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;

  int issued = 0;
  if constexpr (WTMA) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_w0);
      for (; issued < R && issued < cnt; ++issued) issue(issued);
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);
  }

  bool ok = true;
  int done = 0;  // stages consumed
  for (int i = 0; i < cnt; ++i, done = i) {
    uint8_t* st = ring + (i % R) * Cfg::kStageBytes;
    const int s = s_begin + i;
    int nb = 8;  // blocks of this stage inside K
    if constexpr (WTMA) {
      ok = __all_sync(0xffffffffu, mbar_wait(&full[i % R], (i / R) & 1, ctl));
      if (!ok) break;
    } else {
      // General shapes: copy the stage with 2-byte loads, zero past the row
      // end or past N.
      for (int e = lane; e < Cfg::kStageBytes / 2; e += 32) {
        const int mat = e / (16 * S::KPB / 2);
        const int rem = e % (16 * S::KPB / 2);
        const int row = rem / (S::KPB / 2);
        const long long off = (long long)s * S::KPB + 2 * (rem % (S::KPB / 2));
        const int n = n_base + row;
        unsigned short v = 0;
        if (n < p.N && off < p.row_bytes) {
          const uint8_t* base = (SWIGLU && mat == 1) ? p.w1 : p.w0;
          v = __ldg(reinterpret_cast<const unsigned short*>(base + (long long)n * p.row_bytes + off));
        }
        reinterpret_cast<unsigned short*>(st)[e] = v;
      }
      __syncwarp();
      const int left = (p.K - s * S::KP) / S::B;
      nb = left < 8 ? left : 8;
    }
#pragma unroll
    for (int b = 0; b < 8; ++b)
      if (b < nb) gemv_block<C, SWIGLU, MT>(st, b, g, t, s * S::KP + b * S::B, p, acc);
    __syncwarp();
    if constexpr (WTMA) {
      if (lane == 0 && issued < cnt) {
        fence_proxy_async_smem();
        issue(issued);
      }
      ++issued;
      if (issued > cnt) issued = cnt;
      issued = __shfl_sync(0xffffffffu, issued, 0);
    }
  }
  if constexpr (WTMA) {
    if (!ok && lane == 0) {
      // Let the copies still outstanding land before the CTA exits.
      for (int i = done; i < issued; ++i) mbar_wait_drain(&full[i % R], (i / R) & 1, 100000000ull);
    }
  }

  // Cross-warp reduction of the KW partial sums of each row tile.
  float* mine = red + warp * (32 * 2 * 2 * 4) + lane * 16;
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) mine[a * 8 + b * 4 + c] = acc[a][b][c];
  __syncthreads();
  if (part == 0 && !*abort_flag) {
    float sum[2][2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) sum[a][b][c] = 0.f;
    for (int wpart = 0; wpart < kw; ++wpart) {
      const float* src = red + (rt * kw + wpart) * (32 * 2 * 2 * 4) + lane * 16;
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int c = 0; c < 4; ++c) sum[a][b][c] += src[a * 8 + b * 4 + c];
    }
    // c0,c1: row g, columns 2t, 2t+1 of the n8 tile; c2,c3: row g + 8.
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int n = n_base + g + ((c & 2) ? 8 : 0);
        const int m = 8 * mt + 2 * t + (c & 1);
        if (m < p.M && n < p.N) {
          float v = sum[0][mt][c];
          if (SWIGLU) v = (v / (1.0f + __expf(-v))) * sum[1][mt][c];
          p.y[(size_t)m * p.N + n] = __float2half_rn(v);
        }
      }
  }
}

}  // namespace m4q
