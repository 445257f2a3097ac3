// gemv.cuh -- weight-streaming kernel for decode-sized M (1 <= M <= 16):
// Y = X W^T and Y = SiLU(X Wg^T) x (X Wu^T).
//
// Pages: "Releases" v0.3.0 (M4QuantizedLinear sends M = 1 to a GEMV) and
// "v0.1 vs v0.2 comparison" 2.3 (register-level reductions).  At this M the
// packed weights are the whole memory traffic, so the kernel reads every
// weight byte once, in long contiguous row segments, and keeps all
// arithmetic on chip.
//
// Work unit: one 16-row weight tile over the whole of K -- 16 weight rows of
// a GEMM (16 outputs), or 8 gate rows over 8 up rows of SwiGLU (8 outputs, so
// that G and U of one output end up in the same thread).  Units are dealt
// round robin to one persistent CTA per SM.
//
// CTA roles (576 threads):
//   warp 0      producer.  A unit arrives as stages of 16 rows x SB bytes
//               (SB up to about 2.3 KB of whole blocks: one stage holds a
//               whole row when K <= 4096), one bulk copy per row segment,
//               issued by 16 lanes at once, into a ring of shared-memory
//               stages.  Copies of 2 KB and more stream at close to the HBM
//               rate; much shorter ones are limited by the copy issue rate.
//               Rows sit at a pitch of SB + 16 bytes so the 16 rows of a stage
//               fall into different shared-memory banks.
//   warps 2..17 consumers.  Warp c takes blocks c, c + 16, ... of each stage
//               (fully unrolled, alternating between two accumulator sets so
//               that the MMA chains overlap; when a row fits in one stage
//               each warp sees the same k range in every unit, so its X
//               fragments are loaded once), decodes them exactly
//               (codec.cuh) and multiplies them with
//               mma.sync m16n8k16: the weight tile is A (16 rows x 16 k), X^T
//               is B (16 k x 8 activation rows, two n8 tiles when M > 8),
//               fp32 accumulation.  Inside a block the k order of the MMA
//               slots is permuted identically for W and X so that each thread
//               reads contiguous code bytes and contiguous X values.
//   warp 1      reducer.  Adds the 16 consumers' partial tiles of a unit in a
//               fixed order and writes Y (SwiGLU: SiLU(G) x U in registers).
// Every wait is bounded in time; on expiry the CTA records the failure in the
// status word, lets its copies in flight land and returns.
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
  int sb;              // stage bytes per row: whole packed stages, <= kSBMax
  int nst;             // stages per unit (ceil(row_bytes / sb))
  int units;           // 16-row weight tiles
  uint32_t* status;
  unsigned long long limit_ns;
};

template <int C>
struct GemvCfg {
  using S = Stage<C>;
  static constexpr int kConsumers = 16;
  static constexpr int kThreads = 32 * (kConsumers + 2);
  static constexpr int kSBMax = (2400 / S::KPB) * S::KPB;   // 2304 (Q4_0) or 2176 B
  static constexpr int kBlocks = kSBMax / S::BB;             // blocks per full stage
  static constexpr int kBPW = kBlocks / kConsumers;          // blocks per consumer warp
  static constexpr int kPitch = kSBMax + 16;                 // row pitch in a stage
  static constexpr int kStage = 16 * kPitch;
  static constexpr int kRing = 5;
  static constexpr int kRedFloats = 2 * kConsumers * 32 * 8; // [buf][warp][lane][8]
  static constexpr int kBars = 2 * kRing + 4;
  static constexpr int kSmemBytes = kRing * kStage + kRedFloats * 4 + kBars * 8 + 16 + 128;
  static_assert(kPitch % 16 == 0 && kStage % 128 == 0, "bulk-copy alignment");
  static_assert(kBPW * kConsumers == kBlocks, "blocks split evenly over the consumers");
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

// Contiguous global -> shared copy of `bytes` (a multiple of 16, both
// addresses 16-byte aligned), completing on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
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

// X fragments of one block for activation rows g and g + 8 (zero past M).
template <int C>
struct XFrag {
  static constexpr int kRegs = C == kQ4_0 ? 4 : C == kQ8_0 ? 4 : 16;
};

template <int C, int MT>
__device__ __forceinline__ void load_xfrag(const GemvParams& p, int g, int t, int kb,
                                           uint32_t (&xf)[MT][XFrag<C>::kRegs]) {
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
}

// Accumulate block b of a stage into the 16 x 8*MT tile.  `st` is the stage
// ([16 rows][kPitch] bytes); g = lane / 4, t = lane % 4; xf holds the X
// fragments of the block.
template <int C, int MT>
__device__ __forceinline__ void gemv_block(const uint8_t* st, int b, int g, int t,
                                           const uint32_t (&xf)[MT][XFrag<C>::kRegs],
                                           float (&acc)[MT][4]) {
  using S = Stage<C>;
  constexpr int BB = S::BB;
  constexpr int PITCH = GemvCfg<C>::kPitch;

  const uint8_t* r0 = st + g * PITCH + b * BB;  // tile row g
  const uint8_t* r1 = r0 + 8 * PITCH;           // tile row g + 8
  const uint32_t d0 = dup_scale(lds_u16(r0)), d1 = dup_scale(lds_u16(r1));

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
      mma_16816(acc[mt], lo00, lo10, lo01, lo11, xf[mt][0], xf[mt][1]);
      mma_16816(acc[mt], hi00, hi10, hi01, hi11, xf[mt][2], xf[mt][3]);
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
      mma_16816(acc[mt], w[0][0], w[1][0], w[0][1], w[1][1], xf[mt][0], xf[mt][1]);
      mma_16816(acc[mt], w[0][2], w[1][2], w[0][3], w[1][3], xf[mt][2], xf[mt][3]);
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
      for (int mt = 0; mt < MT; ++mt) mma_16816(acc[mt], a0, a1, a2, a3, xf[mt][2 * c], xf[mt][2 * c + 1]);
    }
  }
}

template <int C, bool SWIGLU, int MT, bool WTMA, bool XH>
__global__ void __launch_bounds__(32 * (GemvCfg<C>::kConsumers + 2), 1) gemv_kernel(const GemvParams p) {
  using Cfg = GemvCfg<C>;
  using S = Stage<C>;
  constexpr int R = Cfg::kRing;
  constexpr int NC = Cfg::kConsumers;
  constexpr int OU = SWIGLU ? 8 : 16;  // outputs per unit

  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  float* red = reinterpret_cast<float*>(ring + R * Cfg::kStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + Cfg::kRedFloats);
  uint64_t* empty = full + R;
  uint64_t* red_full = empty + R;
  uint64_t* red_empty = red_full + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&full[i], WTMA ? 1 : 32);
      mbar_init(&empty[i], NC);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&red_full[i], NC);
      mbar_init(&red_empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if constexpr (WTMA) {
      // Lane r < 16 copies tile row r (SwiGLU: rows 8..15 are the up rows).
      int q = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const int n0 = u * OU;
        const int rows = min(OU, p.N - n0);  // weight rows of each matrix inside N
        const int r = lane & 7;
        const bool mine = SWIGLU ? (lane < 16 && r < rows) : (lane < rows);
        const uint8_t* src = (SWIGLU && lane >= 8) ? p.w1 : p.w0;
        src += (long long)(n0 + (SWIGLU ? r : lane)) * p.row_bytes;
        for (int s = 0; s < p.nst; ++s, ++q) {
          const int slot = q % R;
          if (q >= R) {
            ok = __all_sync(0xffffffffu, mbar_wait_idle(&empty[slot], ((q / R) - 1) & 1, ctl));
            if (!ok) break;
          }
          const long long off = (long long)s * p.sb;
          const long long left = p.row_bytes - off;
          const uint32_t bytes = (uint32_t)(left < p.sb ? left : p.sb);
          if (lane == 0) mbar_arrive_expect_tx(&full[slot], bytes * (SWIGLU ? 2 * rows : rows));
          __syncwarp();
          if (mine) bulk_load(ring + slot * Cfg::kStage + lane * Cfg::kPitch, src + off, bytes, &full[slot]);
        }
      }
      if (!ok && lane == 0) {
        // Let the copies still in flight land before the CTA exits.
        for (int i = (q > R ? q - R : 0); i < q; ++i)
          mbar_wait_drain(&full[i % R], (i / R) & 1, 100000000ull);
      }
    } else {
      // Rows that are not 16-byte multiples: the warp copies each stage with
      // 2-byte loads (rows past N and bytes past the row end read as zero).
      int q = 0;
      bool ok = true;
      const int half_sb = p.sb / 2;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        for (int s = 0; s < p.nst; ++s, ++q) {
          const int slot = q % R;
          if (q >= R) {
            ok = __all_sync(0xffffffffu, mbar_wait_idle(&empty[slot], ((q / R) - 1) & 1, ctl));
            if (!ok) break;
          }
          uint8_t* dst = ring + slot * Cfg::kStage;
          const long long off = (long long)s * p.sb;
          for (int e = lane; e < 16 * half_sb; e += 32) {
            const int r = e / half_sb;
            const int c2 = e - r * half_sb;
            const int n = SWIGLU ? u * OU + (r & 7) : u * OU + r;
            const uint8_t* base = (SWIGLU && r >= 8) ? p.w1 : p.w0;
            const long long o = off + 2 * c2;
            unsigned short v = 0;
            if (n < p.N && o < p.row_bytes)
              v = __ldg(reinterpret_cast<const unsigned short*>(base + (long long)n * p.row_bytes + o));
            *reinterpret_cast<unsigned short*>(dst + r * Cfg::kPitch + 2 * c2) = v;
          }
          mbar_arrive(&full[slot]);
        }
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 2;
    const int g = lane >> 2, t = lane & 3;
    const int blocks_per_stage = p.sb / S::BB;
    constexpr int XR = XFrag<C>::kRegs;
    // XH: one stage per unit, so block b of every unit has the same k range.
    uint32_t xh[XH ? Cfg::kBPW : 1][MT][XR];
    if constexpr (XH) {
#pragma unroll
      for (int j = 0; j < Cfg::kBPW; ++j) load_xfrag<C, MT>(p, g, t, (cw + NC * j) * S::B, xh[j]);
    }
    int q = 0, i = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
      float acc[MT][4], acc1[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[mt][c] = acc1[mt][c] = 0.f;
      bool ok = true;
      for (int s = 0; s < p.nst; ++s, ++q) {
        const int slot = q % R;
        ok = __all_sync(0xffffffffu, mbar_wait_idle(&full[slot], (q / R) & 1, ctl, 64));
        if (!ok) break;
        const uint8_t* st = ring + slot * Cfg::kStage;
        const int kb0 = s * blocks_per_stage * S::B;
        const int left = (p.K - kb0) / S::B;
        const int nb = left < blocks_per_stage ? left : blocks_per_stage;
        if (nb == Cfg::kBlocks) {
          // Full stage: every block of this warp is inside K.
#pragma unroll
          for (int j = 0; j < Cfg::kBPW; ++j) {
            const int b = cw + NC * j;
            uint32_t xf[MT][XR];
            if constexpr (XH) {
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < XR; ++r) xf[mt][r] = xh[j][mt][r];
            } else {
              load_xfrag<C, MT>(p, g, t, kb0 + b * S::B, xf);
            }
            if (j & 1) gemv_block<C, MT>(st, b, g, t, xf, acc1);
            else gemv_block<C, MT>(st, b, g, t, xf, acc);
          }
        } else {
          for (int b = cw; b < nb; b += NC) {
            uint32_t xf[MT][XR];
            load_xfrag<C, MT>(p, g, t, kb0 + b * S::B, xf);
            gemv_block<C, MT>(st, b, g, t, xf, acc);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      if (!ok) break;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[mt][c] += acc1[mt][c];
      const int rb = i & 1;
      if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait_idle(&red_empty[rb], ((i >> 1) - 1) & 1, ctl))) break;
      float4* dst = reinterpret_cast<float4*>(red + ((rb * NC + cw) * 32 + lane) * 8);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) dst[mt] = make_float4(acc[mt][0], acc[mt][1], acc[mt][2], acc[mt][3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[rb]);
    }
  } else {
    // ------------------------------------------------------------ reducer
    const int g = lane >> 2, t = lane & 3;
    int i = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
      const int rb = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_idle(&red_full[rb], (i >> 1) & 1, ctl))) break;
      float v[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) v[mt][c] = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float4* src = reinterpret_cast<const float4*>(red + ((rb * NC + w) * 32 + lane) * 8);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const float4 f = src[mt];
          v[mt][0] += f.x; v[mt][1] += f.y; v[mt][2] += f.z; v[mt][3] += f.w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[rb]);
      // v[mt][0..1]: tile row g, activation rows 8mt + 2t + {0,1}; v[mt][2..3]: row g + 8.
      const int n0 = u * OU;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int m = 8 * mt + 2 * t + c;
          if (m >= p.M) continue;
          if (SWIGLU) {
            const int n = n0 + g;
            const float gv = v[mt][c], uv = v[mt][c + 2];
            if (n < p.N) p.y[(size_t)m * p.N + n] = __float2half_rn((gv / (1.0f + __expf(-gv))) * uv);
          } else {
            const int n = n0 + g;
            if (n < p.N) p.y[(size_t)m * p.N + n] = __float2half_rn(v[mt][c]);
            if (n + 8 < p.N) p.y[(size_t)m * p.N + n + 8] = __float2half_rn(v[mt][c + 2]);
          }
        }
    }
  }
}

}  // namespace m4q
