// gemv.cuh -- weight-streaming kernel for decode-sized M (1 <= M <= 16):
// Y = X W^T and Y = SiLU(X Wg^T) x (X Wu^T).
//
// Pages: "Releases" v0.3.0 (M4QuantizedLinear sends M = 1 to a GEMV) and
// "v0.1 vs v0.2 comparison" 2.3 (register-level reductions).  At this M the
// packed weights are the whole memory traffic, so the kernel reads every
// weight byte once, in long contiguous segments, and keeps all arithmetic on
// chip.
//
// Work unit: 16 outputs n0 .. n0+15 over the whole of K.  The MMA tile is 16
// weight rows in which tile row g holds weight row n0 + 2g and tile row g + 8
// holds row n0 + 2g + 1, so each pair of tile rows is one contiguous piece of
// the packed matrix.  SwiGLU runs the gate tile and the up tile of the same
// 16 outputs through the same thread fragments: G and U of an output land in
// the same thread and SiLU(G) x U is formed in registers.
//
// CTA roles (576 threads), one persistent CTA per SM, units dealt round robin:
//   warp 0      producer.  A tile arrives as stages of 8 row pairs, one bulk
//               copy per pair (both rows at once when a row fits one stage:
//               4.6 KB at K = 4096 for Q4_0).  Few, long copies keep the
//               stream at the HBM rate: a bulk copy has a fixed issue cost.
//               Pairs sit 2 SB + 16 bytes apart in shared memory (SB = row
//               bytes per stage), which puts tile rows 0..7 in distinct banks;
//               rows g and g + 8 share banks but are read by different loads.
//   warps 2..17 consumers.  Warp c takes blocks c, c + 16, ... of each stage,
//               decodes them exactly (codec.cuh) and multiplies them with
//               mma.sync m16n8k16 (weight tile = A, X^T = B, two n8 tiles when
//               M > 8, fp32 accumulation, two accumulator sets so that the
//               MMA chains overlap).  When a row is one stage of 16 kXH
//               blocks, each warp keeps the X fragments of its blocks in
//               registers for the whole launch.  Inside a block the k order
//               of the MMA slots is permuted identically for W and X so that
//               each thread reads contiguous code bytes and contiguous X
//               values.
//   warp 1      reducer.  Adds the 16 consumers' partial tiles of a unit in a
//               fixed order and writes Y.
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
  int sb;              // row bytes per stage: row_bytes if a row fits, else kSBMax
  int nst;             // stages per row
  int pp;              // shared-memory pitch of a row pair: 2 sb + 16
  int ring;            // stages in the ring
  int units;           // 16-output units
  int act;             // SwiGLU units: gate activation, 0 SiLU, 1 GELU
  int head_dim;        // GEMM: 0 row-major Y, else head-major Y[N / head_dim][M][head_dim]
  uint32_t* status;
  unsigned long long limit_ns;
};

template <int C, int MT>
struct GemvCfg {
  using S = Stage<C>;
  static constexpr int kConsumers = 16;
  static constexpr int kThreads = 32 * (kConsumers + 2);
  // Largest stage <= 2400 B that splits into 16 equal runs of whole blocks:
  // 2304 (Q4_0), 2176 (Q8_0, Q2_0).  MLX4 takes 2560 B, a whole K = 4096 row,
  // so that rows of that length stay one stage with the X fragments held in
  // registers (11% faster at M = 1 than 2240 + 320 B stages, although the
  // ring then holds only two stages).
  static constexpr int kSBMax = C == kMLX4 ? 2560 : (2400 / (16 * S::BB)) * 16 * S::BB;
  static constexpr int kBlocks = kSBMax / S::BB;             // blocks of a full stage
  static constexpr int kXH = kBlocks / kConsumers;           // blocks per warp of a full stage
  static constexpr int kRingMax = 16;
  static constexpr int kLaneFloats = 2 * MT * 4;                    // [2 mats][MT][4] accumulators
  static constexpr int kRedFloats = 2 * kConsumers * 32 * kLaneFloats;  // [buf][warp][lane][...]
  static constexpr int kBars = 2 * kRingMax + 4;
  // The ring takes all the shared memory the rest leaves: the deeper it is,
  // the more weight bytes are in flight while the consumers work.
  static constexpr int kRingBytes = (227 * 1024 - kRedFloats * 4 - kBars * 8 - 16 - 128) / 128 * 128;
  static constexpr int kSmemBytes = kRingBytes + kRedFloats * 4 + kBars * 8 + 16 + 128;
  static_assert(kXH * kConsumers == kBlocks, "blocks split evenly over the consumers");
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
  static constexpr int kRegs = C == kQ2_0 ? 16 : 4;
};

template <int C, int MT>
__device__ __forceinline__ void load_xfrag(const GemvParams& p, int g, int t, int kb,
                                           uint32_t (&xf)[MT][XFrag<C>::kRegs]) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = g + 8 * mt;
    constexpr int kSpan = C == kQ2_0 ? 128 : 32;   // k values of one block
    const bool ok = m < p.M && in_bounds(kb + kSpan <= p.K, p.status, kSiteGemvX);
    const __half* xr = p.x + (size_t)(ok ? m : 0) * p.K + kb;
    if constexpr (C == kQ4_0) {
      ldx<8>(&xf[mt][0], xr + 4 * t, ok);
      ldx<8>(&xf[mt][2], xr + 16 + 4 * t, ok);
    } else if constexpr (C == kQ8_0 || C == kMLX4) {
      ldx<16>(&xf[mt][0], xr + 8 * t, ok);
    } else {
      ldx<64>(&xf[mt][0], xr + 32 * t, ok);
    }
  }
}

// Accumulate one block into the 16 x 8*MT tile.  r0 points at the block in
// tile row g, r1 at the same block in tile row g + 8; t = lane % 4; xf holds
// the X fragments of the block.
template <int C, int MT>
__device__ __forceinline__ void gemv_block(const uint8_t* r0, const uint8_t* r1, int t,
                                           const uint32_t (&xf)[MT][XFrag<C>::kRegs],
                                           float (&acc)[MT][4], const DecK& K) {
  const uint32_t d0 = dup_scale(lds_u16(r0)), d1 = dup_scale(lds_u16(r1));

  if constexpr (C == kQ4_0) {
    const uint8_t* c0 = r0 + 2 + 4 * t;
    const uint8_t* c1 = r1 + 2 + 4 * t;
    uint32_t lo00, hi00, lo01, hi01, lo10, hi10, lo11, hi11;
    q4_pair(spread16(lds_u16(c0)), d0, K, lo00, hi00);
    q4_pair(spread16(lds_u16(c0 + 2)), d0, K, lo01, hi01);
    q4_pair(spread16(lds_u16(c1)), d1, K, lo10, hi10);
    q4_pair(spread16(lds_u16(c1 + 2)), d1, K, lo11, hi11);
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
      w[0][i] = q8_pair(spread16(lds_u16(c0 + 2 * i)), d0, K);
      w[1][i] = q8_pair(spread16(lds_u16(c1 + 2 * i)), d1, K);
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      mma_16816(acc[mt], w[0][0], w[1][0], w[0][1], w[1][1], xf[mt][0], xf[mt][1]);
      mma_16816(acc[mt], w[0][2], w[1][2], w[0][3], w[1][3], xf[mt][2], xf[mt][3]);
    }
  } else if constexpr (C == kMLX4) {
    // Thread t: code bytes 4t .. 4t+3 = weights 8t .. 8t+7 in natural order,
    // the same k slots as Q8_0 (and the same X fragments).
    const uint32_t b0 = dup_scale(lds_u16(r0 + 2)), b1 = dup_scale(lds_u16(r1 + 2));
    const uint32_t v0 = *reinterpret_cast<const uint32_t*>(r0 + 4 + 4 * t);
    const uint32_t v1 = *reinterpret_cast<const uint32_t*>(r1 + 4 + 4 * t);
    uint32_t w[2][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t sel = 0x4040u | (uint32_t)(i << 8) | (uint32_t)i;  // byte i, replicated
      w[0][i] = mlx_pair(__byte_perm(v0, 0u, sel), d0, b0, K);
      w[1][i] = mlx_pair(__byte_perm(v1, 0u, sel), d1, b1, K);
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
      q2_byte(__byte_perm(v0[c >> 1], 0u, sel), d0, K, a0, a2);
      q2_byte(__byte_perm(v1[c >> 1], 0u, sel), d1, K, a1, a3);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) mma_16816(acc[mt], a0, a1, a2, a3, xf[mt][2 * c], xf[mt][2 * c + 1]);
    }
  }
}

// ---------------------------------------------------------------- X resident
// When a weight row is one stage (XH), every consumer warp works on the same
// blocks of every unit, so its activation fragments are built once per
// launch, in whatever k order suits the decode.  The bodies below read the
// codes as aligned 32-bit words (the 18- and 34-byte blocks are taken in
// pairs: the odd block of a pair starts on a word, the even one on a
// half-word) and decode whole words (codec.cuh); activation pairs follow
// the weight pairs of q4_word / q8_word / mlx_word.
__device__ __forceinline__ uint32_t lds32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
  return v;
}

// In-block k of the activation in half `e` of fragment register `r` of
// thread t, for the even (odd = false) or odd block of a pair (Q4_0, Q8_0)
// or any block (MLX4).  Q4_0 thread t reads code bytes (c0..c3): of the odd
// block 4t..4t+3; of the even block 4t+2..4t+5, or 0, 1, 14, 15 for t = 3
// (from the words that straddle the block's start and end).  Registers:
// (c0, c2), (c1, c3), then the high nibbles 16 later.  Q8_0 reads two words
// (a0..a3), (b0..b3): odd 8t.., 8t+4..; even 8t+2.., 8t+6.., or 26..29 and
// 30, 31, 0, 1 for t = 3; registers (a0, a2), (a1, a3), (b0, b2), (b1, b3).
// MLX4 word 4t..4t+3 holds codes 8t..8t+7; registers (8t, 8t+4),
// (8t+1, 8t+5), (8t+2, 8t+6), (8t+3, 8t+7).
template <int C>
__device__ __forceinline__ int xh_k(bool odd, int t, int r, int e) {
  if constexpr (C == kQ4_0) {
    int c[4];
    for (int i = 0; i < 4; ++i) c[i] = odd ? 4 * t + i : (t < 3 ? 4 * t + 2 + i : (i < 2 ? i : 12 + i));
    const int byte = (r & 1) + 2 * e;         // r 0: (c0, c2), r 1: (c1, c3)
    return c[byte] + (r >= 2 ? 16 : 0);
  } else if constexpr (C == kQ8_0) {
    int a[8];
    for (int i = 0; i < 8; ++i) {
      if (odd) a[i] = 8 * t + i;
      else if (t < 3) a[i] = 8 * t + 2 + i;
      else a[i] = (26 + i) & 31;                 // 26..31, then 0, 1
    }
    const int word = r >> 1, byte = (r & 1) + 2 * e;
    return a[4 * word + byte];
  } else {
    return 8 * t + r + 4 * e;
  }
}

// Q4_0 pair of blocks at shared addresses a0 (tile row g) and a1 (row g + 8).
__device__ __forceinline__ void xh_pair_q4(uint32_t a0, uint32_t a1, uint32_t eoff, uint32_t esel, uint32_t ooff,
                                           const DecK& K, const uint32_t (&xe)[4], const uint32_t (&xo)[4],
                                           float (&acc)[4]) {
  uint32_t l02[2][2], l13[2][2], h02[2][2], h13[2][2];  // [even/odd block][row]
  const uint32_t base[2] = {a0, a1};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t w0 = lds32(base[r]), w4 = lds32(base[r] + 16);
    const uint32_t we = lds32(base[r] + eoff), wo = lds32(base[r] + ooff);
    q4_word(__byte_perm(we, w4, esel), __byte_perm(w0, 0u, 0x1010u), K, l02[0][r], l13[0][r], h02[0][r],
            h13[0][r]);
    q4_word(wo, __byte_perm(w4, 0u, 0x3232u), K, l02[1][r], l13[1][r], h02[1][r], h13[1][r]);
  }
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t(&x)[4] = b ? xo : xe;
    mma_16816(acc, l02[b][0], l02[b][1], l13[b][0], l13[b][1], x[0], x[1]);
    mma_16816(acc, h02[b][0], h02[b][1], h13[b][0], h13[b][1], x[2], x[3]);
  }
}

// Q8_0 pair of blocks (68 bytes, 17 words) at a0 / a1.
__device__ __forceinline__ void xh_pair_q8(uint32_t a0, uint32_t a1, uint32_t eoff_a, uint32_t eoff_b,
                                           uint32_t esel, uint32_t ooff, const DecK& K, const uint32_t (&xe)[4],
                                           const uint32_t (&xo)[4], float (&acc)[4]) {
  uint32_t p[2][2][4];  // [even/odd block][row][(a02, a13, b02, b13)]
  const uint32_t base[2] = {a0, a1};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t w0 = lds32(base[r]), w8 = lds32(base[r] + 32);
    const uint32_t ea = lds32(base[r] + eoff_a), eb = lds32(base[r] + eoff_b);
    const uint32_t oa = lds32(base[r] + ooff), ob = lds32(base[r] + ooff + 4);
    const uint32_t de = __byte_perm(w0, 0u, 0x1010u), dodd = __byte_perm(w8, 0u, 0x3232u);
    q8_word(ea, de, K, p[0][r][0], p[0][r][1]);
    q8_word(__byte_perm(eb, w0, esel), de, K, p[0][r][2], p[0][r][3]);
    q8_word(oa, dodd, K, p[1][r][0], p[1][r][1]);
    q8_word(ob, dodd, K, p[1][r][2], p[1][r][3]);
  }
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t(&x)[4] = b ? xo : xe;
    mma_16816(acc, p[b][0][0], p[b][1][0], p[b][0][1], p[b][1][1], x[0], x[1]);
    mma_16816(acc, p[b][0][2], p[b][1][2], p[b][0][3], p[b][1][3], x[2], x[3]);
  }
}

// MLX4 block (20 bytes: scale, bias, 16 code bytes from byte 4) at a0 / a1.
__device__ __forceinline__ void xh_block_mlx(uint32_t a0, uint32_t a1, uint32_t coff, const DecK& K,
                                             const uint32_t (&x)[4], float (&acc)[4]) {
  uint32_t lo02[2], hi02[2], lo13[2], hi13[2];
  const uint32_t base[2] = {a0, a1};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t sb = lds32(base[r]), w = lds32(base[r] + coff);
    mlx_word(w, __byte_perm(sb, 0u, 0x1010u), __byte_perm(sb, 0u, 0x3232u), K, lo02[r], hi02[r], lo13[r],
             hi13[r]);
  }
  mma_16816(acc, lo02[0], lo02[1], hi02[0], hi02[1], x[0], x[1]);
  mma_16816(acc, lo13[0], lo13[1], hi13[0], hi13[1], x[2], x[3]);
}

template <int C, bool SWIGLU, int MT, bool WTMA, bool XH>
__global__ void __launch_bounds__(GemvCfg<C, MT>::kThreads, 1) gemv_kernel(const GemvParams p) {
  using Cfg = GemvCfg<C, MT>;
  using S = Stage<C>;
  constexpr int NC = Cfg::kConsumers;
  constexpr int NM = SWIGLU ? 2 : 1;  // tiles (matrices) per unit
  const int R = p.ring;
  const int stage_bytes = 8 * p.pp;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = smem_align<128>(smem_raw);
  float* red = reinterpret_cast<float*>(ring + Cfg::kRingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + Cfg::kRedFloats);
  uint64_t* empty = full + Cfg::kRingMax;
  uint64_t* red_full = empty + Cfg::kRingMax;
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
  pdl_launch_dependents();
  pdl_wait();   // every global access below comes after the previous kernel

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Stage order of a unit: for each row segment s, the gate tile then (for
    // SwiGLU) the up tile.
    int q = 0;             // stages issued
    int pslot = 0;         // ring slot of the next stage
    uint32_t pphase = 0;   // parity of the ring lap being filled
    bool ok = true;
    if constexpr (WTMA) {
      // Lane g < 8 copies row pair g (weight rows n0 + 2g, n0 + 2g + 1).
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const int n = u * 16 + 2 * lane;
        const bool mine = lane < 8 && n < p.N;  // N is even: the pair is whole
        const int pairs = __popc(__ballot_sync(0xffffffffu, mine));
        for (int s = 0; s < p.nst && ok; ++s) {
          const long long off = (long long)s * p.sb;
          const long long left = p.row_bytes - off;
          const uint32_t bytes = (uint32_t)(left < p.sb ? left : p.sb);
          for (int mat = 0; mat < NM; ++mat, ++q) {
            const int slot = pslot;
            if (q >= R) {
              ok = __all_sync(0xffffffffu, mbar_wait_idle(&empty[slot], pphase ^ 1u, ctl));
              if (!ok) break;
            }
            if (++pslot == R) {
              pslot = 0;
              pphase ^= 1u;
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2u * bytes * pairs);
            __syncwarp();
            if (mine && in_bounds(n + 1 < p.N && span_ok(off, bytes, p.row_bytes) &&
                                      span_ok((long long)lane * p.pp, (long long)p.sb + bytes, stage_bytes) &&
                                      (p.nst > 1 || (long long)bytes == p.sb),
                                  p.status, kSiteGemvW)) {
              const uint8_t* src = (mat ? p.w1 : p.w0) + (long long)n * p.row_bytes + off;
              uint8_t* dst = ring + slot * stage_bytes + lane * p.pp;
              if (p.nst == 1) {
                bulk_load(dst, src, 2u * bytes, &full[slot]);   // both rows: contiguous
              } else {
                bulk_load(dst, src, bytes, &full[slot]);
                bulk_load(dst + p.sb, src + p.row_bytes, bytes, &full[slot]);
              }
            }
          }
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
      const int half_sb = p.sb / 2;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        for (int s = 0; s < p.nst && ok; ++s) {
          for (int mat = 0; mat < NM; ++mat, ++q) {
            const int slot = pslot;
            if (q >= R) {
              ok = __all_sync(0xffffffffu, mbar_wait_idle(&empty[slot], pphase ^ 1u, ctl));
              if (!ok) break;
            }
            if (++pslot == R) {
              pslot = 0;
              pphase ^= 1u;
            }
            uint8_t* dst = ring + slot * stage_bytes;
            const uint8_t* base = mat ? p.w1 : p.w0;
            const long long off = (long long)s * p.sb;
            for (int e = lane; e < 16 * half_sb; e += 32) {
              const int r = e / half_sb;          // tile row
              const int c2 = e - r * half_sb;
              const int gg = r & 7, hi = r >> 3;  // pair, row within the pair
              const int n = u * 16 + 2 * gg + hi;
              const long long o = off + 2 * c2;
              unsigned short v = 0;
              if (n < p.N && o < p.row_bytes)
                v = __ldg(reinterpret_cast<const unsigned short*>(base + (long long)n * p.row_bytes + o));
              if (in_bounds(span_ok((long long)gg * p.pp + hi * p.sb + 2 * c2, 2, stage_bytes), p.status,
                            kSiteGemvWHalf))
                *reinterpret_cast<unsigned short*>(dst + gg * p.pp + hi * p.sb + 2 * c2) = v;
            }
            mbar_arrive(&full[slot]);
          }
        }
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 2;
    const int g = lane >> 2, t = lane & 3;
    const int bps = p.sb / S::BB;  // blocks per full stage
    constexpr int XR = XFrag<C>::kRegs;
    const DecK K = make_deck();
    // XH (one stage per row, MT = 1): the activation fragments of this
    // warp's blocks for the whole launch, in the k order of the word
    // decoders.  Q4_0 and Q8_0 warps take block pairs cw + 16 j (blocks
    // 2 (cw + 16 j) and the next), MLX4 warps blocks cw + 16 j.
    constexpr bool kPairs = (C == kQ4_0 || C == kQ8_0);
    uint32_t xh[XH ? Cfg::kXH : 1][4];
    if constexpr (XH) {
      static_assert(MT == 1 && C != kQ2_0, "resident activations: one n8 tile, 32-weight blocks");
      const bool ok_m = g < p.M &&  // activation row g is the fragment column
                        in_bounds(p.sb == (int)p.row_bytes && bps * S::B == p.K, p.status, kSiteGemvX);
      const unsigned short* xrow = reinterpret_cast<const unsigned short*>(p.x) + (size_t)(ok_m ? g : 0) * p.K;
#pragma unroll
      for (int j = 0; j < Cfg::kXH; ++j) {
        const int blk = kPairs ? 2 * (cw + NC * (j >> 1)) + (j & 1) : cw + NC * j;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const uint32_t lo = ok_m ? __ldg(xrow + blk * S::B + xh_k<C>(j & 1, t, r, 0)) : 0u;
          const uint32_t hi = ok_m ? __ldg(xrow + blk * S::B + xh_k<C>(j & 1, t, r, 1)) : 0u;
          xh[j][r] = lo | (hi << 16);
        }
      }
    }
    // Per-thread word offsets of the XH bodies (see xh_k).
    const uint32_t q4_eoff = t < 3 ? 4u * (1 + t) : 0u, q4_esel = t < 3 ? 0x3210u : 0x5432u;
    const uint32_t q8_eoff_b = t < 3 ? 4u * (2 + 2 * t) : 32u, q8_esel = t < 3 ? 0x3210u : 0x7610u;
    const int row_off = g * p.pp + cw * S::BB;  // this thread's row g, this warp's first block
    int slot = 0, i = 0;
    uint32_t phase = 0;   // parity of the ring lap being consumed
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
      float acc[NM][MT][4], acc1[NM][MT][4];
#pragma unroll
      for (int mat = 0; mat < NM; ++mat)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[mat][mt][c] = acc1[mat][mt][c] = 0.f;
      bool ok = true;
      for (int s = 0; s < p.nst && ok; ++s) {
        const int kb0 = s * bps * S::B;
        const int left = (p.K - kb0) / S::B;
        const int nb = left < bps ? left : bps;  // blocks of this segment
        // The NM tiles (gate, up) of this segment are adjacent ring slots:
        // wait for both, then run them block by block (independent MMA chains
        // that share the X fragments).
        // The NM stages of this segment are consecutive in the ring (with an
        // odd ring the second may wrap to slot 0 of the next lap).
        int sl[NM];
        uint32_t ph[NM];
        sl[0] = slot;
        ph[0] = phase;
        if constexpr (NM == 2) {
          sl[1] = slot + 1 == R ? 0 : slot + 1;
          ph[1] = slot + 1 == R ? phase ^ 1u : phase;
        }
        for (int mat = 0; mat < NM && ok; ++mat)
          ok = __all_sync(0xffffffffu, mbar_wait_idle(&full[sl[mat]], ph[mat], ctl, 64));
        if (!ok) break;
        if constexpr (XH) {
          if constexpr (kPairs) {
#pragma unroll
            for (int j = 0; j < Cfg::kXH / 2; ++j) {
#pragma unroll
              for (int mat = 0; mat < NM; ++mat) {
                float(&a)[4] = (NM == 1 && (j & 1)) ? acc1[mat][0] : acc[mat][0];
                const uint32_t a0 = smem_u32(ring) + sl[mat] * stage_bytes + g * p.pp + (cw + NC * j) * (2 * S::BB);
                if constexpr (C == kQ4_0)
                  xh_pair_q4(a0, a0 + p.sb, q4_eoff, q4_esel, 20u + 4u * t, K, xh[2 * j], xh[2 * j + 1], a);
                else
                  xh_pair_q8(a0, a0 + p.sb, 4u * (1 + 2 * t), q8_eoff_b, q8_esel, 36u + 8u * t, K, xh[2 * j],
                             xh[2 * j + 1], a);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < Cfg::kXH; ++j) {
#pragma unroll
              for (int mat = 0; mat < NM; ++mat) {
                float(&a)[4] = (NM == 1 && (j & 1)) ? acc1[mat][0] : acc[mat][0];
                const uint32_t a0 = smem_u32(ring) + sl[mat] * stage_bytes + g * p.pp + (cw + NC * j) * S::BB;
                xh_block_mlx(a0, a0 + p.sb, 4u + 4u * t, K, xh[j], a);
              }
            }
          }
        } else {
          const uint8_t* r0 = ring + row_off;   // block cw, row g (plus the stage of each tile)
          const uint8_t* r1 = r0 + p.sb;         // block cw, row g + 8
          if (nb == Cfg::kBlocks) {
            // Full stage: every block of this warp is inside K.
#pragma unroll
            for (int j = 0; j < Cfg::kXH; ++j) {
              const int bo = NC * j * S::BB;
              uint32_t xf[MT][XR];
              load_xfrag<C, MT>(p, g, t, kb0 + (cw + NC * j) * S::B, xf);
#pragma unroll
              for (int mat = 0; mat < NM; ++mat) {
                const int to = sl[mat] * stage_bytes + bo;
                if (NM == 1 && (j & 1)) gemv_block<C, MT>(r0 + to, r1 + to, t, xf, acc1[mat], K);
                else gemv_block<C, MT>(r0 + to, r1 + to, t, xf, acc[mat], K);
              }
            }
          } else {
            for (int b = cw, j = 0; b < nb; b += NC, ++j) {
              const int bo = (b - cw) * S::BB;
              uint32_t xf[MT][XR];
              load_xfrag<C, MT>(p, g, t, kb0 + b * S::B, xf);
#pragma unroll
              for (int mat = 0; mat < NM; ++mat) {
                const int to = sl[mat] * stage_bytes + bo;
                if (NM == 1 && (j & 1)) gemv_block<C, MT>(r0 + to, r1 + to, t, xf, acc1[mat], K);
                else gemv_block<C, MT>(r0 + to, r1 + to, t, xf, acc[mat], K);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0)
          for (int mat = 0; mat < NM; ++mat) mbar_arrive(&empty[sl[mat]]);
        for (int mat = 0; mat < NM; ++mat)
          if (++slot == R) {
            slot = 0;
            phase ^= 1u;
          }
      }
      if (!ok) break;
      const int rb = i & 1;
      if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait_idle(&red_empty[rb], ((i >> 1) - 1) & 1, ctl))) break;
      float4* dst = reinterpret_cast<float4*>(red + ((rb * NC + cw) * 32 + lane) * Cfg::kLaneFloats);
#pragma unroll
      for (int mat = 0; mat < NM; ++mat)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          dst[mat * MT + mt] = make_float4(acc[mat][mt][0] + acc1[mat][mt][0], acc[mat][mt][1] + acc1[mat][mt][1],
                                           acc[mat][mt][2] + acc1[mat][mt][2], acc[mat][mt][3] + acc1[mat][mt][3]);
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
      float v[NM][MT][4];
#pragma unroll
      for (int mat = 0; mat < NM; ++mat)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int c = 0; c < 4; ++c) v[mat][mt][c] = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float4* src = reinterpret_cast<const float4*>(red + ((rb * NC + w) * 32 + lane) * Cfg::kLaneFloats);
#pragma unroll
        for (int mat = 0; mat < NM; ++mat)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const float4 f = src[mat * MT + mt];
            v[mat][mt][0] += f.x; v[mat][mt][1] += f.y; v[mat][mt][2] += f.z; v[mat][mt][3] += f.w;
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[rb]);
      // v[.][mt][c], c < 2: tile row g = output n0 + 2g, activation row
      // 8 mt + 2t + c; v[.][mt][c + 2]: tile row g + 8 = output n0 + 2g + 1.
      const int n = u * 16 + 2 * g;
      if (n < p.N) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int m = 8 * mt + 2 * t + c;
            if (m >= p.M) continue;
            float a = v[0][mt][c], b = v[0][mt][c + 2];
            if constexpr (SWIGLU) {
              a = (p.act ? gelu_f(a) : a / (1.0f + __expf(-a))) * v[NM - 1][mt][c];
              b = (p.act ? gelu_f(b) : b / (1.0f + __expf(-b))) * v[NM - 1][mt][c + 2];
            }
            // outputs n, n + 1 (same head: n is even and head_dim is too)
            const size_t off = p.head_dim == 0 ? (size_t)m * p.N + n
                                               : ((size_t)(n / p.head_dim) * p.M + m) * p.head_dim + n % p.head_dim;
            if (in_bounds(off + 2 <= (size_t)p.M * p.N && (n + 1 < p.N), p.status, kSiteGemvY))
              *reinterpret_cast<__half2*>(p.y + off) = __floats2half2_rn(a, b);
          }
      }
    }
  }
}

}  // namespace m4q
