// tc_small.cuh -- tcgen05 kernel for the projection at small M (M <= 128):
// Y = X W^T and Y = act(X Wg^T) x (X Wu^T).
//
// Pages: "v0.1 vs v0.2 comparison" 2.1 and 2.2 (Bricks 1-3), "Releases"
// v0.3.0 (one linear layer for every M).  With few activation rows the MMA
// shape of tc_proj (M = 128 weight rows read from TMEM, N = the activation
// rows) spends most of each instruction on the weight operand: at N = 64 an
// MMA takes about five times its share of the tensor pipe.  Here the roles
// of the operands are swapped, so that every MMA covers 128 weight rows for
// all activation rows at once:
//   D[128 activation rows (TMEM lanes)][128 weight rows (columns)]
//     += X_tile[128 x 16] * Wdec_tile[128 x 16]^T,   M = N = 128, K = 16,
// with both operands in shared memory (128-byte swizzled, K-major).  An X
// stage holds XR = 32, 64 or 128 rows (the least of them covering M): TMA
// then moves only the rows that exist (128-row boxes that were mostly out of
// bounds were slow).  The MMA still reads a 128-row A window; rows past XR
// are the next stages (or a pad after the ring) and only feed rows of D at
// or past M, which are never stored.
//
// CTA roles (512 threads), one persistent CTA per SM over output tiles of
// 128 weight rows (64 outputs for the gated projection, gate row i and up
// row i at B rows 2i and 2i + 1):
//   warp 0, one lane: TMA producer of X sub-tiles [128 rows x 64 k] (the same
//     sub-tiles for every output tile, re-read from L2).
//   warp 2, one lane: TMA producer of packed weight stages (as tc_proj).
//   warp 1, one lane: issues the MMAs and owns TMEM (two D buffers of 128
//     columns).  The issue loop is the serial step of this kernel, so it
//     takes two 64-k sub-steps at a time (8 MMAs) and frees both with one
//     commit on a per-pair barrier that the X producer and the decode
//     warps both wait on (X and B rings advance together, 2 pairs deep);
//     the X stages and decoded-B slots of a pair are likewise signalled on
//     one barrier each, so the thread waits twice per 8 MMAs.
//   warps 4..11, two decode groups: thread r of a group owns B row r and
//     decodes weights [32 g, 32 g + 32) of each 64-k sub-step (codec.cuh,
//     bit-exact) straight into the swizzled B ring in shared memory.
//   warps 12..15: epilogue.  Thread m owns activation row m = TMEM lane m: it
//     reads its 128 columns of D, forms fp16 outputs (act(g) x u for column
//     pairs), stages them in a 128-byte swizzled tile and one thread stores
//     the tile with TMA (rows past M are clipped by the tensor map).
// Every wait is bounded in time; on expiry the CTA records the failure,
// drains its copies in flight, frees TMEM and returns.
#pragma once

#include "tc_proj.cuh"

namespace m4q {

// D[tmem] (+)= A[smem] * B[smem]^T; fp16 inputs, fp32 accumulator.
__device__ __forceinline__ void tc_mma_ss_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// K split of this kernel: slice q of a staged partial tile holds the W =
// 128 / split weight columns CTA q owns, for every activation row, rows
// W + 4 floats apart (the pad spreads the writes of 32 consecutive rows
// over all banks).  An owner reads a peer's slice as nearly contiguous runs
// (distributed shared memory requests that touch scattered rows were an
// order of magnitude slower), and 4 columns of a row are 4 consecutive
// outputs.
__device__ __forceinline__ int small_split_slot(int m, int c, int W) {
  return ((c / W) * 128 + m) * (W + 4) + (c % W);
}

template <int C, bool SWIGLU, int XR>
struct TsCfg {
  using S = Stage<C>;
  static constexpr int kThreads = 512;
  static constexpr int kRows = 128;                          // B rows (weight rows) per tile = MMA N
  static constexpr int kOutRows = SWIGLU ? 64 : 128;         // outputs per tile
  static constexpr int kXStage = XR * 128;                   // [XR m][64 k] fp16, swizzled
  static constexpr int kXPad = (128 - XR) * 128;             // keeps the last stage's A window inside
  static constexpr int kBStage = 128 * 128;                  // [128 weight rows][64 k] fp16, swizzled
  static constexpr int kSW = S::KPB <= 160 ? 3 : 2;          // packed-W ring depth
  // X and decoded-B rings advance together, 4 slots = 2 pairs of sub-steps:
  // the MMA thread consumes a pair at once and frees it with one commit.
  static constexpr int kSX = 4;                              // X ring depth
  static constexpr int kSB = 4;                              // decoded-B ring depth
  static constexpr int kWStage = kRows * S::KPB;
  static constexpr int kYBytes = 128 * kOutRows * 2;         // 64-output boxes of [128 m][128 B]
  static constexpr int kBars = kSX + 2 * kSW + kSB + 2 + 5;
  static constexpr int kSmemBytes =
      1024 + kSX * kXStage + kXPad + kSB * kBStage + kYBytes + kSW * kWStage + kBars * 8 + 16;
  static constexpr uint32_t kTmemCols = 256;                 // two D buffers
  // K split: each CTA stages its fp32 partial D [128 m][128 cols] over the
  // idle X and B rings, slice-major (small_split_slot).
  static_assert(128 * (128 + 32) * 4 <= kSX * kXStage + kXPad + kSB * kBStage, "D staging fits the rings");
  // Q8_0 / Q2_0 GEMM with 128-row X stages does not fit; the host sends
  // that case to tc_proj (M > 64 with 272-byte packed stages).
  static constexpr bool kFits = kSmemBytes <= 227 * 1024;
  static_assert(XR == 32 || XR == 64 || XR == 128, "X stage rows");
  static_assert(kSX == kSB && kSX % 2 == 0, "paired X and B rings");
  static_assert(kXStage % 1024 == 0, "X stages start on swizzle atoms");
  static_assert(kWStage % 128 == 0 && (64 * S::KPB) % 128 == 0, "TMA destinations 128-byte aligned");
};

template <int C, bool SWIGLU, int ACT, int XR>
__global__ void __launch_bounds__(512, 1)
    tc_small_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w0,
                    const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_y,
                    const TcParams p) {
  using Cfg = TsCfg<C, SWIGLU, XR>;
  using S = Stage<C>;
  static_assert(Cfg::kFits, "shared memory budget");
  constexpr int SX = Cfg::kSX, SW = Cfg::kSW, SB = Cfg::kSB;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* xs = smem_align<1024>(smem_raw);
  uint8_t* bs = xs + SX * Cfg::kXStage + Cfg::kXPad;
  uint8_t* ys = bs + SB * Cfg::kBStage;
  uint8_t* ws = ys + Cfg::kYBytes;
  uint64_t* x_full = reinterpret_cast<uint64_t*>(ws + SW * Cfg::kWStage);
  uint64_t* w_full = x_full + SX;
  uint64_t* w_empty = w_full + SW;
  uint64_t* b_full = w_empty + SW;
  uint64_t* pair_free = b_full + SB;  // [2]: X and B slots 2p, 2p + 1 consumed
  uint64_t* d_full = pair_free + 2;   // [2]
  uint64_t* d_empty = d_full + 2;     // [2]
  uint64_t* drain = d_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nks = (p.K + 63) / 64;
  // K split (p.split > 1): the CTAs of a cluster share one output tile, CTA
  // `rank` taking sub-steps [ks0, ks1) (whole packed stages [pk0, pk1)).
  const int nsplit = p.split;
  const int rank = nsplit > 1 ? (int)cluster_ctarank() : 0;
  const int ks0 = rank * p.ks_per;
  const int ks1 = min(nks, ks0 + p.ks_per);
  const int pk0 = ks0 / S::SUB, pk1 = (ks1 + S::SUB - 1) / S::SUB;
  const int tile0 = blockIdx.x / nsplit, tstep = gridDim.x / nsplit;
  bool split_ok = false;   // epilogue threads: this CTA's partial D is staged

  if (threadIdx.x == 0) {
    for (int i = 0; i < SX; ++i) mbar_init(&x_full[i], 1);   // [0], [1]: stage pairs
    for (int i = 0; i < SW; ++i) { mbar_init(&w_full[i], 1); mbar_init(&w_empty[i], 8); }
    for (int i = 0; i < SB; ++i) mbar_init(&b_full[i], 8);   // [0], [1]: slot pairs, one arrival per decode warp
    for (int i = 0; i < 2; ++i) mbar_init(&pair_free[i], 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&d_full[i], 1); mbar_init(&d_empty[i], 4); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};
  pdl_launch_dependents();
  pdl_wait();   // every global access below comes after the previous kernel

  if (warp == 0) {
    // ------------------------------------------------------------ X producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      int xi = 0;
      bool ok = true;
      for (int tile = tile0; tile < p.tiles && ok; tile += tstep) {
        for (int ks = ks0; ks < ks1; ++ks) {
          // Stages 2p and 2p + 1 land on one barrier (the MMA thread takes
          // them together); every CTA runs an even number of sub-steps here.
          const int sx = xi % SX;
          if ((sx & 1) == 0) {
            if (xi >= SX && !mbar_wait_idle(&pair_free[sx >> 1], ((xi / SX) - 1) & 1, ctl)) { ok = false; break; }
            mbar_arrive_expect_tx(&x_full[sx >> 1], 2 * Cfg::kXStage);
          }
          if (in_bounds(tma_x_ok(ks * 64, 2), p.status, kSiteTcX))
            tma_load_2d(xs + sx * Cfg::kXStage, &tm_x, &x_full[sx >> 1], ks * 64, 0);
          ++xi;
        }
      }
      if (!ok) {
        // (the loop stops only before the first stage of a pair)
        for (int i = (xi > SX ? xi - SX : 0); i < xi; i += 2)
          mbar_wait_drain(&x_full[(i % SX) >> 1], (i / SX) & 1, 100000000ull);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ W producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_w0);
      if (SWIGLU) tma_prefetch_desc(&tm_w1);
      int wi = 0;
      bool ok = true;
      for (int tile = tile0; tile < p.tiles && ok; tile += tstep) {
        const int n0 = tile * Cfg::kOutRows;
        for (int pk = pk0; pk < pk1; ++pk) {
          const int sp = wi % SW;
          if (wi >= SW && !mbar_wait_idle(&w_empty[sp], ((wi / SW) - 1) & 1, ctl)) { ok = false; break; }
          mbar_arrive_expect_tx(&w_full[sp], Cfg::kWStage);
          uint8_t* dst = ws + sp * Cfg::kWStage;
          const int xc = pk * (S::KPB / 2);  // uint16 elements
          if (in_bounds(tma_x_ok(xc, 2) && 2ll * xc < p.row_bytes && n0 >= 0, p.status, kSiteTcW)) {
            tma_load_2d(dst, &tm_w0, &w_full[sp], xc, n0);
            if (SWIGLU) tma_load_2d(dst + 64 * S::KPB, &tm_w1, &w_full[sp], xc, n0);
          }
          ++wi;
        }
      }
      if (!ok) {
        for (int i = (wi > SW ? wi - SW : 0); i < wi; ++i)
          mbar_wait_drain(&w_full[i % SW], (i / SW) & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, 128);
      int ks_g = 0, lt = 0;
      bool ok = true;
      for (int tile = tile0; tile < p.tiles && ok; tile += tstep, ++lt) {
        const int db = lt & 1;
        // D buffer db must have been read out by the epilogue two tiles ago.
        if (lt >= 2 && !mbar_wait(&d_empty[db], ((lt >> 1) - 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        // ks1 - ks0 is even here (K is a multiple of 128 on this path and a
        // split takes whole packed stages)
        for (int ks = ks0; ks < ks1; ks += 2, ks_g += 2) {
          const int s0 = ks_g % SX;   // slots s0, s0 + 1 of both rings (SX == SB)
          if (!mbar_wait(&b_full[s0 >> 1], (ks_g / SB) & 1, ctl) ||
              !mbar_wait(&x_full[s0 >> 1], (ks_g / SX) & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t adesc = sdesc_sw128_kmajor(smem_u32(xs + (s0 + h) * Cfg::kXStage));
            const uint64_t bdesc = sdesc_sw128_kmajor(smem_u32(bs + (s0 + h) * Cfg::kBStage));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_ss_f16(tmem + 128 * db, adesc + 2 * kk, bdesc + 2 * kk, idesc, (ks != ks0) | h | kk);
          }
          tc_commit(&pair_free[s0 >> 1]);
        }
        if (ok) tc_commit(&d_full[db]);
      }
      // Every MMA issued above completes before the CTA frees TMEM.
      tc_commit(drain);
      mbar_wait_drain(drain, 0, 200000000ull);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ decode
    const int G = (warp - 4) >> 2;      // weights [32 G, 32 G + 32) of each sub-step
    const int r = threadIdx.x & 127;    // B row
    const int srow = SWIGLU ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;  // row in the W stage
    bool ok = true;
    int ks_g = 0, pk_g = 0;
    const DecK K = make_deck();
    for (int tile = tile0; tile < p.tiles && ok; tile += tstep) {
      int ks = ks0;
      for (int pk = pk0; pk < pk1 && ok; ++pk, ++pk_g) {
        uint32_t w[S::WORDS];
        const int sp = pk_g % SW;
        ok = __all_sync(0xffffffffu, mbar_wait(&w_full[sp], (pk_g / SW) & 1, ctl));
        if (!ok) break;
        const uint4* src = reinterpret_cast<const uint4*>(ws + sp * Cfg::kWStage + srow * S::KPB);
        const bool rok = in_bounds(span_ok((long long)srow * S::KPB, S::KPB, Cfg::kWStage), p.status, kSiteTcWRow);
#pragma unroll
        for (int i = 0; i < S::KPB / 16; ++i) {
          const uint4 v = rok ? src[i] : make_uint4(0, 0, 0, 0);
          w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
        // The slot is released only after the loop below has used every
        // loaded word: an arrive issued right after the loads let the next
        // TMA fill of the slot land before loads still in flight had read it
        // (seen as stale weights in some rows under shared-memory load).
#pragma unroll
        for (int j = 0; j < S::SUB; ++j) {
          if (ks >= ks1) break;
          const int sb = ks_g % SB;
          if (ks_g >= SB && (sb & 1) == 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&pair_free[sb >> 1], ((ks_g / SB) - 1) & 1, ctl));
            if (!ok) break;
          }
          uint32_t out[16];
          if (G == 0) decode_half<C, 0>(w, j, out, K);
          else decode_half<C, 1>(w, j, out, K);
          // row r of the 128-byte swizzled tile: 16-byte chunk c sits at c ^ (r & 7)
          uint8_t* row = bs + sb * Cfg::kBStage + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = 4 * G + q;
            if (in_bounds(span_ok((long long)r * 128 + ((c ^ (r & 7)) << 4), 16, Cfg::kBStage), p.status,
                          kSiteTcBRing))
              *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
                  make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
          }
          fence_proxy_async_smem();   // generic-proxy writes, read by the tensor core
          if (sb & 1) mbar_arrive_warp(&b_full[sb >> 1]);   // the pair's second slot is written
          ++ks;
          ++ks_g;
        }
        if (ok) mbar_arrive_warp(&w_empty[sp]);
      }
    }
  } else if (warp >= 12 && nsplit > 1) {
    // ------------------------------------------------ epilogue, K split
    // One tile per cluster.  Stage this CTA's partial D (thread m = row m)
    // in its own shared memory; the cluster then reduces it below.
    const int m = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const bool dok = !*ctl.abort && mbar_wait_idle(&d_full[0], 0, ctl, 128);
    split_ok = !named_bar_any(1, 128, !dok || *ctl.abort);
    if (split_ok) {
      tc_fence_after();
      float* stg = reinterpret_cast<float*>(xs);   // X and B rings are idle
      const int W = 128 / nsplit;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        tmem_ld32_wait(tmem + lane_base + 32 * ch, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (in_bounds(span_ok(4ll * small_split_slot(m, 32 * ch + 4 * i, W), 16,
                                (long long)SX * Cfg::kXStage + Cfg::kXPad + SB * Cfg::kBStage),
                        p.status, kSiteTcSplitSlot))
            *reinterpret_cast<float4*>(stg + small_split_slot(m, 32 * ch + 4 * i, W)) =
                make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                            __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
      }
      tc_fence_before();
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int m = 32 * q + lane;        // activation row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const bool leader = threadIdx.x == 384;
    int lt = 0;
    for (int tile = tile0; tile < p.tiles; tile += tstep, ++lt) {
      const int db = lt & 1;
      const int n0 = tile * Cfg::kOutRows;
      bool dok = false;
      if (!*ctl.abort) dok = mbar_wait_idle(&d_full[db], (lt >> 1) & 1, ctl, 128);
      if (named_bar_any(1, 128, !dok || *ctl.abort)) break;
      // The previous tile's store has read the staging tile.
      if (leader) bulk_wait_read<0>();
      named_bar_sync(1, 128);
      tc_fence_after();
      // Staging: [box of 64 outputs][128 m][128 B], 16-byte chunk c of row m
      // at c ^ (m & 7).  Each 32-column chunk of D is converted and written
      // as soon as it is read.
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        tmem_ld32_wait(tmem + lane_base + 128 * db + 32 * ch, v);
        constexpr int NW = SWIGLU ? 8 : 16;   // packed fp16 pairs from this chunk
        uint32_t y2[NW];
        if constexpr (SWIGLU) {
          // columns 2i, 2i + 1: gate and up of output 16 ch + i
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float y[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float g = __uint_as_float(v[2 * (i + h)]), u = __uint_as_float(v[2 * (i + h) + 1]);
              y[h] = (ACT ? gelu_f(g) : __fdividef(g, 1.0f + __expf(-g))) * u;
            }
            const __half2 hy = __floats2half2_rn(y[0], y[1]);
            y2[i / 2] = *reinterpret_cast<const uint32_t*>(&hy);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const __half2 hy = __floats2half2_rn(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
            y2[i / 2] = *reinterpret_cast<const uint32_t*>(&hy);
          }
        }
#pragma unroll
        for (int k = 0; k < NW / 4; ++k) {
          const int c = (NW / 4) * ch + k;          // 16-byte chunk of this row's outputs
          uint8_t* box = ys + (c >> 3) * (128 * 128);
          if (in_bounds(span_ok((long long)(c >> 3) * (128 * 128) + m * 128 + (((c & 7) ^ (m & 7)) << 4), 16,
                                Cfg::kYBytes),
                        p.status, kSiteTcStage))
            *reinterpret_cast<uint4*>(box + m * 128 + (((c & 7) ^ (m & 7)) << 4)) =
                make_uint4(y2[4 * k], y2[4 * k + 1], y2[4 * k + 2], y2[4 * k + 3]);
        }
      }
      // Every column of D has been read: the buffer may take tile lt + 2.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[db]);
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (leader) {
#pragma unroll
        for (int b = 0; b < Cfg::kOutRows / 64; ++b)
          if (in_bounds(tma_x_ok(n0 + 64 * b, 2), p.status, kSiteTcY))
            tma_store_2d(&tm_y, ys + b * (128 * 128), n0 + 64 * b, 0);
        bulk_commit();
      }
    }
    if (leader) bulk_wait_all();
  }

  if (nsplit > 1) {
    // Every thread of the cluster: all partials are staged.
    cluster_sync_all();
    if (warp >= 12 && split_ok) {
      // CTA `rank` owns weight columns [rank W, rank W + W) of the tile for
      // every activation row; the 128 epilogue threads walk its slice a
      // float4 (4 columns of one row) each, add the slices of the cluster's
      // CTAs in rank order (a fixed order: the result does not depend on
      // timing) and write the outputs.
      const int t = threadIdx.x - 384;
      const int W = 128 / nsplit, Q = W / 4;
      const uint32_t slice = smem_u32(reinterpret_cast<float*>(xs) + rank * 128 * (W + 4));
      for (int e = t; e < 128 * Q; e += 128) {
        const int m = e / Q, c = 4 * (e % Q);
        const uint32_t a = slice + 4u * (uint32_t)(m * (W + 4) + c);
        if (!in_bounds(span_ok(4ll * (rank * 128 * (W + 4) + m * (W + 4) + c), 16,
                               (long long)SX * Cfg::kXStage + Cfg::kXPad + SB * Cfg::kBStage),
                       p.status, kSiteTcSplitSlot))
          continue;
        float4 f[8];
#pragma unroll
        for (int src = 0; src < 8; ++src)
          if (src < nsplit) f[src] = ld_dsmem_f4(mapa_shared(a, (uint32_t)src));
        float4 s4 = f[0];
#pragma unroll
        for (int src = 1; src < 8; ++src)
          if (src < nsplit) { s4.x += f[src].x; s4.y += f[src].y; s4.z += f[src].z; s4.w += f[src].w; }
        if (m >= p.M) continue;
        if constexpr (SWIGLU) {
          // columns c, c + 1 (c + 2, c + 3): gate and up of one output
          const int n = tile0 * Cfg::kOutRows + (rank * W + c) / 2;   // 2 outputs, n even
          const float y0 = (ACT ? gelu_f(s4.x) : __fdividef(s4.x, 1.0f + __expf(-s4.x))) * s4.y;
          const float y1 = (ACT ? gelu_f(s4.z) : __fdividef(s4.z, 1.0f + __expf(-s4.z))) * s4.w;
          if (n < p.N && in_bounds(n + 2 <= p.N, p.status, kSiteTcSplitY))
            *reinterpret_cast<__half2*>(p.y + (size_t)m * p.N + n) = __floats2half2_rn(y0, y1);
        } else {
          const int n = tile0 * Cfg::kOutRows + rank * W + c;   // 4 outputs; N % 8 == 0: all in or all out
          if (n < p.N && in_bounds(n + 4 <= p.N, p.status, kSiteTcSplitY)) {
            const __half2 h0 = __floats2half2_rn(s4.x, s4.y), h1 = __floats2half2_rn(s4.z, s4.w);
            *reinterpret_cast<uint2*>(p.y + (size_t)m * p.N + n) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
          }
        }
      }
    }
    // No CTA leaves while a peer may still read its staged partial.
    cluster_sync_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace m4q
