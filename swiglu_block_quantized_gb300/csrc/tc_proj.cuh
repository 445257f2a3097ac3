// tc_proj.cuh -- tcgen05 tensor-core kernel for the quantized projection
// Y = X W^T and the fused gate/up projection Y = SiLU(X Wg^T) x (X Wu^T).
//
// Pages: "v0.1 vs v0.2 comparison" 2.1 (Bricks 1-2: a hardware-MMA GEMM core
// fed by staged, unpacked weight tiles) and 2.2 (Brick 3: gate and up share
// one staged X tile and the SiLU(G) x U epilogue stays on chip).
//
// Mapping onto sm_103a.  One persistent CTA per SM walks output tiles; a
// tile is 128 weight rows (64 outputs for SwiGLU) x NX activation rows.
//   * The MMA computes D^T = W_tile * X_tile^T with M = 128 weight rows and
//     N = NX activation rows: W is the A operand and lives in TMEM, X is the
//     B operand and lives in shared memory (128-byte swizzled, K-major).
//     D (fp32, 128 lanes x NX columns) accumulates in TMEM.
//   * warp 0, one lane: TMA producer of X sub-tiles [NX rows x 64 k].
//     warp 2, one lane: TMA producer of packed weight stages [128 rows x 8
//     blocks].  Independent rings; both run ahead across tile boundaries.
//   * warp 1, one lane: issues tcgen05.mma (4 per 64-k sub-step), commits
//     ring releases to mbarriers.  Warp 1 also owns the TMEM allocation.
//     The A ring is handed over in pairs of sub-steps (64 columns): one
//     a_full wait and one a_empty commit per pair.  Each handover costs the
//     issuing thread a fixed time in which the tensor pipe runs dry, so
//     halving their number gave 5% at the 8B shape (M = 2048) and 8% at
//     M = 64.
//   * warps 4..11, two decode warpgroups.  Thread r of a group owns weight
//     row r = TMEM lane r; group g decodes weights [32g, 32g+32) of every
//     64-k sub-step (codec.cuh) and writes them with tcgen05.st into a TMEM
//     ring of A sub-tiles (32 columns each, taken in pairs): after the
//     second store of a pair the thread waits for its stores and arrives.
//   * warps 12..19, two epilogue warpgroups, each on half of the activation
//     columns: tcgen05.ld of D (D is released to the next tile as soon as it
//     is read), fp16 rounding or SiLU(g)*u, staging in shared memory and TMA
//     bulk stores of Y.
//   * Direct-head output (GEMM, HD = head dim 64 or 128): each staged chunk
//     is laid out [heads][32 m][HD] and stored with a 3-D TMA box into
//     Y[N / HD][M][HD], so a Q/K/V projection needs no transpose afterwards
//     ("v0.1 vs v0.2 comparison" section 4, v0.2.1 direct-head layout).
//   * SwiGLU: A row 2i is gate row n0+i and row 2i+1 the up row of the same
//     output, so one MMA stream computes G and U for 64 outputs and every
//     (G, U) pair sits in adjacent TMEM lanes, i.e. adjacent threads of one
//     warp: the epilogue pairs them with a shuffle and writes only SiLU(G) x U.
// Every mbarrier wait is bounded in time; on expiry the CTA records the
// failure in the status word, drains what it has in flight, frees TMEM and
// returns (results are then undefined and the host reports a timeout).
#pragma once

#include "codec.cuh"

namespace m4q {

struct TcParams {
  const uint8_t* w0;   // weights (gate rows for SwiGLU); read directly when !WTMA
  const uint8_t* w1;   // up weights for SwiGLU, else null
  __half* y;           // output (K-split epilogue of the small-M kernel writes it directly)
  int M, N, K;
  long long row_bytes; // packed bytes per weight row
  int m_tiles, tiles;  // activation tiles, total output tiles
  int split;           // CTAs of a cluster sharing one tile along K (1: no split)
  int ks_per;          // 64-weight sub-steps per CTA of a split (a whole number of packed stages)
  uint32_t* status;    // device status word
  unsigned long long limit_ns;
};

template <int C, bool SWIGLU, int NX, bool WTMA>
struct TcCfg {
  using S = Stage<C>;
  static constexpr int kWarps = 20;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kRows = 128;                               // MMA M
  static constexpr int kOutRows = SWIGLU ? 64 : 128;              // outputs n per tile
  static constexpr int kSW = WTMA ? (S::KPB <= 160 ? 3 : 2) : 0;  // packed-W ring depth
  static constexpr int kSA = 8;                                   // TMEM A ring depth
  static constexpr int kXStage = NX * 128;                        // bytes
  static constexpr int kWStage = kRows * S::KPB;                  // bytes
  static constexpr int kYStage = 32 * kOutRows * 2;               // one staged Y chunk (GEMM)
  static constexpr int kYSlab = (NX / 2) * 16 * 2;                // one warp's Y slab (SwiGLU)
  static constexpr int kYBytes = SWIGLU ? 8 * kYSlab : 4 * kYStage;  // GEMM: 2 groups x 2 buffers
  static constexpr int kFixed = kSW * kWStage + kYBytes + 1024 + 512;  // + align, barriers
  static constexpr int kBudget = 227 * 1024;
  static constexpr int kSX = (kFixed + 8 * kXStage <= kBudget) ? 8
                             : (kFixed + 6 * kXStage <= kBudget) ? 6
                             : (kFixed + 5 * kXStage <= kBudget) ? 5
                             : (kFixed + 4 * kXStage <= kBudget) ? 4 : 3;
  static constexpr int kTmemCols = 512;
  static constexpr int kACol0 = 256;                              // A ring columns
  static constexpr int kSmemBytes =
      (kFixed + kSX * kXStage > 116 * 1024) ? kFixed + kSX * kXStage : 116 * 1024;
  static_assert(NX % 16 == 0 && NX >= 64 && NX <= 256, "MMA N");
  static_assert(kACol0 + 32 * kSA <= kTmemCols && NX <= kACol0, "TMEM budget");
  static_assert(kSmemBytes <= kBudget, "shared memory budget");
  static_assert(kXStage % 1024 == 0 && kWStage % 16 == 0 && kYStage % 1024 == 0 && kYSlab % 1024 == 0,
                "alignment");
};

// Barrier-reduction OR over `count` threads of named barrier `id`.
__device__ __forceinline__ bool named_bar_any(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(count), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// Read this row's packed stage `pk` straight from global memory (2-byte
// loads; rows >= N and bytes past the row end read as zero, which decodes to
// zero weights).
template <int C>
__device__ __forceinline__ void load_stage_global(const uint8_t* __restrict__ row, bool row_ok,
                                                  long long row_bytes, int pk,
                                                  uint32_t (&w)[Stage<C>::WORDS]) {
  using S = Stage<C>;
  const long long b0 = (long long)pk * S::KPB;
#pragma unroll
  for (int i = 0; i < S::WORDS; ++i) {
    uint32_t lo = 0, hi = 0;
    const long long o = b0 + 4 * i;
    if (row_ok && o < row_bytes) lo = __ldg(reinterpret_cast<const unsigned short*>(row + o));
    if (row_ok && o + 2 < row_bytes) hi = __ldg(reinterpret_cast<const unsigned short*>(row + o + 2));
    w[i] = lo | (hi << 16);
  }
}

// Shared state of one CTA.
struct TcSmem {
  uint8_t* xs;  // X ring
  uint8_t* ws;  // packed-W ring
  uint8_t* ys;  // Y staging
  uint64_t *x_full, *x_empty, *w_full, *w_empty, *a_full, *a_empty;
  uint64_t *d_full, *d_empty, *drain;
};

// The part of the K loop a CTA runs.  Without a split (p.split == 1) every
// CTA walks all sub-steps of its tiles (persistent: tiles tile0, tile0 +
// tstep, ...).  With a split the CTAs of a cluster share one tile and CTA
// `rank` takes sub-steps [ks0, ks1), whole packed stages [pk0, pk1).
struct KRange {
  int ks0, ks1, pk0, pk1, tile0, tstep, rank;
};
template <int SUB>
__device__ __forceinline__ KRange k_range(const TcParams& p) {
  KRange r;
  const int nks = (p.K + 63) / 64;
  r.rank = p.split > 1 ? (int)cluster_ctarank() : 0;
  r.ks0 = r.rank * p.ks_per;
  r.ks1 = min(nks, r.ks0 + p.ks_per);
  r.pk0 = r.ks0 / SUB;
  r.pk1 = (r.ks1 + SUB - 1) / SUB;
  r.tile0 = blockIdx.x / p.split;
  r.tstep = gridDim.x / p.split;
  return r;
}

// Decode role of group G (0 or 1): every tile, every sub-step, weights
// [32G, 32G+32) of this thread's row.
template <int C, bool SWIGLU, int NX, bool WTMA, int G>
__device__ __forceinline__ void decode_role(const TcSmem& sm, const TcParams& p, uint32_t tmem,
                                            const WaitCtl& ctl, int warp) {
  using Cfg = TcCfg<C, SWIGLU, NX, WTMA>;
  using S = Stage<C>;
  constexpr int SW = Cfg::kSW, SA = Cfg::kSA;
  const int r = threadIdx.x & 127;  // weight row of the tile == TMEM lane
  const uint32_t lane_addr =
      tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + Cfg::kACol0 + 16 * G;
  // SwiGLU: lane 2i decodes gate row n0+i, lane 2i+1 the up row n0+i.
  const int srow = SWIGLU ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;  // row in the W stage
  const KRange kr = k_range<S::SUB>(p);
  bool ok = true;
  // Pairs of sub-steps share one slot pair of 64 columns (PA of them);
  // pairs start at the CTA's first sub-step of each tile, and the last
  // pair of a tile holds one sub-step if the tile has an odd number.
  constexpr int PA = SA / 2;
  int pg = 0;                  // pairs stored so far
  int ks_g = 0, pk_g = 0;
  const DecK K = make_deck();
  for (int tile = kr.tile0; tile < p.tiles && ok; tile += kr.tstep) {
    const int n0 = (tile / p.m_tiles) * Cfg::kOutRows;
    const uint8_t* grow = nullptr;
    bool grow_ok = false;
    if (!WTMA) {
      const int n = SWIGLU ? n0 + (r >> 1) : n0 + r;
      grow_ok = n < p.N;
      const uint8_t* base = (SWIGLU && (r & 1)) ? p.w1 : p.w0;
      grow = base + (grow_ok ? (long long)n * p.row_bytes : 0);
    }
    int ks = kr.ks0;
    for (int pk = kr.pk0; pk < kr.pk1 && ok; ++pk, ++pk_g) {
      uint32_t w[S::WORDS];
      if constexpr (WTMA) {
        const int sp = pk_g % SW;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.w_full[sp], (pk_g / SW) & 1, ctl));
        if (!ok) break;
        const uint4* src = reinterpret_cast<const uint4*>(sm.ws + sp * Cfg::kWStage + srow * S::KPB);
        const bool rok = in_bounds(span_ok((long long)srow * S::KPB, S::KPB, Cfg::kWStage), p.status, kSiteTcWRow);
#pragma unroll
        for (int i = 0; i < S::KPB / 16; ++i) {
          const uint4 v = rok ? src[i] : make_uint4(0, 0, 0, 0);
          w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
        // Released after the sub-steps below have used the words (an
        // arrive right after the loads could let the slot's next TMA fill
        // overtake loads still in flight).
      } else {
        load_stage_global<C>(grow, grow_ok, p.row_bytes, pk, w);
      }
#pragma unroll
      for (int j = 0; j < S::SUB; ++j) {
        if (ks >= kr.ks1) break;
        const int h = (ks - kr.ks0) & 1;
        const int slot = pg % PA;
        uint32_t out[16];
        decode_half<C, G>(w, j, out, K);
        if (h == 0) {
          if (pg >= PA) {
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.a_empty[slot], ((pg / PA) - 1) & 1, ctl));
            if (!ok) break;
          }
          tc_fence_after();
        }
        tmem_st16(lane_addr + slot * 64 + h * 32, out);
        if (h == 1 || ks + 1 == kr.ks1) {
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&sm.a_full[slot]);
          ++pg;
        }
        ++ks;
        ++ks_g;
      }
      if constexpr (WTMA) {
        if (ok) mbar_arrive(&sm.w_empty[pk_g % SW]);
      }
    }
  }
}

// Epilogue role of group E (0 or 1): columns [E*NX/2, (E+1)*NX/2) of D.
//
// SwiGLU: each warp reads all its columns of D first (SiLU(G) x U halves
// them: every lane keeps 16 outputs per 32 columns as packed fp16), then
// releases D to the next tile, and only then stages its [NX/2 m][16 n] slab
// of Y and stores it with one TMA bulk store.  D is held only for the
// tcgen05.ld round trips.
// GEMM: per 32-column chunk, fp16 rounding, group-wide staging and store;
// D is released after the last chunk load.
template <int C, bool SWIGLU, int NX, bool WTMA, int ACT, int HD>
__device__ __forceinline__ void epilogue_role(const TcSmem& sm, const TcParams& p, uint32_t tmem,
                                              const WaitCtl& ctl, const CUtensorMap* tm_y, int warp,
                                              int E) {
  using Cfg = TcCfg<C, SWIGLU, NX, WTMA>;
  const int lane = threadIdx.x & 31;
  const int r = threadIdx.x & 127;
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  const bool leader = r == 0;
  const uint32_t bar_id = 1 + E;
  const int odd = lane & 1;
  uint8_t* ybuf = sm.ys + E * 2 * Cfg::kYStage;
  if constexpr (SWIGLU) {
    constexpr int NCH = (NX / 2) / 32;  // 32-column chunks of this group
    const int q = warp & 3;             // TMEM lane quadrant = outputs n0 + 16q .. n0 + 16q + 15
    uint8_t* slab = sm.ys + (warp - 12) * Cfg::kYSlab;  // [NX/2 m][16 n] fp16
    int lt = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++lt) {
      const int m0 = (tile % p.m_tiles) * NX;
      const int n0 = (tile / p.m_tiles) * Cfg::kOutRows;
      // The accumulator of a tile takes the whole MMA loop: sleep between
      // polls so the decode warps keep the issue slots.
      const bool dok = !*ctl.abort && mbar_wait_idle(sm.d_full, lt & 1, ctl, 128);
      if (!__all_sync(0xffffffffu, dok)) break;
      tc_fence_after();
      const int c_begin = E * (NX / 2);
      uint32_t y2[NCH][8];  // outputs of columns c_begin + 32 ch + 2 jj + odd, two per register
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t v[32];
        tmem_ld32_wait(tmem + lane_base + c_begin + 32 * ch, v);
        // lane 2i holds G, lane 2i+1 holds U of output n0 + 16q + i; the even
        // lane forms the even columns, the odd lane the odd ones
#pragma unroll
        for (int jj = 0; jj < 16; jj += 2) {
          float y[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float a = __uint_as_float(v[2 * (jj + h)]), b = __uint_as_float(v[2 * (jj + h) + 1]);
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
            const float g = odd ? recv : a;
            const float u = odd ? b : recv;
            y[h] = (ACT ? gelu_f(g) : __fdividef(g, 1.0f + __expf(-g))) * u;
          }
          const __half2 hy = __floats2half2_rn(y[0], y[1]);
          y2[ch][jj / 2] = *reinterpret_cast<const uint32_t*>(&hy);
        }
      }
      // Every column of this warp is in registers: D may be reused.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.d_empty);
      if (m0 + c_begin >= p.M || n0 + 16 * q >= p.N) continue;  // uniform: slab entirely padding
      if (lane == 0) bulk_wait_read<0>();  // the previous store has read the slab
      __syncwarp();
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t w = y2[ch][k];
          const int m = 32 * ch + 4 * k + odd;  // columns 2jj + odd for jj = 2k, 2k + 1
          if (!in_bounds(span_ok((long long)m * 32, 3 * 32, Cfg::kYSlab), p.status, kSiteTcStage)) continue;
          __half* row0 = reinterpret_cast<__half*>(slab + m * 32);
          __half* row1 = reinterpret_cast<__half*>(slab + (m + 2) * 32);
          row0[lane >> 1] = __ushort_as_half((unsigned short)(w & 0xFFFFu));
          row1[lane >> 1] = __ushort_as_half((unsigned short)(w >> 16));
        }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (in_bounds(tma_x_ok(n0 + 16 * q, 2) && m0 + c_begin >= 0, p.status, kSiteTcY))
          tma_store_2d(tm_y, slab, n0 + 16 * q, m0 + c_begin);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();
    return;
  }
  int it = 0, lt = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++lt) {
    const int m0 = (tile % p.m_tiles) * NX;
    const int n0 = (tile / p.m_tiles) * Cfg::kOutRows;
    bool dok = false;
    // The accumulator of a tile takes the whole MMA loop: sleep between
    // polls so the decode warps keep the issue slots.
    if (!*ctl.abort) dok = mbar_wait_idle(sm.d_full, lt & 1, ctl, 128);
    // One decision for both epilogue groups (they synchronise below).
    if (named_bar_any(5, 256, !dok || *ctl.abort)) break;
    tc_fence_after();
    const int c_begin = E * (NX / 2), c_end = c_begin + NX / 2;
    for (int c0 = c_begin; c0 < c_end; c0 += 32) {
      uint32_t v[32];
      tmem_ld32_wait(tmem + lane_base + c0, v);
      if (c0 + 32 == c_end) {
        // This warp has read its last D columns of the tile: D may be reused.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.d_empty);
      }
      if (m0 + c0 >= p.M) continue;  // uniform: columns past M are padding
      uint8_t* stg = ybuf + (it & 1) * Cfg::kYStage;  // [32 m][kOutRows n] fp16
      if (it >= 2 && leader) bulk_wait_read<1>();     // the store of chunk it-2 has read stg
      named_bar_sync(bar_id, 128);
      if (!SWIGLU) {
        // lane r holds Y[m0+c0+j][n0+r]; lanes 2i, 2i+1 write (n, n+1) of rows j, j+1
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float a = __uint_as_float(v[j]), b = __uint_as_float(v[j + 1]);
          const float recv = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
          const __half2 h = odd ? __floats2half2_rn(recv, b) : __floats2half2_rn(a, recv);
          if constexpr (HD == 0) {
            const int o = (j + odd) * (Cfg::kOutRows * 2) + (r - odd) * 2;
            if (in_bounds(span_ok(o, 4, Cfg::kYStage), p.status, kSiteTcStage))
              *reinterpret_cast<__half2*>(stg + o) = h;
          } else {  // [head][32 m][HD]: n and n+1 are in the same head
            const int nl = r - odd;
            const int o = ((nl / HD) * 32 + j + odd) * (HD * 2) + (nl % HD) * 2;
            if (in_bounds(span_ok(o, 4, Cfg::kYStage), p.status, kSiteTcStage))
              *reinterpret_cast<__half2*>(stg + o) = h;
          }
        }
      } else {
        // lane 2i holds G, lane 2i+1 holds U of output n0 + r/2; the even lane
        // forms the even columns, the odd lane the odd ones
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const float a = __uint_as_float(v[2 * jj]), b = __uint_as_float(v[2 * jj + 1]);
          const float recv = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
          const float g = odd ? recv : a;
          const float u = odd ? b : recv;
          const float y = __fdividef(g, 1.0f + __expf(-g)) * u;
          const int o = (2 * jj + odd) * (Cfg::kOutRows * 2) + (r >> 1) * 2;
          if (in_bounds(span_ok(o, 2, Cfg::kYStage), p.status, kSiteTcStage))
            *reinterpret_cast<__half*>(stg + o) = __float2half_rn(y);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (leader) {
        if (in_bounds(tma_x_ok(n0, 2) && m0 + c0 >= 0, p.status, kSiteTcY)) {
          if constexpr (HD == 0) tma_store_2d(tm_y, stg, n0, m0 + c0);
          else tma_store_3d(tm_y, stg, 0, m0 + c0, n0 / HD);
        }
        bulk_commit();
      }
      ++it;
    }
  }
  if (leader) bulk_wait_all();
}

// K split.  Slice q of the staged partial tile holds the W = NX / split
// activation columns CTA q of the cluster owns, column-major: column c's
// 128 weight rows are contiguous.  The staging writes of 32 consecutive rows
// are then conflict-free, an owner reads a peer's slice as contiguous runs
// (distributed shared memory requests that touch scattered rows were an
// order of magnitude slower), and 4 consecutive weight rows of one column
// are 4 consecutive outputs of one activation row: one vector store.
__device__ __forceinline__ int split_slot(int r, int c, int W) {   // float index of (row r, column c)
  return ((c / W) * W + (c % W)) * 128 + r;
}

// K split, epilogue warps (group E of two, lane quadrant warp & 3): stage
// this CTA's partial D [128 weight rows][NX activation columns] in its own,
// now idle, X ring.  Returns false if the tile's accumulator never arrived
// (the CTA gave up).
template <int C, bool SWIGLU, int NX, bool WTMA>
__device__ __forceinline__ bool split_stage_role(const TcSmem& sm, const TcParams& p, uint32_t tmem,
                                                 const WaitCtl& ctl, int warp, int E) {
  using Cfg = TcCfg<C, SWIGLU, NX, WTMA>;
  static_assert(128 * NX * 4 <= Cfg::kSX * Cfg::kXStage, "staged partial fits the X ring");
  const int r = threadIdx.x & 127;
  const int W = NX / p.split;
  const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
  const bool dok = !*ctl.abort && mbar_wait_idle(sm.d_full, 0, ctl, 128);
  if (named_bar_any(5, 256, !dok || *ctl.abort)) return false;
  tc_fence_after();
  float* stg = reinterpret_cast<float*>(sm.xs);
#pragma unroll
  for (int ch = 0; ch < NX / 64; ++ch) {
    const int c0 = E * (NX / 2) + 32 * ch;
    uint32_t v[32];
    tmem_ld32_wait(tmem + lane_base + c0, v);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (in_bounds(split_slot(r, c0 + i, W) < Cfg::kSX * Cfg::kXStage / 4, p.status, kSiteTcSplitSlot))
        stg[split_slot(r, c0 + i, W)] = __uint_as_float(v[i]);
  }
  tc_fence_before();
  return true;
}

// K split, after the cluster barrier: CTA `rank` owns activation columns
// [rank W, rank W + W).  The 256 epilogue threads walk its slice a float4
// (4 consecutive weight rows of one column) each, add the slices of the
// cluster's CTAs in rank order and write the outputs: 4 outputs of one
// activation row (GEMM), or 2 (gated: rows 2i, 2i + 1 are gate and up).
template <int C, bool SWIGLU, int NX, bool WTMA, int ACT>
__device__ __forceinline__ void split_reduce_role(const TcSmem& sm, const TcParams& p, const KRange& kr) {
  using Cfg = TcCfg<C, SWIGLU, NX, WTMA>;
  const int t = threadIdx.x - 384;               // 0 .. 255
  const int W = NX / p.split;
  const int m0 = (kr.tile0 % p.m_tiles) * NX + kr.rank * W;
  const int n0 = (kr.tile0 / p.m_tiles) * Cfg::kOutRows;
  const uint32_t slice = smem_u32(reinterpret_cast<float*>(sm.xs) + kr.rank * W * 128);
  for (int e = t; e < 32 * W; e += 256) {
    const int c = e >> 5, r = 4 * (e & 31);      // column c, weight rows r .. r + 3
    const uint32_t a = slice + 4u * (uint32_t)(c * 128 + r);
    if (!in_bounds(span_ok(4ll * ((kr.rank * W + c) * 128 + r), 16, (long long)Cfg::kSX * Cfg::kXStage), p.status,
                   kSiteTcSplitSlot))
      continue;
    float4 f[8];
#pragma unroll
    for (int src = 0; src < 8; ++src)
      if (src < p.split) f[src] = ld_dsmem_f4(mapa_shared(a, (uint32_t)src));
    float4 s4 = f[0];
#pragma unroll
    for (int src = 1; src < 8; ++src)
      if (src < p.split) { s4.x += f[src].x; s4.y += f[src].y; s4.z += f[src].z; s4.w += f[src].w; }
    const int m = m0 + c;
    if (m >= p.M) continue;
    if constexpr (SWIGLU) {
      const int n = n0 + r / 2;                  // 2 outputs, n even
      const float y0 = (ACT ? gelu_f(s4.x) : __fdividef(s4.x, 1.0f + __expf(-s4.x))) * s4.y;
      const float y1 = (ACT ? gelu_f(s4.z) : __fdividef(s4.z, 1.0f + __expf(-s4.z))) * s4.w;
      if (n < p.N && in_bounds(n + 2 <= p.N, p.status, kSiteTcSplitY))
        *reinterpret_cast<__half2*>(p.y + (size_t)m * p.N + n) = __floats2half2_rn(y0, y1);
    } else {
      const int n = n0 + r;                      // 4 outputs; N % 8 == 0: all in or all out
      if (n < p.N && in_bounds(n + 4 <= p.N, p.status, kSiteTcSplitY)) {
        const __half2 h0 = __floats2half2_rn(s4.x, s4.y), h1 = __floats2half2_rn(s4.z, s4.w);
        *reinterpret_cast<uint2*>(p.y + (size_t)m * p.N + n) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
      }
    }
  }
}

// ACT (gated projections): 0 SiLU, 1 GELU.  HD (GEMM): 0 row-major Y, else
// the head dim of the direct-head output.
template <int C, bool SWIGLU, int NX, bool WTMA, int ACT, int HD>
__global__ void __launch_bounds__(640, 1)
    tc_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w0,
                   const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_y,
                   const TcParams p) {
  using Cfg = TcCfg<C, SWIGLU, NX, WTMA>;
  using S = Stage<C>;
  constexpr int SX = Cfg::kSX, SW = Cfg::kSW, SA = Cfg::kSA;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_align<1024>(smem_raw);
  TcSmem sm;
  sm.xs = base;
  sm.ys = sm.xs + SX * Cfg::kXStage;
  sm.ws = sm.ys + Cfg::kYBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.ws + SW * Cfg::kWStage);
  sm.x_full = bars;
  sm.x_empty = sm.x_full + SX;
  sm.w_full = sm.x_empty + SX;
  sm.w_empty = sm.w_full + SW;
  sm.a_full = sm.w_empty + SW;
  sm.a_empty = sm.a_full + SA;
  sm.d_full = sm.a_empty + SA;
  sm.d_empty = sm.d_full + 1;
  sm.drain = sm.d_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const KRange kr = k_range<S::SUB>(p);      // sub-steps and packed stages of this CTA
  bool staged = false;                       // K split: this CTA's partial tile is staged

  if (threadIdx.x == 0) {
    for (int i = 0; i < SX; ++i) { mbar_init(&sm.x_full[i], 1); mbar_init(&sm.x_empty[i], 1); }
    for (int i = 0; i < SW; ++i) { mbar_init(&sm.w_full[i], 1); mbar_init(&sm.w_empty[i], 256); }
    for (int i = 0; i < SA; ++i) { mbar_init(&sm.a_full[i], 256); mbar_init(&sm.a_empty[i], 1); }
    mbar_init(sm.d_full, 1);
    mbar_init(sm.d_empty, 8);  // one arrival per epilogue warp
    mbar_init(sm.drain, 1);
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
      for (int tile = kr.tile0; tile < p.tiles && ok; tile += kr.tstep) {
        const int m0 = (tile % p.m_tiles) * NX;
        for (int ks = kr.ks0; ks < kr.ks1; ++ks) {
          const int sx = xi % SX;
          if (xi >= SX && !mbar_wait_idle(&sm.x_empty[sx], ((xi / SX) - 1) & 1, ctl)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.x_full[sx], Cfg::kXStage);
          if (in_bounds(tma_x_ok(ks * 64, 2) && m0 >= 0, p.status, kSiteTcX))
            tma_load_2d(sm.xs + sx * Cfg::kXStage, &tm_x, &sm.x_full[sx], ks * 64, m0);
          ++xi;
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA exits.
        for (int i = (xi > SX ? xi - SX : 0); i < xi; ++i)
          mbar_wait_drain(&sm.x_full[i % SX], (i / SX) & 1, 100000000ull);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ W producer
    if constexpr (WTMA) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_w0);
        if (SWIGLU) tma_prefetch_desc(&tm_w1);
        int wi = 0;
        bool ok = true;
        for (int tile = kr.tile0; tile < p.tiles && ok; tile += kr.tstep) {
          const int n0 = (tile / p.m_tiles) * Cfg::kOutRows;
          for (int pk = kr.pk0; pk < kr.pk1; ++pk) {
            const int sp = wi % SW;
            if (wi >= SW && !mbar_wait_idle(&sm.w_empty[sp], ((wi / SW) - 1) & 1, ctl)) { ok = false; break; }
            mbar_arrive_expect_tx(&sm.w_full[sp], Cfg::kWStage);
            uint8_t* dst = sm.ws + sp * Cfg::kWStage;
            const int xc = pk * (S::KPB / 2);  // uint16 elements
            if (in_bounds(tma_x_ok(xc, 2) && 2ll * xc < p.row_bytes && n0 >= 0, p.status, kSiteTcW)) {
              tma_load_2d(dst, &tm_w0, &sm.w_full[sp], xc, n0);
              if (SWIGLU) tma_load_2d(dst + 64 * S::KPB, &tm_w1, &sm.w_full[sp], xc, n0);
            }
            ++wi;
          }
        }
        if (!ok) {
          for (int i = (wi > SW ? wi - SW : 0); i < wi; ++i)
            mbar_wait_drain(&sm.w_full[i % SW], (i / SW) & 1, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, NX);
      int ks_g = 0, lt = 0;
      constexpr int PA = SA / 2;
      int pg = 0;
      bool ok = true;
      for (int tile = kr.tile0; tile < p.tiles && ok; tile += kr.tstep, ++lt) {
        // D must have been read out by the epilogue of the previous tile.
        if (lt > 0 && !mbar_wait(sm.d_empty, (lt - 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        for (int ks = kr.ks0; ks < kr.ks1; ks += 2) {
          const int n = kr.ks1 - ks < 2 ? 1 : 2;
          const int slot = pg % PA;
          if (!mbar_wait(&sm.a_full[slot], (pg / PA) & 1, ctl)) { ok = false; break; }
          // With four or more X stages both of the pair are waited for
          // first, so its 8 MMAs issue back to back (5% at the 8B shape);
          // a ring of three stages must not be held two at a time, so
          // there each stage is waited for just before its MMAs.
          if constexpr (SX >= 4) {
            if (!mbar_wait(&sm.x_full[ks_g % SX], (ks_g / SX) & 1, ctl) ||
                (n == 2 && !mbar_wait(&sm.x_full[(ks_g + 1) % SX], ((ks_g + 1) / SX) & 1, ctl))) {
              ok = false;
              break;
            }
          }
          for (int h = 0; h < n; ++h) {
            const int sx = (ks_g + h) % SX;
            if constexpr (SX < 4) {
              if (!mbar_wait(&sm.x_full[sx], ((ks_g + h) / SX) & 1, ctl)) { ok = false; break; }
            }
            tc_fence_after();
            const uint64_t bdesc = sdesc_sw128_kmajor(smem_u32(sm.xs + sx * Cfg::kXStage));
            const uint32_t acol = tmem + Cfg::kACol0 + slot * 64 + h * 32;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_ts_f16(tmem, acol + kk * 8, bdesc + 2 * kk, idesc, (ks + h != kr.ks0) | kk);
            tc_commit(&sm.x_empty[sx]);
          }
          if (!ok) break;
          tc_commit(&sm.a_empty[slot]);
          ks_g += n;
          ++pg;
        }
        if (ok) tc_commit(sm.d_full);
      }
      // Every MMA issued above completes before the CTA frees TMEM.
      tc_commit(sm.drain);
      mbar_wait_drain(sm.drain, 0, 200000000ull);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    decode_role<C, SWIGLU, NX, WTMA, 0>(sm, p, tmem, ctl, warp);
  } else if (warp >= 8 && warp < 12) {
    decode_role<C, SWIGLU, NX, WTMA, 1>(sm, p, tmem, ctl, warp);
  } else if (warp >= 12) {
    if constexpr (NX <= 128 && HD == 0 && WTMA) {
      if (p.split > 1) staged = split_stage_role<C, SWIGLU, NX, WTMA>(sm, p, tmem, ctl, warp, (warp - 12) >> 2);
      else epilogue_role<C, SWIGLU, NX, WTMA, ACT, HD>(sm, p, tmem, ctl, &tm_y, warp, (warp - 12) >> 2);
    } else {
      epilogue_role<C, SWIGLU, NX, WTMA, ACT, HD>(sm, p, tmem, ctl, &tm_y, warp, (warp - 12) >> 2);
    }
  }

  if constexpr (NX <= 128 && HD == 0 && WTMA) {
    if (p.split > 1) {
      // Every thread of the cluster: all partial tiles are staged; then each
      // CTA reduces its columns; no CTA leaves while a peer may still read
      // its staged partial.
      cluster_sync_all();
      if (warp >= 12 && staged) split_reduce_role<C, SWIGLU, NX, WTMA, ACT>(sm, p, kr);
      cluster_sync_all();
    }
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
