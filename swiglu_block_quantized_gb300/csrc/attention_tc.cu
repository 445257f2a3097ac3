// attention_tc.cu -- softmax attention over an fp16 KV cache on the tcgen05
// tensor cores, for prefill-sized calls (more than 16 rows per KV head, no
// key split).  Same contract as attention.cu, which keeps decode-sized calls
// and the Q8_0 cache.
//
// Pages: "v0.1 vs v0.2 comparison" 2.3 (Brick 4, FlashAttention with an
// online softmax) and "Releases" v0.3.0 (GQA, causal mask with a sequence
// offset, head dims 64 and 128).
//
// One CTA takes 128 rows of one KV head, 128 / G consecutive queries of each
// of its G query heads (row = g (128 / G) + i - q0, head-major, so that each
// head's rows arrive as one TMA box), and walks the key tiles of 128 keys
// its rows can see:
//   S_j = Q K_j^T          tcgen05 MMA, both operands K-major in 128-byte
//                          swizzled shared memory, S_j in TMEM (fp32).
//   softmax warps          two threads per row, 64 keys each: read S_j,
//                          form the running row max m (partial maxima
//                          exchanged), P_j = exp2(S_j scale log2 e - m)
//                          rounded to fp16 and written back over the
//                          thread's own S_j columns in TMEM (keys 64 h ..
//                          64 h + 63 at columns 64 h .. 64 h + 31), the
//                          running sums and the rescale factor alpha_j of
//                          the previous accumulation.
//   O_j = P_j V_j          tcgen05 MMA with P_j as the TMEM operand and the
//                          V_j tile as it lies in the cache ([key][D], the
//                          N-major B operand: D contiguous) in shared
//                          memory, into a fresh TMEM buffer per tile.
//   correction warps       thread = row, half of D each: O = alpha_j O + O_j
//                          in registers; at the end O / l is written.
// Fresh per-tile O buffers keep the online-softmax rescale out of the MMA's
// way: no accumulator is rescaled while the tensor core may still add to it.
// Two S/P and two O buffers (TMEM: 2 x 128 + 2 x D columns), three K and
// two V stages let S_{j+1} and P_j V_j run while the softmax of tile j+1 and
// the correction of tile j proceed.
//
// Warps: 0 MMA (one lane) and TMEM owner; 1 and 2 TMA producers of the K and
// the V tiles (one lane each; 3-D tensor maps [Hkv][T][D], so keys past T
// arrive as zeros); 3 the TMA producer of Q (one box per head and 64-wide
// panel from a 3-D map [H][M][D], rows past M zero); 4-11 softmax, two threads
// per row (warps w and w + 4: keys 0-63 and 64-127 of each tile), which
// exchange their partial row maxima through shared memory; 12-19 correction
// (two groups of four, D/2 columns each).  Every wait is bounded in time; on
// expiry the CTA records the failure in the status word and returns.
#include "codec.cuh"
#include "launch.h"

namespace m4q {

namespace {

constexpr int kTR = 128;   // rows per CTA
constexpr int kTK = 128;   // keys per tile

template <int D>
struct TaCfg {
  static constexpr int kQBytes = kTR * D * 2;        // Q: D / 64 panels of [128 rows][128 B]
  static constexpr int kKBytes = kTK * D * 2;        // K: D / 64 panels of [128 keys][128 B]
  static constexpr int kVBytes = kTK * D * 2;        // V: the same layout
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kThreads = 640;
  static constexpr int kAlphaBytes = 4 * kTR * 4;    // alpha ring of 4 tiles
  static constexpr int kBars = 1 + 3 + 3 + 2 + 2 + 2 + 2 + 2 + 4 + 2 + 2 + 1 + 1;
  static constexpr int kSmem = 1024 + kQBytes + kKStages * kKBytes + kVStages * kVBytes + kAlphaBytes +
                               2 * kTR * 4 + 4 * kTR * 4 + kBars * 8 + 16;
  static constexpr uint32_t kOCol = 256;             // O buffers after the two S/P buffers
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(kOCol + 2 * D <= 512, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kQBytes % 1024 == 0 && kKBytes % 1024 == 0 && kVBytes % 1024 == 0, "swizzle atoms");
};

__device__ __forceinline__ void mma_ss_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane, waited for.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// OR of `pred` over the `count` threads of named barrier `id` (all of them
// arrive; every one gets the result).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
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

// 3-D tile load (x = d, y = row, z = head) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Shared-memory descriptor of an N-major (MN-major) operand in the 128-byte
// swizzled layout: rows of 64 N-elements (128 B) for consecutive k, 8-row
// atoms of 1024 B along k (stride byte offset) and panels of 64 N-elements
// `panel_bytes` apart (leading byte offset).  Checked on a one-hot product.
__device__ __forceinline__ uint64_t sdesc_sw128_nmajor(uint32_t saddr, uint32_t panel_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((panel_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(640, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using Cfg = TaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* qs = smem_align<1024>(smem_raw);
  uint8_t* kst = qs + Cfg::kQBytes;                                 // K stages
  uint8_t* vst = kst + Cfg::kKStages * Cfg::kKBytes;                // V stages
  float* alpha = reinterpret_cast<float*>(vst + Cfg::kVStages * Cfg::kVBytes);   // [4][128]
  float* lfin = alpha + 4 * kTR;                                    // [2][128] partial row sums
  float* pmax = lfin + 2 * kTR;                                     // [2 tiles][2][128] partial row maxima
  uint64_t* q_full = reinterpret_cast<uint64_t*>(pmax + 4 * kTR);
  uint64_t* k_full = q_full + 1;      // [3] producer: K_j in stage j % 3
  uint64_t* k_empty = k_full + 3;     // [3] MMA: S_j done with stage j % 3
  uint64_t* v_full = k_empty + 3;     // [2] producer: V_j in stage j % 2
  uint64_t* v_empty = v_full + 2;     // [2] MMA: P_j V_j done with stage j % 2
  uint64_t* s_full = v_empty + 2;     // [2] MMA: S_j in TMEM buffer j % 2
  uint64_t* s_free = s_full + 2;      // [2] MMA: P_j read from buffer j % 2
  uint64_t* p_full = s_free + 2;      // [2] softmax: P_j written
  uint64_t* a_rdy = p_full + 2;       // [4] softmax: alpha_j written
  uint64_t* o_full = a_rdy + 4;       // [2] MMA: O_j in TMEM
  uint64_t* o_free = o_full + 2;      // [2] correction: O_j consumed
  uint64_t* l_rdy = o_free + 2;       // softmax: final row sums written
  uint64_t* drain = l_rdy + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rt = (int)gridDim.x - 1 - (int)blockIdx.x, hk = blockIdx.y;   // heaviest row tiles first
  const int QPT = kTR / p.G;             // queries per tile (G divides 128)
  const int q0 = rt * QPT;
  // keys [0, kend) are visible to some row of this tile
  int kend = p.T;
  if (CAUSAL) {
    const long long vis = (long long)p.q_offset + min(p.M, q0 + QPT);
    if (vis < kend) kend = (int)vis;
  }
  const int nk = (kend + kTK - 1) / kTK;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 8);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&a_rdy[i], 4);
    mbar_init(l_rdy, 8);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, 2000000000ull};

  if (warp == 0) {
    // ------------------------------------------------------------ MMA
    if (lane == 0 && nk > 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32(128, kTK);
      constexpr uint32_t idesc_o = idesc_f16_f32(128, D) | (1u << 16);   // B (V) N-major
      bool ok = mbar_wait(q_full, 0, ctl);
      auto issue_s = [&](int j) {
        const int st = j & 1, sk = j % 3;
        ok = ok && mbar_wait(&k_full[sk], (j / 3) & 1, ctl);
        if (j >= 2) ok = ok && mbar_wait(&s_free[st], ((j >> 1) - 1) & 1, ctl);
        if (!ok) return;
        tc_fence_after();
        const uint8_t* ks = kst + sk * Cfg::kKBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int panel = kk >> 2;
          const uint64_t a = sdesc_sw128_kmajor(smem_u32(qs + panel * (kTR * 128))) + 2 * (kk & 3);
          const uint64_t b = sdesc_sw128_kmajor(smem_u32(ks + panel * (kTK * 128))) + 2 * (kk & 3);
          mma_ss_f16(tmem + 128 * st, a, b, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[st]);
        tc_commit(&k_empty[sk]);
      };
      auto issue_pv = [&](int j) {
        const int st = j & 1;
        ok = ok && mbar_wait(&v_full[st], (j >> 1) & 1, ctl);
        ok = ok && mbar_wait(&p_full[st], (j >> 1) & 1, ctl);
        if (j >= 2) ok = ok && mbar_wait(&o_free[st], ((j >> 1) - 1) & 1, ctl);
        if (!ok) return;
        tc_fence_after();
        const uint8_t* vs = vst + st * Cfg::kVBytes;
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          // keys 16 kk .. 16 kk + 15: two 8-key atoms, 2 KB into each panel
          const uint64_t b = sdesc_sw128_nmajor(smem_u32(vs + kk * 2048), kTK * 128);
          // P keys 16 kk .. 16 kk + 15: columns 64 (kk / 4) + 8 (kk % 4) of the S/P buffer
          tc_mma_ts_f16(tmem + Cfg::kOCol + D * st, tmem + 128 * st + 64 * (kk >> 2) + 8 * (kk & 3), b, idesc_o,
                        kk > 0 ? 1u : 0u);
        }
        tc_commit(&o_full[st]);
        tc_commit(&v_empty[st]);
        tc_commit(&s_free[st]);
      };
      issue_s(0);
      for (int j = 1; j < nk && ok; ++j) {
        issue_s(j);
        issue_pv(j - 1);
      }
      issue_pv(nk - 1);
      // Every MMA issued above completes before the CTA frees TMEM.
      tc_commit(drain);
      mbar_wait_drain(drain, 0, 200000000ull);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ loaders
    if (warp == 3 && lane == 0) {
      // Q: rows g QPT .. g QPT + QPT - 1 of each 64-wide panel from head
      // hk G + g, queries q0 .. (boxes start on 1024-byte swizzle atoms:
      // QPT is a multiple of 8)
      tma_prefetch_desc(&tm_q);
      mbar_arrive_expect_tx(q_full, Cfg::kQBytes);
      for (int g = 0; g < p.G; ++g)
#pragma unroll
        for (int pn = 0; pn < D / 64; ++pn)
          if (in_bounds(q0 >= 0 && hk * p.G + g < p.H, p.status, kSiteAttnQ))
            tma_load_3d(qs + pn * (kTR * 128) + g * QPT * 128, &tm_q, q_full, 64 * pn, q0, hk * p.G + g);
    }
    if ((warp == 1 || warp == 2) && lane == 0) {
      // warp 1: K_j into stage j % 3 after S_{j-3}; warp 2: V_j into stage
      // j % 2 after P_{j-2} V_{j-2}.  D / 64 boxes of [128 keys][64 d] each.
      const bool isk = warp == 1;
      const CUtensorMap* map = isk ? &tm_k : &tm_v;
      const int ns = isk ? 3 : 2;
      uint64_t* full = isk ? k_full : v_full;
      uint64_t* empty = isk ? k_empty : v_empty;
      uint8_t* ring = isk ? kst : vst;
      tma_prefetch_desc(map);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < nk && ok; ++j, ++issued) {
        const int sl = j % ns, k0 = j * kTK;
        if (j >= ns && !mbar_wait_idle(&empty[sl], ((j / ns) - 1) & 1, ctl, 128)) { ok = false; break; }
        mbar_arrive_expect_tx(&full[sl], Cfg::kKBytes);
#pragma unroll
        for (int pn = 0; pn < D / 64; ++pn)
          if (in_bounds(k0 >= 0, p.status, kSiteAttnKV))
            tma_load_3d(ring + sl * Cfg::kKBytes + pn * (kTK * 128), map, &full[sl], 64 * pn, k0, hk);
      }
      if (!ok) {
        for (int i = (issued > ns ? issued - ns : 0); i < issued; ++i)
          mbar_wait_drain(&full[i % ns], (i / ns) & 1, 100000000ull);
      }
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ softmax
    const int half = (warp - 4) >> 2;   // keys [64 half, 64 half + 64) of each tile
    const int r = 32 * (warp & 3) + lane;
    const int i = q0 + r % QPT;          // query of this row
    const bool valid = i < p.M;
    // last key this row sees (-1: none), one 32-bit bound for validity, the
    // causal limit and T together
    long long lastl = CAUSAL ? (long long)p.q_offset + i : (long long)p.T - 1;
    if (lastl > (long long)p.T - 1) lastl = p.T - 1;
    const int lastk = valid ? (int)lastl : -1;
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t bar_id = 1 + (warp & 3);   // the two warps of these rows
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nk && ok; ++j) {
      const int st = j & 1;
      // one decision for both warps of these rows, which meet at a named
      // barrier below (it has no time limit)
      const bool got = mbar_wait(&s_full[st], (j >> 1) & 1, ctl);
      ok = !bar_red_or(7 + (warp & 3), 64, !got);
      if (!ok) break;
      tc_fence_after();
      const uint32_t scol = tmem + lanes + 128 * st + 64 * half;
      const int kbase = j * kTK + 64 * half;
      const float sc = p.scale_log2;
      // keys e <= cut of chunk c are visible; a chunk with cut >= 31 needs
      // no mask (the warp agrees on it, so the loops below stay uniform)
      const bool full = __all_sync(0xffffffffu, lastk - (kbase + 32) >= 31);
      // row maximum of sc * s over the visible keys: the max of s when
      // sc >= 0, the min when sc < 0 (scaled after)
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32_wait(scol + 32 * c, v);
        const int cut = lastk - (kbase + 32 * c);
        float t = sc >= 0.f ? -INFINITY : INFINITY;
        if (full) {
          if (sc >= 0.f) {
#pragma unroll
            for (int e = 0; e < 32; ++e) t = fmaxf(t, __uint_as_float(v[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) t = fminf(t, __uint_as_float(v[e]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e <= cut) t = sc >= 0.f ? fmaxf(t, __uint_as_float(v[e])) : fminf(t, __uint_as_float(v[e]));
        }
        if (t != INFINITY && t != -INFINITY) mx = fmaxf(mx, t * sc);
      }
      // the row maximum over both halves (buffers by tile parity: a thread
      // rewrites its slot two tiles later, after its partner has passed the
      // next tile's barrier, hence after it has read this value)
      float* pm = pmax + (j & 1) * (2 * kTR);
      pm[half * kTR + r] = mx;
      named_bar_sync(bar_id, 64);
      mx = fmaxf(mx, pm[(half ^ 1) * kTR + r]);
      const float mnew = fmaxf(m, mx);
      const float muse = mnew == -INFINITY ? 0.f : mnew;
      const float a = ex2(m - muse);   // 0 while m = -inf
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32_wait(scol + 32 * c, v);
        const int cut = lastk - (kbase + 32 * c);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0 = ex2(fmaf(__uint_as_float(v[e]), sc, -muse));
          float p1 = ex2(fmaf(__uint_as_float(v[e + 1]), sc, -muse));
          if (!full) {
            p0 = e <= cut ? p0 : 0.f;
            p1 = e + 1 <= cut ? p1 : 0.f;
          }
          sum0 += p0;
          sum1 += p1;
          const __half2 h = __floats2half2_rn(p0, p1);
          w[e >> 1] = *reinterpret_cast<const uint32_t*>(&h);
        }
        // P keys 64 half + 32 c .. + 31 go to columns 64 half + 16 c, inside
        // this thread's own S columns and behind its reads: chunk 0 of S
        // (columns 64 half .. + 31) is read before P chunk 0 overwrites
        // its first half, and P chunk 1 lands on the rest of it
        tmem_st16(scol + 16 * c, w);
      }
      const float sum = sum0 + sum1;
      l = l * a + sum;
      m = mnew;
      if (half == 0) alpha[(j & 3) * kTR + r] = a;
      tmem_wait_st();
      tc_fence_before();
      if (half == 0) mbar_arrive_warp(&a_rdy[j & 3]);
      mbar_arrive_warp(&p_full[st]);
    }
    lfin[half * kTR + r] = l;
    mbar_arrive_warp(l_rdy);
  } else {
    // ------------------------------------------------------------ correction
    const int e = (warp - 12) >> 2;    // columns [e D / 2, (e + 1) D / 2) of O
    const int r = 32 * (warp & 3) + lane;
    const int i = q0 + r % QPT, h = hk * p.G + r / QPT;   // query and head of this row
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    constexpr int HC = D / 2;
    float o[HC];
#pragma unroll
    for (int c = 0; c < HC; ++c) o[c] = 0.f;
    bool ok = true;
    for (int j = 0; j < nk && ok; ++j) {
      const int st = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_idle(&a_rdy[j & 3], (j >> 2) & 1, ctl, 64) &&
                                       mbar_wait_idle(&o_full[st], (j >> 1) & 1, ctl, 64));
      if (!ok) break;
      tc_fence_after();
      const float a = alpha[(j & 3) * kTR + r];
#pragma unroll
      for (int c = 0; c < HC / 16; ++c) {
        uint32_t v[16];
        tmem_ld16_wait(tmem + lanes + Cfg::kOCol + D * st + e * HC + 16 * c, v);
#pragma unroll
        for (int q = 0; q < 16; ++q) o[16 * c + q] = o[16 * c + q] * a + __uint_as_float(v[q]);
      }
      tc_fence_before();
      mbar_arrive_warp(&o_free[st]);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait_idle(l_rdy, 0, ctl, 64)) && i < p.M) {
      const float l = lfin[r] + lfin[kTR + r];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (in_bounds(h < p.H, p.status, kSiteAttnO)) {
        __half* orow = p.o + (long long)i * p.H * D + (long long)h * D + e * HC;
#pragma unroll
        for (int c = 0; c < HC; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __half2 hh = __floats2half2_rn(o[c + 2 * q] * inv, o[c + 2 * q + 1] * inv);
            w[q] = *reinterpret_cast<const uint32_t*>(&hh);
          }
          *reinterpret_cast<uint4*>(orow + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_tc(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                      cudaStream_t s) {
  using Cfg = TaCfg<D>;
  auto kern = attn_tc_kernel<D, CAUSAL>;
  std::atomic<unsigned long long>& configured = attr_flag<std::integer_sequence<int, 4, D, CAUSAL>>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const int qpt = kTR / p.G;
  const dim3 grid((unsigned)((p.M + qpt - 1) / qpt), (unsigned)p.Hkv, 1);
  kern<<<grid, Cfg::kThreads, Cfg::kSmem, s>>>(tm_q, tm_k, tm_v, p);
  return cudaGetLastError();
}

}  // namespace

// fp16 KV cache, more than 16 rows per KV head, one key split, a group size
// that divides 128 rows into whole swizzle atoms per head (G <= 16).
bool attention_tc_applies(const AttnParams& p, bool q8) {
  return !q8 && p.M * p.G > 16 && p.nsplit == 1 && (p.D == 64 || p.D == 128) && (p.kv_row_bytes % 16) == 0 &&
         p.G <= 16 && kTR % p.G == 0;
}

cudaError_t launch_attention_tc(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, cudaStream_t s) {
  if (p.D == 64)
    return p.causal ? launch_tc<64, true>(p, tm_q, tm_k, tm_v, s) : launch_tc<64, false>(p, tm_q, tm_k, tm_v, s);
  return p.causal ? launch_tc<128, true>(p, tm_q, tm_k, tm_v, s) : launch_tc<128, false>(p, tm_q, tm_k, tm_v, s);
}

}  // namespace m4q
