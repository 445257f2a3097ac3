// attention_tc.cu -- softmax attention over an fp16 KV cache on the tcgen05
// tensor cores, for prefill-sized calls (more than 16 rows per KV head) that
// an estimate of the time gives to it; a Q8_0 cache comes here after
// kv_q8_stage_kernel (below) has decoded it to fp16 in the caller's
// workspace.  Same contract as attention.cu, which keeps decode-sized calls
// and the calls the estimate gives to its key split.
//
// Pages: "v0.1 vs v0.2 comparison" 2.3 (Brick 4, FlashAttention with an
// online softmax) and "Releases" v0.3.0 (GQA, causal mask with a sequence
// offset, head dims 64 and 128).
//
// The work items are (128 rows of one KV head: 128 / G consecutive queries
// of each of its G query heads, row = g (128 / G) + i - q0, head-major, so
// that each head's rows arrive as one TMA box).  One persistent CTA per SM
// walks its items one after another, and within an item the key tiles of
// 128 keys its rows can see; the pipeline runs on across items (the next
// item's Q loads once the scores of the last are done, its first P V waits
// until the last item's O is read out):
//   S_j = Q K_j^T          tcgen05 MMA, both operands K-major in 128-byte
//                          swizzled shared memory, S_j in TMEM (fp32), in
//                          buffer j % 3.
//   softmax warps          two teams (tiles j even and odd) of two
//                          threads per row (keys 0-63 and 64-127): each
//                          forms its half's extreme raw score (max, or min
//                          for a negative scale), the pair exchanges them
//                          (shared memory and a named barrier), giving
//                          mu_j; the reference m_j = m_{j-1} unless
//                          mu_j > m_{j-1} + 8, then mu_j (m_{j-1} comes from
//                          the other team through shared memory);
//                          P_j = exp2(S_j scale log2 e - m_j) <= 2^8,
//                          rounded to fp16 and written back over the
//                          thread's own S_j columns (keys 64 h + k at
//                          column 64 h + k / 2); the thread's row sum l,
//                          kept relative to the last reference it used.
//   O += P_j V_j           tcgen05 MMA with P_j as the TMEM operand and the
//                          V_j tile as it lies in the cache ([key][D], the
//                          N-major B operand: D contiguous) in shared
//                          memory; O stays in TMEM for the whole walk.
//   rescale                when m_j > m_{j-1}, the threads of tile j scale
//                          their half of O by 2^(m_{j-1} - m_j) in TMEM
//                          after P_{j-1} V_{j-1} and before they publish P_j
//                          (rare: the reference moves only when a row
//                          maximum jumps by 2^8).
//   epilogue               O / l, l = the four threads' sums of a row
//                          brought to the last reference, written as fp16.
// The lazily raised reference keeps O accumulating in the tensor core's
// TMEM with no per-tile read-out, and frees the softmax of tile j+1 from the
// exponentials of tile j: only the reference, known right after the max,
// passes from one team to the next.  Three S/P buffers and one O (TMEM:
// 3 x 128 + D columns), three K and two V stages: S_{j+3} needs only
// P_j V_j done, so the scores run ahead of the softmax.  The score and the
// P V MMAs come from two issuing threads, each waiting only for its own
// operands: one thread's waits and issue overlap the other thread's MMAs in
// the tensor pipe (a tcgen05.mma is accepted about once per MMA duration, so
// a single issuer's waits leave the pipe idle).
//
// Warps: 0 the score-MMA issuer (one lane) and TMEM owner; 1 the TMA
// producer of each item's Q (one box per head and 64-wide panel from a 3-D
// map [H][M][D], rows past M zero) and of the K tiles, 2 of the V tiles (one
// lane each; 3-D tensor maps [Hkv][T][D], so keys past T arrive as zeros);
// 3 the P V issuer; 4-11 and 12-19 the softmax teams of the even and the
// odd tiles (warps w and w + 4 of a team: the two halves of the same rows),
// which also write each item's output (a quarter of D each).  Items go out
// heaviest first (every head's last row tile, then the one before, ...) in
// a zigzag over the CTAs.  Every wait is bounded in time; on
// expiry the CTA records the failure in the status word and returns, and
// the two halves of a row leave their loop together (a named barrier has no
// time limit).
#include "codec.cuh"
#include "launch.h"

namespace m4q {

namespace {

constexpr int kTR = 128;   // rows per work item
constexpr int kTK = 128;   // keys per tile
constexpr float kLazy = 8.f;   // reference kept while the row max stays within 2^8 of it

template <int D>
struct TaCfg {
  static constexpr int kQBytes = kTR * D * 2;        // Q: D / 64 panels of [128 rows][128 B]
  static constexpr int kKBytes = kTK * D * 2;        // K: D / 64 panels of [128 keys][128 B]
  static constexpr int kVBytes = kTK * D * 2;        // V: the same layout
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kThreads = 640;
  static constexpr int kMlBytes = 4 * kTR * 4 + 8 * kTR * 8 + 8 * kTR * 4;   // references, final (l, m), partial maxima
  static constexpr int kBars = 2 + 3 + 3 + 2 + 2 + 3 + 3 + 3 + 2 + 1 + 1 + 1 + 1;
  static constexpr int kSmem = 1024 + kQBytes + kKStages * kKBytes + kVStages * kVBytes + kMlBytes + kBars * 8 + 16;
  static constexpr uint32_t kOCol = 384;             // O after the three S/P buffers
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(kOCol + D <= 512, "TMEM budget");
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

// 16 consecutive 32-bit TMEM columns of this thread's lane, not waited for:
// v is valid after tmem_wait_ld_tied(v).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
               : "r"(taddr)
               : "memory");
}

// Wait for this thread's TMEM loads; v passes through the wait, so that no
// use of it is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld_tied(uint32_t (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]) : : "memory");
}

// 64 consecutive 32-bit TMEM columns of this thread's lane, waited for.
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, uint32_t (&v)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
               "tcgen05.wait::ld.sync.aligned;"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
               : "r"(taddr)
               : "memory");
}

// Store 8 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// OR of `pred` over the `count` threads of named barrier `id` (all of them
// arrive; every one gets the result).  A named barrier has no time limit,
// so every decision to leave a loop that holds one is taken through it.
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

// Largest (hi) or smallest (!hi) of v[e] over e <= cut (all 32 when cut >=
// 31), four independent chains; +-inf when none.
__device__ __forceinline__ float extreme32(const uint32_t* v, int cut, bool hi) {
  const float init = hi ? -INFINITY : INFINITY;
  float t[4] = {init, init, init, init};
  if (cut >= 31) {
    if (hi) {
#pragma unroll
      for (int e = 0; e < 32; ++e) t[e & 3] = fmaxf(t[e & 3], __uint_as_float(v[e]));
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) t[e & 3] = fminf(t[e & 3], __uint_as_float(v[e]));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float x = e <= cut ? __uint_as_float(v[e]) : init;
      t[e & 3] = hi ? fmaxf(t[e & 3], x) : fminf(t[e & 3], x);
    }
  }
  return hi ? fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3])) : fminf(fminf(t[0], t[1]), fminf(t[2], t[3]));
}

// Two fp32 values in one 64-bit register, for the packed f32x2 FMA and add
// (one instruction for both).
__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long x, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// Work items: (row tile, KV head) in decreasing order of key count (the
// row tile rt of every head, then rt - 1, ...), handed to the persistent
// CTAs in a zigzag: CTA b takes items b, 2 G - 1 - b, 2 G + b, ..., so that
// the heavy and the light items of successive rounds even out.
struct TaItem {
  int q0, hk, nk;
};

__device__ __forceinline__ int ta_item_index(int round, int G) {
  return round * G + ((round & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

template <bool CAUSAL>
__device__ __forceinline__ TaItem ta_item(const AttnParams& p, int n, int QPT, int rtiles) {
  TaItem it;
  it.hk = n % p.Hkv;
  it.q0 = (rtiles - 1 - n / p.Hkv) * QPT;
  // keys [0, kend) are visible to some row of the tile (at least key 0)
  int kend = p.T;
  if (CAUSAL) {
    const long long vis = (long long)p.q_offset + min(p.M, it.q0 + QPT);
    if (vis < kend) kend = (int)vis;
  }
  it.nk = (kend + kTK - 1) / kTK;
  return it;
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
  float* mref = reinterpret_cast<float*>(vst + Cfg::kVStages * Cfg::kVBytes);   // [4][128] reference of tile g
  float2* lfin = reinterpret_cast<float2*>(mref + 4 * kTR);         // [item parity][team][half][128] final (l, m)
  float* pmx = reinterpret_cast<float*>(lfin + 8 * kTR);            // [team][tile parity][half][128] partial extremes
  uint64_t* q_full = reinterpret_cast<uint64_t*>(pmx + 8 * kTR);   // K producer: Q of item w
  uint64_t* q_empty = q_full + 1;     // score issuer: the scores of item w are done with Q
  uint64_t* k_full = q_empty + 1;     // [3] producer: K of tile g in stage g % 3
  uint64_t* k_empty = k_full + 3;     // [3] MMA: S_g done with stage g % 3
  uint64_t* v_full = k_empty + 3;     // [2] producer: V of tile g in stage g % 2
  uint64_t* v_empty = v_full + 2;     // [2] MMA: P_g V_g done with stage g % 2
  uint64_t* s_full = v_empty + 2;     // [3] MMA: S_g in TMEM buffer g % 3
  uint64_t* s_free = s_full + 3;      // [3] MMA: P_g read from buffer g % 3
  uint64_t* p_full = s_free + 3;      // [3] softmax: P_g written
  uint64_t* r_rdy = p_full + 3;       // [2] softmax: reference of tile g written (barrier g % 2)
  uint64_t* l_rdy = r_rdy + 2;        // softmax: final (l, m) of item w written by every thread
  uint64_t* o_done = l_rdy + 1;       // P V issuer: every P V of item w done
  uint64_t* o_free = o_done + 1;      // softmax: O of item w read out
  uint64_t* drain = o_free + 1;       // both issuers: every MMA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int QPT = kTR / p.G;             // queries per tile (G divides 128)
  const int rtiles = (p.M + QPT - 1) / QPT;
  const int NI = rtiles * p.Hkv;         // work items
  const int G = (int)gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 1);
      mbar_init(&p_full[i], 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(&r_rdy[0], 4);
    mbar_init(&r_rdy[1], 4);
    mbar_init(l_rdy, 16);
    mbar_init(o_done, 1);
    mbar_init(o_free, 16);
    mbar_init(drain, 2);   // one commit from each MMA issuer
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
  pdl_launch_dependents();
  pdl_wait();   // every global access below comes after the previous kernel

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing threads: warp 0 the score MMAs, warp 3 the P V MMAs.  Each
    // waits only for its own operands, so the waits and the issue of one
    // overlap the other's MMAs in the tensor pipe.  Tiles are numbered g
    // across the items of this CTA; every ring follows g.
    if (lane == 0) {
      if (warp == 0) {
        // S_g = Q K_g^T into buffer g % 3 once K_g has landed and P_{g-3}
        // V_{g-3} has read that buffer
        constexpr uint32_t idesc_s = idesc_f16_f32(128, kTK);
        // Operand descriptors, formed once: a descriptor is (address / 16)
        // in its low 14 bits, so that of a later slice or stage is a fixed
        // offset from the first.
        const uint64_t qd = sdesc_sw128_kmajor(smem_u32(qs));
        const uint64_t kd = sdesc_sw128_kmajor(smem_u32(kst));
        bool ok = true;
        int g = 0;
        for (int w = 0; ok; ++w) {
          const int n = ta_item_index(w, G);
          if (n >= NI) break;
          const TaItem it = ta_item<CAUSAL>(p, n, QPT, rtiles);
          ok = mbar_wait(q_full, w & 1, ctl);
          for (int j = 0; j < it.nk && ok; ++j, ++g) {
            const int sb = g % 3;   // S buffer and K stage
            ok = mbar_wait(&k_full[sb], (g / 3) & 1, ctl);
            if (g >= 3) ok = ok && mbar_wait(&s_free[sb], ((g / 3) - 1) & 1, ctl);
            if (!ok) break;
            tc_fence_after();
            const uint64_t kds = kd + (uint64_t)(sb * (Cfg::kKBytes >> 4));
            const uint32_t dst = tmem + 128 * sb;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // 16-element slice kk: panel kk / 4, 32 bytes per slice inside it
              constexpr int kPanelA = kTR * 128 >> 4, kPanelB = kTK * 128 >> 4;
              const uint32_t off_a = (kk >> 2) * kPanelA + 2 * (kk & 3);
              const uint32_t off_b = (kk >> 2) * kPanelB + 2 * (kk & 3);
              mma_ss_f16(dst, qd + off_a, kds + off_b, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[sb]);
            tc_commit(&k_empty[sb]);
          }
          if (ok) tc_commit(q_empty);   // Q may be replaced once these MMAs are done
        }
      } else {
        // O (+)= P_g V_g once P_g is written and V_g has landed; the first
        // tile of an item also waits until the previous item's O is read
        // out (a rescale of O, when tile g raised the reference, precedes
        // P_g)
        constexpr uint32_t idesc_o = idesc_f16_f32(128, D) | (1u << 16);   // B (V) N-major
        const uint64_t vd = sdesc_sw128_nmajor(smem_u32(vst), kTK * 128);
        bool ok = true;
        int g = 0;
        for (int w = 0; ok; ++w) {
          const int n = ta_item_index(w, G);
          if (n >= NI) break;
          const TaItem it = ta_item<CAUSAL>(p, n, QPT, rtiles);
          for (int j = 0; j < it.nk && ok; ++j, ++g) {
            const int st = g & 1, sb = g % 3;   // V stage and S/P buffer
            ok = mbar_wait(&v_full[st], (g >> 1) & 1, ctl) && mbar_wait(&p_full[sb], (g / 3) & 1, ctl);
            if (j == 0 && w >= 1) ok = ok && mbar_wait(o_free, (w - 1) & 1, ctl);
            if (!ok) break;
            tc_fence_after();
            const uint64_t vds = vd + (uint64_t)(st * (Cfg::kVBytes >> 4));
            const uint32_t dst = tmem + Cfg::kOCol, pcol = tmem + 128 * sb;
#pragma unroll
            for (int kk = 0; kk < kTK / 16; ++kk) {
              // keys 16 kk .. 16 kk + 15: two 8-key atoms, 2 KB into each V
              // panel; their P at columns 64 (kk / 4) + 8 (kk % 4) of the S/P
              // buffer (each half of the keys written by its own threads)
              tc_mma_ts_f16(dst, pcol + 64 * (kk >> 2) + 8 * (kk & 3), vds + (uint32_t)(kk * (2048 >> 4)), idesc_o,
                            (j | kk) > 0 ? 1u : 0u);
            }
            tc_commit(&v_empty[st]);
            tc_commit(&s_free[sb]);
          }
          if (ok) tc_commit(o_done);   // O of item w complete once these MMAs are done
        }
      }
      // Every MMA of both issuers completes before the CTA frees TMEM.
      tc_commit(drain);
      mbar_wait_drain(drain, 0, 200000000ull);
    }
    __syncwarp();
  } else if (warp < 3) {
    // ------------------------------------------------------------ loaders
    if (lane == 0) {
      // warp 1: per item Q (after the previous item's scores), then K of
      // tile g into stage g % 3 after S_{g-3}; warp 2: V of tile g into
      // stage g % 2 after P_{g-2} V_{g-2}.  D / 64 boxes of [128 keys][64 d]
      // each; Q in one box per head and panel.
      const bool isk = warp == 1;
      const CUtensorMap* map = isk ? &tm_k : &tm_v;
      const int ns = isk ? 3 : 2;
      uint64_t* full = isk ? k_full : v_full;
      uint64_t* empty = isk ? k_empty : v_empty;
      uint8_t* ring = isk ? kst : vst;
      tma_prefetch_desc(map);
      if (isk) tma_prefetch_desc(&tm_q);
      bool ok = true;
      int g = 0, wq = -1;   // tiles issued; the last item whose Q was issued
      for (int w = 0; ok; ++w) {
        const int n = ta_item_index(w, G);
        if (n >= NI) break;
        const TaItem it = ta_item<CAUSAL>(p, n, QPT, rtiles);
        if (isk) {
          // Q: rows g QPT .. g QPT + QPT - 1 of each 64-wide panel from head
          // hk G + g, queries q0 .. (boxes start on 1024-byte swizzle atoms:
          // QPT is a multiple of 8)
          if (w >= 1 && !mbar_wait_idle(q_empty, (w - 1) & 1, ctl, 128)) { ok = false; break; }
          mbar_arrive_expect_tx(q_full, Cfg::kQBytes);
          for (int gq = 0; gq < p.G; ++gq)
#pragma unroll
            for (int pn = 0; pn < D / 64; ++pn)
              if (in_bounds(it.q0 >= 0 && it.hk * p.G + gq < p.H, p.status, kSiteAttnQ))
                tma_load_3d(qs + pn * (kTR * 128) + gq * QPT * 128, &tm_q, q_full, 64 * pn, it.q0,
                            it.hk * p.G + gq);
          wq = w;
        }
        for (int j = 0; j < it.nk; ++j, ++g) {
          const int sl = g % ns, k0 = j * kTK;
          if (g >= ns && !mbar_wait_idle(&empty[sl], ((g / ns) - 1) & 1, ctl, 128)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[sl], Cfg::kKBytes);
#pragma unroll
          for (int pn = 0; pn < D / 64; ++pn)
            if (in_bounds(k0 >= 0, p.status, kSiteAttnKV))
              tma_load_3d(ring + sl * Cfg::kKBytes + pn * (kTK * 128), map, &full[sl], 64 * pn, k0, it.hk);
        }
      }
      if (!ok) {
        // wait for the copies in flight before the CTA can leave
        for (int i = (g > ns ? g - ns : 0); i < g; ++i) mbar_wait_drain(&full[i % ns], (i / ns) & 1, 100000000ull);
        if (isk && wq >= 0) mbar_wait_drain(q_full, wq & 1, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int team = (warp - 4) >> 3;  // tiles g = team, team + 2, ... (S buffer g % 3)
    const int half = (warp >> 2) & 1;  // keys [64 half, 64 half + 64) of each tile
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t bar_id = 1 + 4 * team + (warp & 3);   // the two warps (halves) of these rows
    const float sc = p.scale_log2;
    const bool hi = sc >= 0.f;           // the max of sc s is sc max s, or sc min s when sc < 0
    constexpr int QC = D / 4;            // output columns of this thread: [gq QC, (gq + 1) QC)
    const int gq = team * 2 + half;
    bool bad = false;                    // a wait ran out since the last pair barrier
    bool stop = false;
    int g = 0;
    for (int w = 0; !stop; ++w) {
      const int n = ta_item_index(w, G);
      if (n >= NI) break;
      const TaItem it = ta_item<CAUSAL>(p, n, QPT, rtiles);
      const int i = it.q0 + r % QPT, h = it.hk * p.G + r / QPT;   // query and head of this row
      const bool valid = i < p.M;
      // last key this row sees (-1: none), one 32-bit bound for validity, the
      // causal limit and T together
      long long lastl = CAUSAL ? (long long)p.q_offset + i : (long long)p.T - 1;
      if (lastl > (long long)p.T - 1) lastl = p.T - 1;
      const int lastk = valid ? (int)lastl : -1;
      float lsum = 0.f, lref = -INFINITY;  // this thread's row sum and the reference it is relative to
      const int g0 = g;
      // this team's tiles of the item: those with g = g0 + j of its parity
      for (int j = (team - g0) & 1; j < it.nk; j += 2) {
        const int gt = g0 + j, sb = gt % 3;
        const uint32_t scol = tmem + lanes + 128 * sb + 64 * half;
        const int kbase = j * kTK + 64 * half;
        // S_g and the previous tile's reference (from the other team; also
        // across items, which keeps the hand-off one phase apart)
        const bool got = mbar_wait(&s_full[sb], (gt / 3) & 1, ctl) &&
                         (gt == 0 || mbar_wait(&r_rdy[(gt - 1) & 1], ((gt - 1) >> 1) & 1, ctl));
        const bool okw = __all_sync(0xffffffffu, got && !bad);
        // this half's extreme raw score over its visible keys
        float t = hi ? -INFINITY : INFINITY;
        if (okw) {
          tc_fence_after();
          const bool fullm = __all_sync(0xffffffffu, lastk - kbase >= 63);
          uint32_t v[64];
          tmem_ld64_wait(scol, v);
          const int cut = fullm ? 63 : lastk - kbase;
          const float t0 = extreme32(v, cut, hi), t1 = extreme32(v + 32, cut - 32, hi);
          t = hi ? fmaxf(t0, t1) : fminf(t0, t1);
        }
        float* pm = pmx + (team * 2 + ((gt >> 1) & 1)) * 2 * kTR;   // by tile parity: rewritten two tiles later
        pm[half * kTR + r] = t;
        // both halves leave together or go on together (the barrier has no
        // time limit, so no half may stop short of it)
        if (bar_red_or(bar_id, 64, !okw)) {
          stop = true;
          break;
        }
        const float tp = pm[(half ^ 1) * kTR + r];
        t = hi ? fmaxf(t, tp) : fminf(t, tp);
        // mu: -inf when the row sees no key of this tile
        const float mu = (t == INFINITY || t == -INFINITY) ? -INFINITY : t * sc;
        // Reference of the tile: that of the item's previous tile unless mu
        // exceeds it by more than kLazy (P stays below 2^kLazy).  4 slots:
        // tile g + 4 rewrites slot g % 4 only after both halves of tile g + 1
        // have passed their pair barrier of tile g + 3.
        const float mprev = j >= 1 ? mref[((gt - 1) & 3) * kTR + r] : -INFINITY;
        const float mj = mu > mprev + kLazy ? mu : mprev;
        if (half == 0) {
          mref[(gt & 3) * kTR + r] = mj;
          mbar_arrive_warp(&r_rdy[gt & 1]);
        }
        // A raised reference rescales this half of O (P V of the item's
        // earlier tiles, relative to mprev) by 2^(mprev - mj), after the
        // previous tile's P V is done and before P_g is published.
        const bool resc = mj > mprev && mprev != -INFINITY;
        if (__any_sync(0xffffffffu, resc)) {
          if (!__all_sync(0xffffffffu, mbar_wait(&s_free[(gt - 1) % 3], ((gt - 1) / 3) & 1, ctl))) {
            bad = true;
            continue;
          }
          tc_fence_after();
          const float a = resc ? ex2(mprev - mj) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t v[32];
            const uint32_t oc = tmem + lanes + Cfg::kOCol + (D / 2) * half + 32 * c;
            tmem_ld32_wait(oc, v);
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(__uint_as_float(v[q]) * a);
            tmem_st32(oc, v);
          }
        }
        const float muse = mj == -INFINITY ? 0.f : mj;
        const unsigned long long sc2 = pack2(sc, sc), nm2 = pack2(-muse, -muse);
        unsigned long long s2 = 0ull;          // the two lanes' partial row sums
        // every key of this half visible to every row of the warp: no masks
        const bool full = __all_sync(0xffffffffu, lastk - kbase >= 63);
        // 16-key chunks, the load of chunk c + 1 in flight while chunk c is
        // computed; P of keys 64 half + 16 c .. + 15 goes to columns
        // 64 half + 8 c .. + 7, S columns this thread has already read
        uint32_t v[2][16];
        tmem_ld16_async(scol, v[0]);
        tmem_wait_ld_tied(v[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < 3) tmem_ld16_async(scol + 16 * (c + 1), v[(c + 1) & 1]);
          const uint32_t (&x)[16] = v[c & 1];
          const int cut = lastk - (kbase + 16 * c);
          uint32_t wv[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float a0, a1;
            unpack2(fma2(pack2(__uint_as_float(x[e]), __uint_as_float(x[e + 1])), sc2, nm2), a0, a1);
            float p0 = ex2(a0);
            float p1 = ex2(a1);
            if (!full) {
              p0 = e <= cut ? p0 : 0.f;
              p1 = e + 1 <= cut ? p1 : 0.f;
            }
            s2 = add2(s2, pack2(p0, p1));
            const __half2 hh = __floats2half2_rn(p0, p1);
            wv[e >> 1] = *reinterpret_cast<const uint32_t*>(&hh);
          }
          tmem_st8(scol + 8 * c, wv);
          if (c < 3) tmem_wait_ld_tied(v[(c + 1) & 1]);
        }
        float sum0, sum1;
        unpack2(s2, sum0, sum1);
        // this half's row sum, kept relative to the latest reference it used
        if (mj != -INFINITY) {
          lsum = lsum * ex2(lref - mj) + (sum0 + sum1);
          lref = mj;
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(&p_full[sb]);
      }
      if (stop) break;
      g = g0 + it.nk;
      // ---------------------------------------------------------- epilogue
      // O (relative to the item's last reference M) / l, l = the sum over
      // the four (team, half) threads of the row of l_t 2^(m_t - M), once
      // every P V of the item is done.  Entries by item parity: item w + 2
      // rewrites them only after every thread has passed l_rdy of item
      // w + 1, i.e. after its epilogue of item w.
      lfin[((w & 1) * 4 + gq) * kTR + r] = make_float2(lsum, lref);
      mbar_arrive_warp(l_rdy);
      const bool oke = !bad && __all_sync(0xffffffffu, mbar_wait_idle(l_rdy, w & 1, ctl, 256) &&
                                                            mbar_wait_idle(o_done, w & 1, ctl, 256));
      if (!oke) {
        bad = true;   // leaves at the next pair barrier, with the other half
        continue;
      }
      tc_fence_after();
      const float M = mref[((g - 1) & 3) * kTR + r];
      float l = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = lfin[((w & 1) * 4 + q) * kTR + r];
        if (f.y != -INFINITY) l += f.x * ex2(f.y - M);
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool store = valid && in_bounds(h < p.H, p.status, kSiteAttnO);
      __half* orow = p.o + (long long)(store ? i : 0) * p.H * D + (long long)(store ? h : 0) * D + gq * QC;
#pragma unroll
      for (int c = 0; c < QC / 16; ++c) {
        uint32_t v[16];
        tmem_ld16_wait(tmem + lanes + Cfg::kOCol + gq * QC + 16 * c, v);
        uint32_t wv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const __half2 hh = __floats2half2_rn(__uint_as_float(v[2 * q]) * inv, __uint_as_float(v[2 * q + 1]) * inv);
          wv[q] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        if (store) {
          *reinterpret_cast<uint4*>(orow + 16 * c) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          *reinterpret_cast<uint4*>(orow + 16 * c + 8) = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(o_free);
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

// Q8_0 KV cache -> fp16, the staging of the tensor-core path: one thread per
// 16 values of a row (half of a 32-value block), K for blockIdx.y == 0 and V
// for 1.  Each value is RNE(q d): q is exact in fp16, so one fp16 multiply
// rounds the exact product once.  Blocks start on 2-byte boundaries (34-byte
// blocks), so the codes are read in 2-byte words.
__global__ void __launch_bounds__(256)
    kv_q8_stage_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v, long long rows, int D,
                       __half* __restrict__ kf, __half* __restrict__ vf) {
  pdl_wait();   // the caches may come from the previous kernel
  pdl_launch_dependents();
  const uint8_t* src = blockIdx.y ? v : k;
  __half* dst = blockIdx.y ? vf : kf;
  const int per_row = D / 16;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const long long n = idx / per_row;
  const int c = (int)(idx % per_row);
  const uint8_t* blk = src + n * (D / 32) * 34 + (long long)(c >> 1) * 34;
  const __half2 d2 = __half2half2(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(blk))));
  const unsigned short* q = reinterpret_cast<const unsigned short*>(blk + 2 + 16 * (c & 1));
  uint32_t out[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int two = __ldg(q + e);
    int q0 = two & 0xff, q1 = (two >> 8) & 0xff;
    q0 -= (q0 & 0x80) << 1;   // the codes are signed bytes
    q1 -= (q1 & 0x80) << 1;
    const __half2 h = __hmul2(__halves2half2(__int2half_rn(q0), __int2half_rn(q1)), d2);
    out[e] = *reinterpret_cast<const uint32_t*>(&h);
  }
  uint4* o = reinterpret_cast<uint4*>(dst + n * D + 16 * c);
  o[0] = make_uint4(out[0], out[1], out[2], out[3]);
  o[1] = make_uint4(out[4], out[5], out[6], out[7]);
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
  // one persistent CTA per SM (fewer when there are fewer work items)
  const int qpt = kTR / p.G;
  const long long items = (long long)((p.M + qpt - 1) / qpt) * p.Hkv;
  const dim3 grid((unsigned)std::min<long long>(items, std::max(p.nsm, 1)), 1, 1);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, tm_q, tm_k, tm_v, p);
}

}  // namespace

// Shapes the kernel takes: more than 16 rows per KV head, a group size that
// divides 128 rows into whole swizzle atoms per head (G <= 16), rows of
// 16-byte multiples.
bool attention_tc_shape(const AttnParams& p) {
  return p.M * p.G > 16 && (p.D == 64 || p.D == 128) && (p.kv_row_bytes % 16) == 0 && p.G <= 16 &&
         kTR % p.G == 0;
}

// Whether the tcgen05 kernel (after a Q8_0 staging when q8) beats the
// mma.sync kernel with its key split for this call, by estimated time: the
// tcgen05 kernel takes an item's key tiles in turn on one SM (about 0.9 us
// a tile, at D = 64 as at 128), so its time is the larger of the longest item and the
// SMs' share of all tiles; the split kernel spreads the keys over the SMs
// at about 170 TFLOP/s.  Measured at the 8B shape: for M = 128 to 512 new
// queries over 4096 keys the tcgen05 kernel took 36-37 us against 52-149 us.
bool attention_tc_applies(const AttnParams& p, bool q8) {
  if (!attention_tc_shape(p)) return false;
  const int QPT = kTR / p.G;
  const double rtiles = (double)((p.M + QPT - 1) / QPT), items = rtiles * p.Hkv;
  // visible keys summed over the queries (closed form of sum_i min(T, q_offset + i + 1))
  double vis = (double)p.M * p.T;
  long long last = p.T;   // keys the last row tile sees
  if (p.causal) {
    const long long a = (long long)p.q_offset + 1;
    const long long n1 = std::min<long long>(std::max<long long>((long long)p.T - a + 1, 0), p.M);
    vis = (double)n1 * a + (double)n1 * (n1 - 1) / 2 + (double)(p.M - n1) * p.T;
    last = std::min<long long>(p.T, (long long)p.q_offset + p.M);
  }
  const double longest = (double)((last + kTK - 1) / kTK);
  const double total = p.Hkv * (vis / QPT) / kTK + items;   // key tiles over all items (rounded up once each)
  const double tile_us = 0.9;   // D = 64 tiles cost about as much: the softmax, not the MMA, sets it
  double tc_us = std::max(longest, total / std::max(p.nsm, 1)) * tile_us + 2.0;
  if (q8) tc_us += 2.0 + (double)p.Hkv * p.T * p.D * 6.0 / 5.0e6;   // staging: 3 bytes a value, 5 TB/s
  const double split_us = 4.0 * p.H * p.D * vis / 170.0e6 + 2.0;
  return tc_us <= split_us;
}

cudaError_t launch_kv_q8_stage(const void* k, const void* v, long long rows, int D, void* kf, void* vf,
                               cudaStream_t s) {
  const long long threads = rows * (D / 16);
  if (threads == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)((threads + 255) / 256), 2, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_q8_stage_kernel, static_cast<const uint8_t*>(k), static_cast<const uint8_t*>(v),
                            rows, D, static_cast<__half*>(kf), static_cast<__half*>(vf));
}

cudaError_t launch_attention_tc(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                const CUtensorMap& tm_v, cudaStream_t s) {
  if (p.D == 64)
    return p.causal ? launch_tc<64, true>(p, tm_q, tm_k, tm_v, s) : launch_tc<64, false>(p, tm_q, tm_k, tm_v, s);
  return p.causal ? launch_tc<128, true>(p, tm_q, tm_k, tm_v, s) : launch_tc<128, false>(p, tm_q, tm_k, tm_v, s);
}

}  // namespace m4q
