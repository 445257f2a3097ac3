// attention.cu -- attention of fp16 queries over an fp16 or Q8_0 KV cache.
//
// Pages: "v0.1 vs v0.2 comparison" 2.3 (Brick 4: FlashAttention with the
// Q8_0 KV cache dequantized on the fly, row statistics by register shuffles
// instead of block barriers); "Releases" v0.3.0 (grouped-query attention,
// causal masking with a sequence offset, head dims 64 and 128) and v0.2
// (chunked attention: running max and sum carried between key chunks and
// merged exactly); project page section 4 (Q, K, V arrive head-major).
//
// O[i, h, :] = softmax_j(scale * Q[h, i] . K[h / G, j]) V[h / G, j], keys
// j <= q_offset + i when causal, G = H / Hkv.
//
// One CTA (4 warps) takes one KV head and 64 rows of the query matrix of that
// head's group, row r = (query i = r / G, head h = hk * G + r % G), so every
// decoded K/V tile serves all G query heads of the group.  It walks its key
// range in tiles of 64 keys:
//   1. the 128 threads decode the K and V tile into fp16 shared memory
//      (Q8_0: the same exact decode as the weights, RNE(q * d)); rows past the
//      CTA's last key are zero, so masked products stay finite;
//   2. each warp forms S = Q K^T for its 16 rows with mma.sync m16n8k16 (Q
//      fragments held in registers, K fragments by ldmatrix), fp32;
//   3. online softmax in fp32 on the accumulators: masked scores are -inf,
//      the row maximum is reduced over the 4 threads of a row by shuffles,
//      p = 2^(s * scale * log2 e - m), the O accumulators are rescaled;
//   4. P is repacked in registers as the A operand (fp16) and O += P V with
//      V fragments by ldmatrix.trans.
// Key splits: when the head/row tiles alone would leave SMs idle (decode),
// the key range is split across CTAs; each writes its unnormalised O and
// (max, sum) to a caller workspace and a second kernel merges them exactly
// (the chunked-softmax identity).  Without a workspace the key range is not
// split.
#include "codec.cuh"
#include "launch.h"

namespace m4q {

namespace {

constexpr int kRows = 64;   // query rows per CTA
constexpr int kKeys = 64;   // keys per tile

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <int D, bool Q8>
struct AttnCfg {
  static constexpr int kRowBytes = Q8 ? D / 32 * 34 : 2 * D;   // one key row in the cache
  static constexpr int kPitch = (D + 8) * 2;                   // padded fp16 row in shared memory
  static constexpr int kTile = kKeys * kPitch;                 // one padded fp16 tile
  static constexpr int kRaw = kKeys * kRowBytes;               // one packed Q8_0 tile
  // Q8_0: packed K and V tiles in NS stages, then the decoded K and V
  // tiles.  fp16: the padded K and V tiles in NS stages.
  template <int NS>
  static constexpr int smem() { return Q8 ? 2 * NS * kRaw + 2 * kTile : 2 * NS * kTile; }
};

// Stages of the K/V tile pipeline: three when the warps split the keys of a
// few rows over an fp16 cache (decode: little compute per tile to hide a
// tile's load behind; two CTAs per SM then), else two (the Q8_0 decode is
// bound by its arithmetic, and gains more from a third CTA per SM).
template <bool KS, bool Q8>
constexpr int kAttnStages = (KS && !Q8) ? 3 : 2;

// Start the asynchronous copy of keys [k0, min(k0 + 64, T)) of one KV head:
// packed rows as they are (Q8_0), or fp16 rows into the padded tile, whose
// rows past T are zeroed (they are masked, but V enters P V, where 0 * NaN
// would be NaN).  vec16: every tile start and the cache end are 16-byte
// aligned, so 16-byte copies; otherwise 4-byte copies (Q8_0 rows are 4-byte
// multiples).
template <int D, bool Q8>
__device__ __forceinline__ void issue_tile(uint8_t* kdst, uint8_t* vdst, const uint8_t* khead,
                                           const uint8_t* vhead, int k0, int T, bool vec16, uint32_t* status) {
  using Cfg = AttnCfg<D, Q8>;
  const int rows = min(kKeys, T - k0);
  // keys [k0, k0 + rows) of the head, and whole 16-byte copies when vec16
  if (!in_bounds(k0 >= 0 && rows >= 1 && (!vec16 || (rows * Cfg::kRowBytes) % 16 == 0), status, kSiteAttnKV)) {
    cp_async_commit();
    return;
  }
  const uint8_t* ks = khead + (long long)k0 * Cfg::kRowBytes;
  const uint8_t* vs = vhead + (long long)k0 * Cfg::kRowBytes;
  if constexpr (Q8) {
    const int bytes = rows * Cfg::kRowBytes;
    if (vec16) {
      for (int c = threadIdx.x; c < bytes / 16; c += 128) {
        cp_async16(kdst + 16 * c, ks + 16 * c);
        cp_async16(vdst + 16 * c, vs + 16 * c);
      }
    } else {
      for (int c = threadIdx.x; c < bytes / 4; c += 128) {
        cp_async4(kdst + 4 * c, ks + 4 * c);
        cp_async4(vdst + 4 * c, vs + 4 * c);
      }
    }
  } else {
    constexpr int kChunks = D / 8;
    for (int c = threadIdx.x; c < kKeys * kChunks; c += 128) {
      const int r = c / kChunks, ch = c % kChunks;
      uint8_t* kd = kdst + r * Cfg::kPitch + 16 * ch;
      uint8_t* vd = vdst + r * Cfg::kPitch + 16 * ch;
      if (r < rows) {
        cp_async16(kd, ks + (long long)r * Cfg::kRowBytes + 16 * ch);
        cp_async16(vd, vs + (long long)r * Cfg::kRowBytes + 16 * ch);
      } else {
        *reinterpret_cast<uint4*>(kd) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(vd) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  cp_async_commit();
}

// Decode a packed Q8_0 tile (rows of D / 32 blocks) into the padded fp16
// tile: RNE(q * d) per value, the weights' exact decode.  Rows at or past
// `valid` are written as zeros.  A warp takes 32 consecutive rows of one
// block column, so its reads share one alignment:
//   - rows of a multiple of 8 bytes (D = 128): five 8-byte reads from the
//     8-byte boundary at or before the block, which it starts sh = 34 blk
//     mod 8 bytes into (0, 2, 4 or 6); conflict-free, as the 16 lanes of a
//     half-warp read consecutive rows 34 words apart;
//   - otherwise a block at an even index starts 4-byte aligned (rows are
//     4-byte multiples) and is read as 9 words; one at an odd index starts 2
//     bytes past a word and is read as 10 words and shifted.
// Those reads may run up to 4 bytes past the block (into the next row, or
// the next buffer for the tile's last row); the extra bytes are never used.
template <int D>
__device__ __forceinline__ void decode_q8_tile(uint8_t* dst, const uint8_t* raw, int valid) {
  using Cfg = AttnCfg<D, true>;
  const DecK K = make_deck();
  constexpr int kBlk = D / 32;
  constexpr int kUnits = kKeys * kBlk / 128;
  static_assert(kKeys == 64, "two block columns per 128 threads");
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    // unit = threadIdx.x + 128 u: row unit % 64, block column 2 u + (threadIdx.x >> 6)
    const int h = threadIdx.x >> 6, rr = threadIdx.x & 63, blk = 2 * u + h;
    uint4* out = reinterpret_cast<uint4*>(dst + rr * Cfg::kPitch + 64 * blk);
    if (rr < valid) {
      const int off = rr * Cfg::kRowBytes + 34 * blk;
      uint32_t w[9];
      if constexpr (Cfg::kRowBytes % 8 == 0) {
        // sh = (68 u + 34 h) mod 8 = 4 (u & 1) + 2 h
        const uint2* src = reinterpret_cast<const uint2*>(raw + (off & ~7));
        uint32_t a[10];
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          const uint2 x = src[i];
          a[2 * i] = x.x;
          a[2 * i + 1] = x.y;
        }
        uint32_t b[10];
#pragma unroll
        for (int i = 0; i < 10; ++i) b[i] = (u & 1) ? (i < 9 ? a[i + 1] : 0u) : a[i];
        if (h) {
#pragma unroll
          for (int i = 0; i < 9; ++i) w[i] = __funnelshift_r(b[i], b[i + 1], 16);
        } else {
#pragma unroll
          for (int i = 0; i < 9; ++i) w[i] = b[i];
        }
      } else {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(raw + (off & ~3));
        if ((off & 3) == 0) {
#pragma unroll
          for (int i = 0; i < 9; ++i) w[i] = src[i];
        } else {
          uint32_t a[10];
#pragma unroll
          for (int i = 0; i < 10; ++i) a[i] = src[i];
#pragma unroll
          for (int i = 0; i < 9; ++i) w[i] = __funnelshift_r(a[i], a[i + 1], 16);
        }
      }
      const uint32_t d2 = dup_scale(u16_at(w, 0));
      uint32_t v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = q8_pair(spread_pair(w, 2 + 2 * q), d2, K);
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

// KS (at most 16 query rows, decode): the 4 warps share rows 0..15 of the
// tile and split every key tile, warp w taking keys 16 w .. 16 w + 15; their
// partial (max, sum, O) are merged through shared memory at the end.
template <int D, bool Q8, bool KS>
__global__ void __launch_bounds__(128, KS ? 3 : 2) attn_kernel(const AttnParams p) {
  using Cfg = AttnCfg<D, Q8>;
  constexpr int NT = KS ? 2 : kKeys / 8;   // score n8 tiles per warp and key tile
  constexpr int DK = D / 16;      // k16 steps over the head dim
  constexpr int DN = D / 8;       // output n8 tiles
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  // Row tiles in reverse order: under a causal mask the last tiles see the
  // most keys, so they start first.
  const int rt = (int)gridDim.x - 1 - (int)blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int R = p.M * p.G;
  const int wrow = KS ? 0 : 16 * warp;           // first row of this warp in the tile
  const int kw = KS ? 16 * warp : 0;             // first key of this warp in a key tile
  const bool active = rt * kRows + wrow < R;     // this warp has a row to compute
  pdl_launch_dependents();
  pdl_wait();   // every global access below comes after the previous kernel

  // This thread's two rows (g and g + 8 of the warp's 16).
  int qi[2], qh[2], lim[2];
  bool rok[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = rt * kRows + wrow + g + 8 * h2;
    rok[h2] = r < R;
    qi[h2] = rok[h2] ? r / p.G : 0;
    qh[h2] = hk * p.G + (rok[h2] ? r % p.G : 0);
  }
  // Key range of this CTA: its split, cut at T and, when causal, after the
  // last key its last row can see.
  const int kbeg = split * p.tsplit;
  int kend = min(p.T, kbeg + p.tsplit);
  if (p.causal) {
    const int rlast = min(R - 1, rt * kRows + kRows - 1);
    const long long vis = (long long)p.q_offset + rlast / p.G + 1;
    if (vis < kend) kend = (int)vis;
  }
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    long long l = kend;
    if (p.causal) l = min(l, (long long)p.q_offset + qi[h2] + 1);
    lim[h2] = (int)l;
  }

  // Q fragments (A operand), zero for rows past R.
  uint32_t qa[DK][4];
#pragma unroll
  for (int kk = 0; kk < DK; ++kk)
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const uint32_t* qrow =
          reinterpret_cast<const uint32_t*>(p.q + ((long long)qh[h2] * p.M + qi[h2]) * D + 16 * kk + 2 * t);
      const bool qok = rok[h2] && in_bounds(qh[h2] < p.H && qi[h2] < p.M, p.status, kSiteAttnQ);
      qa[kk][h2] = qok ? __ldg(qrow) : 0u;
      qa[kk][2 + h2] = qok ? __ldg(qrow + 4) : 0u;
    }

  float o[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const uint8_t* khead = p.k + (long long)hk * p.T * Cfg::kRowBytes;
  const uint8_t* vhead = p.v + (long long)hk * p.T * Cfg::kRowBytes;
  // stage s: Q8_0 packed K at 2 s * kRaw, V at (2 s + 1) * kRaw; fp16 padded
  // K at 2 s * kTile, V at (2 s + 1) * kTile
  constexpr int kStage = Q8 ? Cfg::kRaw : Cfg::kTile;
  constexpr int NS = kAttnStages<KS, Q8>;
  uint8_t* dec = smem + 2 * NS * Cfg::kRaw;   // Q8_0: decoded K, then V
  // fp16: tiles 0 .. NS - 2 in flight before the loop; tile it + NS - 1
  // issued once tile it has landed and every warp is done with tile it - 1.
  // Q8_0: a packed stage is free again once its tile is decoded, so tiles
  // 0 .. NS - 1 go before the loop and tile it + NS right after tile it's
  // decode: NS tiles in flight while the warps run the MMAs.
  constexpr int kAhead = Q8 ? NS : NS - 1;
  static_assert(kAhead >= 1 && kAhead <= 2, "copy groups waited for below");
#pragma unroll
  for (int s0 = 0; s0 < kAhead; ++s0)
    if (kbeg + s0 * kKeys < kend)
      issue_tile<D, Q8>(smem + 2 * s0 * kStage, smem + (2 * s0 + 1) * kStage, khead, vhead, kbeg + s0 * kKeys, p.T,
                        p.kv_vec16, p.status);
  int it = 0;
  for (int k0 = kbeg; k0 < kend; k0 += kKeys, ++it) {
    const int st = it % NS;
    // this tile's copy group is the oldest outstanding one: wait for all but
    // the one issued after it
    if (kAhead == 2 && k0 + kKeys < kend) cp_async_wait_one();
    else cp_async_wait_all();
    __syncthreads();   // this tile has landed; every warp is done with the previous one
    const uint8_t* Kt;
    const uint8_t* Vt;
    if constexpr (Q8) {
      decode_q8_tile<D>(dec, smem + 2 * st * kStage, kend - k0);
      decode_q8_tile<D>(dec + Cfg::kTile, smem + (2 * st + 1) * kStage, kend - k0);
      __syncthreads();   // decoded: packed stage st is free
      if (k0 + NS * kKeys < kend)
        issue_tile<D, Q8>(smem + 2 * st * kStage, smem + (2 * st + 1) * kStage, khead, vhead, k0 + NS * kKeys, p.T,
                          p.kv_vec16, p.status);
      Kt = dec;
      Vt = dec + Cfg::kTile;
    } else {
      if (k0 + (NS - 1) * kKeys < kend) {
        const int sn = (it + NS - 1) % NS;
        issue_tile<D, Q8>(smem + 2 * sn * kStage, smem + (2 * sn + 1) * kStage, khead, vhead,
                          k0 + (NS - 1) * kKeys, p.T, p.kv_vec16, p.status);
      }
      Kt = smem + 2 * st * kStage;
      Vt = smem + (2 * st + 1) * kStage;
    }
    if (!active) continue;

    // S = Q K^T (16 rows x 64 keys per warp)
    float s[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DK; ++kk)
#pragma unroll
      for (int j = 0; j < NT; j += 2) {
        uint32_t b[4];
        const int mi = lane >> 3;
        ldsm_x4(b, Kt + (kw + 8 * (j + (mi >> 1)) + (lane & 7)) * Cfg::kPitch + 2 * (16 * kk + 8 * (mi & 1)));
        mma16816(s[j], qa[kk], b[0], b[1]);
        mma16816(s[j + 1], qa[kk], b[2], b[3]);
      }

    // online softmax; accumulator c of tile j: row g + 8 (c >> 1), key 8j + 2t + (c & 1)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = k0 + kw + 8 * j + 2 * t + (c & 1);
        const float x = key < lim[c >> 1] ? s[j][c] * p.scale_log2 : -INFINITY;
        s[j][c] = x;
        mx[c >> 1] = fmaxf(mx[c >> 1], x);
      }
    float corr[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
      mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
      const float mnew = fmaxf(mrow[h2], mx[h2]);
      const float mref = mnew == -INFINITY ? 0.f : mnew;   // a row with no key yet
      corr[h2] = fast_exp2(mrow[h2] - mref);
      mrow[h2] = mnew;
      mx[h2] = mref;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float e = fast_exp2(s[j][c] - mx[c >> 1]);
        s[j][c] = e;
        rs[c >> 1] += e;
      }
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) lrow[h2] = lrow[h2] * corr[h2] + rs[h2];
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      o[dn][0] *= corr[0]; o[dn][1] *= corr[0];
      o[dn][2] *= corr[1]; o[dn][3] *= corr[1];
    }

    // O += P V, P repacked from the score accumulators as the A operand
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
      const uint32_t pa[4] = {pack_h2(s[2 * kk][0], s[2 * kk][1]), pack_h2(s[2 * kk][2], s[2 * kk][3]),
                              pack_h2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                              pack_h2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
      for (int dn = 0; dn < DN; dn += 2) {
        uint32_t b[4];
        const int mi = lane >> 3;
        ldsm_x4_t(b, Vt + (kw + 16 * kk + 8 * (mi & 1) + (lane & 7)) * Cfg::kPitch + 2 * (8 * (dn + (mi >> 1))));
        mma16816(o[dn], pa, b[0], b[1]);
        mma16816(o[dn + 1], pa, b[2], b[3]);
      }
    }
  }

  // row sums over the 4 threads of a row
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    lrow[h2] += __shfl_xor_sync(0xffffffffu, lrow[h2], 1);
    lrow[h2] += __shfl_xor_sync(0xffffffffu, lrow[h2], 2);
  }
  if constexpr (KS) {
    // Merge the 4 warps' partials of rows 0..15: m = max_w m_w,
    // O = sum_w 2^(m_w - m) O_w / sum_w 2^(m_w - m) l_w.  The tile buffers
    // are free (no copy is in flight after the last tile).
    __syncthreads();
    float* Ow = reinterpret_cast<float*>(smem);                   // [4 warps][16 rows][D]
    float2* ML = reinterpret_cast<float2*>(Ow + 4 * 16 * D);      // [4 warps][16 rows]
#pragma unroll
    for (int dn = 0; dn < DN; ++dn)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2)
        *reinterpret_cast<float2*>(Ow + (warp * 16 + g + 8 * h2) * D + 8 * dn + 2 * t) =
            make_float2(o[dn][2 * h2], o[dn][2 * h2 + 1]);
    if (t == 0)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) ML[warp * 16 + g + 8 * h2] = make_float2(mrow[h2], lrow[h2]);
    __syncthreads();
    const int row = threadIdx.x >> 3, seg = threadIdx.x & 7;   // 16 rows x 8 segments of D / 8
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) m = fmaxf(m, ML[w * 16 + row].x);
    const float mref = m == -INFINITY ? 0.f : m;
    float wgt[4], L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      wgt[w] = fast_exp2(ML[w * 16 + row].x - mref);
      L += wgt[w] * ML[w * 16 + row].y;
    }
    const int r = rt * kRows + row;
    constexpr int SEG = D / 8;
    float acc[SEG];
#pragma unroll
    for (int e = 0; e < SEG; ++e) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) a += wgt[w] * Ow[(w * 16 + row) * D + seg * SEG + e];
      acc[e] = a;
    }
    if (p.nsplit == 1) {
      if (r < R && in_bounds(hk * p.G + r % p.G < p.H, p.status, kSiteAttnO)) {
        const float inv = L > 0.f ? 1.f / L : 0.f;
        __half* orow = p.o + (long long)(r / p.G) * p.H * D + (long long)(hk * p.G + r % p.G) * D + seg * SEG;
#pragma unroll
        for (int e = 0; e < SEG; e += 2)
          *reinterpret_cast<__half2*>(orow + e) = __floats2half2_rn(acc[e] * inv, acc[e + 1] * inv);
      }
    } else {
      const long long slot = ((long long)split * p.Hkv + hk) * ((long long)p.rtiles * kRows) + r;
      if (!in_bounds(split < p.nsplit && slot < (long long)p.nsplit * p.Hkv * p.rtiles * kRows, p.status,
                     kSiteAttnWs))
        return;
#pragma unroll
      for (int e = 0; e < SEG; e += 2)
        *reinterpret_cast<float2*>(p.ws_o + slot * D + seg * SEG + e) = make_float2(acc[e], acc[e + 1]);
      if (seg == 0) p.ws_ml[slot] = make_float2(m, L);
    }
    return;
  }
  if (p.nsplit == 1) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      if (!rok[h2] || !in_bounds(qi[h2] < p.M && qh[h2] < p.H, p.status, kSiteAttnO)) continue;
      const float inv = lrow[h2] > 0.f ? 1.f / lrow[h2] : 0.f;
      __half* orow = p.o + (long long)qi[h2] * p.H * D + (long long)qh[h2] * D;
#pragma unroll
      for (int dn = 0; dn < DN; ++dn)
        *reinterpret_cast<__half2*>(orow + 8 * dn + 2 * t) =
            __floats2half2_rn(o[dn][2 * h2] * inv, o[dn][2 * h2 + 1] * inv);
    }
  } else {
    const long long rows_pad = (long long)p.rtiles * kRows;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const long long r = (long long)rt * kRows + wrow + g + 8 * h2;
      const long long slot = ((long long)split * p.Hkv + hk) * rows_pad + r;
      if (!in_bounds(split < p.nsplit && r < rows_pad, p.status, kSiteAttnWs)) continue;
      float* wrow = p.ws_o + slot * D;
#pragma unroll
      for (int dn = 0; dn < DN; ++dn)
        *reinterpret_cast<float2*>(wrow + 8 * dn + 2 * t) = make_float2(o[dn][2 * h2], o[dn][2 * h2 + 1]);
      if (t == 0) p.ws_ml[slot] = make_float2(mrow[h2], lrow[h2]);
    }
  }
}

// Merge the key splits of one row: O = sum_s 2^(m_s - m) O_s / sum_s 2^(m_s - m) l_s.
// One CTA of 8 warps per (KV head, row): the threads take the splits for the
// max; warp w sums splits w, w + 8, ... with its lanes over the head dim (so
// every split's loads are in flight at once); shared memory adds the warps.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p) {
  __shared__ float red_m[8], red_l[8];
  __shared__ float red_o[8][D];
  const long long rows_pad = (long long)p.rtiles * kRows;
  const int R = p.M * p.G;
  const int hk = (int)(blockIdx.x / R), r = (int)(blockIdx.x % R);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long base = (long long)hk * rows_pad + r;          // slot of split s: base + s * stride
  const long long stride = (long long)p.Hkv * rows_pad;
  // No early launch_dependents here: a kernel after this one (the next
  // attention launch) then starts only when these CTAs have left the SMs,
  // so the attention grid, one full wave at three CTAs per SM over a Q8_0
  // cache, is never split by a CTA of this kernel.
  pdl_wait();   // the splits come from the attention kernel before it
  float m = -INFINITY;
  for (int s = threadIdx.x; s < p.nsplit; s += 256) m = fmaxf(m, p.ws_ml[base + s * stride].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red_m[warp] = m;
  __syncthreads();
  m = red_m[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red_m[w]);
  const float mref = m == -INFINITY ? 0.f : m;
  float l = 0.f;
  float acc[D / 32];
#pragma unroll
  for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
#pragma unroll 4
  for (int s = warp; s < p.nsplit; s += 8) {
    const float2 ml = p.ws_ml[base + s * stride];
    const float w = fast_exp2(ml.x - mref);
    l += w * ml.y;
    const float* src = p.ws_o + (base + s * stride) * D + lane;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] += w * src[32 * c];
  }
#pragma unroll
  for (int c = 0; c < D / 32; ++c) red_o[warp][lane + 32 * c] = acc[c];
  if (lane == 0) red_l[warp] = l;
  __syncthreads();
  if (warp == 0) {
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) L += red_l[w];
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int i = r / p.G, h = hk * p.G + r % p.G;
    if (!in_bounds(i < p.M && h < p.H, p.status, kSiteAttnO)) return;
    __half* orow = p.o + (long long)i * p.H * D + (long long)h * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += red_o[w][lane + 32 * c];
      orow[lane + 32 * c] = __float2half_rn(v * inv);
    }
  }
}

// Launch with programmatic dependent launch (unless M4Q_PDL=0): the kernel
// may be scheduled while the previous kernel of the stream finishes, and
// waits for it (griddepcontrol.wait) before its first global access.
template <typename Kern>
cudaError_t launch_pdl(Kern kern, dim3 grid, unsigned block, int smem, cudaStream_t s, const AttnParams& p) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int D, bool Q8, bool KS>
cudaError_t launch_attn_dqk(const AttnParams& p, cudaStream_t s) {
  auto kern = attn_kernel<D, Q8, KS>;
  constexpr int kSmem = AttnCfg<D, Q8>::template smem<kAttnStages<KS, Q8>>();
  static_assert(4 * 16 * D * 4 + 4 * 16 * 8 <= kSmem, "warp merge buffer");
  std::atomic<unsigned long long>& configured = attr_flag<std::integer_sequence<int, 3, D, Q8, KS>>();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  e = launch_pdl(kern, dim3((unsigned)p.rtiles, (unsigned)p.Hkv, (unsigned)p.nsplit), 128, kSmem, s, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  return launch_pdl(attn_combine_kernel<D>, dim3((unsigned)((long long)p.Hkv * p.M * p.G)), 256, 0, s, p);
}

}  // namespace

template <int D, bool Q8>
cudaError_t launch_attn_dq(const AttnParams& p, cudaStream_t s) {
  // at most 16 rows (decode): the warps split the keys instead of the rows
  return p.M * p.G <= 16 ? launch_attn_dqk<D, Q8, true>(p, s) : launch_attn_dqk<D, Q8, false>(p, s);
}

cudaError_t launch_attention(const AttnParams& p, bool q8, cudaStream_t s) {
  if (p.D == 64) return q8 ? launch_attn_dq<64, true>(p, s) : launch_attn_dq<64, false>(p, s);
  return q8 ? launch_attn_dq<128, true>(p, s) : launch_attn_dq<128, false>(p, s);
}

}  // namespace m4q
