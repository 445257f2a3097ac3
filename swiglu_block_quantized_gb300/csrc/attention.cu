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

// Decode keys [k0, k0 + 64) of one KV head into dst[64][D + 8] (fp16); keys
// at or past `kend` are written as zeros.
template <int D, bool Q8>
__device__ __forceinline__ void load_kv_tile(__half (*dst)[D + 8], const uint8_t* __restrict__ head,
                                             long long row_bytes, int k0, int kend) {
  if constexpr (Q8) {
    constexpr int kBlk = D / 32;                  // Q8_0 blocks per key row
    constexpr int kUnits = kKeys * kBlk / 128;    // (row, block) units per thread
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
      const int unit = threadIdx.x + 128 * u;
      const int rr = unit / kBlk, blk = unit % kBlk;
      uint4* out = reinterpret_cast<uint4*>(&dst[rr][32 * blk]);
      if (k0 + rr < kend) {
        const unsigned short* src =
            reinterpret_cast<const unsigned short*>(head + (long long)(k0 + rr) * row_bytes + 34 * blk);
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = (uint32_t)__ldg(src + 2 * i) | ((uint32_t)__ldg(src + 2 * i + 1) << 16);
        w[8] = __ldg(src + 16);
        const uint32_t d2 = dup_scale(u16_at(w, 0));
        uint32_t v[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) v[p] = q8_pair(spread_pair(w, 2 + 2 * p), d2);
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] = make_uint4(0, 0, 0, 0);
      }
    }
  } else {
    constexpr int kChunks = D / 8;                 // 16-byte chunks per key row
    constexpr int kUnits = kKeys * kChunks / 128;
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
      const int unit = threadIdx.x + 128 * u;
      const int rr = unit / kChunks, c = unit % kChunks;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (k0 + rr < kend) val = __ldg(reinterpret_cast<const uint4*>(head + (long long)(k0 + rr) * row_bytes) + c);
      *reinterpret_cast<uint4*>(&dst[rr][8 * c]) = val;
    }
  }
}

template <int D, bool Q8>
__global__ void __launch_bounds__(128, 2) attn_kernel(const AttnParams p) {
  constexpr int NT = kKeys / 8;   // score n8 tiles per key tile
  constexpr int DK = D / 16;      // k16 steps over the head dim
  constexpr int DN = D / 8;       // output n8 tiles
  __shared__ alignas(128) __half Ks[kKeys][D + 8];
  __shared__ alignas(128) __half Vs[kKeys][D + 8];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int rt = blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int R = p.M * p.G;

  // This thread's two rows (g and g + 8 of the warp's 16).
  int qi[2], qh[2], lim[2];
  bool rok[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = rt * kRows + 16 * warp + g + 8 * h2;
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
      qa[kk][h2] = rok[h2] ? __ldg(qrow) : 0u;
      qa[kk][2 + h2] = rok[h2] ? __ldg(qrow + 4) : 0u;
    }

  float o[DN][4];
#pragma unroll
  for (int dn = 0; dn < DN; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const uint8_t* khead = p.k + (long long)hk * p.T * p.kv_row_bytes;
  const uint8_t* vhead = p.v + (long long)hk * p.T * p.kv_row_bytes;
  for (int k0 = kbeg; k0 < kend; k0 += kKeys) {
    __syncthreads();   // the previous tile's fragments have been read
    load_kv_tile<D, Q8>(Ks, khead, p.kv_row_bytes, k0, kend);
    load_kv_tile<D, Q8>(Vs, vhead, p.kv_row_bytes, k0, kend);
    __syncthreads();

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
        ldsm_x4(b, &Ks[8 * (j + (mi >> 1)) + (lane & 7)][16 * kk + 8 * (mi & 1)]);
        mma16816(s[j], qa[kk], b[0], b[1]);
        mma16816(s[j + 1], qa[kk], b[2], b[3]);
      }

    // online softmax; accumulator c of tile j: row g + 8 (c >> 1), key 8j + 2t + (c & 1)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = k0 + 8 * j + 2 * t + (c & 1);
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
    for (int kk = 0; kk < kKeys / 16; ++kk) {
      const uint32_t pa[4] = {pack_h2(s[2 * kk][0], s[2 * kk][1]), pack_h2(s[2 * kk][2], s[2 * kk][3]),
                              pack_h2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                              pack_h2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
      for (int dn = 0; dn < DN; dn += 2) {
        uint32_t b[4];
        const int mi = lane >> 3;
        ldsm_x4_t(b, &Vs[16 * kk + 8 * (mi & 1) + (lane & 7)][8 * (dn + (mi >> 1))]);
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
  if (p.nsplit == 1) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      if (!rok[h2]) continue;
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
      const long long r = (long long)rt * kRows + 16 * warp + g + 8 * h2;
      const long long slot = ((long long)split * p.Hkv + hk) * rows_pad + r;
      float* wrow = p.ws_o + slot * D;
#pragma unroll
      for (int dn = 0; dn < DN; ++dn)
        *reinterpret_cast<float2*>(wrow + 8 * dn + 2 * t) = make_float2(o[dn][2 * h2], o[dn][2 * h2 + 1]);
      if (t == 0) p.ws_ml[slot] = make_float2(mrow[h2], lrow[h2]);
    }
  }
}

// Merge the key splits of one row: O = sum_s 2^(m_s - m) O_s / sum_s 2^(m_s - m) l_s.
// One warp per (KV head, row); lanes over the head dim.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnParams p) {
  const long long rows_pad = (long long)p.rtiles * kRows;
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int R = p.M * p.G;
  if (wid >= (long long)p.Hkv * R) return;
  const int hk = (int)(wid / R), r = (int)(wid % R);
  float m = -INFINITY;
  for (int s = 0; s < p.nsplit; ++s) m = fmaxf(m, p.ws_ml[((long long)s * p.Hkv + hk) * rows_pad + r].x);
  const float mref = m == -INFINITY ? 0.f : m;
  float acc[D / 32], l = 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
  for (int s = 0; s < p.nsplit; ++s) {
    const long long slot = ((long long)s * p.Hkv + hk) * rows_pad + r;
    const float2 ml = p.ws_ml[slot];
    const float w = fast_exp2(ml.x - mref);
    l += w * ml.y;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] += w * p.ws_o[slot * D + lane + 32 * c];
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int i = r / p.G, h = hk * p.G + r % p.G;
  __half* orow = p.o + (long long)i * p.H * D + (long long)h * D;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) orow[lane + 32 * c] = __float2half_rn(acc[c] * inv);
}

template <int D, bool Q8>
cudaError_t launch_attn_dq(const AttnParams& p, cudaStream_t s) {
  const dim3 grid((unsigned)p.rtiles, (unsigned)p.Hkv, (unsigned)p.nsplit);
  attn_kernel<D, Q8><<<grid, 128, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.nsplit == 1) return e;
  const long long warps = (long long)p.Hkv * p.M * p.G;
  attn_combine_kernel<D><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, bool q8, cudaStream_t s) {
  if (p.D == 64) return q8 ? launch_attn_dq<64, true>(p, s) : launch_attn_dq<64, false>(p, s);
  return q8 ? launch_attn_dq<128, true>(p, s) : launch_attn_dq<128, false>(p, s);
}

}  // namespace m4q
