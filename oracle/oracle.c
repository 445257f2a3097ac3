/*
 * oracle.c -- plain CPU reference for the block-quantized projection GEMM
 * and the fused gate/up SwiGLU projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library) shares no code with it and never calls it.
 *
 * Everything is computed in IEEE binary64.  No blocking, fusion or
 * reordering beyond the definitions below: the weights are decoded block by
 * block, each decoded weight is rounded once to fp16 (the operand type the
 * method multiplies, see below), every output is one dot product summed over
 * k in increasing order, and SiLU(g)*u is applied to the two binary64 dot
 * products.
 *
 * Sources (m4-prefill-engine pages):
 *  - "Releases", v0.3.0, PrismML Q2_0 ternary codec: a 128-weight block is
 *    34 bytes, a 2-byte fp16 scale d plus 32 bytes of packed 2-bit codes
 *    (2.125 bits per weight); a weight is (q - 1) * d and the reserved code
 *    q = 3 decodes to +2 * d.
 *  - "Releases", v0.3.0 / v0.2.3 and the project page's Table B: GGUF Q4_0
 *    (block_q4_0) and Q8_0 are the other two codecs.  The pages name them
 *    but do not print their formulas; this oracle takes GGUF's public
 *    definition: 32-weight blocks with an fp16 scale d, Q4_0 w = (q - 8) * d
 *    with a 4-bit q, Q8_0 w = q * d with a signed 8-bit q.
 *  - Project page, section 4 (v0.2.1, "mlx_4bit_planar") and Table B
 *    (both engines of the MLX comparison read the same block_mlx_4bit
 *    weights), and "Releases" v0.2.1
 *    and v0.3.0 (MLX 4-bit among the affine formats of the codec registry):
 *    the MLX 4-bit block is a 20-byte struct.  The pages give its size but
 *    not its fields; this oracle reads it as MLX's affine group quantization
 *    at group size 32: an fp16 scale s, an fp16 bias b and 16 bytes of 4-bit
 *    codes, w = q * s + b.  The planar form of the same weights (section 4:
 *    codes, scales and biases in separate 16-byte aligned arrays) is MLX's
 *    own storage, 32-bit words of eight codes each.
 *  - "v0.1 vs v0.2 comparison", section 2.3 (Brick 4: FlashAttention with a
 *    Q8_0 KV cache, dequantized on the fly), "Releases" v0.3.0
 *    (TransformerBlock: grouped-query attention, causal masking, RoPE
 *    sequence offsets; flash_attn core for head dims 64 and 128) and the
 *    project page, section 4 (Q, K, V projected straight into [H, M, D]):
 *    softmax attention O = softmax(scale * Q K^T) V per head, query head h
 *    reading KV head h / (H / Hkv), query i seeing keys j <= q_offset + i
 *    when causal.  FlashAttention computes exactly this (its online softmax
 *    is a reordering), so the oracle is the definition: scores, one max,
 *    exponentials, one sum, the weighted sum of V.  K and V cache values
 *    are the fp16 operands the attention multiplies: fp16 as stored, or a
 *    Q8_0 block along the head dimension decoded and rounded once to fp16.
 *  - "v0.1 vs v0.2 comparison", section 2.2 (dual-SIMDgroup SwiGLU): the
 *    fused projection is SiLU(X * Wg^T) x (X * Wu^T), with only the final
 *    activation written out.
 *  - "Releases", v0.3.0 (TransformerBlock: GeGLU listed beside SwiGLU,
 *    Gemma 2 configurations): the same gated projection with GELU in place
 *    of SiLU.  The pages do not define GELU; this oracle takes the textbook
 *    definition GELU(g) = g * Phi(g) = g/2 * erfc(-g / sqrt 2).
 *  - "v0.1 vs v0.2 comparison", section 2.1, and "Releases" v0.2.3: the
 *    unpackers feed half-precision MMA fragments (simdgroup_matrix<half,8,8>),
 *    so the weights the projection multiplies are fp16 values.  The oracle
 *    therefore rounds each decoded weight ((q - z) * d, or q * s + b) once to
 *    fp16 (nearest, ties to even) before the binary64 dot product;
 *    oracle_dequant keeps the exact values and oracle_dequant_f16 the rounded
 *    ones.
 *
 * Byte layouts (the reading this library takes; the pages print none):
 *  - Q4_0 (18 B): d (fp16, little-endian) then 16 bytes; byte j holds weight
 *    j in its low nibble and weight j + 16 in its high nibble.
 *  - Q8_0 (34 B): d then 32 signed bytes, weight i in byte i.
 *  - Q2_0 (34 B): d then 32 bytes; weight i is in byte i / 4 at bits
 *    2 * (i % 4) .. 2 * (i % 4) + 1 (least significant pair first).
 *  - MLX4 (20 B): s, then b (both fp16, little-endian), then 16 bytes; weight
 *    i is in byte i / 2, even i in the low nibble.  That is MLX's order: code
 *    k of a row sits at bits 4 * (k % 8) of little-endian 32-bit word k / 8.
 *
 * Parity note: the Q2_0 code order and the Q4_0/Q8_0 byte layouts cannot be
 * checked against real model files (none are available); they are pinned
 * only by hand-decoded golden blocks written from the layouts above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_Q4_0 = 0, ORACLE_Q8_0 = 1, ORACLE_Q2_0 = 2, ORACLE_MLX4 = 3 };

/* Weights per block, by codec. */
long long oracle_block_size(int codec) {
  switch (codec) {
    case ORACLE_Q4_0: return 32;
    case ORACLE_Q8_0: return 32;
    case ORACLE_Q2_0: return 128;
    case ORACLE_MLX4: return 32;
    default: return -1;
  }
}

/* Bytes per block, by codec: a 2-byte scale (and, for MLX4, a 2-byte bias)
 * plus the packed codes. */
long long oracle_block_bytes(int codec) {
  switch (codec) {
    case ORACLE_Q4_0: return 2 + 32 / 2;   /* 16 bytes of nibbles */
    case ORACLE_Q8_0: return 2 + 32;       /* 32 signed bytes */
    case ORACLE_Q2_0: return 2 + 128 / 4;  /* 32 bytes of 2-bit codes */
    case ORACLE_MLX4: return 4 + 32 / 2;   /* 16 bytes of nibbles */
    default: return -1;
  }
}

/* IEEE binary16 -> binary64, exact.  Written from the format definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);   /* 1.f * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* binary64 -> binary16, round to nearest, ties to even (one rounding). */
uint16_t oracle_double_to_half(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return (uint16_t)(sign | 0x7e00);
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: the quantum is 2^-24 */
    double r = nearbyint(a * 16777216.0);    /* exact scaling, then RNE */
    return (uint16_t)(sign | (uint16_t)r);   /* r == 1024 is the smallest normal */
  }
  int e2;
  (void)frexp(a, &e2);                       /* a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;                            /* unbiased half exponent */
  if (E > 15) return (uint16_t)(sign | 0x7c00);
  double r = nearbyint(ldexp(a, 10 - E));    /* significand in [1024, 2048] */
  if (r == 2048.0) { r = 1024.0; E += 1; }
  if (E > 15) return (uint16_t)(sign | 0x7c00);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)r - 1024));
}

/* Decode the integer code of weight i of one block (the byte layouts above). */
static int block_code(const uint8_t* blk, int codec, int i) {
  const uint8_t* qs = blk + (codec == ORACLE_MLX4 ? 4 : 2);
  switch (codec) {
    case ORACLE_Q4_0:
      return (i < 16) ? (qs[i] & 0x0f) : (qs[i - 16] >> 4);
    case ORACLE_Q8_0:
      return (int)(int8_t)qs[i];
    case ORACLE_Q2_0:
      return (qs[i / 4] >> (2 * (i % 4))) & 0x3;
    case ORACLE_MLX4:
      return (qs[i / 2] >> (4 * (i % 2))) & 0x0f;
    default:
      return 0;
  }
}

/* The code value that decodes to zero in the scale-only codecs: Q4_0 8,
 * Q8_0 0, Q2_0 1 (MLX4 has none: its zero point is the bias). */
static int code_zero(int codec) {
  return codec == ORACLE_Q4_0 ? 8 : (codec == ORACLE_Q2_0 ? 1 : 0);
}

/* Dequantize one row of W (K weights) into binary64.  Each weight is
 * (q - z) * d, or q * s + b for MLX4.  Both are exact in binary64: the
 * product of a <= 8-bit integer and an 11-bit significand has at most 19
 * significant bits, and q * s and b are integer multiples of 2^-24 below
 * 2^20 in magnitude, so their sum needs fewer than 53 bits. */
static void dequant_row(const uint8_t* row, int codec, long long K, double* out) {
  long long B = oracle_block_size(codec), BB = oracle_block_bytes(codec);
  int z = code_zero(codec);
  for (long long b = 0; b < K / B; ++b) {
    const uint8_t* blk = row + b * BB;
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    double d = oracle_half_to_double(dbits);
    if (codec == ORACLE_MLX4) {
      double bias = oracle_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
      for (long long i = 0; i < B; ++i) out[b * B + i] = (double)block_code(blk, codec, (int)i) * d + bias;
      continue;
    }
    for (long long i = 0; i < B; ++i) {
      int q = block_code(blk, codec, (int)i);
      out[b * B + i] = (double)(q - z) * d;
    }
  }
}

static int check_shape(int codec, long long N, long long K) {
  long long B = oracle_block_size(codec);
  if (B <= 0) return -2;
  if (N < 0 || K < 0 || K % B != 0) return -3;
  return 0;
}

/* Wd[n*K + k] = exact value of weight (n, k).  Returns 0 or a negative code. */
int oracle_dequant(const uint8_t* W, int codec, long long N, long long K, double* Wd) {
  int rc = check_shape(codec, N, K);
  if (rc) return rc;
  long long row_bytes = (K / oracle_block_size(codec)) * oracle_block_bytes(codec);
  for (long long n = 0; n < N; ++n) dequant_row(W + n * row_bytes, codec, K, Wd + n * K);
  return 0;
}

/* Wh[n*K + k] = binary16 bits of the weight rounded once (RNE) to fp16. */
int oracle_dequant_f16(const uint8_t* W, int codec, long long N, long long K, uint16_t* Wh) {
  int rc = check_shape(codec, N, K);
  if (rc) return rc;
  long long row_bytes = (K / oracle_block_size(codec)) * oracle_block_bytes(codec);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  if (!tmp) return -8;
  for (long long n = 0; n < N; ++n) {
    dequant_row(W + n * row_bytes, codec, K, tmp);
    for (long long k = 0; k < K; ++k) Wh[n * K + k] = oracle_double_to_half(tmp[k]);
  }
  free(tmp);
  return 0;
}

/* MLX planar arrays -> MLX4 blocks.  words [N, K/8]: code k of row n at bits
 * 4 * (k % 8) of words[n * K/8 + k / 8]; scales, biases [N, K/32] fp16 bits.
 * W receives N rows of K/32 blocks laid out as above.  Returns 0, or -3 when
 * K is not a multiple of 32. */
int oracle_mlx4_pack(const uint32_t* words, const uint16_t* scales, const uint16_t* biases,
                     long long N, long long K, uint8_t* W) {
  if (N < 0 || K < 0 || K % 32 != 0) return -3;
  long long nb = K / 32;
  for (long long n = 0; n < N; ++n) {
    for (long long b = 0; b < nb; ++b) {
      uint8_t* blk = W + (n * nb + b) * 20;
      uint16_t s = scales[n * nb + b], t = biases[n * nb + b];
      blk[0] = (uint8_t)(s & 0xff);
      blk[1] = (uint8_t)(s >> 8);
      blk[2] = (uint8_t)(t & 0xff);
      blk[3] = (uint8_t)(t >> 8);
      memset(blk + 4, 0, 16);
      for (int i = 0; i < 32; ++i) {
        long long k = 32 * b + i;
        int q = (int)((words[n * (K / 8) + k / 8] >> (4 * (k % 8))) & 0xf);
        blk[4 + i / 2] |= (uint8_t)(q << (4 * (i % 2)));
      }
    }
  }
  return 0;
}

/* Blocks -> planes: the one-time re-layout that splits the blocks of W into
 * separate arrays ("v0.1 vs v0.2 comparison", section 4, splits MLX 4-bit
 * blocks this way; the same split is taken here for every codec).  P receives,
 * back to back, with no padding:
 *   codes:  for each row n and block b in order, the block's code bytes,
 *           unchanged (16 bytes for Q4_0 and MLX4, 32 for Q8_0 and Q2_0);
 *   scales: fp16 [N, K/B], the scale d of each block (MLX4: s);
 *   biases: fp16 [N, K/B], MLX4 only, the bias b of each block.
 * P has as many bytes as W.  For MLX4 the three arrays are MLX's planar
 * arrays (the inverse of oracle_mlx4_pack).  Returns 0, -2 for an unknown
 * codec, -3 for a bad shape. */
int oracle_repack(const uint8_t* W, int codec, long long N, long long K, uint8_t* P) {
  int rc = check_shape(codec, N, K);
  if (rc) return rc;
  long long nb = K / oracle_block_size(codec), BB = oracle_block_bytes(codec);
  long long head = (codec == ORACLE_MLX4) ? 4 : 2; /* scale (and bias) bytes */
  long long CB = BB - head;                        /* code bytes per block */
  uint8_t* codes = P;
  uint8_t* scales = codes + N * nb * CB;
  uint8_t* biases = scales + 2 * N * nb;
  for (long long n = 0; n < N; ++n) {
    for (long long b = 0; b < nb; ++b) {
      long long i = n * nb + b;
      const uint8_t* blk = W + i * BB;
      memcpy(codes + i * CB, blk + head, (size_t)CB);
      scales[2 * i] = blk[0];
      scales[2 * i + 1] = blk[1];
      if (codec == ORACLE_MLX4) {
        biases[2 * i] = blk[2];
        biases[2 * i + 1] = blk[3];
      }
    }
  }
  return 0;
}

/* SiLU(g) = g * sigmoid(g) = g / (1 + e^-g), in binary64. */
double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* GELU(g) = g * Phi(g), Phi the standard normal CDF, in binary64.
 * Phi(g) = erfc(-g / sqrt 2) / 2, which does not cancel for negative g. */
double oracle_gelu(double g) { return 0.5 * g * erfc(-g / sqrt(2.0)); }

enum { ORACLE_ACT_SILU = 0, ORACLE_ACT_GELU = 1 };

/* ---- projections, split over output columns n across threads ---- */

typedef struct {
  const double* Xd;        /* [nrows, K] widened activations */
  const uint8_t* W0;       /* gate (SwiGLU) or the only weight (GEMM) */
  const uint8_t* W1;       /* up (gated projections) or NULL */
  int codec;
  int act;                 /* ORACLE_ACT_*: activation of the gate */
  long long nrows, N, K, row_bytes;
  long long n_begin, n_end;
  double* Y;               /* [nrows, N] */
  int rc;
} job_t;

static double dot(const double* a, const double* b, long long K) {
  double s = 0.0;
  for (long long k = 0; k < K; ++k) s += a[k] * b[k];
  return s;
}

/* The fp16 operand value of each decoded weight, widened back exactly. */
static void round_row_to_f16(double* w, long long K) {
  for (long long k = 0; k < K; ++k) w[k] = oracle_half_to_double(oracle_double_to_half(w[k]));
}

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  double* w0 = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
  double* w1 = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
  if (!w0 || !w1) { free(w0); free(w1); j->rc = -8; return NULL; }
  for (long long n = j->n_begin; n < j->n_end; ++n) {
    dequant_row(j->W0 + n * j->row_bytes, j->codec, j->K, w0);
    round_row_to_f16(w0, j->K);
    if (j->W1) {
      dequant_row(j->W1 + n * j->row_bytes, j->codec, j->K, w1);
      round_row_to_f16(w1, j->K);
    }
    for (long long r = 0; r < j->nrows; ++r) {
      const double* x = j->Xd + r * j->K;
      double g = dot(x, w0, j->K);
      if (j->W1) {
        double u = dot(x, w1, j->K);
        j->Y[r * j->N + n] = (j->act == ORACLE_ACT_GELU ? oracle_gelu(g) : oracle_silu(g)) * u;
      } else {
        j->Y[r * j->N + n] = g;
      }
    }
  }
  free(w0);
  free(w1);
  j->rc = 0;
  return NULL;
}

static int project(const uint16_t* X, const uint8_t* W0, const uint8_t* W1, int codec, int act,
                   long long M, long long N, long long K, const long long* rows,
                   long long nrows, double* Y, int nthreads) {
  int rc = check_shape(codec, N, K);
  if (rc) return rc;
  if (M < 0 || nrows < 0) return -3;
  if (!rows) nrows = M;
  double* Xd = (double*)malloc(sizeof(double) * (size_t)((nrows * K) > 0 ? nrows * K : 1));
  if (!Xd) return -8;
  for (long long r = 0; r < nrows; ++r) {
    long long m = rows ? rows[r] : r;
    if (m < 0 || m >= M) { free(Xd); return -1; }
    for (long long k = 0; k < K; ++k) Xd[r * K + k] = oracle_half_to_double(X[m * K + k]);
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (N < nthreads) nthreads = (int)(N > 0 ? N : 1);
  job_t jobs[256];
  pthread_t tids[256];
  long long row_bytes = (K / oracle_block_size(codec)) * oracle_block_bytes(codec);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (job_t){Xd, W0, W1, codec, act, nrows, N, K, row_bytes,
                      N * t / nthreads, N * (t + 1) / nthreads, Y, 0};
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, run_job, &jobs[t]) != 0) break;
    started = t;
  }
  run_job(&jobs[0]);
  /* any job whose thread did not start runs here */
  for (int t = started + 1; t < nthreads; ++t) run_job(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  free(Xd);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].rc) return jobs[t].rc;
  return 0;
}

/* Y[r, n] = sum_k X[rows[r], k] * fp16(W[n, k])  (rows == NULL: every row of X).
 * X is fp16 bits [M, K]; W is packed [N, K / block] blocks; Y is [nrows, N]. */
int oracle_gemm(const uint16_t* X, const uint8_t* W, int codec, long long M, long long N,
                long long K, const long long* rows, long long nrows, double* Y, int nthreads) {
  return project(X, W, NULL, codec, ORACLE_ACT_SILU, M, N, K, rows, nrows, Y, nthreads);
}

/* Y[r, n] = SiLU(G) * U with G = X Wg^T, U = X Wu^T, both in binary64. */
int oracle_swiglu(const uint16_t* X, const uint8_t* Wg, const uint8_t* Wu, int codec,
                  long long M, long long N, long long K, const long long* rows,
                  long long nrows, double* Y, int nthreads) {
  if (!Wu) return -1;
  return project(X, Wg, Wu, codec, ORACLE_ACT_SILU, M, N, K, rows, nrows, Y, nthreads);
}

/* Y[r, n] = GELU(G) * U with G = X Wg^T, U = X Wu^T, both in binary64. */
int oracle_geglu(const uint16_t* X, const uint8_t* Wg, const uint8_t* Wu, int codec,
                 long long M, long long N, long long K, const long long* rows,
                 long long nrows, double* Y, int nthreads) {
  if (!Wu) return -1;
  return project(X, Wg, Wu, codec, ORACLE_ACT_GELU, M, N, K, rows, nrows, Y, nthreads);
}

/* ---- attention over a KV cache ---- */

enum { ORACLE_KV_F16 = 16 };

typedef struct {
  const uint16_t* Q;    /* fp16 bits [H, M, D] */
  const uint8_t* K;     /* [Hkv, T] rows of D values: fp16 or Q8_0 blocks */
  const uint8_t* V;
  int kv_codec;
  long long H, Hkv, M, T, D, q_offset;
  int causal;
  double scale;
  const long long* qrows; /* query indices to compute (NULL: all M) */
  long long nq;
  long long h_begin, h_end;
  double* O;            /* [nq, H * D] */
  int rc;
} attn_job_t;

/* Row j of one KV head as binary64 values of the fp16 operands. */
static void kv_row(const uint8_t* base, int kv_codec, long long D, double* out) {
  if (kv_codec == ORACLE_KV_F16) {
    const uint16_t* h = (const uint16_t*)base;
    for (long long d = 0; d < D; ++d) out[d] = oracle_half_to_double(h[d]);
    return;
  }
  dequant_row(base, ORACLE_Q8_0, D, out);
  round_row_to_f16(out, D);
}

static void* run_attn(void* arg) {
  attn_job_t* j = (attn_job_t*)arg;
  const long long D = j->D, T = j->T, G = j->H / j->Hkv;
  const long long kv_bytes = j->kv_codec == ORACLE_KV_F16 ? 2 * D : (D / 32) * 34;
  double* Kd = (double*)malloc(sizeof(double) * (size_t)(T * D > 0 ? T * D : 1));
  double* Vd = (double*)malloc(sizeof(double) * (size_t)(T * D > 0 ? T * D : 1));
  double* s = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  double* q = (double*)malloc(sizeof(double) * (size_t)D);
  if (!Kd || !Vd || !s || !q) { free(Kd); free(Vd); free(s); free(q); j->rc = -8; return NULL; }
  long long cached = -1;
  for (long long h = j->h_begin; h < j->h_end; ++h) {
    const long long hk = h / G;
    if (hk != cached) {
      for (long long t = 0; t < T; ++t) {
        kv_row(j->K + (hk * T + t) * kv_bytes, j->kv_codec, D, Kd + t * D);
        kv_row(j->V + (hk * T + t) * kv_bytes, j->kv_codec, D, Vd + t * D);
      }
      cached = hk;
    }
    for (long long r = 0; r < j->nq; ++r) {
      const long long i = j->qrows ? j->qrows[r] : r;
      for (long long d = 0; d < D; ++d) q[d] = oracle_half_to_double(j->Q[(h * j->M + i) * D + d]);
      long long nvis = T;
      if (j->causal && j->q_offset + i + 1 < nvis) nvis = j->q_offset + i + 1;
      double* o = j->O + r * j->H * D + h * D;
      if (nvis <= 0) {
        for (long long d = 0; d < D; ++d) o[d] = 0.0;
        continue;
      }
      double mx = -INFINITY;
      for (long long t = 0; t < nvis; ++t) {
        s[t] = j->scale * dot(q, Kd + t * D, D);
        if (s[t] > mx) mx = s[t];
      }
      double l = 0.0;
      for (long long t = 0; t < nvis; ++t) {
        s[t] = exp(s[t] - mx);
        l += s[t];
      }
      for (long long d = 0; d < D; ++d) {
        double acc = 0.0;
        for (long long t = 0; t < nvis; ++t) acc += s[t] * Vd[t * D + d];
        o[d] = acc / l;
      }
    }
  }
  free(Kd); free(Vd); free(s); free(q);
  j->rc = 0;
  return NULL;
}

/* O[r, h*D + d] = sum_j softmax_j(scale * Q[h, i] . K[hk, j]) V[hk, j, d] for
 * query i = qrows[r] (all M when qrows is NULL), over the keys the query
 * sees.  kv_codec: ORACLE_KV_F16 (fp16 bits) or ORACLE_Q8_0 (D % 32 == 0).
 * A query that sees no key (causal with q_offset + i < 0) gets O = 0.
 * Returns 0 or a negative code. */
int oracle_attention(const uint16_t* Q, const uint8_t* K, const uint8_t* V, int kv_codec,
                     long long H, long long Hkv, long long M, long long T, long long D,
                     long long q_offset, int causal, double scale, const long long* qrows,
                     long long nq, double* O, int nthreads) {
  if (kv_codec != ORACLE_KV_F16 && kv_codec != ORACLE_Q8_0) return -2;
  if (H < 1 || Hkv < 1 || H % Hkv != 0 || M < 0 || T < 0 || D < 1) return -3;
  if (kv_codec == ORACLE_Q8_0 && D % 32 != 0) return -3;
  if (!qrows) nq = M;
  for (long long r = 0; qrows && r < nq; ++r)
    if (qrows[r] < 0 || qrows[r] >= M) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (H < nthreads) nthreads = (int)H;
  attn_job_t jobs[256];
  pthread_t tids[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (attn_job_t){Q, K, V, kv_codec, H, Hkv, M, T, D, q_offset, causal, scale, qrows, nq,
                           H * t / nthreads, H * (t + 1) / nthreads, O, 0};
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, run_attn, &jobs[t]) != 0) break;
    started = t;
  }
  run_attn(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) run_attn(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].rc) return jobs[t].rc;
  return 0;
}
