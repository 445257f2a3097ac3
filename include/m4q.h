/*
 * m4q.h -- C ABI of the block-quantized projection library for one GB300
 * (sm_103a).  Shared object: swiglu_block_quantized_gb300/_build/libm4q.so.
 *
 * The operation (m4-prefill-engine pages):
 *  - "v0.1 vs v0.2 comparison", section 2.1, and the project page's Pillar 1
 *    (Bricks 1 and 2): the prefill projection Y[M,N] = X[M,K] * W^T with fp16
 *    activations and block-quantized weights unpacked inside the kernel.
 *  - "Releases", v0.3.0 (M4QuantizedLinear): one linear layer dispatches to a
 *    GEMV for decode-sized M and to a GEMM otherwise, across every codec.
 *  - "v0.1 vs v0.2 comparison", section 2.2 (Brick 3): the fused gate/up
 *    projection SiLU(X * Wg^T) x (X * Wu^T), computed on chip, writing only
 *    the final activation.  "Releases" v0.3.0 (TransformerBlock: SwiGLU /
 *    GeGLU activations) adds the GELU-gated form, GELU(g) = g * Phi(g).
 *  - "Releases", v0.3.0, PrismML Q2_0 codec: 128 weights in 34 bytes,
 *    w = (q - 1) * d with the reserved code 3 decoding to +2d.  Q4_0 and Q8_0
 *    are GGUF's 32-weight blocks: w = (q - 8) * d and w = q * d.
 *  - Project page, section 4 (v0.2.1) and Table B: MLX 4-bit weights, a
 *    20-byte block_mlx_4bit and its planar form.  Read as MLX's affine group
 *    quantization at group size 32: w = q * s + b with an fp16 scale s and
 *    bias b per group of 32 weights.
 *
 * Conventions common to every call:
 *  - Pointers X, W, Wg, Wu, Y, Wf16 are DEVICE pointers (cudaMalloc'd or from
 *    PyTorch).  The caller owns every buffer; the library allocates nothing
 *    during a call and keeps no pointer after it returns.
 *  - Layouts are row-major and dense.  X is fp16 [M, K]; Y is fp16 [M, N].
 *    W is [N rows][K / B blocks] of packed blocks (B = 32 for Q4_0, Q8_0 and
 *    MLX4, 128 for Q2_0), block bytes 18 / 34 / 34 / 20, each block a
 *    little-endian fp16 scale d followed by its codes:
 *      Q4_0: byte 2+j holds weight j in its low nibble, weight j+16 high;
 *      Q8_0: byte 2+i holds weight i as a signed byte;
 *      Q2_0: byte 2+i/4 holds weight i at bits 2*(i%4)..2*(i%4)+1;
 *      MLX4: bytes 2-3 hold the fp16 bias b, byte 4+i/2 holds weight i,
 *            even i in the low nibble (MLX's order; m4q_mlx4_pack builds
 *            these blocks from MLX's planar arrays).
 *  - Shapes: M >= 1, N >= 8 with N % 8 == 0, K >= B with K % B == 0.
 *    X, W, Wg, Wu, Y must be 16-byte aligned.
 *  - Arithmetic: every weight is decoded to fp16 as (q - z) * d (MLX4:
 *    q * s + b) rounded once to nearest even, products are accumulated in
 *    fp32, and each output is
 *    rounded once to fp16 (SiLU(g) * u or GELU(g) * u is formed in fp32
 *    first).
 *  - Asynchrony: calls enqueue work on `stream` and return; argument errors
 *    are returned before anything is enqueued.  Launch failures return
 *    M4Q_ERR_CUDA.  Device-side failures (a pipeline wait that gave up) are
 *    recorded in a device status word that m4q_check_device_status() reads.
 *  - Threading: calls may be made from several host threads.
 */
#ifndef M4Q_H_
#define M4Q_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t.  NULL means the legacy default stream. */
typedef struct CUstream_st* m4q_stream_t;

/* Weight codecs. */
enum m4q_codec { M4Q_Q4_0 = 0, M4Q_Q8_0 = 1, M4Q_Q2_0 = 2, M4Q_MLX4 = 3 };

/* Execution paths for m4q_gemm_ex / m4q_swiglu_ex. */
enum m4q_path {
  M4Q_PATH_AUTO = 0, /* M <= 16: streaming GEMV; otherwise the tensor-core GEMM */
  M4Q_PATH_GEMV = 1, /* weight-streaming GEMV (requires M <= 16) */
  M4Q_PATH_TC = 2    /* tcgen05 tensor-core GEMM (any M) */
};

/* Activations of the gated projection (m4q_glu_ex). */
enum m4q_act {
  M4Q_ACT_SILU = 0, /* SiLU(g) = g / (1 + e^-g): SwiGLU */
  M4Q_ACT_GELU = 1  /* GELU(g) = g * Phi(g) = g/2 * erfc(-g / sqrt 2): GeGLU */
};

/* Status codes returned by every call. */
enum m4q_status {
  M4Q_OK = 0,
  M4Q_ERR_INVALID_ARG = -1,        /* null pointer, M/N/K out of range, bad path */
  M4Q_ERR_UNSUPPORTED_CODEC = -2,  /* codec not one of enum m4q_codec */
  M4Q_ERR_BAD_SHAPE = -3,          /* K % B != 0 or N % 8 != 0 */
  M4Q_ERR_MISALIGNED = -4,         /* a pointer is not 16-byte aligned */
  M4Q_ERR_CUDA = -5,               /* a CUDA runtime call or launch failed */
  M4Q_ERR_NONFINITE = -6,          /* m4q_check_finite found NaN/Inf */
  M4Q_ERR_TIMEOUT = -7,            /* a device pipeline wait gave up */
  M4Q_ERR_UNSUPPORTED_DEVICE = -8, /* the current device is not sm_103 */
  M4Q_ERR_SCRATCH_LIMIT = -9,      /* m4q_mlp_noalloc: M * F above its fixed scratch */
  M4Q_ERR_BOUNDS = -10             /* bounds-checked build: an access was out of range */
};

/* Y = X * W^T.  Dispatch: M <= 16 takes the GEMV path, else the tcgen05
 * path.  Errors as listed in enum m4q_status. */
int m4q_gemm(const void* X, const void* W, int codec, int64_t M, int64_t N, int64_t K,
             void* Y, m4q_stream_t stream);

/* Y = SiLU(X * Wg^T) x (X * Wu^T); Wg and Wu share codec and shape [N, K].
 * Neither intermediate product is written to memory. */
int m4q_swiglu(const void* X, const void* Wg, const void* Wu, int codec, int64_t M,
               int64_t N, int64_t K, void* Y, m4q_stream_t stream);

/* Y = X * W^T written head-major: Y[h][m][d] = (X * W^T)[m][h * head_dim + d],
 * Y fp16 [N / head_dim][M][head_dim], so each head's [M, head_dim] block is
 * contiguous and attention reads it without a transpose ("v0.1 vs v0.2
 * comparison" section 4 and "Releases" v0.2.1: direct-head [H, M, D]
 * projection).  head_dim is 64 or 128 (else M4Q_ERR_INVALID_ARG) and must
 * divide N (else M4Q_ERR_BAD_SHAPE).  A fused Q/K/V projection is one call
 * on the row concatenation of Wq, Wk and Wv (packed rows are independent, so
 * concatenating the packed matrices concatenates the rows): the first
 * N_q / head_dim heads of Y are Q, then K, then V.  Otherwise as m4q_gemm. */
int m4q_gemm_heads(const void* X, const void* W, int codec, int64_t M, int64_t N, int64_t K,
                   int64_t head_dim, void* Y, m4q_stream_t stream);

/* Y = GELU(X * Wg^T) x (X * Wu^T) ("Releases" v0.3.0, GeGLU); otherwise as
 * m4q_swiglu. */
int m4q_geglu(const void* X, const void* Wg, const void* Wu, int codec, int64_t M,
              int64_t N, int64_t K, void* Y, m4q_stream_t stream);

/* As m4q_gemm / m4q_swiglu, with the path chosen by the caller (enum m4q_path). */
int m4q_gemm_ex(const void* X, const void* W, int codec, int64_t M, int64_t N, int64_t K,
                void* Y, int path, m4q_stream_t stream);
int m4q_swiglu_ex(const void* X, const void* Wg, const void* Wu, int codec, int64_t M,
                  int64_t N, int64_t K, void* Y, int path, m4q_stream_t stream);

/* The gated projection Y = act(X * Wg^T) x (X * Wu^T) with the activation
 * (enum m4q_act) and the path (enum m4q_path) chosen by the caller.  An
 * unknown act returns M4Q_ERR_INVALID_ARG. */
int m4q_glu_ex(const void* X, const void* Wg, const void* Wu, int codec, int64_t M, int64_t N,
               int64_t K, void* Y, int act, int path, m4q_stream_t stream);

/* The gated MLP block of a transformer layer ("Releases" v0.3.0:
 * TransformerBlock with SwiGLU / GeGLU activations):
 *     H = act(X * Wg^T) x (X * Wu^T)      fp16 [M, F]
 *     Y = H * Wd^T                         fp16 [M, D]
 * enqueued as two launches on `stream` (the gated projection, then the down
 * projection), each with the M <= 16 / tcgen05 dispatch of m4q_gemm.
 * X is fp16 [M, D]; Wg, Wu are packed [F, D] in codec_gu; Wd is packed
 * [D, F] in codec_d.  H is caller-provided device scratch of M * F fp16
 * (16-byte aligned) that receives the intermediate activation; it may be
 * reused once the call's work on `stream` has completed.  Shape rules of
 * m4q_gemm apply to both projections (D and F multiples of 8 and of the
 * block sizes).  act: enum m4q_act. */
int m4q_mlp(const void* X, const void* Wg, const void* Wu, const void* Wd, int codec_gu,
            int codec_d, int64_t M, int64_t D, int64_t F, void* H, void* Y, int act,
            m4q_stream_t stream);

/* m4q_mlp for callers that cannot allocate device memory (a runtime that
 * owns all device memory and gives plug-ins no allocator, or a loop that must
 * not call cudaMalloc, which may synchronize the device).  The pages have no
 * counterpart: this is a deployment variant of m4q_mlp.  Same arguments and
 * result as m4q_mlp without H: the fp16 intermediate is kept in one fixed
 * device array of the library, 1 << 20 elements (2 MiB, held on every GPU
 * that loads the library until the process exits).  M * F above that returns
 * M4Q_ERR_SCRATCH_LIMIT before anything is enqueued.  The call allocates
 * nothing.  The first call on a device checks that it is an sm_103 part
 * (else M4Q_ERR_UNSUPPORTED_DEVICE), looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process; it should
 * come before any stream capture on that device.  cudaDeviceReset() on a
 * device makes the kept address stale: do not call this entry point on that
 * device afterwards.  All calls share the array: each one overwrites the part
 * it uses before reading it, but calls whose work overlaps on the GPU (no
 * stream order between them) race. */
int m4q_mlp_noalloc(const void* X, const void* Wg, const void* Wu, const void* Wd, int codec_gu,
                    int codec_d, int64_t M, int64_t D, int64_t F, void* Y, int act,
                    m4q_stream_t stream);

/* The projection of m4q_gemm (W1 == NULL) or the gated projection of
 * m4q_glu_ex (W1 != NULL, activation `act`) with the activations in host
 * memory and the result written to host memory: the end-to-end call of a
 * caller whose inputs arrive from the host.  M is cut into chunks of
 * `chunk_rows` rows (0: about a quarter of M, rounded up to 128 rows); each
 * chunk's activations are copied to the device on `h2d_stream`, projected on
 * `stream` (the dispatch of m4q_gemm / m4q_glu_ex with path AUTO) and
 * copied back on `d2h_stream`, so the copies of one chunk overlap the
 * kernels of its neighbours.  The copies overlap only if X_host and Y_host
 * are page-locked (cudaHostAlloc / pinned); otherwise the result is the same
 * and the copies serialize.
 *  - X_host: fp16 [M, K]; Y_host: fp16 [M, N] (host memory).
 *  - X_dev, Y_dev: device staging buffers of M * K and M * N fp16, 16-byte
 *    aligned, owned by the caller (the library allocates no memory).
 *  - W0, W1: packed device weights as for m4q_gemm / m4q_glu_ex.
 *  - Ordering: the copies start after the work already enqueued on
 *    `stream`, and `stream` waits for the last copy back, so work enqueued
 *    on `stream` after this call, and a synchronization of `stream`, see
 *    Y_host complete.  The three streams should be distinct for overlap.
 *  - The call records CUDA events of a per-device pool, created by the first
 *    call on a device; calls from several host threads are serialized while
 *    they enqueue.
 * Errors: those of m4q_gemm / m4q_glu_ex (checked before anything is
 * enqueued), M4Q_ERR_INVALID_ARG for a null host or staging pointer or a
 * negative chunk_rows, M4Q_ERR_MISALIGNED for unaligned staging buffers. */
int m4q_project_host(const void* X_host, const void* W0, const void* W1, int codec, int act, int64_t M,
                     int64_t N, int64_t K, void* Y_host, void* X_dev, void* Y_dev, int64_t chunk_rows,
                     m4q_stream_t stream, m4q_stream_t h2d_stream, m4q_stream_t d2h_stream);

/* Repack MLX 4-bit weights from MLX's planar arrays into MLX4 blocks
 * (project page, section 4: the deinterleaved "mlx_4bit_planar" layout of
 * the 20-byte block_mlx_4bit).  words: uint32 [N, K/8], code k of row n at
 * bits 4*(k%8) of word k/8 (little-endian); scales, biases: fp16 [N, K/32],
 * one per group of 32 weights.  W receives [N, K/32] 20-byte blocks
 * (m4q_weight_bytes(M4Q_MLX4, N, K) bytes) for any call above.  A one-time
 * layout step, not part of a projection: the tensor-core path moves whole
 * 160-byte stages of 8 blocks by TMA, so the 20-byte block stride never
 * splits a copy.  Requires N >= 1, K >= 32 with K % 32 == 0 (else
 * M4Q_ERR_BAD_SHAPE); words and W 16-byte aligned, scales and biases 2-byte
 * aligned (else M4Q_ERR_MISALIGNED).  Device pointers; enqueued on stream. */
int m4q_mlx4_pack(const void* words, const void* scales, const void* biases, int64_t N, int64_t K,
                  void* W, m4q_stream_t stream);

/* Split packed weights into planes ("v0.1 vs v0.2 comparison", section 4:
 * the v0.2.1 planar layout, which moves the codes of the 20-byte MLX 4-bit
 * blocks into their own 16-byte aligned array; the same split is offered for
 * every codec).  W: packed [N, K/B] blocks in `codec`.  Wplanar receives, back
 * to back with no padding, m4q_weight_bytes(codec, N, K) bytes in all:
 *   codes:  the code bytes of every block, unchanged, in row-major block
 *           order (16 bytes per block for Q4_0 and MLX4, 32 for Q8_0 and
 *           Q2_0), at offset 0;
 *   scales: fp16 [N, K/B], each block's scale d (MLX4: s), right after;
 *   biases: fp16 [N, K/B], MLX4 only, each block's bias b, after the scales.
 * For MLX4 the three arrays are MLX's own planar arrays (the inverse of
 * m4q_mlx4_pack).  The projections above read the packed blocks, never the
 * planes: this is an export for callers that store or hand on weights in
 * planar form.  Requires a known codec (else M4Q_ERR_UNSUPPORTED_CODEC),
 * N >= 1, K >= 1 (else M4Q_ERR_INVALID_ARG) with K % B == 0 (else
 * M4Q_ERR_BAD_SHAPE), W and Wplanar 16-byte aligned (else
 * M4Q_ERR_MISALIGNED) and not overlapping (not checked).  Device pointers;
 * enqueued on stream; the caller owns both buffers. */
int m4q_repack(const void* W, int codec, int64_t N, int64_t K, void* Wplanar, m4q_stream_t stream);

/* KV cache value formats for m4q_attention: fp16 values, or M4Q_Q8_0 blocks
 * along the head dimension. */
enum m4q_kv_codec { M4Q_KV_F16 = 16 };

/* Attention of fp16 queries over a KV cache ("v0.1 vs v0.2 comparison" 2.3:
 * FlashAttention with the Q8_0 KV cache dequantized on the fly; "Releases"
 * v0.3.0: grouped-query attention, causal masking with a sequence offset,
 * head dims 64 and 128; v0.2: chunked attention, running max and sum merged
 * exactly across key chunks):
 *   O[i, h*D + d] = sum_j softmax_j(scale * Q[h, i, :] . K[h / G, j, :]) V[h / G, j, d]
 * with G = H / Hkv, over keys j < T, and, when causal != 0, j <= q_offset + i.
 *  - Q: fp16 [H, M, D] (head-major, as m4q_gemm_heads writes it).
 *  - K, V: [Hkv, T] rows of D values: fp16 (kv_codec M4Q_KV_F16, 2 D bytes a
 *    row) or Q8_0 (kv_codec M4Q_Q8_0: D / 32 blocks of 34 bytes a row, the
 *    same block as the Q8_0 weights).  Each value enters the products as
 *    fp16 (Q8_0: RNE(q * d)).
 *  - O: fp16 [M, H * D] (token-major: the o-projection's input).
 *  - D is 64 or 128, H % Hkv == 0 (else M4Q_ERR_BAD_SHAPE); M, T >= 1,
 *    q_offset >= 0, scale finite (else M4Q_ERR_INVALID_ARG; the usual scale
 *    is 1 / sqrt(D)); Q, K, V, O and workspace 16-byte aligned.
 *  - Scores and the softmax are fp32; the probabilities are rounded to fp16
 *    for the P V product, which accumulates in fp32; O is rounded once.
 *  - workspace (m4q_attention_workspace() bytes of device memory, owned by
 *    the caller): when the query rows alone would leave SMs idle (decode),
 *    the keys are split across CTAs and merged by a second kernel, which
 *    keeps its partial results there; for a Q8_0 cache under a prefill-sized
 *    call (more than 16 rows per KV head) both caches are first decoded to
 *    fp16 there (RNE(q * d), as above), since every key tile is read by each
 *    row tile of its KV head, and the fp16 tensor-core path runs on them.
 *    NULL (or a smaller size) runs without either: the same result up to
 *    fp32 rounding, slower.  The library allocates nothing. */
int m4q_attention(const void* Q, const void* K, const void* V, int kv_codec, int64_t H, int64_t Hkv,
                  int64_t M, int64_t T, int64_t D, int64_t q_offset, int causal, float scale, void* O,
                  void* workspace, size_t workspace_bytes, m4q_stream_t stream);

/* Bytes of the key split's partial results m4q_attention keeps in its
 * workspace for this shape on the current device (0: no key split; also 0
 * for an invalid shape).  m4q_attention_workspace covers the Q8_0 staging
 * as well. */
size_t m4q_attention_workspace_bytes(int64_t H, int64_t Hkv, int64_t M, int64_t T, int64_t D);

/* Workspace bytes m4q_attention uses for this cache format and shape on the
 * current device: the key split's partial results, or for a Q8_0 cache
 * under a prefill-sized call 2 Hkv T D fp16 values (the decoded caches);
 * 0 when it uses none, or for an invalid shape. */
size_t m4q_attention_workspace(int kv_codec, int64_t H, int64_t Hkv, int64_t M, int64_t T, int64_t D);

/* Decode W [N, K] to fp16 Wf16 [N, K] (row-major): each weight (q - z) * d
 * (MLX4: q * s + b) rounded once to nearest even.  The test hook for
 * bit-exact decoding. */
int m4q_dequant(const void* W, int codec, int64_t N, int64_t K, void* Wf16,
                m4q_stream_t stream);

/* Bytes of a packed [N, K] weight matrix: N * (K / B) * block_bytes, or 0 for
 * an unknown codec or a K that is not a multiple of B. */
size_t m4q_weight_bytes(int codec, int64_t N, int64_t K);

/* NaN/Inf tripwire (the pages' "Releases" v0.3.0 bridge and the "v0.1 vs
 * v0.2 comparison" metrology table: a non-finite output is a hard failure).
 * Scans the device fp16 array x[n], synchronizes `stream` and returns
 * M4Q_ERR_NONFINITE if any element is NaN or +-Inf, M4Q_OK otherwise. */
int m4q_check_finite(const void* x, int64_t n, m4q_stream_t stream);

/* Synchronize `stream`, read and clear the current device's status word.
 * Returns M4Q_ERR_BOUNDS if, in a bounds-checked build, a kernel found an
 * index out of range since the last check (the site stays readable through
 * m4q_bounds_site until then), else M4Q_ERR_TIMEOUT if a kernel's bounded
 * pipeline wait gave up, else M4Q_OK. */
int m4q_check_device_status(m4q_stream_t stream);

/* Bounds-checked build (compiled with -DM4Q_BOUNDS=1, for tests): every
 * computed global access, every TMA coordinate and every computed
 * shared-memory staging offset of the projection and attention kernels is
 * tested against the extents the kernel was given before it is made; a
 * failing access is skipped and reported (M4Q_ERR_BOUNDS above) instead of
 * faulting.  m4q_build_flags() returns M4Q_BUILD_BOUNDS for such a build,
 * 0 for the normal one.  m4q_bounds_site() synchronizes `stream` and returns
 * the site number of the first failed check since the previous call (0: none;
 * the numbers are listed in the library source), clearing it; it returns
 * M4Q_ERR_CUDA (negative) if the status word cannot be read. */
#define M4Q_BUILD_BOUNDS 1
int m4q_build_flags(void);
int m4q_bounds_site(m4q_stream_t stream);

/* Self-test of the bounded wait: launches one block that waits on a barrier
 * nothing will complete, with a limit of `limit_ns` nanoseconds; the kernel
 * records the timeout in the status word and returns.  The caller then sees
 * M4Q_ERR_TIMEOUT from m4q_check_device_status().  Nothing faults or hangs. */
int m4q_selftest_wait_timeout(int64_t limit_ns, m4q_stream_t stream);

/* Human-readable text of a status code (static storage). */
const char* m4q_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int m4q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* M4Q_H_ */
