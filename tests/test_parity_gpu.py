"""GPU parity: every call of the C ABI against the CPU oracle on the same
seeded inputs.

Tolerance: per element |gpu - ref| <= 1e-2 * max(1, |ref|) with ref the
binary64 oracle (fp32 accumulation, one fp16 rounding of the output).  The
fp16 decode (m4q_dequant, and the tcgen05 path read out through X = I) must
equal the oracle's once-rounded weights bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
import swiglu_block_quantized_gb300 as m
from _helpers import TOL, assert_close, dev, host, sample_rows

pytestmark = pytest.mark.gpu

CODECS = [synth.Q4_0, synth.Q8_0, synth.Q2_0, synth.MLX4]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load()
    yield
    assert m.check_device_status() == m.OK


def kvals(codec, general):
    """K values: multiples of the packed stage (TMA weights) or not (plain loads)."""
    if codec == synth.Q2_0:
        return [1024, 2048] if not general else [128, 384, 1152]
    if codec == synth.MLX4:
        # 384: 240-byte rows, TMA-able, the last 160-byte stage half past the row end
        return [256, 384] if not general else [32, 96, 288]
    return [256, 512] if not general else [32, 96, 288]


# ------------------------------------------------------------ dequant export

@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("K", [128, 256, 1024, 1152])
def test_dequant_bit_exact(codec, K):
    N = 40
    W = synth.weights(codec, N, K, seed=K)
    got = host(m.dequant(dev(W), codec, N, K)).view(np.uint16)
    assert np.array_equal(got, oracle.dequant_f16(W, codec, N, K))


@pytest.mark.parametrize("codec", CODECS)
def test_dequant_special_scales(codec):
    # subnormal, zero, negative, large (overflow to inf) and NaN scales
    B = synth.BLOCK[codec]
    specials = np.array([0x0001, 0x03FF, 0x0000, 0x8000, 0xBC00, 0x7BFF, 0x7800, 0x7E00, 0x3C00],
                        dtype=np.uint16).view(np.float16)
    N, K = 8, B * len(specials)
    q = synth.codes(codec, N, K, seed=1, name="W")
    d = np.tile(specials, (N, 1))
    W = synth.pack(codec, q, d)
    got = host(m.dequant(dev(W), codec, N, K)).view(np.uint16)
    ref = oracle.dequant_f16(W, codec, N, K)
    nan = (ref & 0x7C00) == 0x7C00
    nan &= (ref & 0x03FF) != 0
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(((got[nan] & 0x7C00) == 0x7C00) & ((got[nan] & 0x3FF) != 0))


@pytest.mark.parametrize("K", [32, 256, 384])
def test_mlx4_dequant_special_biases(K):
    # Biases that are subnormal, signed zeros, large (q * s + b overflows to
    # inf for the larger codes) or NaN, with ordinary and zero scales.
    N = 16
    specials = np.array([0x0001, 0x8000, 0x0000, 0x7BFF, 0xFBFF, 0x7E00, 0x3555, 0xB001],
                        dtype=np.uint16).view(np.float16)
    nb = K // 32
    q = synth.codes(synth.MLX4, N, K, seed=K, name="W")
    d = np.where(np.arange(N * nb).reshape(N, nb) % 3 == 0, np.float16(0), np.float16(2.0)).astype(np.float16)
    b = specials[np.arange(N * nb).reshape(N, nb) % len(specials)]
    W = synth.pack(synth.MLX4, q, d, b)
    got = host(m.dequant(dev(W), synth.MLX4, N, K)).view(np.uint16)
    ref = oracle.dequant_f16(W, synth.MLX4, N, K)
    nan = ((ref & 0x7C00) == 0x7C00) & ((ref & 0x03FF) != 0)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(((got[nan] & 0x7C00) == 0x7C00) & ((got[nan] & 0x3FF) != 0))


@pytest.mark.parametrize("N,K", [(8, 32), (40, 256), (264, 4096), (3000, 2048)])
def test_mlx4_pack_bit_exact(N, K):
    # MLX planar arrays -> blocks on the GPU equals the oracle's repack byte
    # for byte, and the repacked weights project like the generator's blocks.
    import torch
    q = synth.codes(synth.MLX4, N, K, seed=N, name="W")
    d = synth.scales(synth.MLX4, N, K, seed=N, name="W")
    b = synth.biases(synth.MLX4, N, K, seed=N, name="W", d=d)
    words, s, bb = synth.planar(q, d, b)
    wt = torch.from_numpy(words.view(np.int32)).cuda()
    got = host(m.mlx4_pack(wt, dev(s), dev(bb), N, K))
    assert np.array_equal(got, oracle.mlx4_pack(words, s, bb, N, K))
    if N <= 264:
        X = synth.activations(20, K, seed=5)
        Y = host(m.gemm(dev(X), dev(got), synth.MLX4, N, K))
        assert_close(Y, oracle.gemm(X, synth.pack(synth.MLX4, q, d, b), synth.MLX4, 20, N, K), "packed mlx4")


# ------------------------------------------------------------ tcgen05 path

@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("general", [False, True])
def test_tc_identity_readout_bit_exact(codec, general):
    # X = I (M = K): every output is one exact product 1 * w, so Y^T must be
    # the fp16 weights bit for bit -- checks decode, TMEM operand layout and
    # the epilogue indexing of the tensor-core path at once.
    K = kvals(codec, general)[0]
    N = 136   # two weight tiles, the second ragged
    W = synth.weights(codec, N, K, seed=3)
    X = np.eye(K, dtype=np.float16)
    Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_TC)).view(np.uint16)
    assert np.array_equal(Y.T, oracle.dequant_f16(W, codec, N, K))


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("general", [False, True])
@pytest.mark.parametrize("M", [17, 64, 129, 300])
def test_tc_gemm_parity(codec, general, M):
    for K in kvals(codec, general):
        N = 264
        X = synth.activations(M, K, seed=M)
        W = synth.weights(codec, N, K, seed=K)
        Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_TC))
        assert_close(Y, oracle.gemm(X, W, codec, M, N, K), "tc gemm %s M=%d K=%d" % (codec, M, K))


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("general", [False, True])
@pytest.mark.parametrize("M", [20, 128, 257])
def test_tc_swiglu_parity(codec, general, M):
    for K in kvals(codec, general):
        N = 200
        X = synth.activations(M, K, seed=M + 1)
        Wg = synth.weights(codec, N, K, seed=K, name="Wg")
        Wu = synth.weights(codec, N, K, seed=K, name="Wu")
        Y = host(m.swiglu(dev(X), dev(Wg), dev(Wu), codec, N, K, path=m.PATH_TC))
        assert_close(Y, oracle.swiglu(X, Wg, Wu, codec, M, N, K), "tc swiglu %s M=%d K=%d" % (codec, M, K))


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("M", [1, 5, 16, 33, 100, 128])
def test_tc_small_m_parity(codec, M):
    # M <= 128 on the tensor-core path: the activations are the A operand and
    # the decoded weights the B operand (N = 264: ragged last tiles).
    K = kvals(codec, False)[-1]
    N = 264
    X = synth.activations(M, K, seed=M + 60)
    W = synth.weights(codec, N, K, seed=61)
    Wu = synth.weights(codec, N, K, seed=61, name="Wu")
    Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_TC))
    assert_close(Y, oracle.gemm(X, W, codec, M, N, K), "tc small gemm %s M=%d" % (codec, M))
    Ys = host(m.glu(dev(X), dev(W), dev(Wu), codec, N, K, m.ACT_SILU, path=m.PATH_TC))
    assert_close(Ys, oracle.swiglu(X, W, Wu, codec, M, N, K), "tc small swiglu %s M=%d" % (codec, M))
    Yg = host(m.glu(dev(X), dev(W), dev(Wu), codec, N, K, m.ACT_GELU, path=m.PATH_TC))
    assert_close(Yg, oracle.geglu(X, W, Wu, codec, M, N, K), "tc small geglu %s M=%d" % (codec, M))


@pytest.mark.parametrize("codec", CODECS)
def test_tc_small_m_one_hot_readout_bit_exact(codec):
    # X rows are unit vectors at permuted columns: every output is one exact
    # product 1 * w, so Y must be columns of the fp16 weights bit for bit --
    # checks the decode, the swizzled operand layouts and the epilogue.
    K = kvals(codec, False)[0]
    M, N = 128, 200
    cols = np.random.default_rng(codec).permutation(K)[:M]
    X = np.zeros((M, K), dtype=np.float16)
    X[np.arange(M), cols] = 1
    W = synth.weights(codec, N, K, seed=62)
    Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_TC)).view(np.uint16)
    assert np.array_equal(Y, oracle.dequant_f16(W, codec, N, K)[:, cols].T)


@pytest.mark.parametrize("codec", CODECS)
def test_tc_small_m_k_split_one_hot_readout_bit_exact(codec):
    # Few output tiles and a long K: the small-M kernel splits K over a
    # cluster of CTAs and adds their partial tiles.  With one-hot X rows each
    # output is one exact product, held by exactly one CTA of the split, so
    # the sum is still exact: Y must be columns of the fp16 weights.
    K = 8 * 8 * synth.BLOCK[codec]           # eight packed stages: a split of 8
    M, N = 40, 136
    cols = np.random.default_rng(codec + 7).permutation(K)[:M]
    X = np.zeros((M, K), dtype=np.float16)
    X[np.arange(M), cols] = 1
    W = synth.weights(codec, N, K, seed=63)
    Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_TC)).view(np.uint16)
    assert np.array_equal(Y, oracle.dequant_f16(W, codec, N, K)[:, cols].T)


@pytest.mark.parametrize("N", [136, 9728])
def test_tc_small_m_with_and_without_k_split(N):
    # N = 136: 3 gated / 2 plain tiles, K split 8 ways over clusters.
    # N = 9728: 152 gated tiles, a full wave with no split, and 76 plain
    # tiles, split 2 ways.  All match the oracle.
    M, K = 40, 2048
    X = synth.activations(M, K, seed=64)
    Wg = synth.weights(synth.Q4_0, N, K, seed=65, name="Wg")
    Wu = synth.weights(synth.Q4_0, N, K, seed=65, name="Wu")
    Y = host(m.swiglu(dev(X), dev(Wg), dev(Wu), synth.Q4_0, N, K))
    assert_close(Y, oracle.swiglu(X, Wg, Wu, synth.Q4_0, M, N, K), "small-M swiglu N=%d" % N)
    Yl = host(m.gemm(dev(X), dev(Wg), synth.Q4_0, N, K))
    assert_close(Yl, oracle.gemm(X, Wg, synth.Q4_0, M, N, K), "small-M gemm N=%d" % N)


@pytest.mark.parametrize("M", [40, 200, 600])
def test_k_split_with_a_partial_last_stage(M):
    # MLX4 with K % 256 == 128: the last packed stage of a row is half past
    # the row end, and a K split must still cover every sub-step (both
    # tensor-core kernels split K here: few output tiles).
    K, N = 2176, 136
    X = synth.activations(M, K, seed=90 + M)
    W = synth.weights(synth.MLX4, N, K, seed=91, name="Wg")
    Wu = synth.weights(synth.MLX4, N, K, seed=91, name="Wu")
    rows = sample_rows(M)
    Y = host(m.gemm(dev(X), dev(W), synth.MLX4, N, K))
    assert_close(Y[rows], oracle.gemm(X, W, synth.MLX4, M, N, K, rows=rows), "split mlx4 gemm M=%d" % M)
    Ys = host(m.swiglu(dev(X), dev(W), dev(Wu), synth.MLX4, N, K))
    assert_close(Ys[rows], oracle.swiglu(X, W, Wu, synth.MLX4, M, N, K, rows=rows), "split mlx4 swiglu M=%d" % M)


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("M,N", [(300, 512), (1000, 136), (512, 2048)])
def test_prefill_k_split_parity(codec, M, N):
    # M > 128 with few 128-row output tiles: the prefill kernel splits K
    # over a cluster per tile (GEMM and SwiGLU), against the oracle on
    # sampled rows, every column.
    K = 2048 if codec != synth.Q2_0 else 4096
    X = synth.activations(M, K, seed=92 + M)
    W = synth.weights(codec, N, K, seed=93, name="Wg")
    Wu = synth.weights(codec, N, K, seed=93, name="Wu")
    rows = sample_rows(M)
    Y = host(m.gemm(dev(X), dev(W), codec, N, K))
    assert_close(Y[rows], oracle.gemm(X, W, codec, M, N, K, rows=rows), "prefill split gemm M=%d N=%d" % (M, N))
    Ys = host(m.swiglu(dev(X), dev(W), dev(Wu), codec, N, K))
    assert_close(Ys[rows], oracle.swiglu(X, W, Wu, codec, M, N, K, rows=rows),
                 "prefill split swiglu M=%d N=%d" % (M, N))


def test_tc_tile_widths():
    # M large enough for 256- and 128-wide activation tiles on a full GPU.
    import torch
    for M, N in ((2048, 8192), (512, 2048), (1000, 4096)):
        K = 256
        X = synth.activations(M, K, seed=5)
        W = synth.weights(synth.Q4_0, N, K, seed=6)
        Y = host(m.gemm(dev(X), dev(W), synth.Q4_0, N, K, path=m.PATH_TC))
        rows = sample_rows(M)
        assert_close(Y[rows], oracle.gemm(X, W, synth.Q4_0, M, N, K, rows=rows), "tile M=%d" % M)


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("general", [False, True])
@pytest.mark.parametrize("M", [1, 9, 20, 257])
def test_geglu_parity(codec, general, M):
    # GELU-gated projection on both paths (M <= 16: GEMV, else tcgen05).
    for K in kvals(codec, general)[:1]:
        N = 200
        X = synth.activations(M, K, seed=M + 3)
        Wg = synth.weights(codec, N, K, seed=K + 5, name="Wg")
        Wu = synth.weights(codec, N, K, seed=K + 5, name="Wu")
        Y = host(m.geglu(dev(X), dev(Wg), dev(Wu), codec, N, K))
        assert_close(Y, oracle.geglu(X, Wg, Wu, codec, M, N, K), "geglu %s M=%d K=%d" % (codec, M, K))
        # the same through the explicit-activation entry point on the other path
        path = m.PATH_TC if M <= 16 else m.PATH_AUTO
        Y2 = host(m.glu(dev(X), dev(Wg), dev(Wu), codec, N, K, m.ACT_GELU, path=path))
        assert_close(Y2, oracle.geglu(X, Wg, Wu, codec, M, N, K), "glu gelu %s M=%d" % (codec, M))


def test_quant_glu_layer():
    K, N = 256, 64
    Wg = synth.weights(synth.Q8_0, N, K, seed=18, name="Wg")
    Wu = synth.weights(synth.Q8_0, N, K, seed=18, name="Wu")
    X = synth.activations(2 * 7, K, seed=19)
    for act, ref in ((m.ACT_SILU, oracle.swiglu), (m.ACT_GELU, oracle.geglu)):
        layer = m.QuantGLU(dev(Wg), dev(Wu), synth.Q8_0, N, K, act=act)
        y = layer(dev(X).reshape(2, 7, K))
        assert tuple(y.shape) == (2, 7, N)
        assert_close(host(y).reshape(-1, N), ref(X, Wg, Wu, synth.Q8_0, 14, N, K), "QuantGLU act=%d" % act)


def mlp_reference(X, Wg, Wu, Wd, cgu, cd, M, D, F, act):
    """Oracle composition of the MLP block: the gated projection, its output
    rounded to fp16 (the intermediate the library materialises), then the
    down projection."""
    glu_ref = oracle.geglu if act == m.ACT_GELU else oracle.swiglu
    H16 = glu_ref(X, Wg, Wu, cgu, M, F, D).astype(np.float16)
    return oracle.gemm(H16, Wd, cd, M, D, F)


@pytest.mark.parametrize("M", [1, 3, 40])
@pytest.mark.parametrize("cgu,cd", [(synth.Q4_0, synth.Q4_0), (synth.Q4_0, synth.Q8_0), (synth.Q2_0, synth.Q8_0),
                                    (synth.MLX4, synth.MLX4)])
@pytest.mark.parametrize("act", [0, 1])
def test_mlp_parity(M, cgu, cd, act):
    D, F = 256, 1024
    X = synth.activations(M, D, seed=M + 30)
    Wg = synth.weights(cgu, F, D, seed=31, name="Wg")
    Wu = synth.weights(cgu, F, D, seed=31, name="Wu")
    Wd = synth.weights(cd, D, F, seed=32, name="Wd")
    layer = m.QuantMLP(dev(Wg), dev(Wu), dev(Wd), cgu, cd, D, F, act=act)
    Y = host(layer(dev(X)))
    assert_close(Y, mlp_reference(X, Wg, Wu, Wd, cgu, cd, M, D, F, act), "mlp M=%d %s/%s act=%d" % (M, cgu, cd, act))


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("M", [1, 9, 70, 300])
@pytest.mark.parametrize("hd", [64, 128])
def test_direct_head_output(codec, M, hd):
    # "v0.1 vs v0.2 comparison" section 4 (v0.2.1): Q/K/V projected straight
    # into [H, M, D].  The head-major output is the row-major GEMM output
    # permuted, bit for bit, and matches the oracle.
    K = kvals(codec, False)[0]
    N = 5 * hd   # e.g. 3 query heads + 1 key head + 1 value head
    X = synth.activations(M, K, seed=M + 40)
    W = synth.weights(codec, N, K, seed=41)
    Yh = host(m.gemm_heads(dev(X), dev(W), codec, N, K, hd))
    assert Yh.shape == (N // hd, M, hd)
    Yr = host(m.gemm(dev(X), dev(W), codec, N, K))
    assert np.array_equal(Yh.view(np.uint16), Yr.reshape(M, N // hd, hd).transpose(1, 0, 2).view(np.uint16))
    ref = oracle.gemm(X, W, codec, M, N, K).reshape(M, N // hd, hd).transpose(1, 0, 2)
    assert_close(Yh, ref, "heads %s M=%d hd=%d" % (codec, M, hd))


def test_fused_qkv_views():
    K, hd, hq, hkv = 256, 64, 4, 2
    Wq = synth.weights(synth.Q8_0, hq * hd, K, seed=42, name="Wq")
    Wk = synth.weights(synth.Q8_0, hkv * hd, K, seed=42, name="Wk")
    Wv = synth.weights(synth.Q8_0, hkv * hd, K, seed=42, name="Wv")
    X = synth.activations(37, K, seed=43)
    q, k, v = m.QuantQKV(dev(Wq), dev(Wk), dev(Wv), synth.Q8_0, K, hd, hq, hkv)(dev(X))
    for got, W, h in ((q, Wq, hq), (k, Wk, hkv), (v, Wv, hkv)):
        assert tuple(got.shape) == (h, 37, hd)
        ref = oracle.gemm(X, W, synth.Q8_0, 37, h * hd, K).reshape(37, h, hd).transpose(1, 0, 2)
        assert_close(host(got), ref, "qkv")


# ------------------------------------------------------------ GEMV path

@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("general", [False, True])
@pytest.mark.parametrize("M", [1, 2, 8, 9, 16])
def test_gemv_parity(codec, general, M):
    for K in kvals(codec, general):
        N = 264
        X = synth.activations(M, K, seed=M + 2)
        W = synth.weights(codec, N, K, seed=K + 1)
        Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_GEMV))
        assert_close(Y, oracle.gemm(X, W, codec, M, N, K), "gemv %s M=%d K=%d" % (codec, M, K))
        Wu = synth.weights(codec, N, K, seed=K + 2, name="Wu")
        Ys = host(m.swiglu(dev(X), dev(W), dev(Wu), codec, N, K, path=m.PATH_GEMV))
        assert_close(Ys, oracle.swiglu(X, W, Wu, codec, M, N, K), "gemv swiglu %s M=%d" % (codec, M))


# Rows of exactly one streamed stage (Q4_0 K = 4096, Q8_0 K = 2048, MLX4
# K = 4096) with M <= 8: the activation fragments stay in registers for the
# launch and the codes are read as aligned words (Q4_0 and Q8_0 as block
# pairs), with the activations permuted to the weight pairs' k order.
RESIDENT_X = [(synth.Q4_0, 4096), (synth.Q8_0, 2048), (synth.MLX4, 4096)]


@pytest.mark.parametrize("codec,K", RESIDENT_X)
@pytest.mark.parametrize("M", [1, 5, 8])
def test_gemv_resident_x_parity(codec, K, M):
    N = 264
    X = synth.activations(M, K, seed=M + 30)
    W = synth.weights(codec, N, K, seed=K + 5)
    Wu = synth.weights(codec, N, K, seed=K + 5, name="Wu")
    Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_GEMV))
    assert_close(Y, oracle.gemm(X, W, codec, M, N, K), "gemv resident %s M=%d" % (codec, M))
    Ys = host(m.swiglu(dev(X), dev(W), dev(Wu), codec, N, K, path=m.PATH_GEMV))
    assert_close(Ys, oracle.swiglu(X, W, Wu, codec, M, N, K), "gemv resident swiglu %s M=%d" % (codec, M))


@pytest.mark.parametrize("codec,K", RESIDENT_X)
def test_gemv_resident_x_one_hot_readout_bit_exact(codec, K):
    # Eight one-hot activation rows at spread-out columns (every k position
    # class of a block: even and odd blocks, both halves, the straddling
    # words): each output is one exact product, so Y must be columns of the
    # fp16 weights bit for bit -- a wrong activation permutation or a wrong
    # code word shows up as a wrong column.
    N = 136
    W = synth.weights(codec, N, K, seed=K + 6)
    ref = oracle.dequant_f16(W, codec, N, K)
    rng = np.random.default_rng(K)
    for rep in range(8):
        cols = rng.permutation(K)[:8] if rep else np.array([0, 1, 14, 15, 16, 30, 31, 32 + 26])
        X = np.zeros((8, K), dtype=np.float16)
        X[np.arange(8), cols] = 1
        Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_GEMV)).view(np.uint16)
        assert np.array_equal(Y, ref[:, cols].T), "columns %s" % cols.tolist()


@pytest.mark.parametrize("codec,K", [(synth.Q4_0, 4352), (synth.Q8_0, 2304), (synth.Q2_0, 5120),
                                     (synth.MLX4, 4096),
                                     (synth.Q4_0, 2400), (synth.Q8_0, 2080), (synth.Q2_0, 5248),
                                     (synth.MLX4, 4000)])
@pytest.mark.parametrize("M", [1, 11])
def test_gemv_long_rows(codec, K, M):
    # Rows longer than one streamed stage, with a ragged last stage; the
    # second three K values give rows that are not 16-byte multiples.
    N = 200
    X = synth.activations(M, K, seed=M + 20)
    W = synth.weights(codec, N, K, seed=K + 3)
    Y = host(m.gemm(dev(X), dev(W), codec, N, K, path=m.PATH_GEMV))
    assert_close(Y, oracle.gemm(X, W, codec, M, N, K), "gemv long %s M=%d K=%d" % (codec, M, K))
    Wu = synth.weights(codec, N, K, seed=K + 4, name="Wu")
    Ys = host(m.swiglu(dev(X), dev(W), dev(Wu), codec, N, K, path=m.PATH_GEMV))
    assert_close(Ys, oracle.swiglu(X, W, Wu, codec, M, N, K), "gemv long swiglu %s M=%d" % (codec, M))


def test_auto_dispatch_matches_explicit_paths():
    K, N = 512, 256
    W = synth.weights(synth.Q8_0, N, K, seed=9)
    for M in (16, 17):
        X = synth.activations(M, K, seed=10)
        auto = host(m.gemm(dev(X), dev(W), synth.Q8_0, N, K))
        path = m.PATH_GEMV if M <= 16 else m.PATH_TC
        explicit = host(m.gemm(dev(X), dev(W), synth.Q8_0, N, K, path=path))
        assert np.array_equal(auto.view(np.uint16), explicit.view(np.uint16))


def test_results_are_repeatable():
    M, N, K = 300, 512, 1024
    X = synth.activations(M, K, seed=11)
    Wg = synth.weights(synth.Q4_0, N, K, seed=12, name="Wg")
    Wu = synth.weights(synth.Q4_0, N, K, seed=12, name="Wu")
    a = host(m.swiglu(dev(X), dev(Wg), dev(Wu), synth.Q4_0, N, K)).view(np.uint16)
    b = host(m.swiglu(dev(X), dev(Wg), dev(Wu), synth.Q4_0, N, K)).view(np.uint16)
    assert np.array_equal(a, b)
    x1 = dev(X[:4])
    c = host(m.gemm(x1, dev(Wg), synth.Q4_0, N, K)).view(np.uint16)
    d = host(m.gemm(x1, dev(Wg), synth.Q4_0, N, K)).view(np.uint16)
    assert np.array_equal(c, d)


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("M", [20, 64, 300])
def test_repeated_calls_are_bit_identical(codec, M):
    # Many back-to-back calls on the same inputs, on the tensor-core paths
    # with a long K (64 sub-steps, so the packed-weight rings wrap many
    # times): every call must give the same bits, within tolerance of the
    # oracle.  A packed-weight slot released to its producer before its
    # decoders had finished reading it showed up here as occasional stale
    # weights in a few output columns.
    import torch
    N, K = 136, 4096
    X = synth.activations(M, K, seed=13)
    Wg = synth.weights(codec, N, K, seed=14, name="Wg")
    Wu = synth.weights(codec, N, K, seed=14, name="Wu")
    x, wg, wu = dev(X), dev(Wg), dev(Wu)
    rows = sample_rows(M) if M > 64 else list(range(M))
    for glu in (True, False):
        ref = (oracle.swiglu(X, Wg, Wu, codec, M, N, K, rows=rows) if glu
               else oracle.gemm(X, Wg, codec, M, N, K, rows=rows))
        outs = [m.swiglu(x, wg, wu, codec, N, K) if glu else m.gemm(x, wg, codec, N, K) for _ in range(24)]
        torch.cuda.synchronize()
        first = host(outs[0])
        assert_close(first[rows], ref, "repeat %s M=%d glu=%d" % (synth.CODEC_NAMES[codec], M, glu))
        for i, o in enumerate(outs[1:], 1):
            assert np.array_equal(host(o).view(np.uint16), first.view(np.uint16)), \
                "call %d differs from call 0 (%s M=%d glu=%d)" % (i, synth.CODEC_NAMES[codec], M, glu)


def test_zero_code_weights_give_zero():
    # Q4_0 all q=8 -> W = 0 -> Y = 0 and SwiGLU = 0 exactly, on both paths.
    K, N = 256, 128
    W = synth.constant_weights(synth.Q4_0, N, K, 8, np.float16(0.5))
    for M in (3, 100):
        X = synth.activations(M, K, seed=13)
        Y = host(m.gemm(dev(X), dev(W), synth.Q4_0, N, K))
        S = host(m.swiglu(dev(X), dev(W), dev(W), synth.Q4_0, N, K))
        assert np.all(Y == 0) and np.all(S == 0)


def test_quant_linear_flattens_leading_dims():
    import torch
    K, N = 256, 64
    W = synth.weights(synth.Q4_0, N, K, seed=14)
    X = synth.activations(2 * 3 * 5, K, seed=15)
    layer = m.QuantLinear(dev(W), synth.Q4_0, N, K)
    y = layer(dev(X).reshape(2, 3, 5, K))
    assert tuple(y.shape) == (2, 3, 5, N)
    assert_close(host(y).reshape(-1, N), oracle.gemm(X, W, synth.Q4_0, 30, N, K), "QuantLinear")


# ------------------------------------------------------------ status words

def test_wait_timeout_is_reported_and_context_survives():
    m.selftest_wait_timeout(1_000_000)   # 1 ms limit on a barrier nothing completes
    assert m.check_device_status() == m.ERR_TIMEOUT
    assert m.check_device_status() == m.OK   # cleared
    K, N, M = 256, 64, 4
    X = synth.activations(M, K, seed=16)
    W = synth.weights(synth.Q4_0, N, K, seed=17)
    assert_close(host(m.gemm(dev(X), dev(W), synth.Q4_0, N, K)), oracle.gemm(X, W, synth.Q4_0, M, N, K))


def test_finite_tripwire():
    import torch
    t = torch.zeros(1000, dtype=torch.float16, device="cuda")
    assert m.check_finite(t)
    t[777] = float("inf")
    assert not m.check_finite(t)
    t[777] = float("nan")
    assert not m.check_finite(t)
