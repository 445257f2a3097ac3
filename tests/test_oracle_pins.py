"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against something it cannot agree with by
construction: hand-decoded golden blocks, numpy's IEEE conversions, exact
rational arithmetic on tiny inputs, closed forms, the identity matrix, and
invariants of SiLU and GELU.  A second group compiles copies of the oracle with a
planted mistake and checks that at least one pin fails for each.
"""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

CODEC_BY_NAME = {"Q4_0": synth.Q4_0, "Q8_0": synth.Q8_0, "Q2_0": synth.Q2_0, "MLX4": synth.MLX4}
# The code that decodes to zero (MLX4: with a zero bias).
ZERO_CODE = {synth.Q4_0: 8, synth.Q8_0: 0, synth.Q2_0: 1, synth.MLX4: 0}


def golden_packed(blk):
    d = blk["d_bits"]
    head = [d & 0xFF, d >> 8]
    if "b_bits" in blk:
        head += [blk["b_bits"] & 0xFF, blk["b_bits"] >> 8]
    return np.array(head + blk["code_bytes"], dtype=np.uint8)


# ------------------------------------------------------------ block layout

def test_block_sizes():
    # "Releases" v0.3.0: Q2_0 is 128 weights in 34 bytes, 2.125 bits per weight.
    assert oracle.block_size(synth.Q2_0) == 128
    assert oracle.block_bytes(synth.Q2_0) == 34
    assert oracle.block_bytes(synth.Q2_0) * 8 / oracle.block_size(synth.Q2_0) == 2.125
    assert (oracle.block_size(synth.Q4_0), oracle.block_bytes(synth.Q4_0)) == (32, 18)
    assert (oracle.block_size(synth.Q8_0), oracle.block_bytes(synth.Q8_0)) == (32, 34)
    # Project page section 4 (v0.2.1): the MLX 4-bit block is a 20-byte struct.
    assert (oracle.block_size(synth.MLX4), oracle.block_bytes(synth.MLX4)) == (32, 20)
    assert oracle.block_size(7) == -1


def check_golden(blocks):
    for blk in blocks:
        codec = CODEC_BY_NAME[blk["codec"]]
        B = oracle.block_size(codec)
        w = oracle.dequant(golden_packed(blk), codec, 1, B)[0]
        assert list(w) == blk["weights"], (blk["codec"], blk["name"])


def test_golden_blocks(golden_blocks):
    check_golden(golden_blocks)


def test_q2_0_reserved_code_is_plus_two_d():
    # "Releases" v0.3.0: q = 3 decodes to +2d (not clamped to +d).
    for dbits, d in ((0x3C00, 1.0), (0x2E66, float(np.array([0x2E66], np.uint16).view(np.float16)[0]))):
        W = synth.constant_weights(synth.Q2_0, 1, 128, 3, np.array([dbits], np.uint16).view(np.float16)[0])
        assert np.all(oracle.dequant(W, synth.Q2_0, 1, 128) == 2 * d)


def test_encoder_matches_golden(golden_blocks):
    # The generator's encoder writes the same bytes as the hand-built blocks.
    for blk in golden_blocks:
        codec = CODEC_BY_NAME[blk["codec"]]
        B = oracle.block_size(codec)
        d = np.array([blk["d_bits"]], np.uint16).view(np.float16)
        dval = float(d[0])
        if codec == synth.MLX4:
            b = np.array([blk["b_bits"]], np.uint16).view(np.float16)
            q = np.array([[round((w - float(b[0])) / dval) for w in blk["weights"]]], dtype=np.int16)
            packed = synth.pack(codec, q, d.reshape(1, 1), b.reshape(1, 1))
        else:
            z = ZERO_CODE[codec]
            q = np.array([[round(w / dval) + z for w in blk["weights"]]], dtype=np.int16)
            packed = synth.pack(codec, q, d.reshape(1, 1))
        assert np.array_equal(packed, golden_packed(blk).reshape(1, -1))


# ------------------------------------------------------------ fp16 conversions

def test_half_to_double_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_double_to_half_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        # exact ties between neighbouring fp16 values, normal and subnormal
        (np.arange(1, 4000) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 2048) + 0.5) * 2.0 ** -10,
        (np.arange(1024, 2048) + 0.5) * 2.0 ** 5,
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25,
                  2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12)]),
    ])
    ours = oracle.double_to_half(vals)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------ projections

def f16_weights(q, d, codec, b=None):
    """Each weight (q - z) * d, or q * s + b for MLX4 (exact in binary64),
    rounded once to fp16 by numpy, as binary64 -- the operand values the
    method multiplies."""
    B = synth.BLOCK[codec]
    scale = np.repeat(d.astype(np.float64), B, axis=1)
    if codec == synth.MLX4:
        exact = q.astype(np.float64) * scale + np.repeat(b.astype(np.float64), B, axis=1)
    else:
        exact = (q.astype(np.float64) - ZERO_CODE[codec]) * scale
    return exact.astype(np.float16).astype(np.float64)


def exact_gemm(q, d, codec, X16, b=None):
    """Exact rational Y = X W16^T from the generator's codes and scales."""
    M, K = X16.shape
    N = q.shape[0]
    W16 = f16_weights(q, d, codec, b)
    Xf = [[Fraction(float(v)) for v in row] for row in X16.astype(np.float64)]
    Wf = [[Fraction(float(W16[n, k])) for k in range(K)] for n in range(N)]
    return [[sum(Xf[m][k] * Wf[n][k] for k in range(K)) for n in range(N)] for m in range(M)]


@pytest.mark.parametrize("codec", synth.CODECS)
def test_brute_force_exact(codec):
    M, N = 4, 32
    K = 32 if codec != synth.Q2_0 else 128
    X = synth.activations(M, K, seed=11)
    q = synth.codes(codec, N, K, seed=12, name="W")
    d = synth.scales(codec, N, K, seed=12, name="W")
    b = synth.biases(codec, N, K, seed=12, name="W", d=d)
    W = synth.pack(codec, q, d, b)
    Y = oracle.gemm(X, W, codec, M, N, K)
    E = exact_gemm(q, d, codec, X, b)
    W16 = f16_weights(q, d, codec, b)
    for m in range(M):
        for n in range(N):
            # recursive fp64 summation: |err| <= K * 2^-52 * sum |x w| (loose)
            bound = K * 2.0 ** -52 * float(np.abs(X[m].astype(np.float64) * W16[n]).sum())
            assert abs(Fraction(Y[m, n]) - E[m][n]) <= Fraction(bound) + Fraction(1, 10 ** 30)


@pytest.mark.parametrize("codec", synth.CODECS)
def test_zero_code_gives_zero(codec):
    # Q4_0 all q=8, Q8_0 all q=0, Q2_0 all q=1 decode to 0, so Y == 0 and SwiGLU == 0.
    K = 256
    X = synth.activations(8, K, seed=3)
    W = synth.constant_weights(codec, 16, K, ZERO_CODE[codec], np.float16(0.37))
    assert np.all(oracle.gemm(X, W, codec, 8, 16, K) == 0.0)
    assert np.all(oracle.swiglu(X, W, W, codec, 8, 16, K) == 0.0)


@pytest.mark.parametrize("codec,code", [(synth.Q4_0, 13), (synth.Q8_0, -57), (synth.Q2_0, 3), (synth.Q2_0, 0),
                                        (synth.MLX4, 13)])
def test_constant_code_closed_form(codec, code):
    # Constant code c and scale d: Y[m, n] = fp16((c - z) * d) * sum_k X[m, k].
    M, N, K = 5, 8, 256
    X = synth.activations(M, K, seed=4)
    dv = np.float16(0.0173)
    w16 = float(np.float16((code - ZERO_CODE[codec]) * float(dv)))
    W = synth.constant_weights(codec, N, K, code, dv)
    Y = oracle.gemm(X, W, codec, M, N, K)
    for m in range(M):
        exact = w16 * math.fsum(X[m].astype(np.float64))
        scale = abs(w16) * np.abs(X[m].astype(np.float64)).sum()
        assert np.all(np.abs(Y[m] - exact) <= K * 2.0 ** -52 * scale + 1e-300)


@pytest.mark.parametrize("codec", synth.CODECS)
def test_identity_and_permutation_readout(codec):
    # X = I (M = K): Y[k, n] = W16[n, k] exactly -- one nonzero product per sum.
    # X = a permutation P: Y[m, n] = W16[n, p(m)], which a transposed operand breaks.
    K = 128
    N = 24
    W = synth.weights(codec, N, K, seed=5)
    Wd = oracle.dequant_f16(W, codec, N, K).view(np.float16).astype(np.float64)
    I = np.eye(K, dtype=np.float16)
    assert np.array_equal(oracle.gemm(I, W, codec, K, N, K), Wd.T)
    perm = np.random.default_rng(2).permutation(K)
    P = np.zeros((K, K), dtype=np.float16)
    P[np.arange(K), perm] = 1
    assert np.array_equal(oracle.gemm(P, W, codec, K, N, K), Wd[:, perm].T)


def test_row_subset_matches_full():
    M, N, K = 40, 16, 64
    X = synth.activations(M, K, seed=6)
    W = synth.weights(synth.Q4_0, N, K, seed=7)
    full = oracle.gemm(X, W, synth.Q4_0, M, N, K)
    rows = [39, 0, 17, 17, 5]
    assert np.array_equal(oracle.gemm(X, W, synth.Q4_0, M, N, K, rows=rows), full[rows])


def test_threads_do_not_change_results():
    M, N, K = 9, 37, 96
    X = synth.activations(M, K, seed=8)
    W = synth.weights(synth.Q8_0, N, K, seed=9)
    a = oracle.gemm(X, W, synth.Q8_0, M, N, K, nthreads=1)
    b = oracle.gemm(X, W, synth.Q8_0, M, N, K, nthreads=7)
    assert np.array_equal(a, b)


# ------------------------------------------------------------ MLX 4-bit affine

def check_mlx4_affine_closed_form():
    # Constant code c, scale s, bias b: every weight is fp16(c * s + b), so
    # Y[m, n] = fp16(c s + b) * sum_k X[m, k].
    M, N, K = 4, 8, 256
    X = synth.activations(M, K, seed=21)
    for c, s, b in ((13, 0.0173, -0.1), (0, 0.5, 0.3125), (15, -0.02, 0.15), (7, 0.0, -0.25)):
        sv, bv = np.float16(s), np.float16(b)
        w16 = float(np.float16(c * float(sv) + float(bv)))
        W = synth.constant_weights(synth.MLX4, N, K, c, sv, bv)
        Y = oracle.gemm(X, W, synth.MLX4, M, N, K)
        for m in range(M):
            exact = w16 * math.fsum(X[m].astype(np.float64))
            scale = abs(w16) * np.abs(X[m].astype(np.float64)).sum()
            assert np.all(np.abs(Y[m] - exact) <= K * 2.0 ** -52 * scale + 1e-300), (c, s, b)


def test_mlx4_affine_closed_form():
    check_mlx4_affine_closed_form()


def check_mlx4_one_rounding():
    # Block C of the golden file at the projection level: with s = 1 + 2^-10,
    # b = -3 and code 3, each fp16 operand is 3 * 2^-10, so X = all ones gives
    # Y = K * 3 * 2^-10 exactly (a product rounded to fp16 before the bias is
    # added would give K * 2^-8).
    K = 64
    s = np.array([0x3C01], np.uint16).view(np.float16)[0]
    b = np.array([0xC200], np.uint16).view(np.float16)[0]
    W = synth.constant_weights(synth.MLX4, 2, K, 3, s, b)
    assert np.all(oracle.dequant_f16(W, synth.MLX4, 2, K) == np.float16(3 * 2.0 ** -10).view(np.uint16))
    X = np.ones((1, K), dtype=np.float16)
    assert np.all(oracle.gemm(X, W, synth.MLX4, 1, 2, K) == K * 3 * 2.0 ** -10)


def test_mlx4_one_rounding():
    check_mlx4_one_rounding()


def check_mlx4_pack():
    # MLX's planar arrays (codes in uint32 words, code k at bits 4 (k % 8) of
    # word k // 8; scales and biases in their own arrays) repack into exactly
    # the blocks the layout writer produces from the same codes.
    for N, K in ((3, 32), (5, 256), (2, 1024)):
        q = synth.codes(synth.MLX4, N, K, seed=N, name="W")
        d = synth.scales(synth.MLX4, N, K, seed=N, name="W")
        b = synth.biases(synth.MLX4, N, K, seed=N, name="W", d=d)
        words, s, bb = synth.planar(q, d, b)
        assert np.array_equal(oracle.mlx4_pack(words, s, bb, N, K), synth.pack(synth.MLX4, q, d, b))


def test_mlx4_pack():
    check_mlx4_pack()
    with pytest.raises(ValueError):
        oracle.mlx4_pack(np.zeros((1, 2), np.uint32), np.zeros(1, np.float16), np.zeros(1, np.float16), 1, 16)


# ------------------------------------------------------------ blocks -> planes

def check_repack_golden(blocks):
    # Hand-built blocks of one codec, laid out as two rows (the second in
    # reverse order): the codes plane is each block's code bytes in row-major
    # block order, then the scale bits, then (MLX4) the bias bits.
    by_codec = {}
    for blk in blocks:
        by_codec.setdefault(CODEC_BY_NAME[blk["codec"]], []).append(blk)
    for codec, blks in by_codec.items():
        B = oracle.block_size(codec)
        order = blks + blks[::-1]
        nb = len(blks)
        W = np.concatenate([golden_packed(b) for b in order])
        P = oracle.repack(W, codec, 2, nb * B)
        codes = [c for b in order for c in b["code_bytes"]]
        expect = codes + [v for b in order for v in (b["d_bits"] & 0xFF, b["d_bits"] >> 8)]
        if codec == synth.MLX4:
            expect += [v for b in order for v in (b["b_bits"] & 0xFF, b["b_bits"] >> 8)]
        assert P.tolist() == expect, codec


def check_repack_planes():
    # The scale plane is the generator's scale array; for MLX4 the three
    # planes are the generator's own MLX planar arrays (words, scales, biases).
    for codec in synth.CODECS:
        for N, K in ((3, 256), (2, 1024)):
            q = synth.codes(codec, N, K, seed=N, name="W")
            d = synth.scales(codec, N, K, seed=N, name="W")
            b = synth.biases(codec, N, K, seed=N, name="W", d=d)
            W = synth.pack(codec, q, d, b)
            P = oracle.repack(W, codec, N, K)
            nb = K // oracle.block_size(codec)
            cb = oracle.block_bytes(codec) - (4 if codec == synth.MLX4 else 2)
            scales = P[N * nb * cb: N * nb * (cb + 2)].view(np.float16).reshape(N, nb)
            assert np.array_equal(scales.view(np.uint16), d.view(np.uint16)), codec
            if codec == synth.MLX4:
                words, s, bb = synth.planar(q, d, b)
                assert np.array_equal(P[:N * nb * cb].view("<u4").reshape(N, K // 8), words)
                assert np.array_equal(P[N * nb * (cb + 2):].view(np.uint16).reshape(N, nb), bb.view(np.uint16))
                assert np.array_equal(oracle.mlx4_pack(words, s, bb, N, K), W)


def test_repack(golden_blocks):
    check_repack_golden(golden_blocks)
    check_repack_planes()
    with pytest.raises(ValueError):
        oracle.repack(np.zeros(18, np.uint8), synth.Q4_0, 1, 16)


def test_mlx4_scale_zero_gives_bias():
    # s = 0: every weight equals the block's bias whatever its code.
    K = 64
    q = synth.codes(synth.MLX4, 4, K, seed=3, name="W")
    d = np.zeros((4, 2), np.float16)
    b = np.array([[0.125, -2.5], [3.0, 0.0], [-0.0078125, 1.5], [7.0, -7.0]], np.float16)
    W = synth.pack(synth.MLX4, q, d, b)
    assert np.array_equal(oracle.dequant(W, synth.MLX4, 4, K), np.repeat(b.astype(np.float64), 32, axis=1))


# ------------------------------------------------------------ SiLU and SwiGLU

def sigmoid_decimal(x):
    getcontext().prec = 50
    return Decimal(1) / (Decimal(1) + (-Decimal(x)).exp())


def test_silu_values_and_invariants():
    assert oracle.silu(0.0) == 0.0
    for x in (1.0, -1.0, 0.5, -3.25, 7.0, 20.0, -20.0):
        ref = float(Decimal(x) * sigmoid_decimal(x))
        assert abs(oracle.silu(x) - ref) <= 4e-16 * max(1.0, abs(ref))
    # SiLU(x) - SiLU(-x) = x; SiLU(x) -> x for large x, -> 0 for very negative x
    for x in np.linspace(-30, 30, 241):
        assert abs(oracle.silu(x) - oracle.silu(-x) - x) <= 1e-14 * max(1.0, abs(x))
    assert oracle.silu(60.0) == 60.0
    assert abs(oracle.silu(-60.0)) < 1e-24


@pytest.mark.parametrize("codec", synth.CODECS)
def test_swiglu_fused_equals_unfused(codec):
    # "v0.1 vs v0.2 comparison" section 2.2: fusion must not change the result.
    M, N = 6, 20
    K = 256
    X = synth.activations(M, K, seed=10)
    Wg = synth.weights(codec, N, K, seed=10, name="Wg")
    Wu = synth.weights(codec, N, K, seed=10, name="Wu")
    fused = oracle.swiglu(X, Wg, Wu, codec, M, N, K)
    G = oracle.gemm(X, Wg, codec, M, N, K)
    U = oracle.gemm(X, Wu, codec, M, N, K)
    unfused = np.vectorize(oracle.silu)(G) * U
    assert np.array_equal(fused, unfused)
    # and against an independent SiLU (math.exp) within rounding
    ind = G / (1.0 + np.exp(-G)) * U
    assert np.allclose(fused, ind, rtol=1e-13, atol=1e-300)


def phi_decimal(x, digits=40):
    """Standard normal CDF in exact decimal arithmetic, independent of the C
    library's erf: the Maclaurin series of erf for |x| <= 8, the asymptotic
    tail series phi(x)/|x| * sum (-1)^n (2n-1)!! / x^(2n) beyond."""
    getcontext().prec = digits + 10
    xd = Decimal(x)
    if abs(xd) > 8:
        t = abs(xd)
        dens = (-(t * t) / 2).exp() / (2 * _sqrt_pi() / Decimal(2).sqrt())  # phi(t) = e^(-t^2/2) / sqrt(2 pi)
        term, total, n = Decimal(1), Decimal(1), 0
        while n < 30:
            n += 1
            term = -term * (2 * n - 1) / (t * t)
            total += term
        tail = dens / t * total                          # Phi(-t)
        return tail if xd < 0 else 1 - tail
    z = xd / Decimal(2).sqrt()
    term, total, n = z, z, 0
    while True:
        n += 1
        term = -term * z * z / n                      # (-1)^n z^(2n+1) / n!
        add = term / (2 * n + 1)
        total += add
        if abs(add) < Decimal(10) ** (-(digits + 5)):
            break
    erf = 2 * total / _sqrt_pi()
    return (1 + erf) / 2


def _sqrt_pi():
    # pi from Machin's formula, exact to the working precision
    def arctan_inv(k):
        x = Decimal(1) / k
        x2, term, total, n = x * x, x, x, 1
        while True:
            term = -term * x2
            add = term / (2 * n + 1)
            if abs(add) < Decimal(10) ** (-(getcontext().prec + 2)):
                return total
            total += add
            n += 1
    return (4 * (4 * arctan_inv(5) - arctan_inv(239))).sqrt()


def test_gelu_values_and_invariants():
    # "Releases" v0.3.0 names GeGLU; GELU(g) = g * Phi(g) (textbook reading).
    assert oracle.gelu(0.0) == 0.0
    for x in (1.0, -1.0, 0.5, -2.25, 3.0, 6.0, -6.0):
        ref = float(Decimal(x) * phi_decimal(x))
        assert abs(oracle.gelu(x) - ref) <= 4e-15 * max(1.0, abs(ref)), x
    # tabulated value: Phi(1) = 0.8413447460685429...
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) <= 2e-16
    # GELU(x) - GELU(-x) = x; GELU(x) -> x for large x, -> 0 for very negative x
    for x in np.linspace(-12, 12, 97):
        assert abs(oracle.gelu(x) - oracle.gelu(-x) - x) <= 1e-14 * max(1.0, abs(x))
    assert oracle.gelu(40.0) == 40.0
    assert abs(oracle.gelu(-40.0)) < 1e-300


@pytest.mark.parametrize("codec", synth.CODECS)
def test_geglu_fused_equals_unfused(codec):
    M, N = 5, 24
    K = 256
    X = synth.activations(M, K, seed=11)
    Wg = synth.weights(codec, N, K, seed=11, name="Wg")
    Wu = synth.weights(codec, N, K, seed=11, name="Wu")
    fused = oracle.geglu(X, Wg, Wu, codec, M, N, K)
    G = oracle.gemm(X, Wg, codec, M, N, K)
    U = oracle.gemm(X, Wu, codec, M, N, K)
    assert np.array_equal(fused, np.vectorize(oracle.gelu)(G) * U)
    # and against an independent GELU (the series above) within rounding
    ind = np.array([[float(Decimal(g) * phi_decimal(g, 60)) for g in row] for row in G]) * U
    assert np.allclose(fused, ind, rtol=1e-13, atol=1e-300)
    # the activation is applied to the gate, not to the up projection
    assert not np.allclose(fused, G * np.vectorize(oracle.gelu)(U))


# ------------------------------------------------------------ planted mistakes

MUTATIONS = {
    # each: (text in oracle.c, replacement) -- plausible slips the pins must catch
    "nibble_order": ("(i < 16) ? (qs[i] & 0x0f) : (qs[i - 16] >> 4)",
                     "(i % 2 == 0) ? (qs[i / 2] & 0x0f) : (qs[i / 2] >> 4)"),
    "q4_offset": ("return codec == ORACLE_Q4_0 ? 8 :", "return codec == ORACLE_Q4_0 ? 7 :"),
    "q2_offset": ("(codec == ORACLE_Q2_0 ? 1 : 0)", "(codec == ORACLE_Q2_0 ? 0 : 0)"),
    "q2_msb_first": ("(qs[i / 4] >> (2 * (i % 4))) & 0x3", "(qs[i / 4] >> (6 - 2 * (i % 4))) & 0x3"),
    "q2_clamp_reserved": ("return (qs[i / 4] >> (2 * (i % 4))) & 0x3;",
                          "{ int c = (qs[i / 4] >> (2 * (i % 4))) & 0x3; return c == 3 ? 2 : c; }"),
    "q8_unsigned": ("return (int)(int8_t)qs[i];", "return (int)qs[i];"),
    "scale_position": ("uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));",
                       "uint16_t dbits = (uint16_t)(blk[1] | (blk[0] << 8));"),
    "transposed_sum": ("const double* x = j->Xd + r * j->K;",
                       "const double* x = j->Xd + ((r + 1) % (j->nrows ? j->nrows : 1)) * j->K;"),
    "dropped_term": ("for (long long k = 0; k < K; ++k) s += a[k] * b[k];",
                     "for (long long k = 1; k < K; ++k) s += a[k] * b[k];"),
    "silu_sign": ("return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    "silu_on_up": ("(j->act == ORACLE_ACT_GELU ? oracle_gelu(g) : oracle_silu(g)) * u;",
                   "(j->act == ORACLE_ACT_GELU ? oracle_gelu(g) : g * oracle_silu(u) / u) * u;"),
    "half_rounding": ("double r = nearbyint(ldexp(a, 10 - E));", "double r = floor(ldexp(a, 10 - E));"),
    "unrounded_operands": ("    round_row_to_f16(w0, j->K);\n", "\n"),
    "gelu_scale": ("return 0.5 * g * erfc(-g / sqrt(2.0));", "return 0.5 * g * erfc(-g / 2.0);"),
    "gelu_half_missing": ("return 0.5 * g * erfc(-g / sqrt(2.0));", "return g * erfc(-g / sqrt(2.0));"),
    "gelu_sign": ("return 0.5 * g * erfc(-g / sqrt(2.0));", "return 0.5 * g * erfc(g / sqrt(2.0));"),
    "geglu_uses_silu": ("(j->act == ORACLE_ACT_GELU ? oracle_gelu(g) : oracle_silu(g))", "oracle_silu(g)"),
    "mlx4_q4_0_nibble_order": ("return (qs[i / 2] >> (4 * (i % 2))) & 0x0f;",
                               "return (i < 16) ? (qs[i] & 0x0f) : (qs[i - 16] >> 4);"),
    "mlx4_high_nibble_first": ("return (qs[i / 2] >> (4 * (i % 2))) & 0x0f;",
                               "return (qs[i / 2] >> (4 - 4 * (i % 2))) & 0x0f;"),
    "mlx4_bias_dropped": ("(double)block_code(blk, codec, (int)i) * d + bias;",
                          "(double)block_code(blk, codec, (int)i) * d;"),
    "mlx4_bias_subtracted": ("(double)block_code(blk, codec, (int)i) * d + bias;",
                             "(double)block_code(blk, codec, (int)i) * d - bias;"),
    "mlx4_centred_codes": ("(double)block_code(blk, codec, (int)i) * d + bias;",
                           "(double)(block_code(blk, codec, (int)i) - 8) * d + bias;"),
    "mlx4_product_rounded_first": (
        "(double)block_code(blk, codec, (int)i) * d + bias;",
        "oracle_half_to_double(oracle_double_to_half((double)block_code(blk, codec, (int)i) * d)) + bias;"),
    "mlx4_scale_bias_swapped": ("double bias = oracle_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));",
                                "double bias = d; d = oracle_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));"),
    "mlx4_codes_after_scale_only": ("const uint8_t* qs = blk + (codec == ORACLE_MLX4 ? 4 : 2);",
                                    "const uint8_t* qs = blk + 2;"),
    "mlx4_pack_word_order": ("int q = (int)((words[n * (K / 8) + k / 8] >> (4 * (k % 8))) & 0xf);",
                             "int q = (int)((words[n * (K / 8) + k / 8] >> (28 - 4 * (k % 8))) & 0xf);"),
    "mlx4_pack_bias_scale_swapped": ("uint16_t s = scales[n * nb + b], t = biases[n * nb + b];",
                                     "uint16_t t = scales[n * nb + b], s = biases[n * nb + b];"),
    "repack_codes_with_header": ("memcpy(codes + i * CB, blk + head, (size_t)CB);",
                                 "memcpy(codes + i * CB, blk, (size_t)CB);"),
    "repack_blocks_column_major": ("memcpy(codes + i * CB, blk + head, (size_t)CB);",
                                   "memcpy(codes + (b * N + n) * CB, blk + head, (size_t)CB);"),
    "repack_scale_byte_order": ("scales[2 * i] = blk[0];\n      scales[2 * i + 1] = blk[1];",
                                "scales[2 * i] = blk[1];\n      scales[2 * i + 1] = blk[0];"),
    "repack_bias_from_scale": ("biases[2 * i] = blk[2];\n        biases[2 * i + 1] = blk[3];",
                               "biases[2 * i] = blk[0];\n        biases[2 * i + 1] = blk[1];"),
}


def all_pins_pass(golden_blocks):
    checks = [
        lambda: check_golden(golden_blocks),
        test_half_to_double_all_patterns,
        test_double_to_half_matches_numpy,
        lambda: [test_brute_force_exact(c) for c in synth.CODECS],
        lambda: [test_zero_code_gives_zero(c) for c in synth.CODECS],
        lambda: [test_identity_and_permutation_readout(c) for c in synth.CODECS],
        test_silu_values_and_invariants,
        lambda: [test_swiglu_fused_equals_unfused(c) for c in synth.CODECS],
        test_gelu_values_and_invariants,
        lambda: [test_geglu_fused_equals_unfused(c) for c in synth.CODECS],
        lambda: test_q2_0_reserved_code_is_plus_two_d(),
        check_mlx4_affine_closed_form,
        check_mlx4_one_rounding,
        check_mlx4_pack,
        lambda: check_repack_golden(golden_blocks),
        check_repack_planes,
    ]
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, golden_blocks):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, name
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / ("mut_%s.so" % name)))
    with oracle.use_library(path):
        assert not all_pins_pass(golden_blocks), "mutation %s survived every pin" % name
