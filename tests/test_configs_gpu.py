"""Parity at the full sizes of the pages' workloads (LLaMA-1B/8B-shaped
projections), in the launch configuration the benchmark times.  Outputs of
sampled activation rows (always 0, 1, 127, 128, 129, M/2, M-1 and random
rows, every output column) are compared element by element with the oracle.
"""
import numpy as np
import pytest

import oracle
import synth
import swiglu_block_quantized_gb300 as m
from _helpers import assert_close, dev, host, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    yield
    assert m.check_device_status() == m.OK


def check_gemm(codec, M, N, K, seed):
    X = synth.activations(M, K, seed=seed)
    W = synth.weights(codec, N, K, seed=seed)
    Y = host(m.gemm(dev(X), dev(W), codec, N, K))
    rows = sample_rows(M) if M > 16 else list(range(M))
    assert_close(Y[rows], oracle.gemm(X, W, codec, M, N, K, rows=rows),
                 "gemm %s %dx%dx%d" % (synth.CODEC_NAMES[codec], M, N, K))


def check_swiglu(codec, M, N, K, seed):
    X = synth.activations(M, K, seed=seed)
    Wg = synth.weights(codec, N, K, seed=seed, name="Wg")
    Wu = synth.weights(codec, N, K, seed=seed, name="Wu")
    Y = host(m.swiglu(dev(X), dev(Wg), dev(Wu), codec, N, K))
    rows = sample_rows(M) if M > 16 else list(range(M))
    assert_close(Y[rows], oracle.swiglu(X, Wg, Wu, codec, M, N, K, rows=rows),
                 "swiglu %s %dx%dx%d" % (synth.CODEC_NAMES[codec], M, N, K))


def test_tiny_q4_0_full_compare():
    M, N, K = 64, 256, 256
    X = synth.activations(M, K, seed=0)
    W = synth.weights(synth.Q4_0, N, K, seed=0)
    Y = host(m.gemm(dev(X), dev(W), synth.Q4_0, N, K))
    assert_close(Y, oracle.gemm(X, W, synth.Q4_0, M, N, K), "tiny")


@pytest.mark.parametrize("codec", [synth.Q4_0, synth.Q8_0])
def test_1b_projection(codec):
    check_gemm(codec, 2048, 8192, 2048, seed=1)


def test_8b_swiglu_m2048():
    check_swiglu(synth.Q4_0, 2048, 14336, 4096, seed=2)


def test_8b_swiglu_m1():
    check_swiglu(synth.Q4_0, 1, 14336, 4096, seed=2)


@pytest.mark.parametrize("M", [1, 16, 512, 2048])
def test_q2_0_sweep(M):
    check_gemm(synth.Q2_0, M, 4096, 4096, seed=3)


@pytest.mark.parametrize("M", [1, 128, 512, 2048])
def test_llama1b_layer_set(M):
    for i, (name, kind, codec, m_, n, k) in enumerate(synth.llama1b_layer(M)):
        if kind == "gemm":
            check_gemm(codec, m_, n, k, seed=40 + i)
        else:
            check_swiglu(codec, m_, n, k, seed=40 + i)
