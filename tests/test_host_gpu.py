"""m4q_project_host: the projection with activations and results in host
memory, chunked so that copies overlap kernels.  Same results as the device
call (within the tests' tolerance of the oracle) for every chunking."""
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


@pytest.mark.parametrize("M,chunk", [(300, 0), (300, 128), (300, 100), (37, 16), (1, 0)])
@pytest.mark.parametrize("gated", [True, False])
def test_project_host_matches_the_oracle(M, chunk, gated):
    import torch
    N, K = 264, 1024
    codec = synth.Q4_0 if gated else synth.Q8_0
    X = synth.activations(M, K, seed=70 + M)
    W = synth.weights(codec, N, K, seed=71, name="Wg")
    Wu = synth.weights(codec, N, K, seed=71, name="Wu")
    xh = torch.from_numpy(X).pin_memory()
    y = m.project_host(xh, dev(W), codec, N, K, wu=dev(Wu) if gated else None, chunk_rows=chunk)
    torch.cuda.current_stream().synchronize()
    Y = y.numpy()
    rows = sample_rows(M) if M > 16 else list(range(M))
    ref = (oracle.swiglu(X, W, Wu, codec, M, N, K, rows=rows) if gated
           else oracle.gemm(X, W, codec, M, N, K, rows=rows))
    assert_close(Y[rows], ref, "project_host M=%d chunk=%d gated=%d" % (M, chunk, gated))
    # the device call on the same data, within tolerance (chunks may take other kernels)
    yd = host(m.swiglu(dev(X), dev(W), dev(Wu), codec, N, K) if gated else m.gemm(dev(X), dev(W), codec, N, K))
    assert_close(Y, yd.astype(np.float64), "project_host vs device M=%d" % M)


def test_project_host_pageable_and_repeated():
    # pageable host memory gives the same result (the copies serialize), and
    # two calls in a row on reused staging buffers are independent
    import torch
    M, N, K = 129, 136, 512
    X1 = synth.activations(M, K, seed=80)
    X2 = synth.activations(M, K, seed=81)
    W = synth.weights(synth.MLX4, N, K, seed=82, name="Wg")
    Wu = synth.weights(synth.MLX4, N, K, seed=82, name="Wu")
    w, wu = dev(W), dev(Wu)
    xd = torch.empty((M, K), dtype=torch.float16, device="cuda")
    yd = torch.empty((M, N), dtype=torch.float16, device="cuda")
    outs = []
    for X, pinned in ((X1, False), (X2, True)):
        xh = torch.from_numpy(X)
        if pinned:
            xh = xh.pin_memory()
        outs.append(m.project_host(xh, w, synth.MLX4, N, K, wu=wu, x_dev=xd, y_dev=yd, chunk_rows=64))
    torch.cuda.current_stream().synchronize()
    for X, y in zip((X1, X2), outs):
        assert_close(y.numpy(), oracle.swiglu(X, W, Wu, synth.MLX4, M, N, K), "pageable/pinned")
