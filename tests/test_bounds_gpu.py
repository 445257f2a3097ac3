"""Every kernel run through the bounds-checked build (-DM4Q_BOUNDS=1): each
computed global access, TMA coordinate and shared-memory staging offset is
tested before it is made, so an index out of range is reported (status
M4Q_ERR_BOUNDS and the failing site) instead of faulting.  The sweep covers
every path (GEMV with and without resident activations and with 2-byte
weight copies, the small-M kernel with and without a K split, the prefill
kernel at every tile width, with a K split, head-major output and 2-byte
weight loads, GeGLU and the MLP chain, attention prefill and split decode)
on ragged shapes, and requires results bit-identical to the normal build."""
import contextlib

import numpy as np
import pytest

import swiglu_block_quantized_gb300 as m
import synth

from _helpers import dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    m.build()
    m.build(bounds=True)
    normal = m.load()
    checked = m.load(m.LIB_BOUNDS_PATH)
    assert checked.m4q_build_flags() == m.BUILD_BOUNDS
    return normal, checked


@contextlib.contextmanager
def using(lib):
    old = m._lib
    m._lib = lib
    try:
        yield
    finally:
        m._lib = old


def run_both(libs, fn):
    """fn() with the normal and the bounds-checked library: identical bits,
    no failed check, no timeout."""
    outs = []
    for lib in libs:
        with using(lib):
            y = host(fn())
            assert m.check_device_status() == m.OK
            assert m.bounds_site() == 0
        outs.append(y)
    assert outs[0].dtype == outs[1].dtype
    assert np.array_equal(outs[0].view(np.uint8), outs[1].view(np.uint8))


PROJ_CASES = [
    # (codec, M, N, K, path): GEMV (resident X at M <= 8, K = 4096), 2-byte
    # weight copies (rows not 16-byte multiples), small-M kernel with and
    # without a K split, prefill kernel (64, 128 and 256 wide, K split)
    (synth.Q4_0, 1, 264, 4096, m.PATH_AUTO),
    (synth.Q8_0, 9, 136, 2048, m.PATH_AUTO),
    (synth.MLX4, 5, 200, 4096, m.PATH_AUTO),
    (synth.Q2_0, 16, 264, 4096, m.PATH_AUTO),
    (synth.Q4_0, 3, 136, 2080, m.PATH_AUTO),
    (synth.Q4_0, 17, 264, 4096, m.PATH_AUTO),
    (synth.Q8_0, 64, 2048, 2048, m.PATH_AUTO),
    (synth.MLX4, 100, 136, 2048, m.PATH_AUTO),
    (synth.Q4_0, 128, 512, 8192, m.PATH_AUTO),
    (synth.Q4_0, 129, 264, 2048, m.PATH_AUTO),
    (synth.Q8_0, 300, 520, 2048, m.PATH_AUTO),
    (synth.Q2_0, 257, 1024, 4096, m.PATH_AUTO),
    (synth.Q4_0, 300, 200, 2080, m.PATH_TC),
    (synth.Q4_0, 2048, 2048, 2048, m.PATH_AUTO),
]


@pytest.mark.parametrize("codec,M,N,K,path", PROJ_CASES)
def test_projection_in_bounds(libs, codec, M, N, K, path):
    X = dev(synth.activations(M, K, seed=M))
    W = dev(synth.weights(codec, N, K, seed=N))
    Wu = dev(synth.weights(codec, N, K, seed=N, name="Wu"))
    run_both(libs, lambda: m.gemm(X, W, codec, N, K, path=path))
    run_both(libs, lambda: m.swiglu(X, W, Wu, codec, N, K, path=path))


@pytest.mark.parametrize("M", [1, 40, 300])
@pytest.mark.parametrize("hd", [64, 128])
def test_head_major_output_in_bounds(libs, M, hd):
    N, K = 3 * 256, 2048
    X = dev(synth.activations(M, K, seed=M))
    W = dev(synth.weights(synth.Q8_0, N, K, seed=hd))
    run_both(libs, lambda: m.gemm_heads(X, W, synth.Q8_0, N, K, hd))


@pytest.mark.parametrize("M", [4, 96, 384])
def test_geglu_and_mlp_in_bounds(libs, M):
    d, f = 2048, 1024
    X = dev(synth.activations(M, d, seed=M))
    Wg = dev(synth.weights(synth.Q4_0, f, d, seed=1, name="Wg"))
    Wu = dev(synth.weights(synth.Q4_0, f, d, seed=1, name="Wu"))
    Wd = dev(synth.weights(synth.Q8_0, d, f, seed=2, name="Wd"))
    run_both(libs, lambda: m.glu(X, Wg, Wu, synth.Q4_0, f, d, m.ACT_GELU))
    run_both(libs, lambda: m.mlp(X, Wg, Wu, Wd, synth.Q4_0, synth.Q8_0, d, f))


@pytest.mark.parametrize("kv", [m.KV_F16, m.Q8_0])
@pytest.mark.parametrize("H,Hkv,M,T,D", [(8, 2, 200, 200, 64), (4, 4, 33, 161, 128), (8, 2, 1, 4096, 128),
                                         (32, 8, 4, 3000, 64), (32, 8, 1100, 1200, 128)])
def test_attention_in_bounds(libs, kv, H, Hkv, M, T, D):
    Q = dev(synth.queries(H, M, D, seed=T))
    K = dev(synth.kv_cache(kv, Hkv, T, D, seed=T + 1, name="K"))
    V = dev(synth.kv_cache(kv, Hkv, T, D, seed=T + 1, name="V"))
    run_both(libs, lambda: m.attention(Q, K, V, kv, Hkv, T))
