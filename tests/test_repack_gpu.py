"""GPU parity of m4q_repack (packed blocks -> planes) with the oracle's
repack, byte for byte, through the C ABI: every codec, one block to the 8B
gate matrix, a guard region after the output that must stay untouched, and
the MLX4 planes turned back into the same blocks by m4q_mlx4_pack."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
import swiglu_block_quantized_gb300 as m

pytestmark = pytest.mark.gpu

CODECS = [synth.Q4_0, synth.Q8_0, synth.Q2_0, synth.MLX4]
GUARD = 64


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    yield m.load()
    assert m.check_device_status() == m.OK


def _repack_c(lib, W, codec, N, K):
    """m4q_repack through the C ABI into a buffer with a guard region after
    the planes; returns (planes, guard bytes)."""
    import torch
    w = torch.from_numpy(np.ascontiguousarray(W).reshape(-1)).cuda()
    nbytes = m.weight_bytes(codec, N, K)
    out = torch.full((nbytes + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.m4q_repack(ctypes.c_void_p(w.data_ptr()), codec, N, K, ctypes.c_void_p(out.data_ptr()), s)
    assert rc == m.OK, m.status_string(rc)
    torch.cuda.synchronize()
    host = out.cpu().numpy()
    return host[:nbytes], host[nbytes:]


@pytest.mark.parametrize("codec", CODECS)
def test_repack_bit_exact(lib, codec):
    B = synth.BLOCK[codec]
    for N, K in ((1, B), (3, 3 * B), (264, 4096), (1000, 2048)):
        W = synth.weights(codec, N, K, seed=N + K, name="W")
        P, guard = _repack_c(lib, W, codec, N, K)
        assert np.array_equal(P, oracle.repack(W, codec, N, K)), (codec, N, K)
        assert np.all(guard == 0xA5), "repack wrote past its output"


def test_repack_8b_gate_matrix(lib):
    N, K = 14336, 4096
    W = synth.weights(synth.Q4_0, N, K, seed=2, name="Wg")
    P, guard = _repack_c(lib, W, synth.Q4_0, N, K)
    assert np.array_equal(P, oracle.repack(W, synth.Q4_0, N, K))
    assert np.all(guard == 0xA5)


def test_mlx4_planes_pack_back_to_blocks(lib):
    import torch
    N, K = 300, 2048
    W = synth.weights(synth.MLX4, N, K, seed=5, name="W")
    P = m.repack(torch.from_numpy(W).cuda(), synth.MLX4, N, K)
    nb = K // 32
    words = P[:N * nb * 16]
    scales = P[N * nb * 16:N * nb * 18].view(torch.float16)
    biases = P[N * nb * 18:].view(torch.float16)
    back = m.mlx4_pack(words, scales, biases, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), W)
