"""m4q_mlp_noalloc: the gated MLP block for callers that cannot allocate
device memory (a runtime that owns all device memory and gives plug-ins no
allocator, or a loop that must not call cudaMalloc).  Its intermediate lives
in a fixed array of the library instead of a caller buffer; its results must
match m4q_mlp, which takes that buffer from the caller.

The file name puts it last in collection order; it passes alone and after
the other tests.
"""
import ctypes

import numpy as np
import pytest

import synth
import swiglu_block_quantized_gb300 as m
from _helpers import assert_close, dev, host

pytestmark = pytest.mark.gpu

MAX_H = 1 << 20  # fp16 elements of the library's fixed scratch


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    return m.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _mlp_pair(lib, X, Wg, Wu, Wd, cgu, cd, M, D, F, act):
    """m4q_mlp with a caller intermediate, then m4q_mlp_noalloc on the same
    inputs; returns both outputs on the host."""
    import torch
    H = torch.empty((M, F), dtype=torch.float16, device="cuda")
    Y_ref = torch.empty((M, D), dtype=torch.float16, device="cuda")
    rc = lib.m4q_mlp(_p(X), _p(Wg), _p(Wu), _p(Wd), cgu, cd, M, D, F, _p(H), _p(Y_ref), act, _stream())
    assert rc == m.OK, m.status_string(rc)
    # inputs and output only: the intermediate stays inside the library
    Y = torch.full((M, D), float("nan"), dtype=torch.float16, device="cuda")
    rc = lib.m4q_mlp_noalloc(_p(X), _p(Wg), _p(Wu), _p(Wd), cgu, cd, M, D, F, _p(Y), act, _stream())
    assert rc == m.OK, m.status_string(rc)
    return host(Y), host(Y_ref)


# M = 4 runs both projections on the streaming GEMV, M = 64 on the small-M
# tcgen05 kernel and M = 256 on the prefill tcgen05 kernel, whose TMA stores
# write the intermediate into the library's array.  At F = 4096, M = 256 uses
# the whole array (M * F = 1 << 20).
@pytest.mark.parametrize("M,D,F", [(4, 256, 1024), (64, 256, 4096), (256, 256, 4096)])
def test_noalloc_matches_mlp_on_two_calls_in_a_row(lib, M, D, F):
    cgu, cd = synth.Q4_0, synth.Q8_0
    Wg = dev(synth.weights(cgu, F, D, seed=51, name="Wg"))
    Wu = dev(synth.weights(cgu, F, D, seed=51, name="Wu"))
    Wd = dev(synth.weights(cd, D, F, seed=52, name="Wd"))
    for call, (seed, act) in enumerate(((53, m.ACT_SILU), (54, m.ACT_GELU))):
        X = dev(synth.activations(M, D, seed=seed + M))
        Y, Y_ref = _mlp_pair(lib, X, Wg, Wu, Wd, cgu, cd, M, D, F, act)
        # Both entry points run the same kernels on the same inputs: only the
        # address of the intermediate differs, so the outputs agree bit for
        # bit, and both stay within the tests' tolerance of each other.
        assert np.array_equal(Y.view(np.uint16), Y_ref.view(np.uint16)), "noalloc call %d, M = %d" % (call, M)
        assert_close(Y, Y_ref.astype(np.float64), "noalloc call %d, M = %d" % (call, M))
    assert m.check_device_status() == m.OK


def test_noalloc_rejects_an_intermediate_above_its_scratch(lib):
    import torch
    D = 256
    F = 4096
    M = MAX_H // F + 1  # one row too many
    X = torch.zeros((M, D), dtype=torch.float16, device="cuda")
    Y = torch.zeros((M, D), dtype=torch.float16, device="cuda")
    w = torch.zeros(16, dtype=torch.uint8, device="cuda")  # never read: rejected first
    rc = lib.m4q_mlp_noalloc(_p(X), _p(w), _p(w), _p(w), 0, 0, M, D, F, _p(Y), 0, _stream())
    assert rc == m.ERR_SCRATCH_LIMIT
    assert "scratch" in m.status_string(rc)
