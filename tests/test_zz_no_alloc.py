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


def test_noalloc_matches_mlp_on_two_calls_in_a_row(lib):
    import torch
    M, D, F = 4, 256, 1024
    cgu, cd = synth.Q4_0, synth.Q8_0
    Wg = dev(synth.weights(cgu, F, D, seed=51, name="Wg"))
    Wu = dev(synth.weights(cgu, F, D, seed=51, name="Wu"))
    Wd = dev(synth.weights(cd, D, F, seed=52, name="Wd"))
    for call, (seed, act) in enumerate(((53, m.ACT_SILU), (54, m.ACT_GELU))):
        X = dev(synth.activations(M, D, seed=seed))
        # the existing entry point, with a caller-provided intermediate
        H = torch.empty((M, F), dtype=torch.float16, device="cuda")
        Y_ref = torch.empty((M, D), dtype=torch.float16, device="cuda")
        rc = lib.m4q_mlp(_p(X), _p(Wg), _p(Wu), _p(Wd), cgu, cd, M, D, F, _p(H), _p(Y_ref), act, _stream())
        assert rc == m.OK, m.status_string(rc)
        # the no-allocation entry point: inputs and output only
        Y = torch.full((M, D), float("nan"), dtype=torch.float16, device="cuda")
        rc = lib.m4q_mlp_noalloc(_p(X), _p(Wg), _p(Wu), _p(Wd), cgu, cd, M, D, F, _p(Y), act, _stream())
        assert rc == m.OK, m.status_string(rc)
        torch.cuda.synchronize()
        assert_close(host(Y), host(Y_ref).astype(np.float64), "noalloc call %d" % call)
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
