"""The C ABI library loads, exports every symbol include/m4q.h declares, and
rejects bad arguments before touching the GPU (runs without a GPU)."""
import ctypes
import os
import re

import pytest

import swiglu_block_quantized_gb300 as m


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    m.build()
    return m.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "m4q.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(m4q_\w+)\s*\(", text)))


def test_header_declares_the_core_calls():
    fns = header_functions()
    for name in ("m4q_gemm", "m4q_swiglu", "m4q_dequant", "m4q_weight_bytes", "m4q_status_string"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert name in m.SIGNATURES, name
    assert sorted(m.SIGNATURES) == header_functions()


def test_weight_bytes(lib):
    assert m.weight_bytes(m.Q4_0, 8192, 2048) == 8192 * 64 * 18
    assert m.weight_bytes(m.Q8_0, 8192, 2048) == 8192 * 64 * 34
    assert m.weight_bytes(m.Q2_0, 4096, 4096) == 4096 * 32 * 34
    assert m.weight_bytes(m.Q2_0, 4096, 4000) == 0      # K not a multiple of 128
    assert m.weight_bytes(m.MLX4, 8192, 2048) == 8192 * 64 * 20
    assert m.weight_bytes(7, 16, 32) == 0


def test_status_strings(lib):
    assert m.status_string(m.OK) == "ok"
    assert "aligned" in m.status_string(m.ERR_MISALIGNED)
    assert m.status_string(12345) == "unknown status"
    assert m.version() == 100


def P(v):
    return ctypes.c_void_p(v)


def test_argument_errors_return_before_any_cuda_call(lib):
    good = 0x100000   # 16-byte aligned, never dereferenced: every case fails validation first
    s = None
    assert lib.m4q_gemm(None, P(good), 0, 4, 8, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_gemm(P(good), P(good), 9, 4, 8, 32, P(good), s) == m.ERR_UNSUPPORTED_CODEC
    assert lib.m4q_gemm(P(good), P(good), 0, 0, 8, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_gemm(P(good), P(good), 0, 4, 8, 48, P(good), s) == m.ERR_BAD_SHAPE   # K % 32
    assert lib.m4q_gemm(P(good), P(good), 2, 4, 8, 64, P(good), s) == m.ERR_BAD_SHAPE   # K % 128
    assert lib.m4q_gemm(P(good), P(good), 0, 4, 12, 32, P(good), s) == m.ERR_BAD_SHAPE  # N % 8
    assert lib.m4q_gemm(P(good + 2), P(good), 0, 4, 8, 32, P(good), s) == m.ERR_MISALIGNED
    assert lib.m4q_gemm(P(good), P(good), 0, 4, 8, 32, P(good + 8), s) == m.ERR_MISALIGNED
    assert lib.m4q_swiglu(P(good), P(good), None, 0, 4, 8, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_swiglu(P(good), P(good), P(good + 4), 0, 4, 8, 32, P(good), s) == m.ERR_MISALIGNED
    assert lib.m4q_gemm_ex(P(good), P(good), 0, 17, 8, 32, P(good), m.PATH_GEMV, s) == m.ERR_INVALID_ARG
    assert lib.m4q_gemm_ex(P(good), P(good), 0, 4, 8, 32, P(good), 7, s) == m.ERR_INVALID_ARG
    assert lib.m4q_glu_ex(P(good), P(good), P(good), 0, 4, 8, 32, P(good), 2, 0, s) == m.ERR_INVALID_ARG  # act
    assert lib.m4q_glu_ex(P(good), P(good), P(good), 0, 4, 8, 32, P(good), -1, 0, s) == m.ERR_INVALID_ARG
    assert lib.m4q_geglu(P(good), P(good), None, 0, 4, 8, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_geglu(P(good), P(good), P(good), 0, 4, 12, 32, P(good), s) == m.ERR_BAD_SHAPE
    assert lib.m4q_gemm_heads(P(good), P(good), 0, 4, 128, 32, 96, P(good), s) == m.ERR_INVALID_ARG   # head dim
    assert lib.m4q_gemm_heads(P(good), P(good), 0, 4, 128, 32, 0, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_gemm_heads(P(good), P(good), 0, 4, 192, 32, 128, P(good), s) == m.ERR_BAD_SHAPE  # N % hd
    # m4q_mlp validates both projections before enqueueing anything
    assert lib.m4q_mlp(P(good), P(good), P(good), P(good), 0, 1, 4, 64, 128, None, P(good), 0, s) == m.ERR_INVALID_ARG
    assert lib.m4q_mlp(P(good), P(good), P(good), P(good), 0, 1, 4, 64, 132, P(good), P(good), 0, s) == m.ERR_BAD_SHAPE
    assert lib.m4q_mlp(P(good), P(good), P(good), P(good), 0, 2, 4, 64, 192, P(good), P(good), 0, s) == m.ERR_BAD_SHAPE
    assert lib.m4q_mlp(P(good), P(good), P(good), P(good), 0, 1, 4, 64, 128, P(good + 8), P(good), 0, s) == m.ERR_MISALIGNED
    assert lib.m4q_mlp(P(good), P(good), P(good), P(good), 0, 1, 4, 64, 128, P(good), P(good), 5, s) == m.ERR_INVALID_ARG
    assert lib.m4q_dequant(None, 0, 8, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_dequant(P(good), 0, 8, 40, P(good), s) == m.ERR_BAD_SHAPE
    assert lib.m4q_dequant(P(good), 4, 8, 32, P(good), s) == m.ERR_UNSUPPORTED_CODEC
    assert lib.m4q_gemm(P(good), P(good), 3, 4, 8, 48, P(good), s) == m.ERR_BAD_SHAPE   # MLX4 K % 32
    assert lib.m4q_mlx4_pack(None, P(good), P(good), 8, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_mlx4_pack(P(good), P(good), P(good), 0, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_mlx4_pack(P(good), P(good), P(good), 8, 48, P(good), s) == m.ERR_BAD_SHAPE
    assert lib.m4q_mlx4_pack(P(good + 4), P(good), P(good), 8, 32, P(good), s) == m.ERR_MISALIGNED
    assert lib.m4q_mlx4_pack(P(good), P(good + 1), P(good), 8, 32, P(good), s) == m.ERR_MISALIGNED
    assert lib.m4q_mlx4_pack(P(good), P(good), P(good + 3), 8, 32, P(good), s) == m.ERR_MISALIGNED
    assert lib.m4q_mlx4_pack(P(good), P(good), P(good), 8, 32, P(good + 4), s) == m.ERR_MISALIGNED
    assert lib.m4q_repack(None, 0, 8, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_repack(P(good), 0, 8, 32, None, s) == m.ERR_INVALID_ARG
    assert lib.m4q_repack(P(good), 4, 8, 32, P(good), s) == m.ERR_UNSUPPORTED_CODEC
    assert lib.m4q_repack(P(good), 0, 0, 32, P(good), s) == m.ERR_INVALID_ARG
    assert lib.m4q_repack(P(good), 2, 8, 64, P(good), s) == m.ERR_BAD_SHAPE   # Q2_0 K % 128
    assert lib.m4q_repack(P(good + 2), 0, 8, 32, P(good), s) == m.ERR_MISALIGNED
    assert lib.m4q_repack(P(good), 3, 8, 32, P(good + 8), s) == m.ERR_MISALIGNED
    assert lib.m4q_check_finite(None, 10, s) == m.ERR_INVALID_ARG
    att = lambda q, k, v, codec, H, Hkv, M, T, D, off, sc, o, ws=None, wsb=0: lib.m4q_attention(
        q, k, v, codec, H, Hkv, M, T, D, off, 1, sc, o, ws, wsb, s)
    assert att(None, P(good), P(good), m.KV_F16, 4, 2, 8, 8, 64, 0, 0.125, P(good)) == m.ERR_INVALID_ARG
    assert att(P(good), P(good), P(good), m.Q4_0, 4, 2, 8, 8, 64, 0, 0.125, P(good)) == m.ERR_UNSUPPORTED_CODEC
    assert att(P(good), P(good), P(good), m.KV_F16, 4, 3, 8, 8, 64, 0, 0.125, P(good)) == m.ERR_BAD_SHAPE
    assert att(P(good), P(good), P(good), m.Q8_0, 4, 2, 8, 8, 96, 0, 0.125, P(good)) == m.ERR_BAD_SHAPE
    assert att(P(good), P(good), P(good), m.Q8_0, 4, 2, 0, 8, 64, 0, 0.125, P(good)) == m.ERR_INVALID_ARG
    assert att(P(good), P(good), P(good), m.Q8_0, 4, 2, 8, 8, 64, -1, 0.125, P(good)) == m.ERR_INVALID_ARG
    assert att(P(good), P(good), P(good), m.Q8_0, 4, 2, 8, 8, 64, 0, float("nan"), P(good)) == m.ERR_INVALID_ARG
    assert att(P(good), P(good + 2), P(good), m.Q8_0, 4, 2, 8, 8, 64, 0, 0.125, P(good)) == m.ERR_MISALIGNED
    assert att(P(good), P(good), P(good), m.Q8_0, 4, 2, 8, 8, 64, 0, 0.125, P(good + 8)) == m.ERR_MISALIGNED
    assert lib.m4q_attention_workspace_bytes(4, 3, 8, 8, 64) == 0
    assert lib.m4q_selftest_wait_timeout(10, s) == m.ERR_INVALID_ARG


def test_python_binding_rejects_non_cuda_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 32, dtype=torch.float16)
    w = torch.zeros(m.weight_bytes(m.Q4_0, 8, 32), dtype=torch.uint8)
    with pytest.raises(TypeError):
        m.gemm(x, w, m.Q4_0, 8, 32)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        m.load(str(tmp_path / "nope.so"))


def test_project_host_argument_errors(lib):
    good = 0x100000
    s = None
    # null host or staging pointers, negative chunk
    assert lib.m4q_project_host(None, P(good), None, 0, 0, 4, 8, 32, P(good), P(good), P(good), 0, s, s, s) \
        == m.ERR_INVALID_ARG
    assert lib.m4q_project_host(P(good), P(good), None, 0, 0, 4, 8, 32, P(good), None, P(good), 0, s, s, s) \
        == m.ERR_INVALID_ARG
    assert lib.m4q_project_host(P(good), P(good), None, 0, 0, 4, 8, 32, P(good), P(good), P(good), -1, s, s, s) \
        == m.ERR_INVALID_ARG
    assert lib.m4q_project_host(P(good), P(good), P(good), 0, 5, 4, 8, 32, P(good), P(good), P(good), 0, s, s, s) \
        == m.ERR_INVALID_ARG   # activation
    assert lib.m4q_project_host(P(good), P(good), None, 0, 0, 4, 12, 32, P(good), P(good), P(good), 0, s, s, s) \
        == m.ERR_BAD_SHAPE
    assert lib.m4q_project_host(P(good), P(good), None, 0, 0, 4, 8, 32, P(good), P(good + 8), P(good), 0, s, s, s) \
        == m.ERR_MISALIGNED
