"""The Python binding rejects activations that are not whole rows and output
buffers of the wrong size before anything reaches the library (a kernel
writes every element of its result, so a short buffer would be overrun).
Runs without a GPU: the device checks are replaced by dtype checks and the
library by a stand-in that fails the test if a compute call is made."""
import pytest

import swiglu_block_quantized_gb300 as m

torch = pytest.importorskip("torch")


class _NoLaunch:
    """Library stand-in: sizes work, every other call fails the test."""

    def m4q_weight_bytes(self, codec, n, k):
        b, bb = m.BLOCK[codec], m.BLOCK_BYTES[codec]
        return n * (k // b) * bb if k % b == 0 else 0

    def __getattr__(self, name):
        raise AssertionError("%s was called: the binding did not reject its arguments" % name)


@pytest.fixture
def cpu_binding(monkeypatch):
    def require(t, dtype, what):
        if not isinstance(t, torch.Tensor) or t.dtype != dtype:
            raise TypeError(what)
    monkeypatch.setattr(m, "_require", require)
    monkeypatch.setattr(m, "load", lambda path=None: _NoLaunch())
    return m


def f16(*shape):
    return torch.zeros(shape, dtype=torch.float16)


def packed(codec, n, k):
    return torch.zeros(m.BLOCK_BYTES[codec] * n * (k // m.BLOCK[codec]), dtype=torch.uint8)


def test_rows_counts_whole_rows():
    assert m._rows(f16(3, 64), 64) == 3
    assert m._rows(f16(2, 3, 64), 64) == 6
    assert m._rows(f16(0, 64), 64) == 0
    assert m._rows(f16(3, 64), 48) == 4   # any shape: the element count decides
    with pytest.raises(ValueError):
        m._rows(f16(3, 64), 50)
    with pytest.raises(ValueError):
        m._rows(f16(1, 100), 64)


def test_gemm_rejects_ragged_activations(cpu_binding):
    w = packed(m.Q4_0, 64, 64)
    with pytest.raises(ValueError, match="whole number of rows"):
        m.gemm(f16(1, 100), w, m.Q4_0, 64, 64)


@pytest.mark.parametrize("shape", [(3, 63), (3, 65), (2, 64)])
def test_gemm_rejects_a_wrong_size_output(cpu_binding, shape):
    w = packed(m.Q4_0, 64, 64)
    with pytest.raises(ValueError, match="out holds"):
        m.gemm(f16(3, 64), w, m.Q4_0, 64, 64, out=f16(*shape))


def test_gated_projection_rejects_a_wrong_size_output(cpu_binding):
    w = packed(m.Q8_0, 64, 64)
    with pytest.raises(ValueError, match="out holds"):
        m.swiglu(f16(5, 64), w, w, m.Q8_0, 64, 64, out=f16(4, 64))
    with pytest.raises(ValueError, match="out holds"):
        m.geglu(f16(5, 64), w, w, m.Q8_0, 64, 64, out=f16(5, 72))
    with pytest.raises(ValueError, match="whole number of rows"):
        m.glu(f16(5 * 64 + 8), w, w, m.Q8_0, 64, 64, m.ACT_SILU)


def test_gemm_heads_rejects_a_wrong_size_output(cpu_binding):
    w = packed(m.Q4_0, 256, 64)
    with pytest.raises(ValueError, match="out holds"):
        m.gemm_heads(f16(3, 64), w, m.Q4_0, 256, 64, 128, out=f16(2, 3, 64))
    with pytest.raises(ValueError, match="head_dim"):
        m.gemm_heads(f16(3, 64), w, m.Q4_0, 256, 64, 96)


def test_mlp_rejects_wrong_sizes(cpu_binding):
    d, f = 64, 128
    wg = packed(m.Q4_0, f, d)
    wd = packed(m.Q4_0, d, f)
    with pytest.raises(ValueError, match="out holds"):
        m.mlp(f16(2, d), wg, wg, wd, m.Q4_0, m.Q4_0, d, f, out=f16(3, d))
    with pytest.raises(ValueError, match="h holds"):
        m.mlp(f16(2, d), wg, wg, wd, m.Q4_0, m.Q4_0, d, f, h=f16(1, f), out=f16(2, d))
    with pytest.raises(ValueError, match="whole number of rows"):
        m.mlp(f16(2 * d + 1), wg, wg, wd, m.Q4_0, m.Q4_0, d, f)


def test_dequant_rejects_a_wrong_size_output(cpu_binding):
    w = packed(m.Q2_0, 8, 256)
    with pytest.raises(ValueError, match="out holds"):
        m.dequant(w, m.Q2_0, 8, 256, out=f16(8, 255))


def test_empty_batch_returns_without_a_launch(cpu_binding):
    w = packed(m.Q4_0, 64, 64)
    assert m.gemm(f16(0, 64), w, m.Q4_0, 64, 64).shape == (0, 64)
    assert m.swiglu(f16(0, 64), w, w, m.Q4_0, 64, 64).shape == (0, 64)
    assert m.gemm_heads(f16(0, 64), w, m.Q4_0, 64, 64, 64).shape == (1, 0, 64)
    y = m.mlp(f16(0, 64), w, w, w, m.Q4_0, m.Q4_0, 64, 64)
    assert y.shape == (0, 64)
    lin = m.QuantLinear(w, m.Q4_0, 64, 64)
    assert lin(f16(2, 0, 64)).shape == (2, 0, 64)
