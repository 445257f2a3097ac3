"""Python binding of libm4q.so: the block-quantized projection GEMM and the
fused gate/up SwiGLU projection for one GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libm4q.so (see include/m4q.h).  PyTorch supplies device memory and
streams.  There is no fallback: if the library is missing or the device is not
sm_103, calls raise.

Functions mirror the C ABI (same names without the ``m4q_`` prefix):
    gemm(x, w, codec, n, k, out=None, path=PATH_AUTO)
    gemm_heads(x, w, codec, n, k, head_dim, out=None)
    swiglu(x, wg, wu, codec, n, k, out=None, path=PATH_AUTO)
    geglu(x, wg, wu, codec, n, k, out=None, path=PATH_AUTO)
    glu(x, wg, wu, codec, n, k, act, out=None, path=PATH_AUTO)
    mlp(x, wg, wu, wd, codec_gu, codec_d, d, f, act=ACT_SILU, h=None, out=None)
    project_host(x_host, w, codec, n, k, wu=None, act=ACT_SILU, out=None, ...)
    dequant(w, codec, n, k, out=None)
    mlx4_pack(words, scales, biases, n, k, out=None)
    attention(q, k, v, kv_codec, hkv, t, q_offset=None, causal=True, scale=None, out=None)
    weight_bytes(codec, n, k), check_finite(t), check_device_status(),
    selftest_wait_timeout(limit_ns), status_string(code), version()
Activations are read as M whole rows (their element count must be a multiple
of the row length) and a caller's ``out`` must hold exactly the result's
element count; both are checked before anything is launched.  M = 0 (an
empty batch) returns an empty result without a launch.

``QuantLinear`` is the layer wrapper (leading batch dimensions are
flattened into M; M <= 16 streams the weights, larger M uses tcgen05), the
analogue of the pages' M4QuantizedLinear ("Releases" v0.3.0); ``QuantGLU``
wraps the gated gate/up projection (SwiGLU or GeGLU), ``QuantMLP`` the
whole gated MLP block (gate/up then down, one stream) and ``QuantQKV`` the
fused Q/K/V projection with head-major outputs.
"""
from __future__ import annotations

import ctypes
import os
import threading

Q4_0, Q8_0, Q2_0, MLX4 = 0, 1, 2, 3
CODECS = (Q4_0, Q8_0, Q2_0, MLX4)
BLOCK = {Q4_0: 32, Q8_0: 32, Q2_0: 128, MLX4: 32}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q2_0: 34, MLX4: 20}
KV_F16 = 16   # fp16 KV cache values (the quantized KV cache uses Q8_0)
PATH_AUTO, PATH_GEMV, PATH_TC = 0, 1, 2
ACT_SILU, ACT_GELU = 0, 1

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_CODEC = -2
ERR_BAD_SHAPE = -3
ERR_MISALIGNED = -4
ERR_CUDA = -5
ERR_NONFINITE = -6
ERR_TIMEOUT = -7
ERR_UNSUPPORTED_DEVICE = -8
ERR_SCRATCH_LIMIT = -9
ERR_BOUNDS = -10
BUILD_BOUNDS = 1

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libm4q.so")
LIB_BOUNDS_PATH = os.path.join(HERE, "_build", "libm4q_bounds.so")   # bounds-checked build

# Every symbol declared in include/m4q.h, with its ctypes signature.
_i64, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
SIGNATURES = {
    "m4q_gemm": (_i32, [_vp, _vp, _i32, _i64, _i64, _i64, _vp, _vp]),
    "m4q_swiglu": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _i64, _vp, _vp]),
    "m4q_gemm_ex": (_i32, [_vp, _vp, _i32, _i64, _i64, _i64, _vp, _i32, _vp]),
    "m4q_swiglu_ex": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _i64, _vp, _i32, _vp]),
    "m4q_geglu": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _i64, _vp, _vp]),
    "m4q_gemm_heads": (_i32, [_vp, _vp, _i32, _i64, _i64, _i64, _i64, _vp, _vp]),
    "m4q_glu_ex": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _i64, _vp, _i32, _i32, _vp]),
    "m4q_mlp": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i64, _i64, _i64, _vp, _vp, _i32, _vp]),
    "m4q_mlp_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i64, _i64, _i64, _vp, _i32, _vp]),
    "m4q_project_host": (_i32, [_vp, _vp, _vp, _i32, _i32, _i64, _i64, _i64, _vp, _vp, _vp, _i64, _vp, _vp,
                                _vp]),
    "m4q_dequant": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp]),
    "m4q_mlx4_pack": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp, _vp]),
    "m4q_repack": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp]),
    "m4q_attention": (_i32, [_vp, _vp, _vp, _i32, _i64, _i64, _i64, _i64, _i64, _i64, _i32,
                             ctypes.c_float, _vp, _vp, _sz, _vp]),
    "m4q_attention_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _i64]),
    "m4q_attention_workspace": (_sz, [_i32, _i64, _i64, _i64, _i64, _i64]),
    "m4q_weight_bytes": (_sz, [_i32, _i64, _i64]),
    "m4q_check_finite": (_i32, [_vp, _i64, _vp]),
    "m4q_check_device_status": (_i32, [_vp]),
    "m4q_build_flags": (_i32, []),
    "m4q_bounds_site": (_i32, [_vp]),
    "m4q_selftest_wait_timeout": (_i32, [_i64, _vp]),
    "m4q_status_string": (ctypes.c_char_p, [_i32]),
    "m4q_version": (_i32, []),
}

_lock = threading.Lock()
_lib = None


class M4QError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, status_string(code), code))


def load(path: str | None = None):
    """Load libm4q.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError("libm4q.so not built (run python -m swiglu_block_quantized_gb300.buildlib): %s" % p)
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def build(force: bool = False, bounds: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force, bounds=bounds)


def status_string(code: int) -> str:
    try:
        return load().m4q_status_string(code).decode()
    except ImportError:
        return "status %d" % code


def version() -> int:
    return int(load().m4q_version())


def weight_bytes(codec: int, n: int, k: int) -> int:
    return int(load().m4q_weight_bytes(codec, n, k))


def _check(rc: int, what: str):
    if rc != OK:
        raise M4QError(rc, what)


def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _require(t, dtype, what):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % what)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)


def _rows(x, k: int, what: str = "x") -> int:
    """Rows M of an activation tensor read as [M, k]; its element count must
    be a whole number of rows (M = 0 is allowed: an empty batch)."""
    if k < 1 or x.numel() % k != 0:
        raise ValueError("%s holds %d elements, not a whole number of rows of %d"
                         % (what, x.numel(), k))
    return x.numel() // k


def _result(out, shape, device, what="out"):
    """The caller's output tensor, checked to hold exactly prod(shape) fp16
    values, or a new one of that shape.  A kernel writes every element of the
    result, so a smaller buffer would be overrun and a larger one only partly
    written: both are rejected before anything is launched."""
    import torch
    need = 1
    for s in shape:
        need *= int(s)
    if out is None:
        return torch.empty(tuple(int(s) for s in shape), dtype=torch.float16, device=device)
    _require(out, torch.float16, what)
    if out.numel() != need:
        raise ValueError("%s holds %d elements, expected %d for shape %s"
                         % (what, out.numel(), need, tuple(int(s) for s in shape)))
    return out


def _packed_check(w, codec, n, k, what):
    import torch
    _require(w, torch.uint8, what)
    need = weight_bytes(codec, n, k)
    if need == 0 or w.numel() != need:
        raise ValueError("%s holds %d bytes, expected %d for %s [%d, %d]"
                         % (what, w.numel(), need, codec, n, k))


def gemm(x, w, codec: int, n: int, k: int, out=None, path: int = PATH_AUTO, stream=None):
    """Y[M, n] = X[M, k] . W^T with W packed [n, k] (uint8 blocks).  X holds
    M whole rows of k values; out, if given, exactly M * n values."""
    import torch
    _require(x, torch.float16, "x")
    _packed_check(w, codec, n, k, "w")
    m = _rows(x, k)
    out = _result(out, (m, n), x.device)
    if m == 0:
        return out
    _check(load().m4q_gemm_ex(x.data_ptr(), w.data_ptr(), codec, m, n, k, out.data_ptr(),
                              path, _stream_ptr(stream)), "m4q_gemm")
    return out


def gemm_heads(x, w, codec: int, n: int, k: int, head_dim: int, out=None, stream=None):
    """Y[n / head_dim, M, head_dim] with Y[h, m, d] = (X . W^T)[m, h * head_dim + d]."""
    import torch
    _require(x, torch.float16, "x")
    _packed_check(w, codec, n, k, "w")
    if head_dim < 1 or n % head_dim != 0:
        raise ValueError("head_dim %d must divide n = %d" % (head_dim, n))
    m = _rows(x, k)
    out = _result(out, (n // head_dim, m, head_dim), x.device)
    if m == 0:
        return out
    _check(load().m4q_gemm_heads(x.data_ptr(), w.data_ptr(), codec, m, n, k, head_dim, out.data_ptr(),
                                 _stream_ptr(stream)), "m4q_gemm_heads")
    return out


def glu(x, wg, wu, codec: int, n: int, k: int, act: int, out=None, path: int = PATH_AUTO, stream=None):
    """Y[M, n] = act(X . Wg^T) * (X . Wu^T), act = ACT_SILU or ACT_GELU."""
    import torch
    _require(x, torch.float16, "x")
    _packed_check(wg, codec, n, k, "wg")
    _packed_check(wu, codec, n, k, "wu")
    m = _rows(x, k)
    out = _result(out, (m, n), x.device)
    if m == 0:
        return out
    _check(load().m4q_glu_ex(x.data_ptr(), wg.data_ptr(), wu.data_ptr(), codec, m, n, k,
                             out.data_ptr(), act, path, _stream_ptr(stream)), "m4q_glu_ex")
    return out


def swiglu(x, wg, wu, codec: int, n: int, k: int, out=None, path: int = PATH_AUTO, stream=None):
    """Y[M, n] = SiLU(X . Wg^T) * (X . Wu^T)."""
    return glu(x, wg, wu, codec, n, k, ACT_SILU, out=out, path=path, stream=stream)


def geglu(x, wg, wu, codec: int, n: int, k: int, out=None, path: int = PATH_AUTO, stream=None):
    """Y[M, n] = GELU(X . Wg^T) * (X . Wu^T)."""
    return glu(x, wg, wu, codec, n, k, ACT_GELU, out=out, path=path, stream=stream)


def mlp(x, wg, wu, wd, codec_gu: int, codec_d: int, d: int, f: int, act: int = ACT_SILU,
        h=None, out=None, stream=None):
    """Y[M, d] = (act(X Wg^T) * (X Wu^T)) Wd^T; Wg, Wu packed [f, d], Wd packed
    [d, f].  h (fp16 [M, f]) receives the intermediate; allocated if None."""
    import torch
    _require(x, torch.float16, "x")
    _packed_check(wg, codec_gu, f, d, "wg")
    _packed_check(wu, codec_gu, f, d, "wu")
    _packed_check(wd, codec_d, d, f, "wd")
    m = _rows(x, d)
    out = _result(out, (m, d), x.device)
    if h is None:
        h = torch.empty((m, f), dtype=torch.float16, device=x.device)
    _require(h, torch.float16, "h")
    if h.numel() < m * f:
        raise ValueError("h holds %d elements, needs %d" % (h.numel(), m * f))
    if m == 0:
        return out
    _check(load().m4q_mlp(x.data_ptr(), wg.data_ptr(), wu.data_ptr(), wd.data_ptr(), codec_gu, codec_d,
                          m, d, f, h.data_ptr(), out.data_ptr(), act, _stream_ptr(stream)), "m4q_mlp")
    return out


_host_streams_by_device = {}


def _host_streams(device):
    """Two copy streams per device, created once, for project_host."""
    import torch
    key = torch.device(device).index
    if key not in _host_streams_by_device:
        _host_streams_by_device[key] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    return _host_streams_by_device[key]


def project_host(x, w, codec: int, n: int, k: int, wu=None, act: int = ACT_SILU, out=None, x_dev=None,
                 y_dev=None, chunk_rows: int = 0, stream=None):
    """Y = X W^T (wu None) or act(X W^T) * (X Wu^T) with X and Y in host
    memory: chunks of rows are copied in, projected and copied back with the
    copies overlapping the kernels (m4q_project_host).  x: CPU fp16 [..., k]
    (page-locked for overlap); out: CPU fp16 [M, n], page-locked when
    allocated here.  x_dev / y_dev: device staging [M, k] / [M, n], allocated
    if not given.  The result is complete once the current stream (or
    `stream`) has reached this point: synchronize it before reading out."""
    import torch
    if not isinstance(x, torch.Tensor) or x.is_cuda or x.dtype != torch.float16 or not x.is_contiguous():
        raise TypeError("x must be a contiguous fp16 host tensor")
    _packed_check(w, codec, n, k, "w")
    if wu is not None:
        _packed_check(wu, codec, n, k, "wu")
    m = _rows(x, k)
    if out is None:
        out = torch.empty((m, n), dtype=torch.float16, pin_memory=True)
    elif (not isinstance(out, torch.Tensor) or out.is_cuda or out.dtype != torch.float16
          or not out.is_contiguous() or out.numel() != m * n):
        raise ValueError("out must be a contiguous fp16 host tensor of %d elements" % (m * n))
    x_dev = _result(x_dev, (m, k), w.device, "x_dev")
    y_dev = _result(y_dev, (m, n), w.device, "y_dev")
    if m == 0:
        return out
    s_in, s_out = _host_streams(w.device)
    _check(load().m4q_project_host(x.data_ptr(), w.data_ptr(), wu.data_ptr() if wu is not None else None, codec,
                                   act, m, n, k, out.data_ptr(), x_dev.data_ptr(), y_dev.data_ptr(), chunk_rows,
                                   _stream_ptr(stream), ctypes.c_void_p(s_in.cuda_stream),
                                   ctypes.c_void_p(s_out.cuda_stream)), "m4q_project_host")
    return out


def dequant(w, codec: int, n: int, k: int, out=None, stream=None):
    """fp16 [n, k] decode of the packed weights (bit-exact test hook)."""
    import torch
    _packed_check(w, codec, n, k, "w")
    out = _result(out, (n, k), w.device)
    _check(load().m4q_dequant(w.data_ptr(), codec, n, k, out.data_ptr(), _stream_ptr(stream)),
           "m4q_dequant")
    return out


def mlx4_pack(words, scales, biases, n: int, k: int, out=None, stream=None):
    """MLX planar arrays -> MLX4 blocks uint8 [n, (k/32) * 20].  words holds
    the [n, k/8] little-endian uint32 code words (any contiguous CUDA tensor
    of n * k / 2 bytes, e.g. int32 [n, k/8]); scales and biases are fp16
    [n, k/32]."""
    import torch
    if not isinstance(words, torch.Tensor) or not words.is_cuda or not words.is_contiguous():
        raise TypeError("words must be a contiguous CUDA tensor")
    if k % 32 or words.numel() * words.element_size() != n * k // 2:
        raise ValueError("words must hold n * k / 2 bytes with k % 32 == 0")
    for t, what in ((scales, "scales"), (biases, "biases")):
        _require(t, torch.float16, what)
        if t.numel() != n * (k // 32):
            raise ValueError("%s must hold n * k / 32 values" % what)
    if out is None:
        out = torch.empty((n, (k // 32) * 20), dtype=torch.uint8, device=words.device)
    _packed_check(out, MLX4, n, k, "out")
    _check(load().m4q_mlx4_pack(words.data_ptr(), scales.data_ptr(), biases.data_ptr(), n, k,
                                out.data_ptr(), _stream_ptr(stream)), "m4q_mlx4_pack")
    return out


def repack(w, codec: int, n: int, k: int, out=None, stream=None):
    """Packed blocks [n, k] -> planes, uint8 [weight_bytes(codec, n, k)]: the
    code bytes of every block in row-major block order, then the fp16 scales
    [n, k/B], then (MLX4) the fp16 biases [n, k/B]."""
    import torch
    _packed_check(w, codec, n, k, "w")
    if out is None:
        out = torch.empty(weight_bytes(codec, n, k), dtype=torch.uint8, device=w.device)
    _require(out, torch.uint8, "out")
    if out.numel() != weight_bytes(codec, n, k):
        raise ValueError("out must hold %d bytes" % weight_bytes(codec, n, k))
    _check(load().m4q_repack(w.data_ptr(), codec, n, k, out.data_ptr(), _stream_ptr(stream)), "m4q_repack")
    return out


def attention(q, k, v, kv_codec: int, hkv: int, t: int, q_offset: int | None = None,
              causal: bool = True, scale: float | None = None, out=None, workspace=None, stream=None):
    """O fp16 [M, H * D] = attention of q fp16 [H, M, D] over the KV cache k,
    v [hkv, t, D] (fp16 for KV_F16; uint8 Q8_0 blocks [hkv, t, D / 32 * 34]
    for Q8_0).  q_offset defaults to t - M (the queries are the last M
    positions); scale to 1 / sqrt(D).  The workspace (the key split's
    partial results, or the Q8_0 caches decoded to fp16 for a prefill-sized
    call) is allocated here when not given; workspace=False runs without
    one."""
    import torch
    _require(q, torch.float16, "q")
    if q.dim() != 3:
        raise ValueError("q must be [H, M, D]")
    h, m_, d = q.shape
    row = 2 * d if kv_codec == KV_F16 else (d // 32) * 34
    for x, what in ((k, "k"), (v, "v")):
        _require(x, torch.float16 if kv_codec == KV_F16 else torch.uint8, what)
        if x.numel() * x.element_size() != hkv * t * row:
            raise ValueError("%s must hold [%d, %d] rows of %d bytes" % (what, hkv, t, row))
    if q_offset is None:
        q_offset = t - m_
    if scale is None:
        scale = float(d) ** -0.5
    if out is None:
        out = torch.empty((m_, h * d), dtype=torch.float16, device=q.device)
    _require(out, torch.float16, "out")
    if out.numel() != m_ * h * d:
        raise ValueError("out must hold M * H * D values")
    lib = load()
    if workspace is None:
        need = int(lib.m4q_attention_workspace(kv_codec, h, hkv, m_, t, d))
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device) if need else None
    elif workspace is False:
        workspace = None
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.m4q_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), kv_codec, h, hkv, m_, t, d,
                             q_offset, int(bool(causal)), float(scale), out.data_ptr(), ws_ptr, ws_bytes,
                             _stream_ptr(stream)), "m4q_attention")
    return out


def check_finite(t, stream=None) -> bool:
    """True if every element of the fp16 tensor is finite (synchronizes)."""
    import torch
    _require(t, torch.float16, "t")
    rc = load().m4q_check_finite(t.data_ptr(), t.numel(), _stream_ptr(stream))
    if rc == ERR_NONFINITE:
        return False
    _check(rc, "m4q_check_finite")
    return True


def check_device_status(stream=None) -> int:
    """Synchronize and return (and clear) the device status: OK, ERR_BOUNDS or ERR_TIMEOUT."""
    return int(load().m4q_check_device_status(_stream_ptr(stream)))


def build_flags() -> int:
    """BUILD_BOUNDS for the bounds-checked build, else 0."""
    return int(load().m4q_build_flags())


def bounds_site(stream=None) -> int:
    """Synchronize and return (and clear) the site of the first failed bounds
    check (0: none; bounds-checked build only)."""
    rc = int(load().m4q_bounds_site(_stream_ptr(stream)))
    if rc < 0:
        _check(rc, "m4q_bounds_site")
    return rc


def selftest_wait_timeout(limit_ns: int, stream=None):
    _check(load().m4q_selftest_wait_timeout(int(limit_ns), _stream_ptr(stream)),
           "m4q_selftest_wait_timeout")


class QuantLinear:
    """A linear layer over block-quantized weights [out_features, in_features]
    (GEMV for M <= 16, tcgen05 otherwise); leading dims of x are flattened."""

    def __init__(self, weight, codec: int, out_features: int, in_features: int):
        _packed_check(weight, codec, out_features, in_features, "weight")
        self.weight, self.codec = weight, codec
        self.out_features, self.in_features = out_features, in_features

    def __call__(self, x):
        lead = x.shape[:-1]
        if x.shape[-1] != self.in_features:
            raise ValueError("last dim of x must be %d" % self.in_features)
        x2 = x.reshape(-1, self.in_features)
        y = gemm(x2, self.weight, self.codec, self.out_features, self.in_features)
        return y.reshape(*lead, self.out_features)


class QuantGLU:
    """The fused gate/up projection act(x Wg^T) * (x Wu^T) (SwiGLU or GeGLU);
    leading dims of x are flattened."""

    def __init__(self, wg, wu, codec: int, out_features: int, in_features: int, act: int = ACT_SILU):
        _packed_check(wg, codec, out_features, in_features, "wg")
        _packed_check(wu, codec, out_features, in_features, "wu")
        self.wg, self.wu, self.codec, self.act = wg, wu, codec, act
        self.out_features, self.in_features = out_features, in_features

    def __call__(self, x):
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features)
        y = glu(x2, self.wg, self.wu, self.codec, self.out_features, self.in_features, self.act)
        return y.reshape(*lead, self.out_features)


class QuantSwiGLU(QuantGLU):
    """The fused gate/up projection SiLU(x Wg^T) * (x Wu^T)."""

    def __init__(self, wg, wu, codec: int, out_features: int, in_features: int):
        super().__init__(wg, wu, codec, out_features, in_features, ACT_SILU)


class QuantMLP:
    """The gated MLP block: down(act(x Wg^T) * (x Wu^T)).  Wg, Wu: packed
    [hidden_ff, hidden]; Wd: packed [hidden, hidden_ff].  The fp16
    intermediate buffer is kept and reused across calls of the same M."""

    def __init__(self, wg, wu, wd, codec_gu: int, codec_d: int, hidden: int, hidden_ff: int,
                 act: int = ACT_SILU):
        _packed_check(wg, codec_gu, hidden_ff, hidden, "wg")
        _packed_check(wu, codec_gu, hidden_ff, hidden, "wu")
        _packed_check(wd, codec_d, hidden, hidden_ff, "wd")
        self.wg, self.wu, self.wd = wg, wu, wd
        self.codec_gu, self.codec_d, self.act = codec_gu, codec_d, act
        self.hidden, self.hidden_ff = hidden, hidden_ff
        self._h = None

    def __call__(self, x):
        import torch
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.hidden)
        m = x2.shape[0]
        if self._h is None or self._h.shape[0] != m or self._h.device != x2.device:
            self._h = torch.empty((m, self.hidden_ff), dtype=torch.float16, device=x2.device)
        y = mlp(x2, self.wg, self.wu, self.wd, self.codec_gu, self.codec_d, self.hidden, self.hidden_ff,
                act=self.act, h=self._h)
        return y.reshape(*lead, self.hidden)


class QuantQKV:
    """Fused Q/K/V projection: one GEMM on the row concatenation of Wq [hq * hd,
    hidden], Wk and Wv [hkv * hd, hidden], written head-major, returning the
    views q [hq, M, hd], k [hkv, M, hd], v [hkv, M, hd] (no transposes)."""

    def __init__(self, wq, wk, wv, codec: int, hidden: int, head_dim: int, q_heads: int, kv_heads: int):
        import torch
        _packed_check(wq, codec, q_heads * head_dim, hidden, "wq")
        _packed_check(wk, codec, kv_heads * head_dim, hidden, "wk")
        _packed_check(wv, codec, kv_heads * head_dim, hidden, "wv")
        self.w = torch.cat([wq, wk, wv]).contiguous()
        self.codec, self.hidden, self.head_dim = codec, hidden, head_dim
        self.q_heads, self.kv_heads = q_heads, kv_heads

    def __call__(self, x):
        x2 = x.reshape(-1, self.hidden)
        n = (self.q_heads + 2 * self.kv_heads) * self.head_dim
        y = gemm_heads(x2, self.w, self.codec, n, self.hidden, self.head_dim)
        hq, hk = self.q_heads, self.kv_heads
        return y[:hq], y[hq:hq + hk], y[hq + hk:]
