"""CPU oracle for the block-quantized projection GEMM and fused SwiGLU.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never imports, links or calls it, and this package imports nothing from the
CUDA side.

The arithmetic lives in ``oracle.c`` (plain C, binary64).  This module builds
it with gcc on first use and marshals numpy arrays through ctypes.  Sources
for each function are cited in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

Q4_0, Q8_0, Q2_0, MLX4 = 0, 1, 2, 3
KV_F16 = 16   # fp16 KV cache values (the other KV cache codec is Q8_0)
CODEC_NAMES = {Q4_0: "Q4_0", Q8_0: "Q8_0", Q2_0: "Q2_0", MLX4: "MLX4"}


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (plain gcc, no fast-math,
    no floating-point contraction so x86 and Arm hosts round alike)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p
    lib.oracle_block_size.argtypes = [i32]
    lib.oracle_block_size.restype = i64
    lib.oracle_block_bytes.argtypes = [i32]
    lib.oracle_block_bytes.restype = i64
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_double_to_half.argtypes = [ctypes.c_double]
    lib.oracle_double_to_half.restype = ctypes.c_uint16
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_dequant.argtypes = [vp, i32, i64, i64, vp]
    lib.oracle_dequant.restype = i32
    lib.oracle_dequant_f16.argtypes = [vp, i32, i64, i64, vp]
    lib.oracle_dequant_f16.restype = i32
    lib.oracle_gemm.argtypes = [vp, vp, i32, i64, i64, i64, vp, i64, vp, i32]
    lib.oracle_gemm.restype = i32
    lib.oracle_swiglu.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, i64, vp, i32]
    lib.oracle_swiglu.restype = i32
    lib.oracle_geglu.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, i64, vp, i32]
    lib.oracle_geglu.restype = i32
    lib.oracle_gelu.argtypes = [ctypes.c_double]
    lib.oracle_gelu.restype = ctypes.c_double
    lib.oracle_mlx4_pack.argtypes = [vp, vp, vp, i64, i64, vp]
    lib.oracle_mlx4_pack.restype = i32
    lib.oracle_repack.argtypes = [vp, i32, i64, i64, vp]
    lib.oracle_repack.restype = i32
    lib.oracle_attention.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i64, i64, i32,
                                     ctypes.c_double, vp, i64, vp, i32]
    lib.oracle_attention.restype = i32
    return lib


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile another copy of the oracle source (used by the tests that
    plant a mistake in the oracle and check that the pins catch it)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-D_DEFAULT_SOURCE", "-ffp-contract=off",
                    "-fPIC", "-shared", "-pthread", src, "-o", out_path, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


_override = threading.local()


class use_library:
    """Context manager: route this module's functions to another compiled
    oracle (a planted-mistake variant) for the current thread."""

    def __init__(self, path: str):
        self.lib = _bind(path)

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.lib
        return self

    def __exit__(self, *exc):
        _override.lib = self.prev
        return False


def _L():
    lib = getattr(_override, "lib", None)
    return lib if lib is not None else _load()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def block_size(codec: int) -> int:
    return int(_L().oracle_block_size(codec))


def block_bytes(codec: int) -> int:
    return int(_L().oracle_block_bytes(codec))


def half_to_double(bits) -> np.ndarray:
    lib = _L()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_half_to_double(int(v)) for v in b], dtype=np.float64)


def double_to_half(vals) -> np.ndarray:
    lib = _L()
    v = np.asarray(vals, dtype=np.float64).ravel()
    return np.array([lib.oracle_double_to_half(float(x)) for x in v], dtype=np.uint16)


def silu(g: float) -> float:
    return float(_L().oracle_silu(float(g)))


def gelu(g: float) -> float:
    return float(_L().oracle_gelu(float(g)))


def _as_packed(W: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(W, dtype=np.uint8))


def _as_xbits(X: np.ndarray) -> np.ndarray:
    X = np.asarray(X)
    if X.dtype == np.float16:
        X = X.view(np.uint16)
    return np.ascontiguousarray(X, dtype=np.uint16)


def dequant(W: np.ndarray, codec: int, N: int, K: int) -> np.ndarray:
    """Exact binary64 weights [N, K]."""
    Wp = _as_packed(W)
    out = np.empty((N, K), dtype=np.float64)
    _check(_L().oracle_dequant(_ptr(Wp), codec, N, K, _ptr(out)), "dequant")
    return out


def dequant_f16(W: np.ndarray, codec: int, N: int, K: int) -> np.ndarray:
    """fp16 bits [N, K] of each weight rounded once, to nearest even."""
    Wp = _as_packed(W)
    out = np.empty((N, K), dtype=np.uint16)
    _check(_L().oracle_dequant_f16(_ptr(Wp), codec, N, K, _ptr(out)), "dequant_f16")
    return out


def mlx4_pack(words, scales, biases, N: int, K: int) -> np.ndarray:
    """MLX planar arrays (uint32 words [N, K/8], fp16 scales and biases
    [N, K/32]) -> MLX4 blocks uint8 [N, (K/32) * 20]."""
    w = np.ascontiguousarray(np.asarray(words, dtype=np.uint32))
    s = np.ascontiguousarray(np.asarray(scales, dtype=np.float16)).view(np.uint16)
    b = np.ascontiguousarray(np.asarray(biases, dtype=np.float16)).view(np.uint16)
    out = np.zeros((N, (K // 32) * 20), dtype=np.uint8)
    _check(_L().oracle_mlx4_pack(_ptr(w), _ptr(s), _ptr(b), N, K, _ptr(out)), "mlx4_pack")
    return out


def repack(W: np.ndarray, codec: int, N: int, K: int) -> np.ndarray:
    """Blocks -> planes, uint8 [weight bytes]: the code bytes of every block
    in order, then the fp16 scales [N, K/B], then (MLX4) the fp16 biases."""
    Wp = _as_packed(W)
    out = np.zeros(Wp.size, dtype=np.uint8)
    _check(_L().oracle_repack(_ptr(Wp), codec, N, K, _ptr(out)), "repack")
    return out


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, int(r.size)


def gemm(X, W, codec: int, M: int, N: int, K: int, rows=None, nthreads: int | None = None):
    """binary64 Y[len(rows) or M, N] = X[rows] . W^T."""
    Xb, Wp = _as_xbits(X), _as_packed(W)
    r, nrows = _rows_arg(rows, M)
    out = np.empty((nrows, N), dtype=np.float64)
    rc = _L().oracle_gemm(_ptr(Xb), _ptr(Wp), codec, M, N, K,
                             None if r is None else _ptr(r), nrows, _ptr(out),
                             nthreads or default_threads())
    _check(rc, "gemm")
    return out


def swiglu(X, Wg, Wu, codec: int, M: int, N: int, K: int, rows=None,
           nthreads: int | None = None):
    """binary64 Y = SiLU(X Wg^T) * (X Wu^T) for the selected rows."""
    Xb, Gp, Up = _as_xbits(X), _as_packed(Wg), _as_packed(Wu)
    r, nrows = _rows_arg(rows, M)
    out = np.empty((nrows, N), dtype=np.float64)
    rc = _L().oracle_swiglu(_ptr(Xb), _ptr(Gp), _ptr(Up), codec, M, N, K,
                               None if r is None else _ptr(r), nrows, _ptr(out),
                               nthreads or default_threads())
    _check(rc, "swiglu")
    return out


def geglu(X, Wg, Wu, codec: int, M: int, N: int, K: int, rows=None,
          nthreads: int | None = None):
    """binary64 Y = GELU(X Wg^T) * (X Wu^T) for the selected rows."""
    Xb, Gp, Up = _as_xbits(X), _as_packed(Wg), _as_packed(Wu)
    r, nrows = _rows_arg(rows, M)
    out = np.empty((nrows, N), dtype=np.float64)
    rc = _L().oracle_geglu(_ptr(Xb), _ptr(Gp), _ptr(Up), codec, M, N, K,
                              None if r is None else _ptr(r), nrows, _ptr(out),
                              nthreads or default_threads())
    _check(rc, "geglu")
    return out


def attention(Q, K, V, kv_codec: int, H: int, Hkv: int, M: int, T: int, D: int,
              q_offset: int = 0, causal: bool = True, scale: float | None = None, rows=None,
              nthreads: int | None = None):
    """binary64 O [len(rows) or M, H * D]: softmax attention of fp16 Q
    [H, M, D] over the KV cache K, V [Hkv, T, D] (fp16 values for KV_F16, or
    Q8_0 blocks along D as uint8 [Hkv, T, D / 32 * 34])."""
    Qb = _as_xbits(Q)
    if kv_codec == KV_F16:
        Kb = np.ascontiguousarray(np.asarray(K, dtype=np.float16)).view(np.uint8)
        Vb = np.ascontiguousarray(np.asarray(V, dtype=np.float16)).view(np.uint8)
    else:
        Kb, Vb = _as_packed(K), _as_packed(V)
    r, nrows = _rows_arg(rows, M)
    out = np.empty((nrows, H * D), dtype=np.float64)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    rc = _L().oracle_attention(_ptr(Qb), _ptr(Kb), _ptr(Vb), kv_codec, H, Hkv, M, T, D, q_offset,
                               int(bool(causal)), sc, None if r is None else _ptr(r), nrows, _ptr(out),
                               nthreads or default_threads())
    _check(rc, "attention")
    return out
