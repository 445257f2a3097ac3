"""Seeded synthetic inputs for the quantized projection workloads.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds no arithmetic of the method (no decoding, no products, no activation):
it only draws random numbers and writes them into the block byte layouts.

Random numbers: a counter-based SplitMix64 stream (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014; constants as
published with the reference generator).  Value i of a stream with key s is
``mix(s + (i + 1) * GAMMA)``.  Uniforms in [0, 1) take the top 53 bits;
normals come from Box-Muller on consecutive uniform pairs (the cosine branch
only).  Every stream key is derived from (seed, stream name) so each tensor
of a workload has an independent stream.

Block layouts written here (little-endian fp16 scale d first):
  Q4_0  18 B: byte 2+j holds code j (low nibble) and code j+16 (high nibble)
  Q8_0  34 B: byte 2+i holds code i as a signed byte
  Q2_0  34 B: byte 2+i//4 holds code i at bits 2*(i%4)..2*(i%4)+1
  MLX4  20 B: scale s, then bias b (fp16), then byte 4+i//2 holds code i,
        even i in the low nibble (MLX's packing order: code k of a row sits
        at bits 4*(k%8) of little-endian 32-bit word k//8)
MLX's own planar arrays (``planar``): codes as uint32 words [N, K/8] with
code k at bits 4*(k%8) of word k//8, scales and biases fp16 [N, K/32].

Value recipes of the pages' LLaMA-shaped workloads (synthetic weights, as the
m4-prefill-engine v0.2 notes describe): X ~ N(0,1) rounded to fp16;
Q4_0 d = |N(0,1)|*0.02, q uniform on 0..15; Q8_0 d = |N(0,1)|*0.01,
q = clip(round(40*N(0,1)), -127, 127) with halves rounded away from zero;
Q2_0 d = |N(0,1)|*0.02, q in {0,1,2} with probabilities 0.3/0.4/0.3, then each
code independently replaced by the reserved code 3 with probability 0.01;
MLX4 s = |N(0,1)|*0.02, q uniform on 0..15, b = -s*(7.5 + 0.5*N(0,1)) (the
shape of an affine min/max fit of a zero-mean group: b near the group minimum
-7.5 s).  Scales and biases are drawn in binary64 and rounded to fp16 (round to
nearest even).
"""
from __future__ import annotations

import zlib

import numpy as np

Q4_0, Q8_0, Q2_0, MLX4 = 0, 1, 2, 3
CODECS = (Q4_0, Q8_0, Q2_0, MLX4)
CODEC_NAMES = {Q4_0: "Q4_0", Q8_0: "Q8_0", Q2_0: "Q2_0", MLX4: "MLX4"}
BLOCK = {Q4_0: 32, Q8_0: 32, Q2_0: 128, MLX4: 32}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q2_0: 34, MLX4: 20}

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, name: str) -> int:
    """Key of the named stream for a seed (stable across hosts)."""
    tag = zlib.crc32(name.encode("utf-8")) & 0xFFFFFFFF
    z = np.array([(int(seed) * 0x100000001 + tag) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return int(_mix(z)[0])


def u64(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    """Values offset .. offset+n-1 of the stream, as uint64."""
    key = np.uint64(stream_key(seed, name))
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * _GAMMA)


def uniform(seed: int, name: str, n: int) -> np.ndarray:
    """n uniforms in [0, 1) (53-bit)."""
    return (u64(seed, name, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, name: str, n: int) -> np.ndarray:
    """n standard normals, Box-Muller on uniform pairs (u1, u2)."""
    u = uniform(seed, name, 2 * n).reshape(n, 2)
    r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
    return r * np.cos(2.0 * np.pi * u[:, 1])


def to_f16(v: np.ndarray) -> np.ndarray:
    """binary64 -> fp16, round to nearest even (numpy's conversion)."""
    return np.asarray(v, dtype=np.float64).astype(np.float16)


# ---------------------------------------------------------------- tensors

def activations(M: int, K: int, seed: int, name: str = "X") -> np.ndarray:
    """X fp16 [M, K] ~ N(0, 1)."""
    return to_f16(normal(seed, name, M * K)).reshape(M, K)


def codes(codec: int, N: int, K: int, seed: int, name: str) -> np.ndarray:
    """Integer codes [N, K] drawn by the codec's recipe (int16)."""
    n = N * K
    if codec in (Q4_0, MLX4):
        words = u64(seed, name + ".q", (n + 15) // 16)
        nib = np.empty((words.size, 16), dtype=np.uint8)
        for j in range(16):
            nib[:, j] = ((words >> np.uint64(4 * j)) & np.uint64(0xF)).astype(np.uint8)
        return nib.ravel()[:n].astype(np.int16).reshape(N, K)
    if codec == Q8_0:
        z = normal(seed, name + ".q", n) * 40.0
        r = np.sign(z) * np.floor(np.abs(z) + 0.5)      # halves away from zero
        return np.clip(r, -127, 127).astype(np.int16).reshape(N, K)
    if codec == Q2_0:
        u = uniform(seed, name + ".q", n)
        q = np.where(u < 0.3, 0, np.where(u < 0.7, 1, 2)).astype(np.int16)
        v = uniform(seed, name + ".q3", n)
        q[v < 0.01] = 3
        return q.reshape(N, K)
    raise ValueError("unknown codec %r" % codec)


_SCALE = {Q4_0: 0.02, Q8_0: 0.01, Q2_0: 0.02, MLX4: 0.02}


def scales(codec: int, N: int, K: int, seed: int, name: str, scale: float | None = None):
    """Block scales d fp16 [N, K / block] = |N(0,1)| * scale."""
    nb = K // BLOCK[codec]
    c = _SCALE[codec] if scale is None else scale
    return to_f16(np.abs(normal(seed, name + ".d", N * nb)) * c).reshape(N, nb)


def biases(codec: int, N: int, K: int, seed: int, name: str, d) -> np.ndarray | None:
    """Block biases fp16 [N, K / block] for the affine codec (MLX4):
    b = -s * (7.5 + 0.5 * N(0,1)) with s the block's scale.  None for the
    scale-only codecs."""
    if codec != MLX4:
        return None
    nb = K // BLOCK[codec]
    s = np.asarray(d, dtype=np.float16).astype(np.float64).reshape(N, nb)
    z = normal(seed, name + ".b", N * nb).reshape(N, nb)
    return to_f16(-s * (7.5 + 0.5 * z))


def _f16_bytes(v, N: int, nb: int) -> np.ndarray:
    """fp16 values [N, nb] as their little-endian bytes [N, nb, 2]."""
    b = np.ascontiguousarray(np.asarray(v, dtype=np.float16).reshape(N, nb)).view("<u2")
    return b.view(np.uint8).reshape(N, nb, 2)


def pack(codec: int, q: np.ndarray, d: np.ndarray, b=None) -> np.ndarray:
    """Write codes q [N, K] and fp16 scales d [N, K/block] (and, for MLX4,
    fp16 biases b [N, K/block], zero when omitted) into packed blocks,
    returned as uint8 [N, (K/block) * block_bytes]."""
    q = np.asarray(q)
    N, K = q.shape
    B = BLOCK[codec]
    if K % B:
        raise ValueError("K must be a multiple of the block size")
    nb = K // B
    head = [_f16_bytes(d, N, nb)]
    qb = q.reshape(N, nb, B)
    if codec == Q4_0:
        if qb.min(initial=0) < 0 or qb.max(initial=0) > 15:
            raise ValueError("Q4_0 codes are 0..15")
        u = qb.astype(np.uint8)
        body = (u[:, :, :16] | (u[:, :, 16:] << 4)).astype(np.uint8)
    elif codec == Q8_0:
        if qb.min(initial=0) < -128 or qb.max(initial=0) > 127:
            raise ValueError("Q8_0 codes are -128..127")
        body = qb.astype(np.int8).view(np.uint8)
    elif codec == Q2_0:
        if qb.min(initial=0) < 0 or qb.max(initial=0) > 3:
            raise ValueError("Q2_0 codes are 0..3")
        u = qb.astype(np.uint8).reshape(N, nb, 32, 4)
        body = (u[..., 0] | (u[..., 1] << 2) | (u[..., 2] << 4) | (u[..., 3] << 6)).astype(np.uint8)
    elif codec == MLX4:
        if qb.min(initial=0) < 0 or qb.max(initial=0) > 15:
            raise ValueError("MLX4 codes are 0..15")
        u = qb.astype(np.uint8)
        body = (u[:, :, 0::2] | (u[:, :, 1::2] << 4)).astype(np.uint8)
        head.append(_f16_bytes(np.zeros((N, nb)) if b is None else b, N, nb))
    else:
        raise ValueError("unknown codec %r" % codec)
    out = np.concatenate(head + [body], axis=2)
    return np.ascontiguousarray(out.reshape(N, nb * BLOCK_BYTES[codec]))


def planar(q: np.ndarray, d: np.ndarray, b: np.ndarray):
    """MLX's own planar arrays for 4-bit codes q [N, K] (K % 32 == 0) with
    group scales d and biases b [N, K/32]: (words uint32 [N, K/8] with code k
    at bits 4*(k%8) of word k//8, scales fp16, biases fp16)."""
    q = np.asarray(q)
    N, K = q.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    if q.min(initial=0) < 0 or q.max(initial=0) > 15:
        raise ValueError("codes are 0..15")
    u = q.astype(np.uint32).reshape(N, K // 8, 8)
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for e in range(8):
        words |= u[:, :, e] << np.uint32(4 * e)
    nb = K // 32
    return (words, np.ascontiguousarray(np.asarray(d, np.float16).reshape(N, nb)),
            np.ascontiguousarray(np.asarray(b, np.float16).reshape(N, nb)))


def weights(codec: int, N: int, K: int, seed: int, name: str = "W", scale: float | None = None):
    """Packed weights uint8 [N, row_bytes] by the codec's recipe."""
    d = scales(codec, N, K, seed, name, scale)
    return pack(codec, codes(codec, N, K, seed, name), d, biases(codec, N, K, seed, name, d))


def row_bytes(codec: int, K: int) -> int:
    return (K // BLOCK[codec]) * BLOCK_BYTES[codec]


def constant_weights(codec: int, N: int, K: int, code: int, d_f16, b_f16=0.0) -> np.ndarray:
    """Every code equal to ``code``, every scale equal to ``d_f16`` (and,
    for MLX4, every bias equal to ``b_f16``)."""
    q = np.full((N, K), code, dtype=np.int16)
    d = np.full((N, K // BLOCK[codec]), d_f16, dtype=np.float16)
    b = np.full((N, K // BLOCK[codec]), b_f16, dtype=np.float16)
    return pack(codec, q, d, b if codec == MLX4 else None)


# ---------------------------------------------------------------- KV cache

KV_F16 = 16   # fp16 KV cache values; the quantized KV cache uses Q8_0


def kv_cache(codec: int, Hkv: int, T: int, D: int, seed: int, name: str) -> np.ndarray:
    """One KV cache tensor [Hkv, T, D] by token rows: fp16 values ~ N(0,1)
    (KV_F16), or Q8_0 blocks along D by the Q8_0 recipe, uint8 [Hkv, T,
    D / 32 * 34]."""
    if codec == KV_F16:
        return activations(Hkv * T, D, seed, name).reshape(Hkv, T, D)
    if codec == Q8_0:
        return weights(Q8_0, Hkv * T, D, seed, name).reshape(Hkv, T, row_bytes(Q8_0, D))
    raise ValueError("KV cache codec must be KV_F16 or Q8_0")


def queries(H: int, M: int, D: int, seed: int, name: str = "Q") -> np.ndarray:
    """Q fp16 [H, M, D] ~ N(0,1) (head-major, as the direct-head projection
    writes it)."""
    return activations(H * M, D, seed, name).reshape(H, M, D)


# ---------------------------------------------------------------- workloads
# Shapes of the pages' LLaMA-shaped layers (1B tier: hidden 2048, MLP 8192;
# 8B tier: hidden 4096, MLP 14336).  Each entry: (kind, codec, M, N, K).

WORKLOADS = {
    "tiny_q4_0": [("gemm", Q4_0, 64, 256, 256)],
    "1b_proj_q4_0": [("gemm", Q4_0, 2048, 8192, 2048)],
    "1b_proj_q8_0": [("gemm", Q8_0, 2048, 8192, 2048)],
    "8b_swiglu_m2048": [("swiglu", Q4_0, 2048, 14336, 4096)],
    "q2_0_sweep": [("gemm", Q2_0, m, 4096, 4096) for m in (1, 16, 512, 2048)],
}


def llama1b_layer(M: int):
    """The 1B layer's projection set at M tokens: q/k/v/o Q8_0, fused
    gate/up SwiGLU Q4_0 and down Q4_0 (hidden 2048, 8 kv heads of 64)."""
    return [
        ("q", "gemm", Q8_0, M, 2048, 2048),
        ("k", "gemm", Q8_0, M, 512, 2048),
        ("v", "gemm", Q8_0, M, 512, 2048),
        ("o", "gemm", Q8_0, M, 2048, 2048),
        ("gate_up", "swiglu", Q4_0, M, 8192, 2048),
        ("down", "gemm", Q4_0, M, 2048, 8192),
    ]
