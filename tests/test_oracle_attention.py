"""Pins of the oracle's attention over a KV cache ("v0.1 vs v0.2
comparison" 2.3: FlashAttention with a Q8_0 KV cache; "Releases" v0.3.0:
grouped-query attention, causal masking with sequence offsets).

Each check compares the oracle with something it cannot agree with by
construction: softmax in 50-digit decimal arithmetic on tiny inputs, closed
forms (equal scores average V; one visible key returns it; a dominant score
selects its row), grouped-query attention written as multi-head attention
over repeated KV heads, and causal invariances.  A planted-mistake group
checks that each plausible slip fails at least one of them.
"""
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
import synth

F16, Q8 = synth.KV_F16, synth.Q8_0


def kv_values(K, codec, D):
    """fp16 operand values of a KV cache tensor, decoded with numpy from the
    Q8_0 layout (d then 32 signed bytes per block), independent of the oracle."""
    if codec == F16:
        return np.asarray(K, np.float16).astype(np.float64)
    Hkv, T, rb = K.shape
    blocks = K.reshape(Hkv, T, D // 32, 34)
    d = blocks[..., 0:2].copy().view("<f2")[..., 0].astype(np.float64)
    q = blocks[..., 2:].view(np.int8).astype(np.float64)
    return (q * d[..., None]).astype(np.float16).astype(np.float64).reshape(Hkv, T, D)


def decimal_attention(Q, Kv, Vv, H, Hkv, M, T, D, q_offset, causal, scale):
    getcontext().prec = 50
    G = H // Hkv
    O = np.zeros((M, H * D))
    for h in range(H):
        hk = h // G
        for i in range(M):
            vis = T if not causal else min(T, q_offset + i + 1)
            if vis <= 0:
                continue
            qv = [Decimal(float(x)) for x in Q[h, i].astype(np.float64)]
            s = [Decimal(scale) * sum(qv[d] * Decimal(float(Kv[hk, j, d])) for d in range(D)) for j in range(vis)]
            mx = max(s)
            e = [(x - mx).exp() for x in s]
            tot = sum(e)
            for d in range(D):
                O[i, h * D + d] = float(sum(e[j] * Decimal(float(Vv[hk, j, d])) for j in range(vis)) / tot)
    return O


def check_decimal_brute_force():
    for codec in (F16, Q8):
        H, Hkv, M, T, D = 4, 2, 3, 7, 32
        Q = synth.queries(H, M, D, seed=1)
        K = synth.kv_cache(codec, Hkv, T, D, seed=2, name="K")
        V = synth.kv_cache(codec, Hkv, T, D, seed=2, name="V")
        for causal, off in ((True, T - M), (True, 1), (False, 0)):
            scale = D ** -0.5
            got = oracle.attention(Q, K, V, codec, H, Hkv, M, T, D, off, causal, scale)
            ref = decimal_attention(Q, kv_values(K, codec, D), kv_values(V, codec, D), H, Hkv, M, T, D,
                                    off, causal, scale)
            assert np.allclose(got, ref, rtol=1e-13, atol=1e-15), (codec, causal, off)


def test_decimal_brute_force():
    check_decimal_brute_force()


def check_closed_forms():
    H, Hkv, M, T, D = 2, 2, 6, 10, 64
    Q = synth.queries(H, M, D, seed=3)
    V = synth.kv_cache(F16, Hkv, T, D, seed=3, name="V")
    Vd = V.astype(np.float64)
    # zero keys: every visible score is 0, so O is the mean of the visible V rows
    K0 = np.zeros((Hkv, T, D), np.float16)
    off = T - M
    O = oracle.attention(Q, K0, V, F16, H, Hkv, M, T, D, off, True).reshape(M, H, D)
    for i in range(M):
        for h in range(H):
            assert np.allclose(O[i, h], Vd[h, : off + i + 1].mean(axis=0), rtol=1e-14, atol=1e-15)
    # offset 0: query 0 sees only key 0, so its output is V[0] exactly
    K = synth.kv_cache(F16, Hkv, T, D, seed=4, name="K")
    O = oracle.attention(Q, K, V, F16, H, Hkv, M, T, D, 0, True).reshape(M, H, D)
    for h in range(H):
        assert np.array_equal(O[0, h], Vd[h, 0])
    # a dominant score (s = 2048 against 0) selects its V row; e^2048 overflows
    # binary64, so this also requires the max to be subtracted first
    Kb = np.zeros((Hkv, T, D), np.float16)
    Kb[:, 3, :] = 1.0
    Qb = np.full((H, M, D), 8.0, np.float16)
    O = oracle.attention(Qb, Kb, V, F16, H, Hkv, M, T, D, 0, False, 4.0).reshape(M, H, D)
    assert np.all(np.isfinite(O))
    for h in range(H):
        assert np.allclose(O[:, h], np.broadcast_to(Vd[h, 3], (M, D)), rtol=0, atol=1e-200)


def test_closed_forms():
    check_closed_forms()


def check_gqa_is_repeated_mha():
    H, Hkv, M, T, D = 8, 2, 5, 12, 32
    for codec in (F16, Q8):
        Q = synth.queries(H, M, D, seed=5)
        K = synth.kv_cache(codec, Hkv, T, D, seed=6, name="K")
        V = synth.kv_cache(codec, Hkv, T, D, seed=6, name="V")
        gqa = oracle.attention(Q, K, V, codec, H, Hkv, M, T, D, T - M, True)
        Kr, Vr = np.repeat(K, H // Hkv, axis=0), np.repeat(V, H // Hkv, axis=0)   # head h reads kv head h // 4
        mha = oracle.attention(Q, Kr, Vr, codec, H, H, M, T, D, T - M, True)
        assert np.array_equal(gqa, mha)


def test_gqa_is_repeated_mha():
    check_gqa_is_repeated_mha()


def check_causal_invariances():
    H, Hkv, M, T, D = 2, 1, 6, 9, 64
    Q = synth.queries(H, M, D, seed=7)
    K = synth.kv_cache(Q8, Hkv, T, D, seed=8, name="K")
    V = synth.kv_cache(Q8, Hkv, T, D, seed=8, name="V")
    off = T - M
    base = oracle.attention(Q, K, V, Q8, H, Hkv, M, T, D, off, True)
    # keys and values after a query's position do not change its output
    K2, V2 = K.copy(), V.copy()
    K2[:, off + 2:], V2[:, off + 2:] = K[:, :T - off - 2][:, ::-1], V[:, :T - off - 2][:, ::-1]
    moved = oracle.attention(Q, K2, V2, Q8, H, Hkv, M, T, D, off, True)
    assert np.array_equal(moved[:2], base[:2])
    assert not np.array_equal(moved[2:], base[2:])
    # every key visible: causal with a large offset equals non-causal
    assert np.array_equal(oracle.attention(Q, K, V, Q8, H, Hkv, M, T, D, T, True),
                          oracle.attention(Q, K, V, Q8, H, Hkv, M, T, D, 0, False))
    # a row subset equals the same rows of the full result
    assert np.array_equal(oracle.attention(Q, K, V, Q8, H, Hkv, M, T, D, off, True, rows=[5, 0, 3]),
                          base[[5, 0, 3]])


def test_causal_invariances():
    check_causal_invariances()


def check_q8_is_f16_of_decoded():
    H, Hkv, M, T, D = 4, 4, 3, 8, 128
    Q = synth.queries(H, M, D, seed=9)
    K = synth.kv_cache(Q8, Hkv, T, D, seed=10, name="K")
    V = synth.kv_cache(Q8, Hkv, T, D, seed=10, name="V")
    Kf = oracle.dequant_f16(K.reshape(Hkv * T, -1), Q8, Hkv * T, D).view(np.float16).reshape(Hkv, T, D)
    Vf = oracle.dequant_f16(V.reshape(Hkv * T, -1), Q8, Hkv * T, D).view(np.float16).reshape(Hkv, T, D)
    assert np.array_equal(oracle.attention(Q, K, V, Q8, H, Hkv, M, T, D, T - M, True),
                          oracle.attention(Q, Kf, Vf, F16, H, Hkv, M, T, D, T - M, True))


def test_q8_is_f16_of_decoded():
    check_q8_is_f16_of_decoded()


def test_argument_errors():
    Q = np.zeros((2, 1, 32), np.float16)
    K = np.zeros((1, 4, 32), np.float16)
    with pytest.raises(ValueError):
        oracle.attention(Q, K, K, F16, 2, 3, 1, 4, 32)        # H % Hkv
    with pytest.raises(ValueError):
        oracle.attention(Q, K, K, 5, 2, 1, 1, 4, 32)          # codec


MUTATIONS = {
    "scale_ignored": ("s[t] = j->scale * dot(q, Kd + t * D, D);", "s[t] = dot(q, Kd + t * D, D);"),
    "causal_strict": ("if (j->causal && j->q_offset + i + 1 < nvis) nvis = j->q_offset + i + 1;",
                      "if (j->causal && j->q_offset + i < nvis) nvis = j->q_offset + i;"),
    "offset_ignored": ("if (j->causal && j->q_offset + i + 1 < nvis) nvis = j->q_offset + i + 1;",
                       "if (j->causal && i + 1 < nvis) nvis = i + 1;"),
    "gqa_modulo": ("const long long hk = h / G;", "const long long hk = h % j->Hkv;"),
    "v_is_k": ("acc += s[t] * Vd[t * D + d];", "acc += s[t] * Kd[t * D + d];"),
    "no_max_shift": ("s[t] = exp(s[t] - mx);", "s[t] = exp(s[t]);"),
    "kv_unrounded": ("  dequant_row(base, ORACLE_Q8_0, D, out);\n  round_row_to_f16(out, D);",
                     "  dequant_row(base, ORACLE_Q8_0, D, out);"),
    "q_row_of_head0": ("q[d] = oracle_half_to_double(j->Q[(h * j->M + i) * D + d]);",
                       "q[d] = oracle_half_to_double(j->Q[(hk * j->M + i) * D + d]);"),
}


def all_pins_pass():
    for check in (check_decimal_brute_force, check_closed_forms, check_gqa_is_repeated_mha,
                  check_causal_invariances, check_q8_is_f16_of_decoded):
        try:
            with np.errstate(all="ignore"):
                check()
        except AssertionError:
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, name
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / ("attn_%s.so" % name)))
    with oracle.use_library(path):
        assert not all_pins_pass(), "mutation %s survived every pin" % name
