"""GPU parity of m4q_attention (fp16 or Q8_0 KV cache) against the oracle.

Tolerance as for the projections: per element |gpu - ref| <= 1e-2 *
max(1, |ref|), ref the binary64 oracle.  The GPU computes scores and the
softmax in fp32 and rounds the probabilities to fp16 for the P V product.
"""
import numpy as np
import pytest

import oracle
import synth
import swiglu_block_quantized_gb300 as m
from _helpers import assert_close, dev, host, sample_rows

pytestmark = pytest.mark.gpu

F16, Q8 = synth.KV_F16, synth.Q8_0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load()
    yield
    assert m.check_device_status() == m.OK


def run(codec, H, Hkv, M, T, D, q_offset, causal, seed=0, workspace="auto", rows=None):
    Q = synth.queries(H, M, D, seed=seed)
    K = synth.kv_cache(codec, Hkv, T, D, seed=seed + 1, name="K")
    V = synth.kv_cache(codec, Hkv, T, D, seed=seed + 1, name="V")
    kw = {} if workspace == "auto" else {"workspace": workspace}
    O = host(m.attention(dev(Q), dev(K), dev(V), codec, Hkv, T, q_offset=q_offset, causal=causal, **kw))
    ref = oracle.attention(Q, K, V, codec, H, Hkv, M, T, D, q_offset, causal, rows=rows)
    return (O if rows is None else O[rows]), ref


@pytest.mark.parametrize("codec", [F16, Q8])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 2)])
@pytest.mark.parametrize("M,T", [(1, 1), (1, 200), (5, 63), (64, 64), (130, 1000), (77, 77)])
def test_attention_parity(codec, D, H, Hkv, M, T):
    for causal in (True, False):
        O, ref = run(codec, H, Hkv, M, T, D, T - M, causal, seed=M + T)
        assert_close(O, ref, "attn codec=%d D=%d H=%d/%d M=%d T=%d causal=%d" % (codec, D, H, Hkv, M, T, causal))


@pytest.mark.parametrize("codec", [F16, Q8])
def test_attention_offsets(codec):
    # queries past the end of the cache (q_offset + i >= T see every key) and
    # a zero offset (query i sees keys 0..i)
    for M, T, off in ((9, 4, 0), (40, 100, 0), (3, 50, 10)):
        O, ref = run(codec, 4, 2, M, T, 64, off, True, seed=M)
        assert_close(O, ref, "offset M=%d T=%d off=%d" % (M, T, off))


@pytest.mark.parametrize("codec", [F16, Q8])
def test_key_split_matches_single_pass(codec):
    # M = 1 over a long cache: the key range is split across CTAs and merged;
    # without a workspace one CTA per row tile walks every key.
    import torch
    H, Hkv, M, T, D = 8, 2, 1, 4096, 128
    assert m.load().m4q_attention_workspace_bytes(H, Hkv, M, T, D) > 0
    Osplit, ref = run(codec, H, Hkv, M, T, D, T - M, True, seed=3)
    Oone, _ = run(codec, H, Hkv, M, T, D, T - M, True, seed=3, workspace=False)
    assert_close(Osplit, ref, "split")
    assert_close(Oone, ref, "single pass")
    assert np.abs(Osplit.astype(np.float64) - Oone.astype(np.float64)).max() < 2e-3


def test_8b_prefill_sampled_rows():
    # The 8B layer's attention at the prefill size: H = 32, 8 KV heads,
    # D = 128, M = T = 2048, causal, Q8_0 cache; sampled query rows.
    H, Hkv, M, T, D = 32, 8, 2048, 2048, 128
    rows = sample_rows(M)
    O, ref = run(Q8, H, Hkv, M, T, D, 0, True, seed=7, rows=rows)
    assert_close(O, ref, "8b prefill")


@pytest.mark.parametrize("codec", [F16, Q8])
def test_decode_long_context(codec):
    # one new token over a 32K cache (split keys), 8B shape
    H, Hkv, M, T, D = 32, 8, 1, 32768, 128
    O, ref = run(codec, H, Hkv, M, T, D, T - 1, True, seed=11)
    assert_close(O, ref, "decode 32K")


def test_direct_head_q_feeds_attention():
    # Q projected straight into [H, M, D] by m4q_gemm_heads feeds attention
    # without a transpose; O [M, H * D] feeds the o-projection.
    K_, hd, H, Hkv, M, T = 256, 64, 4, 2, 40, 40
    W = synth.weights(synth.Q4_0, H * hd, K_, seed=50, name="Wq")
    X = synth.activations(M, K_, seed=51)
    q = m.gemm_heads(dev(X), dev(W), synth.Q4_0, H * hd, K_, hd)
    Kc = synth.kv_cache(Q8, Hkv, T, hd, seed=52, name="K")
    Vc = synth.kv_cache(Q8, Hkv, T, hd, seed=52, name="V")
    O = host(m.attention(q, dev(Kc), dev(Vc), Q8, Hkv, T))
    ref = oracle.attention(host(q), Kc, Vc, Q8, H, Hkv, M, T, hd, 0, True)
    assert_close(O, ref, "heads -> attention")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("scale", [None, -0.2])
def test_attention_growing_scores(D, scale):
    # Key rows scaled up along the sequence (x1 .. x13), so the scaled row
    # maximum grows by far more than 2^8 across the key tiles: a kernel that
    # keeps a reference maximum per row must raise it, and rescale what it
    # has accumulated, several times within a row.  A negative scale makes
    # the smallest raw scores the largest scaled ones.
    H, Hkv, M, T = 8, 2, 300, 700
    Q = synth.queries(H, M, D, seed=21)
    ramp = (1.0 + 12.0 * np.arange(T) / T).astype(np.float32)
    K = (synth.kv_cache(F16, Hkv, T, D, seed=22, name="K").astype(np.float32) * ramp[None, :, None]).astype(np.float16)
    V = synth.kv_cache(F16, Hkv, T, D, seed=22, name="V")
    for causal in (True, False):
        O = host(m.attention(dev(Q), dev(K), dev(V), F16, Hkv, T, q_offset=T - M, causal=causal, scale=scale))
        ref = oracle.attention(Q, K, V, F16, H, Hkv, M, T, D, T - M, causal, scale=scale)
        assert_close(O, ref, "growing scores D=%d scale=%s causal=%d" % (D, scale, causal))


@pytest.mark.parametrize("G", [1, 2, 8, 16])
def test_attention_group_sizes(G):
    # prefill-sized calls for each query group size the tensor-core path
    # takes (rows of G heads per KV head), with ragged M and T
    Hkv, D, M, T = 2, 128, 83, 451
    H = G * Hkv
    for causal in (True, False):
        O, ref = run(F16, H, Hkv, M, T, D, T - M, causal, seed=G)
        assert_close(O, ref, "G=%d causal=%d" % (G, causal))


@pytest.mark.parametrize("G,D", [(1, 64), (4, 128)])
def test_attention_many_row_tiles(G, D):
    # More (row tile, KV head) work items than SMs, so that a CTA walks
    # several items in turn (a persistent grid): rows spread over every row
    # tile, causal and not, and with key rows scaled up along the sequence
    # (the reference maximum raised within an item after a previous item
    # of the same CTA ended high).
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv = 16 if G == 1 else 8
    H = G * Hkv
    rows_per_tile = 128 // G
    M = ((2 * sms + 40) // Hkv + 1) * rows_per_tile - 37     # > 2 items per SM, ragged last tile
    T = M + 90
    rows = list(range(0, M, 19)) + [M - 1]
    Q = synth.queries(H, M, D, seed=41)
    Kf = synth.kv_cache(F16, Hkv, T, D, seed=42, name="K")
    V = synth.kv_cache(F16, Hkv, T, D, seed=42, name="V")
    ramp = (1.0 + 6.0 * np.arange(T) / T).astype(np.float32)
    Kr = (Kf.astype(np.float32) * ramp[None, :, None]).astype(np.float16)
    for K, tag in ((Kf, "plain"), (Kr, "growing")):
        for causal in (True, False):
            O = host(m.attention(dev(Q), dev(K), dev(V), F16, Hkv, T, q_offset=T - M, causal=causal))
            ref = oracle.attention(Q, K, V, F16, H, Hkv, M, T, D, T - M, causal, rows=rows)
            assert_close(O[rows], ref, "many tiles G=%d D=%d %s causal=%d" % (G, D, tag, causal))


@pytest.mark.parametrize("D", [64, 128])
def test_q8_prefill_staged_equals_f16_on_decoded_cache(D):
    # A prefill-sized call on a Q8_0 cache (enough row tiles that the keys
    # are not split) decodes both caches to fp16 in the workspace and runs
    # the fp16 tensor-core path: bit for bit the fp16 call on the decoded
    # cache.  Without a workspace the Q8_0 cache is decoded tile by tile in
    # the attention kernel (oracle tolerance).
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H, Hkv = 16, 4
    M = (2 * sms * 64) // (4 * Hkv) + 53
    T = M + 70
    rows = list(range(0, M, 29)) + [M - 1]
    Q = dev(synth.queries(H, M, D, seed=61))
    K8 = synth.kv_cache(Q8, Hkv, T, D, seed=62, name="K")
    V8 = synth.kv_cache(Q8, Hkv, T, D, seed=62, name="V")
    lib = m.load()
    assert lib.m4q_attention_workspace(Q8, H, Hkv, M, T, D) == 2 * Hkv * T * D * 2
    assert lib.m4q_attention_workspace(F16, H, Hkv, M, T, D) == 0
    Kf = m.dequant(dev(K8.reshape(Hkv * T, -1)), Q8, Hkv * T, D).reshape(Hkv, T, D)
    Vf = m.dequant(dev(V8.reshape(Hkv * T, -1)), Q8, Hkv * T, D).reshape(Hkv, T, D)
    ref = oracle.attention(host(Q), K8, V8, Q8, H, Hkv, M, T, D, T - M, True, rows=rows)
    O8 = host(m.attention(Q, dev(K8), dev(V8), Q8, Hkv, T))
    Of = host(m.attention(Q, Kf, Vf, F16, Hkv, T))
    On = host(m.attention(Q, dev(K8), dev(V8), Q8, Hkv, T, workspace=False))
    assert np.array_equal(O8.view(np.uint16), Of.view(np.uint16))
    assert_close(O8[rows], ref, "q8 staged D=%d" % D)
    assert_close(On[rows], ref, "q8 in-kernel decode D=%d" % D)
