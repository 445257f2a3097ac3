"""Cross-file consistency that needs no GPU: the C header and the Python
binding agree on every enum value, and the ncu summaries that bench.py
quotes were taken on the kernel sources as they are now."""
import os
import re

import bench
import synth
import oracle
import swiglu_block_quantized_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_enums():
    text = open(os.path.join(ROOT, "include", "m4q.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    vals = {}
    for body in re.findall(r"enum\s+\w+\s*\{(.*?)\}", text, flags=re.S):
        for name, v in re.findall(r"(M4Q_\w+)\s*=\s*(-?\d+)", body):
            vals[name] = int(v)
    return vals


def test_header_enums_match_the_binding():
    e = header_enums()
    pairs = {
        "M4Q_Q4_0": m.Q4_0, "M4Q_Q8_0": m.Q8_0, "M4Q_Q2_0": m.Q2_0, "M4Q_MLX4": m.MLX4,
        "M4Q_KV_F16": m.KV_F16,
        "M4Q_PATH_AUTO": m.PATH_AUTO, "M4Q_PATH_GEMV": m.PATH_GEMV, "M4Q_PATH_TC": m.PATH_TC,
        "M4Q_ACT_SILU": m.ACT_SILU, "M4Q_ACT_GELU": m.ACT_GELU,
        "M4Q_OK": m.OK, "M4Q_ERR_INVALID_ARG": m.ERR_INVALID_ARG,
        "M4Q_ERR_UNSUPPORTED_CODEC": m.ERR_UNSUPPORTED_CODEC, "M4Q_ERR_BAD_SHAPE": m.ERR_BAD_SHAPE,
        "M4Q_ERR_MISALIGNED": m.ERR_MISALIGNED, "M4Q_ERR_CUDA": m.ERR_CUDA,
        "M4Q_ERR_NONFINITE": m.ERR_NONFINITE, "M4Q_ERR_TIMEOUT": m.ERR_TIMEOUT,
        "M4Q_ERR_UNSUPPORTED_DEVICE": m.ERR_UNSUPPORTED_DEVICE, "M4Q_ERR_SCRATCH_LIMIT": m.ERR_SCRATCH_LIMIT,
        "M4Q_ERR_BOUNDS": m.ERR_BOUNDS,
    }
    assert set(pairs) == set(e), sorted(set(pairs) ^ set(e))
    for name, v in pairs.items():
        assert e[name] == v, name


def test_codec_tables_agree():
    # the binding, the generators and the oracle describe the same blocks
    for c in m.CODECS:
        assert m.BLOCK[c] == synth.BLOCK[c] == oracle.block_size(c)
        assert m.BLOCK_BYTES[c] == synth.BLOCK_BYTES[c] == oracle.block_bytes(c)
    assert m.KV_F16 == synth.KV_F16 == oracle.KV_F16


def test_bench_ncu_summaries():
    # bench.py reports DRAM traffic from committed summaries, and only when
    # they were taken on the current kernel sources (else null); a stale
    # summary is reported as a skip, not a failure.
    import json
    import pytest
    stale = []
    for name, srcs in (("tc_swiglu_q4_0_8b_m2048", bench.KERNEL_SOURCES),
                       ("gemv_swiglu_q4_0_8b_m1", bench.GEMV_SOURCES)):
        with open(os.path.join(ROOT, "profiles", name + ".json")) as f:
            d = json.load(f)
        assert {"kernel", "command", "source_hash", "dram_bytes_per_launch"} <= set(d)
        assert d["dram_bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(ROOT, "profiles", name + ".md"))
        if bench.recorded_traffic(name, srcs) is None:
            stale.append(name)
    if stale:
        pytest.skip("ncu summaries older than the kernel sources: %s" % ", ".join(stale))
