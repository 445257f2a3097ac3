"""The bounds-checked build (-DM4Q_BOUNDS=1) compiles, loads without a GPU and
identifies itself; the normal build does not (no GPU needed: both calls are
host-only)."""
import swiglu_block_quantized_gb300 as m


def test_bounds_build_compiles_and_identifies_itself():
    m.build()
    path = m.build(bounds=True)
    assert path == m.LIB_BOUNDS_PATH
    assert m.load(path).m4q_build_flags() == m.BUILD_BOUNDS
    assert m.load().m4q_build_flags() == 0


def test_bounds_status_string():
    m.build()
    assert "bounds" in m.status_string(m.ERR_BOUNDS)
