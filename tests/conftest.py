import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden_blocks(fname):
    """Parse a golden block file: blocks of 'key value...' lines ended by 'end'."""
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "block":
                cur = {"name": vals[0]}
            elif key == "end":
                blocks.append(cur)
                cur = None
            elif key == "codec":
                cur["codec"] = vals[0]
            elif key == "d_bits":
                cur["d_bits"] = int(vals[0], 16)
            elif key == "b_bits":
                cur["b_bits"] = int(vals[0], 16)
            elif key == "code_bytes":
                cur["code_bytes"] = [int(v, 16) for v in vals]
            elif key == "weights":
                cur["weights"] = [float(v) for v in vals]
    return blocks


@pytest.fixture(scope="session")
def golden_blocks():
    out = []
    for f in ("q4_0_blocks.txt", "q8_0_blocks.txt", "q2_0_blocks.txt", "mlx4_blocks.txt"):
        out.extend(read_golden_blocks(f))
    return out
