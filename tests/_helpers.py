"""Shared helpers of the GPU parity tests."""
import numpy as np

TOL = 1e-2   # |gpu - ref| <= TOL * max(1, |ref|), per element (fp32 accumulate, fp16 out)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close(y_gpu, ref, what=""):
    y = np.asarray(y_gpu).astype(np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), "%s: non-finite output" % what
    err = np.abs(y - ref)
    bound = TOL * np.maximum(1.0, np.abs(ref))
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d of %d elements out of tolerance; first at %s: gpu %r ref %r"
                             % (what, int(bad.sum()), bad.size, tuple(i), y[tuple(i)], ref[tuple(i)]))
    return float((err / np.maximum(1.0, np.abs(ref))).max()) if err.size else 0.0


def sample_rows(M, extra=8, seed=0):
    rows = {0, 1, M - 1}
    for r in (127, 128, 129, 255, 256, M // 2):
        if 0 <= r < M:
            rows.add(r)
    rng = np.random.default_rng(seed)
    rows.update(int(v) for v in rng.integers(0, M, size=extra))
    return sorted(rows)
