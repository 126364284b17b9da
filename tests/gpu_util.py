"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import oracle

TOL = 1e-5  # |y_gpu - y_ref| <= TOL * sum_k |What x Xhat| (fp32 accumulation of exact block sums)


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def assert_within(y_gpu, y_ref, sabs, tol=TOL, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = tol * sabs + 1e-30
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of tolerance; first at {tuple(i)}: "
                             f"gpu {y_gpu[tuple(i)]!r} ref {y_ref[tuple(i)]!r} bound {bound[tuple(i)]!r}")


def sample_rows(M, n=48, seed=0):
    """Rows worth checking: both ends, tile and unit boundaries, random."""
    r = np.random.default_rng(seed)
    rows = {0, 1, 7, 8, 31, 32, 33, M - 1, M - 2, M - 8, M - 9, M // 2}
    rows |= set(int(v) for v in r.integers(0, M, n))
    return np.array(sorted(v for v in rows if 0 <= v < M))


def oracle_rows(fmt, W_np, rows, x, K):
    y, sabs = oracle.qmv(fmt, W_np[rows], x, K)
    return y, sabs
