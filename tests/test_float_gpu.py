"""GPU parity of the F16 / F32 matvecs (unquantized rows, fp32 activations
used as they are) against the oracle: the weight conversion bit for bit, the
matvec within 1e-5 * sum_k |w x| per output, exact-sum cases bit for bit, and
the variants (split-K, residual add, siblings, token passes)."""
import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import synth
from tests.gpu_util import TOL, assert_within, dev, sample_rows

pytestmark = pytest.mark.gpu

FLOAT = (oracle.F16, oracle.F32)


def _weights(fmt, M, K, seed):
    w = synth.weights(seed, M, K)
    if fmt == oracle.F16:
        w[0, :8] = [2.0 ** -24, 3 * 2.0 ** -26, 65504.0, 65519.0, -0.0, 1e-8, 2049.0, 2051.0]  # subnormal, ties, max
    return w


@pytest.mark.parametrize("fmt", FLOAT)
def test_convert_weights_bit_exact(lib, fmt):
    M, K = 300, 2080
    w = _weights(fmt, M, K, 70 + fmt)
    w[5, :4] = [7e4, -7e4, 65520.0, 1e30]   # overflow to infinity in F16
    W = lib.quantize_weights(fmt, dev(w)).cpu().numpy()
    assert np.array_equal(W, oracle.quantize(fmt, w))


SMALL = []
for fmt in FLOAT:
    for M, K, ns in [(1, 32, (1, 3)), (37, 1056, (1, 2, 5)), (333, 3072, (1, 4, 8, 16)),
                     (1000, 1024, (7, 17, 33, 64)), (64, 7200, (2, 13))]:
        for n in ns:
            SMALL.append((fmt, M, K, n))


@pytest.mark.parametrize("fmt,M,K,n", SMALL)
def test_float_qmv_small(lib, fmt, M, K, n):
    seed = 1000 * fmt + M + K + n
    w = _weights(fmt, M, K, seed)
    x = synth.activations(seed, n, K)
    Wn = oracle.quantize(fmt, w)
    y = lib.run(fmt, dev(Wn), dev(x), M, K).cpu().numpy()
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    assert_within(y, yr, sabs, what=f"fmt{fmt} M{M} K{K} n{n}")
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("fmt", FLOAT)
def test_float_qmv_exact_sums(lib, fmt):
    # weights k * 2^-6 (|k| <= 60) and activations j * 2^-3 (|j| <= 100):
    # every product is a multiple of 2^-9 and every partial sum stays below
    # 2^24 of those, so fp32 sums in any order are exact
    r = np.random.default_rng(fmt)
    M, K, n = 100, 2048, 6
    w = (r.integers(-60, 61, (M, K)) * 2.0 ** -6).astype(np.float32)
    x = (r.integers(-100, 101, (n, K)) * 2.0 ** -3).astype(np.float32)
    Wn = oracle.quantize(fmt, w)
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    assert np.all(sabs < 2.0 ** 24 * 2.0 ** -9)
    for S in (1, 3):
        y = lib.splitk_run(fmt, dev(Wn), dev(x), M, K, n_split=S).cpu().numpy()
        assert np.array_equal(y.astype(np.float64), yr)


@pytest.mark.parametrize("fmt,M,K,n,S", [(oracle.F16, 64, 8192, 3, 4), (oracle.F32, 100, 16384, 16, 0),
                                         (oracle.F16, 40, 6144, 2, 3), (oracle.F32, 17, 4096, 1, 16),
                                         (oracle.F16, 2000, 5120, 16, 0)])
def test_float_splitk(lib, fmt, M, K, n, S):
    seed = 77 + fmt + M
    Wn = oracle.quantize(fmt, _weights(fmt, M, K, seed))
    x = synth.activations(seed, n, K)
    Wd, xd = dev(Wn), dev(x)
    y = lib.splitk_run(fmt, Wd, xd, M, K, n_split=S)
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    assert_within(y.cpu().numpy(), yr, sabs, what=f"splitk S{S}")
    assert torch.equal(y, lib.splitk_run(fmt, Wd, xd, M, K, n_split=S))   # deterministic


def test_long_rows_need_split_k(lib):
    # 65536 fp32 activations do not fit in shared memory for one CTA's range:
    # the plain call refuses the shape, split-K (chosen split) computes it
    fmt, M, K, n = oracle.F32, 48, 65536, 2
    Wn = oracle.quantize(fmt, _weights(fmt, M, K, 5))
    x = synth.activations(6, n, K)
    Wd, xd = dev(Wn), dev(x)
    with pytest.raises(lib.QmvError):
        lib.run(fmt, Wd, xd, M, K)
    S = lib.splitk_choose(fmt, M, K, n)
    assert S >= 3
    y = lib.splitk_run(fmt, Wd, xd, M, K, n_split=0).cpu().numpy()
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    assert_within(y, yr, sabs, what="long rows")


@pytest.mark.parametrize("fmt", FLOAT)
def test_float_residual_and_siblings(lib, fmt):
    M, K, n = 700, 3072, 5
    Wn = oracle.quantize(fmt, _weights(fmt, M, K, 11 + fmt))
    x = synth.activations(12, n, K)
    r = synth.activations(13, n, M)
    Wd, xd = dev(Wn), dev(x)
    y = lib.run_residual(fmt, Wd, xd, dev(r), M, K).cpu().numpy()
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    ref = yr + r.astype(np.float64)
    assert_within(y, ref, sabs + np.abs(ref) * (2.0 ** -23 / TOL), what="residual")
    # siblings: a float matrix next to a quantized one, at 1 and 5 tokens
    Wq = dev(oracle.quantize(1, synth.weights(14, 256, K)))
    for nn in (1, n):
        ys = lib.run_siblings([(fmt, Wd, M), (1, Wq, 256)], xd[:nn], K)
        assert torch.equal(ys[0], lib.run(fmt, Wd, xd[:nn], M, K))
        assert torch.equal(ys[1], lib.run(1, Wq, xd[:nn], 256, K))
    assert lib.get_device_error() == 0


@pytest.mark.parametrize("fmt,n", [(oracle.F16, 1), (oracle.F16, 4), (oracle.F16, 16), (oracle.F32, 16)])
def test_float_full_size_sampled(lib, fmt, n):
    # the benchmark's workload and launch configuration (split chosen from the
    # shape, workspace given), sampled rows
    M, K = (17408, 5120) if fmt == oracle.F16 else (4096, 4096)
    Wn = oracle.quantize(fmt, synth.weights(5000 + fmt, M, K))
    x = synth.activations(5100 + n, n, K)
    S = lib.splitk_choose(fmt, M, K, n)
    ws = torch.empty(max(16, lib.splitk_workspace_fast_bytes(M, K, n, S)), dtype=torch.uint8, device="cuda")
    y = lib.splitk_run(fmt, dev(Wn), dev(x), M, K, n_split=S, ws=ws).cpu().numpy()
    rows = sample_rows(M)
    yr, sabs = oracle.qmv(fmt, Wn[rows], x, K)
    assert_within(y[:, rows], yr, sabs, what=f"fmt{fmt} n{n} S{S}")
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("M,K,n,S", [(4200, 2048, 16, 0), (4200, 2048, 8, 0), (5000, 3072, 12, 0),
                                     (4104, 1056, 21, 2), (6000, 5120, 16, 0)])
def test_f16_tensor_core_matvec(lib, M, K, n, S):
    # F16 rows, passes of 5-16 tokens, tall matrices, split ranges: the
    # tensor-core kernel (activations scaled per token by a power of two and
    # split into two f16 parts).  Tokens over a wide range of magnitudes, a
    # zero token, special weights; every output against the oracle.
    seed = 5000 + M + K + n
    w = _weights(oracle.F16, M, K, seed)
    x = synth.activations(seed + 1, n, K)
    x[1] *= np.float32(1e-30)
    x[2] *= np.float32(1e30)
    x[3] = 0.0
    x[4, :100] *= np.float32(1e-20)      # small elements beside large ones in one range
    Wn = oracle.quantize(oracle.F16, w)
    y = lib.splitk_run(oracle.F16, dev(Wn), dev(x), M, K, n_split=S).cpu().numpy()
    yr, sabs = oracle.qmv(oracle.F16, Wn, x, K)
    assert np.all(np.isfinite(y))
    assert_within(y, yr, sabs, what=f"F16 M{M} K{K} n{n} S{S}")
    assert np.all(y[3] == 0.0)


def test_f16_tensor_core_exact_sums(lib):
    # weights k * 2^-6 and activations j * 2^-3 (as the exact-sum test
    # above) on a tall matrix: the tensor-core kernel's products and fp32
    # accumulation are exact, so the result is bit for bit the oracle's
    r = np.random.default_rng(11)
    M, K, n = 4200, 2048, 16
    w = (r.integers(-60, 61, (M, K)) * 2.0 ** -6).astype(np.float32)
    x = (r.integers(-100, 101, (n, K)) * 2.0 ** -3).astype(np.float32)
    Wn = oracle.quantize(oracle.F16, w)
    yr, sabs = oracle.qmv(oracle.F16, Wn, x, K)
    assert np.all(sabs < 2.0 ** 24 * 2.0 ** -9)
    y = lib.splitk_run(oracle.F16, dev(Wn), dev(x), M, K, n_split=0).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), yr)
