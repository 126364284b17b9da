"""GPU parity of the epilogue fusions: matvec + residual add, and sibling
matvecs sharing one quantized x."""
import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import api, synth
from tests.gpu_util import TOL, assert_within, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,M,K,n,S", [(0, 300, 2048, 1, 1), (1, 1000, 4096, 5, 1), (2, 72, 8192, 3, 4),
                                         (0, 64, 16384, 16, 8), (1, 17408, 5120, 16, 1)])
@pytest.mark.parametrize("in_place", [False, True])
def test_residual_add(lib, fmt, M, K, n, S, in_place):
    seed = 1100 + fmt + n + S
    Wn = oracle.quantize(fmt, synth.weights(seed, M, K))
    x = synth.activations(seed + 1, n, K)
    r = synth.activations(seed + 2, n, M)
    Wd, xd, rd = dev(Wn), dev(x), dev(r)
    out = rd if in_place else None
    y = api.run_residual(fmt, Wd, xd, rd, M, K, out=out, n_split=S).cpu().numpy()
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    ref = yr + r.astype(np.float64)
    # the matvec's tolerance plus the rounding of the one fp32 addition
    assert_within(y, ref, sabs + np.abs(ref) * (2.0 ** -23 / TOL), what=f"residual fmt{fmt} S{S}")


def test_residual_of_zero_is_the_plain_matvec(lib):
    M, K, n = 500, 4096, 6
    Wd = dev(oracle.quantize(1, synth.weights(1200, M, K)))
    xd = dev(synth.activations(1201, n, K))
    for S in (1, 4):
        y0 = api.splitk_run(1, Wd, xd, M, K, n_split=S)
        y1 = api.run_residual(1, Wd, xd, torch.zeros((n, M), device="cuda"), M, K, n_split=S)
        assert torch.equal(y0, y1)


@pytest.mark.parametrize("n", [1, 2, 5, 16])
def test_siblings_equal_separate_matvecs(lib, n):
    # q/k/v-style siblings of three formats and sizes over one x
    K = 2048
    mats = []
    for i, (fmt, M) in enumerate([(0, 512), (1, 1000), (2, 96)]):
        mats.append((fmt, dev(oracle.quantize(fmt, synth.weights(1300 + i, M, K))), M))
    xd = dev(synth.activations(1310 + n, n, K))
    ys = api.run_siblings(mats, xd, K)
    for (fmt, W, M), y in zip(mats, ys):
        assert torch.equal(y, api.run(fmt, W, xd, M, K))
    assert lib.get_device_error() == 0


def test_siblings_match_the_oracle(lib):
    K, n = 4096, 4
    Ws = [oracle.quantize(f, synth.weights(1400 + f, M, K)) for f, M in [(0, 128), (1, 256)]]
    x = synth.activations(1410, n, K)
    ys = api.run_siblings([(0, dev(Ws[0]), 128), (1, dev(Ws[1]), 256)], dev(x), K)
    for fmt, Wn, y in zip((0, 1), Ws, ys):
        yr, sabs = oracle.qmv(fmt, Wn, x, K)
        assert_within(y.cpu().numpy(), yr, sabs, what=f"sibling fmt{fmt}")
