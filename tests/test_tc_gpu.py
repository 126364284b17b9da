"""The tensor-core building block and the measured pipe rates.

qmv_tc_probe multiplies a 128 x 32 tile of int8 codes by an N x 32 one
through the tcgen05 tensor cores, the codes held as f16 and accumulated in
fp32: every product (|c| <= 128) and every partial sum of 32 of them is an
integer far below 2^24, so the result must be the exact integer dot product.
This pins the operand layout (core matrices, descriptors) and the exactness
that a quantized contraction on the tensor cores relies on."""
import numpy as np
import pytest
import torch

from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N", [16, 32, 48, 64, 128, 256])
def test_tc_probe_gives_exact_integer_dot_products(lib, N):
    r = np.random.default_rng(N)
    A = r.integers(-127, 128, (128, 32)).astype(np.int8)
    B = r.integers(-127, 128, (N, 32)).astype(np.int8)
    A[0] = 127
    B[0] = -127                       # the largest magnitude of a block sum
    A[1, ::2], A[1, 1::2] = -128, 127  # the codes' full int8 range converts exactly
    got = lib.tc_probe(dev(A), dev(B)).cpu().numpy()
    ref = A.astype(np.int64) @ B.astype(np.int64).T
    assert np.array_equal(got.astype(np.int64), ref)
    assert np.array_equal(got, ref.astype(np.float32))
    assert lib.get_device_error() == 0


def test_measured_pipe_rates_are_plausible(lib):
    r = lib.measure_pipes()
    assert set(r) == set(lib.PIPE_NAMES)
    assert all(v > 0 for v in r.values())
    assert 8 <= r["dp4a"] <= 128            # per SM per clock (four schedulers x 32 lanes at most)
    assert r["tcgen05_f16_n256_mac"] > 4 * r["dp4a"] * 4   # the tensor core outruns dp4a's MACs
