"""GPU parity of the dense quantized matvec, the activation quantizer, the
weight quantizer and split-K, against the CPU oracle on the same seeded
inputs.  Integer work is compared bit for bit; fp32 results within
1e-5 * sum_k |What x Xhat| per output."""
import functools

import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import synth
from tests import layout_ref as L
from tests.gpu_util import TOL, assert_within, dev, sample_rows

pytestmark = pytest.mark.gpu

GW = {0: 256, 1: 256, 2: 512, 3: 256, 4: 256, 5: 512, 6: 1024}


# --------------------------------------------------------------------------
# activation quantizer: bit-exact
# --------------------------------------------------------------------------

def _tricky_activations(n, K, seed):
    x = synth.activations(seed, n, K)
    x[0, :32] = 0.0                                     # zero block
    x[0, 32:64] = np.arange(-16, 16, dtype=np.float32) * 8.0   # exact halves after scaling
    x[0, 64] = 127 * 3.0
    x[min(1, n - 1), 96:128] *= 1e-30                    # tiny but normal
    x[n - 1, -32:] = np.float32(1e30)                    # huge, all equal
    if K >= 512:
        x[n - 1, 224:256] *= np.float32(1e-38)           # 1 / d overflows to infinity ...
        x[n - 1, 230] = 0.0                              # ... and 0 * inf gives code 0
    return x


def test_branch_free_rounding_is_ieee_on_every_input(lib):
    # the staging's a / 127 and 1 / d against div.rn / rcp.rn, all 2^31 inputs
    assert lib.check_rounding() == [0, 0]


@pytest.mark.parametrize("fmt,n,K", [(f, n, K) for f in (0, 1, 2) for n, K in ((1, 1024), (5, 2048), (16, 4096))])
def test_fused_staging_matches_standalone_quantizer(lib, fmt, n, K):
    # the in-kernel quantization of x must produce exactly the codes and scales
    # of the standalone quantizer (itself bit-exact against the oracle): the
    # two paths then run the same arithmetic and agree bit for bit
    M = 96
    x = _tricky_activations(n, K, seed=n + K + fmt)
    x[n // 2, 256:288] *= 1e-38          # blocks far below 2^-100 take the exact slow path
    Wd = dev(oracle.quantize(fmt, synth.weights(40 + fmt, M, K)))
    xd = dev(x)
    q, d, s = lib.quantize_act(xd)
    rq, rd, rs = oracle.act_quant(x)
    assert np.array_equal(L.q8_codes_natural(q.cpu().numpy()), rq) and np.array_equal(s.cpu().numpy(), rs)
    assert torch.equal(lib.run(fmt, Wd, xd, M, K), lib.run_q8(fmt, Wd, q, d, s, M, K))


@pytest.mark.parametrize("n,K", [(1, 256), (3, 4096), (16, 5120), (64, 2048)])
def test_act_quant_bit_exact(lib, n, K):
    x = _tricky_activations(n, K, seed=n + K)
    q, d, s = lib.quantize_act(dev(x))
    rq, rd, rs = oracle.act_quant(x)
    assert np.array_equal(L.q8_codes_natural(q.cpu().numpy()), rq)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(s.cpu().numpy(), rs)


# --------------------------------------------------------------------------
# weight quantizer: bit-exact bytes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4, 5, 6])
def test_quantize_weights_bit_exact(lib, fmt):
    K = 2048
    w = synth.weights(70 + fmt, 300, K)
    w[3] = 0.0
    w[4] *= 1e-4                                          # subnormal fp16 scales
    w[5, :256] = np.abs(w[5, :256])                       # one-signed blocks
    w[6, :256] = -np.abs(w[6, :256])
    w[7] *= 100.0
    W = lib.quantize_weights(fmt, dev(w))
    ref = oracle.quantize(fmt, w)
    got = W.cpu().numpy()
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# dense matvec on small shapes (several tiles and ragged tails)
# --------------------------------------------------------------------------

SMALL = []
for fmt in (0, 1, 2, 3, 4, 5, 6):
    for M, K, ns in [(1, 512, (1, 3)), (37, 1536, (1, 2, 5)), (333, 3072, (1, 4, 8, 16)),
                     (1000, 1024, (7, 17, 33, 64)), (64, 7168, (2, 13))]:
        if K % GW[fmt]:
            continue
        for n in ns:
            SMALL.append((fmt, M, K, n))


@pytest.mark.parametrize("fmt,M,K,n", SMALL)
def test_qmv_small(lib, fmt, M, K, n):
    seed = 1000 * fmt + M + K + n
    w = synth.weights(seed, M, K)
    x = synth.activations(seed, n, K)
    Wn = oracle.quantize(fmt, w)
    y = lib.run(fmt, dev(Wn), dev(x), M, K).cpu().numpy()
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    assert_within(y, yr, sabs, what=f"fmt{fmt} M{M} K{K} n{n}")


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4, 5, 6])
def test_qmv_prequantized_input_matches_fused(lib, fmt):
    M, K, n = 200, 2048, 5
    w = synth.weights(5 + fmt, M, K)
    x = synth.activations(6, n, K)
    Wd = dev(oracle.quantize(fmt, w))
    xd = dev(x)
    y1 = lib.run(fmt, Wd, xd, M, K)
    q, d, s = lib.quantize_act(xd)
    y2 = lib.run_q8(fmt, Wd, q, d, s, M, K)
    assert torch.equal(y1, y2)
    assert torch.equal(y1, lib.run(fmt, Wd, xd, M, K))     # bitwise reproducible


def _exact_case(fmt, r):
    """Weights and activations whose products and sums are exact in fp32:
    power-of-two scales, small integer codes, K = 512 (one group where larger)."""
    K, M, n = max(512, GW[fmt]), 40, 3
    groups = []
    for m in range(M):
        row = b""
        for gi in range(K // GW[fmt]):
            if fmt == 0:
                row += L.pack_q8_0([L.f16_bits(2.0 ** -3)] * 8, r.integers(-127, 128, (8, 32)).tolist())
            elif fmt == 1:
                row += L.pack_q4_k(L.f16_bits(2.0 ** -4), L.f16_bits(2.0 ** -5), r.integers(0, 4, 8).tolist(),
                                   r.integers(0, 4, 8).tolist(), r.integers(0, 16, (8, 32)).tolist())
            elif fmt in (5, 6):
                gs = 64 if fmt == 5 else 128
                row += L.pack_q8_g([L.f16_bits(2.0 ** -3)] * 8, r.integers(-63, 64, 8 * gs).tolist(), gs)
            elif fmt == 4:
                row += L.pack_q6_k(L.f16_bits(2.0 ** -4), r.integers(0, 4, 16).tolist(),
                                   r.integers(24, 41, 256).tolist())
            elif fmt == 3:
                row += L.pack_q5_k(L.f16_bits(2.0 ** -4), L.f16_bits(2.0 ** -5), r.integers(0, 4, 8).tolist(),
                                   r.integers(0, 4, 8).tolist(), r.integers(0, 32, (8, 32)).tolist())
            else:
                row += L.pack_iq4_xs([L.f16_bits(2.0 ** -6)] * 2, r.integers(31, 34, (2, 8)).tolist(),
                                     r.integers(0, 16, (2, 8, 32)).tolist())
        groups.append(np.frombuffer(row, np.uint8))
    W = np.stack(groups)
    kx = r.integers(-127, 128, (n, K))
    kx[:, ::32] = 127
    x = (kx * 2.0 ** -2).astype(np.float32)
    return W, x, K, M


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4, 5, 6])
def test_qmv_exact_integer_sums(lib, fmt):
    # every partial sum is an integer multiple of 2^-8 below 2^24 * 2^-8, so an
    # exact int32 block sum gives a bit-exact fp32 result in any order
    W, x, K, M = _exact_case(fmt, np.random.default_rng(fmt))
    yr, sabs = oracle.qmv(fmt, W, x, K)
    unit = {0: 2.0 ** -5, 1: 2.0 ** -7, 2: 2.0 ** -8, 3: 2.0 ** -7, 4: 2.0 ** -6, 5: 2.0 ** -5, 6: 2.0 ** -5}[fmt]   # d_w * d_x (and dmin * d_x)
    assert np.all(sabs < 2.0 ** 22 * unit)
    y = lib.run(fmt, dev(W), dev(x), M, K).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), yr)


@pytest.mark.parametrize("M,K,n,S", [(7171, 1024, 5, 1), (7171, 1024, 8, 1), (9000, 2048, 13, 1), (7171, 1024, 16, 1),
                                     (7171, 1024, 33, 1), (7200, 6144, 8, 3), (8192, 1792, 16, 2)])
def test_q4_k_tensor_core_matvec(lib, M, K, n, S):
    # the tensor-core kernel (Q4_K, passes of 5-16 tokens, tall matrices):
    # ragged tiles, token passes with a partial last one, split ranges with
    # odd numbers of superblocks; every output against the oracle, the
    # pre-quantized path bitwise equal to the fused one
    seed = 7000 + M + K + n
    w = synth.weights(seed, M, K)
    x = synth.activations(seed + 1, n, K)
    Wn = oracle.quantize(1, w)
    Wd, xd = dev(Wn), dev(x)
    y = lib.run(1, Wd, xd, M, K) if S == 1 else lib.splitk_run(1, Wd, xd, M, K, n_split=S)
    yr, sabs = oracle.qmv(1, Wn, x, K)
    assert_within(y.cpu().numpy(), yr, sabs, what=f"M{M} K{K} n{n} S{S}")
    q, d, s = lib.quantize_act(xd)
    if S == 1:
        assert torch.equal(lib.run_q8(1, Wd, q, d, s, M, K), y)


@pytest.mark.parametrize("n", [5, 8, 12, 16, 21])
def test_q4_k_block_sums_exact_at_their_extremes(lib, n):
    # Q4_K from 5 tokens forms its block sums on the tensor cores, with the
    # weights entering as 1024 + q: the largest sums (all codes 15 against
    # all +-127, and the mixed rows) must still come out exact.  Scales are
    # powers of two, so the fp32 result is bit-exact in any order.
    r = np.random.default_rng(n)
    K, M = 1024, 8200   # tall enough for the tensor-core kernel, with a ragged last tile
    rows = []
    for m in range(M):
        row = b""
        for gi in range(K // 256):
            if m % 3 == 0:
                codes = [[15] * 32] * 8
            elif m % 3 == 1:
                codes = [[0] * 32] * 8
            else:
                codes = r.integers(0, 16, (8, 32)).tolist()
            row += L.pack_q4_k(L.f16_bits(2.0 ** -4), L.f16_bits(2.0 ** -5), r.integers(0, 4, 8).tolist(),
                               r.integers(0, 4, 8).tolist(), codes)
        rows.append(np.frombuffer(row, np.uint8))
    W = np.stack(rows)
    kx = r.integers(-127, 128, (n, K))
    kx[0] = 127
    kx[1] = -127
    kx[2, :512] = 127
    kx[2, 512:] = -127
    kx[:, ::32] = np.where(kx[:, ::32] < 0, -127, 127)   # every block's amax is 127: d_x = 2^-2
    x = (kx * 2.0 ** -2).astype(np.float32)
    yr, _ = oracle.qmv(1, W, x, K)
    y = lib.run(1, dev(W), dev(x), M, K).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), yr)
    q, d, s = lib.quantize_act(dev(x))
    y8 = lib.run_q8(1, dev(W), q, d, s, M, K).cpu().numpy()
    assert np.array_equal(y8, y)


# --------------------------------------------------------------------------
# full-size workloads, sampled rows, in the benchmark's launch configuration
# --------------------------------------------------------------------------

@functools.lru_cache(maxsize=2)
def _full_weights(fmt, M, K, seed):
    w = synth.weights(seed, M, K)
    return oracle.quantize(fmt, w)


FULL = []
for c in synth.DENSE_CASES:
    if c.workload == "splitk_q8_0":
        continue
    for i, n in enumerate(c.n_toks):
        FULL.append((c.workload, c.fmt, c.M, c.K, n, synth.seed_for(c.index, c.shape_index, i),
                     synth.seed_for(c.index, c.shape_index, 0)))


@pytest.mark.parametrize("name,fmt,M,K,n,seed,wseed", FULL)
def test_qmv_full_size_sampled(lib, name, fmt, M, K, n, seed, wseed):
    Wn = _full_weights(fmt, M, K, wseed)
    x = synth.activations(seed, n, K)
    y = lib.run(fmt, dev(Wn), dev(x), M, K).cpu().numpy()
    rows = sample_rows(M)
    yr, sabs = oracle.qmv(fmt, Wn[rows], x, K)
    assert_within(y[:, rows], yr, sabs, what=f"{name} n{n}")
    assert np.all(np.isfinite(y))


BENCH_CASE = next(c for c in synth.DENSE_CASES if c.workload == "q4_k")


@pytest.mark.parametrize("n_idx,n", list(enumerate(BENCH_CASE.n_toks)))
def test_bench_call_full_size(lib, n_idx, n):
    # the exact call the benchmark times for Q4_K 17408 x 5120: qmv_splitk_run
    # with the split chosen from the shape and a workspace with room for the
    # once-quantized activations (above 4 tokens: the standalone quantizer,
    # then the matvec kernel with pre-quantized input), checked element by
    # element on the first and last 512 rows (every tile and 8-row unit of
    # the first and last CTAs' ranges) and 256 random rows
    c = BENCH_CASE
    Wn = _full_weights(c.fmt, c.M, c.K, synth.seed_for(c.index, c.shape_index, 0))
    x = synth.activations(synth.seed_for(c.index, c.shape_index, n_idx), n, c.K)
    S = lib.splitk_choose(c.fmt, c.M, c.K, n)
    ws = torch.empty(max(16, lib.splitk_workspace_fast_bytes(c.M, c.K, n, S)), dtype=torch.uint8, device="cuda")
    y = lib.splitk_run(c.fmt, dev(Wn), dev(x), c.M, c.K, n_split=S, ws=ws).cpu().numpy()
    r = np.random.default_rng(n)
    rows = np.unique(np.concatenate([np.arange(512), np.arange(c.M - 512, c.M), r.integers(0, c.M, 256)]))
    yr, sabs = oracle.qmv(c.fmt, Wn[rows], x, c.K, nthreads=8)
    assert_within(y[:, rows], yr, sabs, what=f"bench call n{n} S{S}")
    assert np.all(np.isfinite(y))
    assert lib.get_device_error() == 0


# --------------------------------------------------------------------------
# split-K
# --------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,M,K,n,S", [(0, 64, 8192, 3, 4), (0, 100, 16384, 16, 0), (1, 40, 6144, 2, 3),
                                         (2, 72, 8192, 5, 8), (0, 17, 4096, 1, 16)])
def test_splitk_small(lib, fmt, M, K, n, S):
    seed = 77 + fmt + M
    w = synth.weights(seed, M, K)
    x = synth.activations(seed, n, K)
    Wn = oracle.quantize(fmt, w)
    Wd, xd = dev(Wn), dev(x)
    y = lib.splitk_run(fmt, Wd, xd, M, K, n_split=S)
    yr, sabs = oracle.qmv(fmt, Wn, x, K)
    assert_within(y.cpu().numpy(), yr, sabs, what=f"splitk S{S}")
    assert torch.equal(y, lib.splitk_run(fmt, Wd, xd, M, K, n_split=S))   # deterministic
    y1 = lib.run(fmt, Wd, xd, M, K).cpu().numpy()
    assert_within(y1, yr, sabs, what="unsplit")


SPLITK_FULL = []
for c in synth.DENSE_CASES:
    if c.workload != "splitk_q8_0":
        continue
    for i, n in enumerate(c.n_toks):
        SPLITK_FULL.append((c.M, c.K, n, synth.seed_for(c.index, c.shape_index, i),
                            synth.seed_for(c.index, c.shape_index, 0)))


@pytest.mark.parametrize("M,K,n,seed,wseed", SPLITK_FULL)
def test_splitk_full_size_sampled(lib, M, K, n, seed, wseed):
    Wn = _full_weights(0, M, K, wseed)
    x = synth.activations(seed, n, K)
    Wd, xd = dev(Wn), dev(x)
    y = lib.splitk_run(0, Wd, xd, M, K, n_split=0).cpu().numpy()
    rows = sample_rows(M)
    yr, sabs = oracle.qmv(0, Wn[rows], x, K)
    assert_within(y[:, rows], yr, sabs, what=f"splitk {M}x{K} n{n}")


@pytest.mark.parametrize("fmt,M,K,n,S", [(0, 64, 8192, 4, 4), (1, 40, 6144, 7, 3), (2, 72, 8192, 5, 8),
                                         (0, 100, 4096, 16, 1), (1, 24, 4096, 9, 2), (1, 17408, 5120, 16, 1)])
def test_splitk_quantized_once_is_bitwise_equal(lib, fmt, M, K, n, S):
    # a workspace with room for the activations makes split-K quantize them
    # once instead of per CTA: the same arithmetic, so the same bits
    w = synth.weights(90 + fmt + S, M, K)
    x = synth.activations(91 + n, n, K)
    Wd, xd = dev(oracle.quantize(fmt, w)), dev(x)
    small = torch.empty(max(16, lib.splitk_workspace_bytes(M, n, S) if S > 1 else 16), dtype=torch.uint8,
                        device="cuda")
    y_per_cta = lib.splitk_run(fmt, Wd, xd, M, K, n_split=S, ws=small)
    y_once = lib.splitk_run(fmt, Wd, xd, M, K, n_split=S)
    assert torch.equal(y_per_cta, y_once)
    yr, sabs = oracle.qmv(fmt, oracle.quantize(fmt, w), x, K)
    assert_within(y_once.cpu().numpy(), yr, sabs, what=f"splitk once S{S}")
