"""Pins of the CPU oracle against things other than itself: numpy's binary16
rounding, brute-force argmins, hand-worked blocks, closed forms, a library
matmul, and invariants of the method.  CPU only."""
import os

import numpy as np
import pytest

import oracle
from moe_matvec_gb300 import synth
from tests import layout_ref as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng0 = np.random.default_rng(12345)


# --------------------------------------------------------------------------
# binary16 conversions (reduce to numpy's IEEE conversion)
# --------------------------------------------------------------------------

def test_f16_decode_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(h)) for h in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_encode_matches_numpy_including_ties_and_subnormals():
    vals = []
    # random magnitudes over the whole fp16 range, both signs
    vals += list(np.exp(rng0.uniform(np.log(1e-9), np.log(7e4), 20000)) * rng0.choice([-1, 1], 20000))
    # exact midpoints between neighbouring fp16 values (ties), normal and subnormal
    hs = np.arange(1, 0x7BFF, 7, dtype=np.uint16)
    lo = hs.view(np.float16).astype(np.float64)
    hi = (hs + 1).view(np.float16).astype(np.float64)
    vals += list((lo + hi) / 2)
    vals += [65504.0, 65519.99, 65520.0, 65536.0, 1e6, 2 ** -24, 2 ** -25, 3 * 2 ** -26, 2 ** -26,
             6.1e-5, 0.0, -0.0]
    for v in vals:
        ref = int(np.array(v, np.float64).astype(np.float16).view(np.uint16))
        assert oracle.f64_to_f16(v) == ref, (v, hex(ref))


# --------------------------------------------------------------------------
# activation quantizer
# --------------------------------------------------------------------------

def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = [float(t) for t in v.split()]
    return out


def test_act_quant_golden_block():
    g = _read_golden("act_quant_block.txt")
    x = np.array(g["x"], np.float32)[None, :]
    q, d, s = oracle.act_quant(x)
    assert d[0, 0] == np.float32(g["d"][0])
    assert q[0].tolist() == [int(v) for v in g["q"]]
    assert s[0, 0] == int(g["s"][0])


def test_act_quant_integer_block_is_exact():
    # amax = 127 gives d = 1 and id = 1, so q = x exactly
    x = rng0.integers(-127, 128, size=(3, 256)).astype(np.float32)
    x[:, ::32] = 127.0
    q, d, s = oracle.act_quant(x)
    assert np.all(d == 1.0)
    assert np.array_equal(q.astype(np.float32), x)
    assert np.array_equal(s, x.reshape(3, 8, 32).sum(-1).astype(np.int32))


def test_act_quant_power_of_two_scale():
    k = rng0.integers(-127, 128, size=(2, 512))
    k[:, ::32] = -127
    x = (k * 2.0 ** -9).astype(np.float32)
    q, d, s = oracle.act_quant(x)
    assert np.all(d == np.float32(2.0 ** -9))
    assert np.array_equal(q.astype(np.int64), k)


def test_act_quant_zero_block():
    x = rng0.standard_normal((1, 128)).astype(np.float32)
    x[0, 32:64] = 0.0
    q, d, s = oracle.act_quant(x)
    assert d[0, 1] == 0.0 and s[0, 1] == 0 and not q[0, 32:64].any()


@pytest.mark.parametrize("scale", [1.0, 1e-3, 37.0])
def test_act_quant_invariants(scale):
    x = (rng0.standard_normal((4, 1024)) * scale).astype(np.float32)
    x[1] = rng0.standard_cauchy(1024).astype(np.float32) * np.float32(scale)
    q, d, s = oracle.act_quant(x)
    qb = q.reshape(4, 32, 32).astype(np.int64)
    xb = x.reshape(4, 32, 32).astype(np.float64)
    amax = np.abs(xb).max(-1)
    assert np.all(d == (amax.astype(np.float32) / np.float32(127)))
    assert np.all(np.abs(qb) <= 127)
    assert np.all(np.abs(qb).max(-1) == 127)           # the largest element maps to 127
    assert np.array_equal(s, qb.sum(-1).astype(np.int32))
    assert np.all(np.sign(qb) * np.sign(xb) >= 0)       # never flips a sign
    err = np.abs(xb - d[..., None].astype(np.float64) * qb)
    assert np.all(err <= d[..., None] * (0.5 + 1e-5))   # nearest grid point


def _act_quant_numpy(x):
    """The activation rule restated with numpy fp32 element-wise operations,
    one line per step of the rule (amax; d = amax / 127; id = 1 / d or 0;
    q = clamp(rne(x * id)); s = sum q), independently of the oracle's C."""
    xb = np.ascontiguousarray(x, np.float32).reshape(-1, 32)
    amax = np.abs(xb).max(axis=1)
    d = amax / np.float32(127.0)
    pos = d > 0
    with np.errstate(divide="ignore", over="ignore"):
        inv = np.where(pos, np.float32(1.0) / np.where(pos, d, np.float32(1.0)), np.float32(0.0))
    inv = inv.astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        p = xb * inv[:, None]                     # fp32 products, round to nearest
        r = np.clip(np.rint(p), -127.0, 127.0)    # round half to even, clamp
    r = np.where(np.isnan(p), 0.0, r)             # 0 * inf (1 / d overflowed): code 0
    q = r.astype(np.int8)
    return q, d, q.astype(np.int32).sum(axis=1)


def _near_tie_blocks(nb, seed):
    """Blocks whose products x * id fall on or within two ulps of k + 1/2:
    the largest element a fixes d = a / 127 and id = 1 / d, every other
    element is (k + 1/2) / id (k a random integer) moved by -2..2 ulps."""
    r = np.random.default_rng(seed)
    a = (r.uniform(0.5, 2.0, nb) * 2.0 ** r.integers(-100, 100, nb)).astype(np.float32)
    d = a / np.float32(127.0)
    inv = (np.float32(1.0) / d).astype(np.float32)
    k = r.integers(-127, 127, (nb, 32)).astype(np.float64)
    x = ((k + 0.5) / inv[:, None].astype(np.float64)).astype(np.float32)
    x = (x.view(np.int32) + r.integers(-2, 3, (nb, 32)).astype(np.int32)).view(np.float32)
    x = np.clip(x, -a[:, None], a[:, None])
    x[np.arange(nb), r.integers(0, 32, nb)] = a * np.where(r.random(nb) < 0.5, 1, -1).astype(np.float32)
    return x


def test_act_quant_matches_a_naive_numpy_restatement_on_a_million_blocks():
    # random blocks over a wide range of scales, blocks crowded with near and
    # exact .5 ties, tiny blocks (subnormal d, 1/d overflowing) with zeros,
    # zero blocks: the oracle's codes, scales and sums must be those of the
    # rule written out with numpy's IEEE fp32 operations, bit for bit
    r = np.random.default_rng(12345)
    nb_rand, nb_tie = 600_000, 400_000
    xr = r.standard_normal((nb_rand, 32)).astype(np.float32)
    xr *= (2.0 ** r.integers(-120, 120, nb_rand)).astype(np.float32)[:, None]
    xr[:1000] = 0.0
    tiny = r.standard_normal((2000, 32)).astype(np.float32) * np.float32(1e-38)
    tiny[:, 5] = 0.0
    xr[1000:3000] = tiny
    xt = _near_tie_blocks(nb_tie, 54321)
    x = np.concatenate([xr, xt]).reshape(-1, 1024)    # 1e6 blocks as rows of 32 blocks
    q, d, s = oracle.act_quant(x)
    nq, nd, ns = _act_quant_numpy(x)
    assert np.array_equal(q.reshape(-1, 32), nq)
    assert np.array_equal(d.reshape(-1).view(np.uint32), nd.view(np.uint32))
    assert np.array_equal(s.reshape(-1), ns)
    # the tie-heavy blocks really do hit exact halves (where the rounding
    # direction decides the code) and land on both sides of them
    _, dt, _ = _act_quant_numpy(xt)
    inv = (np.float32(1.0) / dt).astype(np.float32)
    pt = (xt * inv[:, None]).astype(np.float64)
    assert (np.abs(pt - np.floor(pt)) == 0.5).sum() > 10_000
    assert (np.abs(np.abs(pt - np.floor(pt)) - 0.5) < 1e-6 * np.abs(pt)).sum() > 100_000


# --------------------------------------------------------------------------
# weight quantizers
# --------------------------------------------------------------------------

def _rand_w(M, K, std=0.02, seed=7):
    return synth.weights(seed, M, K, std)


def test_q8_0_scales_and_codes_are_argmins():
    w = _rand_w(3, 512)
    W = oracle.quantize(0, w)
    for m in range(3):
        for gi in range(2):
            d_bits, q = L.unpack_q8_0(W[m, 272 * gi:272 * (gi + 1)])
            for j in range(8):
                wb = w[m, 256 * gi + 32 * j: 256 * gi + 32 * j + 32].astype(np.float64)
                assert d_bits[j] == L.f16_bits(np.abs(wb).max() / 127.0)
                dv = L.f16_value(d_bits[j])
                cand = np.arange(-127, 128)
                err = np.abs(wb[:, None] - dv * cand[None, :])
                best = cand[np.argmin(err, axis=1)]
                assert q[j] == best.tolist()


def test_q8_0_ties_go_to_even():
    # d = 2^-7 exactly (amax = 127 * 2^-7); weights on exact half-steps
    w = np.zeros((1, 256), np.float32)
    w[0, 0] = 127 * 2.0 ** -7
    w[0, 1:6] = np.array([2.5, 3.5, -2.5, -3.5, 0.5]) * 2.0 ** -7
    W = oracle.quantize(0, w)
    d_bits, q = L.unpack_q8_0(W[0])
    assert L.f16_value(d_bits[0]) == 2.0 ** -7
    assert q[0][:6] == [127, 2, 4, -2, -4, 0]


def test_q8_0_requantization_is_idempotent():
    w = _rand_w(4, 1024)
    W = oracle.quantize(0, w)
    wh = oracle.dequant(0, W, 1024).astype(np.float32)
    assert np.array_equal(oracle.quantize(0, wh), W)


def test_q4_k_fields_follow_the_rule_and_codes_are_argmins():
    w = _rand_w(2, 512)
    w[1, :32] = np.abs(w[1, :32])          # a sub-block with no negative weight
    w[1, 32:64] = -np.abs(w[1, 32:64])     # and one with no positive weight
    W = oracle.quantize(1, w)
    for m in range(2):
        for gi in range(2):
            d_bits, dmin_bits, sc, mm, q = L.unpack_q4_k(W[m, 144 * gi:144 * (gi + 1)])
            wg = w[m, 256 * gi:256 * (gi + 1)].astype(np.float64).reshape(8, 32)
            lo = np.minimum(0.0, wg.min(1))
            a = (wg.max(1) - lo) / 15.0
            b = -lo
            assert d_bits == L.f16_bits(a.max() / 63.0)
            assert dmin_bits == L.f16_bits(b.max() / 63.0)
            d, dmin = L.f16_value(d_bits), L.f16_value(dmin_bits)
            assert sc == np.clip(np.rint(a / d), 0, 63).astype(int).tolist()
            assert mm == np.clip(np.rint(b / dmin), 0, 63).astype(int).tolist()
            for j in range(8):
                grid = d * sc[j] * np.arange(16) - dmin * mm[j]
                err = np.abs(wg[j][:, None] - grid[None, :])
                assert q[j] == np.argmin(err, axis=1).tolist()   # argmin keeps the lower q on ties


def test_iq4_xs_fields_follow_the_rule_and_codes_are_argmins():
    w = _rand_w(2, 1024)
    W = oracle.quantize(2, w)
    for m in range(2):
        for gi in range(2):
            d_bits, ls, c = L.unpack_iq4_xs(W[m, 272 * gi:272 * (gi + 1)])
            for s in range(2):
                wg = w[m, 512 * gi + 256 * s: 512 * gi + 256 * (s + 1)].astype(np.float64).reshape(8, 32)
                sj = np.abs(wg).max(1) / 113.0
                assert d_bits[s] == L.f16_bits(sj.max() / 31.0)
                d = L.f16_value(d_bits[s])
                assert ls[s] == (32 + np.clip(np.rint(sj / d), 0, 31)).astype(int).tolist()
                for j in range(8):
                    grid = d * (ls[s][j] - 32) * L.CODEBOOK
                    err = np.abs(wg[j][:, None] - grid[None, :])
                    assert c[s][j] == np.argmin(err, axis=1).tolist()


def test_q5_k_fields_follow_the_rule_and_codes_are_argmins():
    w = _rand_w(2, 512, seed=11)
    w[1, :32] = np.abs(w[1, :32])
    w[1, 32:64] = -np.abs(w[1, 32:64])
    W = oracle.quantize(3, w)
    assert W.shape[1] == 2 * 176
    for m in range(2):
        for gi in range(2):
            d_bits, dmin_bits, sc, mm, q = L.unpack_q5_k(W[m, 176 * gi:176 * (gi + 1)])
            wg = w[m, 256 * gi:256 * (gi + 1)].astype(np.float64).reshape(8, 32)
            lo = np.minimum(0.0, wg.min(1))
            a = (wg.max(1) - lo) / 31.0
            b = -lo
            assert d_bits == L.f16_bits(a.max() / 63.0)
            assert dmin_bits == L.f16_bits(b.max() / 63.0)
            d, dmin = L.f16_value(d_bits), L.f16_value(dmin_bits)
            assert sc == np.clip(np.rint(a / d), 0, 63).astype(int).tolist()
            assert mm == np.clip(np.rint(b / dmin), 0, 63).astype(int).tolist()
            for j in range(8):
                grid = d * sc[j] * np.arange(32) - dmin * mm[j]
                err = np.abs(wg[j][:, None] - grid[None, :])
                assert q[j] == np.argmin(err, axis=1).tolist()


def test_q6_k_fields_follow_the_rule_and_codes_are_argmins():
    w = _rand_w(2, 512, seed=13)
    w[1, :16] = np.abs(w[1, :16])
    W = oracle.quantize(4, w)
    assert W.shape[1] == 2 * 208
    for m in range(2):
        for gi in range(2):
            d_bits, sc, q = L.unpack_q6_k(W[m, 208 * gi:208 * (gi + 1)])
            wg = w[m, 256 * gi:256 * (gi + 1)].astype(np.float64).reshape(16, 16)
            s_i = np.abs(wg).max(1) / 31.0
            assert d_bits == L.f16_bits(s_i.max() / 127.0)
            d = L.f16_value(d_bits)
            assert sc == np.clip(np.rint(s_i / d), 0, 127).astype(int).tolist()
            for i in range(16):
                grid = d * sc[i] * (np.arange(64) - 32)
                err = np.abs(wg[i][:, None] - grid[None, :])
                assert q[16 * i:16 * i + 16] == np.argmin(err, axis=1).tolist()


@pytest.mark.parametrize("fmt,gs", [(5, 64), (6, 128)])
def test_q8_group_scales_and_codes_are_argmins(fmt, gs):
    K = 2048
    w = _rand_w(2, K, seed=fmt)
    W = oracle.quantize(fmt, w)
    gb = 16 + 8 * gs
    assert W.shape[1] == K // (8 * gs) * gb
    cand = np.arange(-127, 128)
    for m in range(2):
        for gi in range(K // (8 * gs)):
            d_bits, q = L.unpack_q8_g(W[m, gb * gi:gb * (gi + 1)], gs)
            wg = w[m, 8 * gs * gi:8 * gs * (gi + 1)].astype(np.float64).reshape(8, gs)
            for s_ in range(8):
                assert d_bits[s_] == L.f16_bits(np.abs(wg[s_]).max() / 127.0)
                dv = L.f16_value(d_bits[s_])
                err = np.abs(wg[s_][:, None] - dv * cand[None, :])
                assert q[gs * s_:gs * (s_ + 1)] == cand[np.argmin(err, axis=1)].tolist()
    # requantizing the dequantized weights gives the same bytes
    wh = oracle.dequant(fmt, W, K).astype(np.float32)
    assert np.array_equal(oracle.quantize(fmt, wh), W)


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4, 5, 6])
def test_zero_weights_dequantize_to_zero(fmt):
    w = _rand_w(2, 1024)
    w[0] = 0.0
    W = oracle.quantize(fmt, w)
    wh = oracle.dequant(fmt, W, 1024)
    assert np.all(wh[0] == 0.0)


def test_round_trip_error_bounds():
    w = _rand_w(8, 1024).astype(np.float64)
    # Q8_0: at most half a step of the stored scale, plus the scale's own rounding
    W = oracle.quantize(0, w.astype(np.float32))
    err = np.abs(oracle.dequant(0, W, 1024) - w).reshape(8, 32, 32)
    amax = np.abs(w).reshape(8, 32, 32).max(-1)
    d = amax / 127.0
    assert np.all(err.max(-1) <= d * (0.5 + 127 * 2.0 ** -11) + 1e-12)
    # Q4_K: codes land on a 16-point grid covering [lo, hi] of each sub-block
    W = oracle.quantize(1, w.astype(np.float32))
    err = np.abs(oracle.dequant(1, W, 1024) - w).reshape(8, 32, 32)
    rngb = (w.reshape(8, 32, 32).max(-1) - np.minimum(0, w.reshape(8, 32, 32).min(-1)))
    assert np.all(err.max(-1) <= rngb / 15.0 * 0.5 * 1.2 + 1e-4)
    # Q5_K: within half a step of the stored grid, or the distance from the
    # grid's ends to a weight outside them; smaller on average than Q4_K
    W = oracle.quantize(3, w.astype(np.float32))
    err = np.abs(oracle.dequant(3, W, 1024) - w).reshape(8, 4, 8, 32)
    wb = w.reshape(8, 4, 8, 32)
    for m in range(8):
        for gi in range(4):
            d_bits, dmin_bits, sc, mm, _ = L.unpack_q5_k(W[m, 176 * gi:176 * (gi + 1)])
            d, dmin = L.f16_value(d_bits), L.f16_value(dmin_bits)
            for j in range(8):
                lo_g = -dmin * mm[j]
                hi_g = lo_g + 31 * d * sc[j]
                bound = max(d * sc[j] / 2, lo_g - wb[m, gi, j].min(), wb[m, gi, j].max() - hi_g)
                assert err[m, gi, j].max() <= bound * (1 + 1e-12) + 1e-15
    assert err.mean() < np.abs(oracle.dequant(1, oracle.quantize(1, w.astype(np.float32)), 1024) - w).mean()
    # Q6_K: within half a step of the stored grid (it covers +-31 steps of s_i = amax / 31)
    W = oracle.quantize(4, w.astype(np.float32))
    err = np.abs(oracle.dequant(4, W, 1024) - w).reshape(8, 4, 16, 16)
    for m in range(8):
        for gi in range(4):
            d_bits, sc, _ = L.unpack_q6_k(W[m, 208 * gi:208 * (gi + 1)])
            d = L.f16_value(d_bits)
            wb = np.abs(w.reshape(8, 4, 16, 16)[m, gi])
            for i in range(16):
                step = d * sc[i]
                bound = max(step / 2, wb[i].max() - 31 * step)
                assert err[m, gi, i].max() <= bound * (1 + 1e-12) + 1e-15
    # IQ4_XS: the largest codebook gap is 24 (89 -> 113), so half a gap is 12 steps
    W = oracle.quantize(2, w.astype(np.float32))
    err = np.abs(oracle.dequant(2, W, 1024) - w).reshape(8, 32, 32)
    s = np.abs(w).reshape(8, 32, 32).max(-1) / 113.0
    assert np.all(err.max(-1) <= 14.5 * s * 1.1 + 1e-4)


# --------------------------------------------------------------------------
# dequantizers: hand-worked groups
# --------------------------------------------------------------------------

def test_dequant_q8_0_hand_worked():
    d_bits = [0x3800] * 8          # 0.5
    d_bits[3] = 0xB400             # -0.25
    q = [[(i - 16) for i in range(32)] for _ in range(8)]
    g = np.frombuffer(L.pack_q8_0(d_bits, q), np.uint8)[None, :]
    wh = oracle.dequant(0, g, 256)
    assert wh[0, 0] == -8.0 and wh[0, 31] == 7.5 and wh[0, 17] == 0.5
    assert wh[0, 96] == 4.0 and wh[0, 127] == -3.75          # block 3 scaled by -0.25


def test_dequant_q4_k_hand_worked():
    sc = [1, 2, 3, 4, 5, 6, 7, 63]
    m = [0, 1, 2, 3, 4, 5, 62, 63]
    q = [[i % 16 for i in range(32)] for _ in range(8)]
    q[7] = [15 - (i % 16) for i in range(32)]
    g = np.frombuffer(L.pack_q4_k(0x3400, 0x3000, sc, m, q), np.uint8)[None, :]   # d 0.25, dmin 0.125
    wh = oracle.dequant(1, g, 256)
    # weight 5 of sub-block 1: 0.25*2*5 - 0.125*1
    assert wh[0, 32 + 5] == 2.375
    # weight 20 of sub-block 6 (high nibble of byte 4): 0.25*7*4 - 0.125*62
    assert wh[0, 6 * 32 + 20] == 7.0 - 7.75
    # weight 0 of sub-block 7: q = 15: 0.25*63*15 - 0.125*63
    assert wh[0, 224] == 236.25 - 7.875


def test_dequant_iq4_xs_hand_worked():
    ls = [[32, 33, 31, 63, 0, 40, 32, 34], [35] * 8]
    c = [[[i % 16 for i in range(32)] for _ in range(8)] for _ in range(2)]
    g = np.frombuffer(L.pack_iq4_xs([0x2400, 0x3C00], ls, c), np.uint8)[None, :]   # 2^-6, 1.0
    wh = oracle.dequant(2, g, 512)
    assert wh[0, 0] == 0.0                                   # ls 32 -> zero scale
    assert wh[0, 32 + 3] == 2.0 ** -6 * 1 * -65              # ls 33, code 3
    assert wh[0, 64 + 17] == 2.0 ** -6 * -1 * -104           # ls 31 (negative scale), code 1
    assert wh[0, 96 + 31] == 2.0 ** -6 * 31 * 113            # ls 63, code 15
    assert wh[0, 128 + 8] == 2.0 ** -6 * -32 * 1             # ls 0, code 8
    assert wh[0, 256 + 100] == 3.0 * L.CODEBOOK[100 % 32 % 16]


def test_dequant_q5_k_hand_worked():
    q = [[0] * 32 for _ in range(8)]
    q[0][0], q[0][17], q[3][31], q[7][5] = 31, 16, 15, 1
    g = L.pack_q5_k(L.f16_bits(0.5), L.f16_bits(0.25), [1, 2, 3, 4, 5, 6, 7, 63], [0, 1, 2, 3, 4, 5, 6, 63], q)
    wh = oracle.dequant(3, np.frombuffer(g, np.uint8)[None, :], 256)[0]
    assert wh[0] == 0.5 * 1 * 31                     # fifth bit set, low bits 15
    assert wh[17] == 0.5 * 1 * 16                    # fifth bit only, high-nibble half
    assert wh[32 * 3 + 31] == 0.5 * 4 * 15 - 0.25 * 3
    assert wh[32 * 7 + 5] == 0.5 * 63 * 1 - 0.25 * 63
    assert wh[32 * 2 + 4] == -0.25 * 2


def test_dequant_q6_k_hand_worked():
    q = [32] * 256
    q[0], q[17], q[40], q[255] = 63, 0, 33, 31
    sc = list(range(1, 17))
    sc[15] = 127
    g = L.pack_q6_k(L.f16_bits(0.5), sc, q)
    wh = oracle.dequant(4, np.frombuffer(g, np.uint8)[None, :], 256)[0]
    assert wh[0] == 0.5 * 1 * 31
    assert wh[17] == 0.5 * 2 * -32                   # sub-block 1 (weights 16..31)
    assert wh[40] == 0.5 * 3 * 1
    assert wh[255] == 0.5 * 127 * -1
    assert wh[100] == 0.0


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4, 5, 6])
def test_dequant_random_fields(fmt):
    r = np.random.default_rng(fmt + 100)
    if fmt == 0:
        d = [L.f16_bits(v) for v in r.uniform(-1, 1, 8)]
        q = r.integers(-128, 128, (8, 32)).tolist()
        g = L.pack_q8_0(d, q)
        exp = np.concatenate([L.f16_value(d[j]) * np.array(q[j], float) for j in range(8)])
        K = 256
    elif fmt == 1:
        d, dm = L.f16_bits(r.uniform(0, 1)), L.f16_bits(r.uniform(0, 1))
        sc, m = r.integers(0, 64, 8).tolist(), r.integers(0, 64, 8).tolist()
        q = r.integers(0, 16, (8, 32)).tolist()
        g = L.pack_q4_k(d, dm, sc, m, q)
        exp = np.concatenate([L.f16_value(d) * sc[j] * np.array(q[j], float) - L.f16_value(dm) * m[j]
                              for j in range(8)])
        K = 256
    elif fmt in (5, 6):
        gs = 64 if fmt == 5 else 128
        d = [L.f16_bits(v) for v in r.uniform(-1, 1, 8)]
        q = r.integers(-128, 128, 8 * gs).tolist()
        g = L.pack_q8_g(d, q, gs)
        exp = np.array([L.f16_value(d[e // gs]) * q[e] for e in range(8 * gs)], float)
        K = 8 * gs
    elif fmt == 4:
        d = L.f16_bits(r.uniform(-1, 1))
        sc = r.integers(0, 128, 16).tolist()
        q = r.integers(0, 64, 256).tolist()
        g = L.pack_q6_k(d, sc, q)
        exp = np.array([L.f16_value(d) * sc[e // 16] * (q[e] - 32) for e in range(256)], float)
        K = 256
    elif fmt == 3:
        d, dm = L.f16_bits(r.uniform(0, 1)), L.f16_bits(r.uniform(0, 1))
        sc, m = r.integers(0, 64, 8).tolist(), r.integers(0, 64, 8).tolist()
        q = r.integers(0, 32, (8, 32)).tolist()
        g = L.pack_q5_k(d, dm, sc, m, q)
        exp = np.concatenate([L.f16_value(d) * sc[j] * np.array(q[j], float) - L.f16_value(dm) * m[j]
                              for j in range(8)])
        K = 256
    else:
        d = [L.f16_bits(v) for v in r.uniform(-1, 1, 2)]
        ls = r.integers(0, 64, (2, 8)).tolist()
        c = r.integers(0, 16, (2, 8, 32)).tolist()
        g = L.pack_iq4_xs(d, ls, c)
        exp = np.concatenate([L.f16_value(d[s]) * (ls[s][j] - 32) * L.CODEBOOK[np.array(c[s][j])]
                              for s in range(2) for j in range(8)])
        K = 512
    wh = oracle.dequant(fmt, np.frombuffer(g, np.uint8)[None, :], K)
    assert np.array_equal(wh[0], exp)


# --------------------------------------------------------------------------
# matvec
# --------------------------------------------------------------------------

def _xhat(x):
    q, d, _ = oracle.act_quant(x)
    return q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)


@pytest.mark.parametrize("fmt,K", [(0, 512), (1, 768), (2, 1024), (3, 768), (4, 512), (5, 1024), (6, 2048)])
def test_qmv_matches_library_matmul(fmt, K):
    w = _rand_w(37, K, seed=fmt)
    x = synth.activations(fmt, 5, K)
    W = oracle.quantize(fmt, w)
    y, sabs = oracle.qmv(fmt, W, x, K)
    wh = oracle.dequant(fmt, W, K)
    xh = _xhat(x)
    ref = xh @ wh.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(sabs, np.abs(xh) @ np.abs(wh).T, rtol=1e-12)
    assert np.all(sabs >= np.abs(y))


def test_qmv_closed_form_power_of_two():
    r = np.random.default_rng(3)
    K = 512
    q = r.integers(-127, 128, (2, 16, 32))
    W = np.stack([np.concatenate([np.frombuffer(L.pack_q8_0([0x3000] * 8, q[m, 8 * gi:8 * gi + 8]), np.uint8)
                                  for gi in range(2)]) for m in range(2)])   # d = 2^-3
    kx = r.integers(-127, 128, (3, K))
    kx[:, ::32] = 127
    x = (kx * 2.0 ** -2).astype(np.float32)    # d_x = 2^-2, q_x = kx
    y, _ = oracle.qmv(0, W, x, K)
    exact = (kx @ q.reshape(2, K).T) * 2.0 ** -5
    assert np.array_equal(y, exact.astype(np.float64))


def test_qmv_one_hot_row_selects_xhat():
    K = 256
    q = [[0] * 32 for _ in range(8)]
    q[5][7] = 1
    W = np.frombuffer(L.pack_q8_0([0x3C00] * 8, q), np.uint8)[None, :]
    x = synth.activations(11, 4, K)
    y, _ = oracle.qmv(0, W, x, K)
    assert np.array_equal(y[:, 0], _xhat(x)[:, 5 * 32 + 7])


def test_qmv_tokens_are_independent_and_threads_agree():
    K = 1024
    W = oracle.quantize(2, _rand_w(50, K))
    x = synth.activations(3, 6, K)
    y, _ = oracle.qmv(2, W, x, K)
    for t in range(6):
        yt, _ = oracle.qmv(2, W, x[t:t + 1], K)
        assert np.array_equal(yt[0], y[t])
    y4, _ = oracle.qmv(2, W, x, K, nthreads=4)
    assert np.array_equal(y4, y)


# --------------------------------------------------------------------------
# unquantized rows (F16, F32): plain conversions, no activation rule
# --------------------------------------------------------------------------

def _float_w(M, K, seed):
    r = np.random.default_rng(seed)
    w = (r.standard_normal((M, K)) * 0.05).astype(np.float32)
    # values at binary16 ties, subnormals, overflow, signed zeros
    ties = (np.arange(1, 64, dtype=np.uint16) * 37).view(np.float16).astype(np.float64)
    nxt = (np.arange(1, 64, dtype=np.uint16) * 37 + 1).view(np.float16).astype(np.float64)
    special = np.concatenate([(ties + nxt) / 2, [2.0 ** -24, 3 * 2.0 ** -26, 65519.0, 65520.0, 7e4, -0.0, 0.0]])
    w.reshape(-1)[:special.size] = special.astype(np.float32)
    return w


def test_f16_rows_are_numpy_binary16_and_f32_rows_the_bits():
    M, K = 5, 96
    w = _float_w(M, K, 1)
    W16 = oracle.quantize(oracle.F16, w)
    assert W16.shape == (M, 2 * K)
    assert np.array_equal(W16.view(np.uint16), w.astype(np.float16).view(np.uint16))
    d16 = oracle.dequant(oracle.F16, W16, K)
    assert np.array_equal(d16, w.astype(np.float16).astype(np.float64))
    W32 = oracle.quantize(oracle.F32, w)
    assert np.array_equal(W32, w.view(np.uint8).reshape(M, 4 * K))
    assert np.array_equal(oracle.dequant(oracle.F32, W32, K).view(np.uint64),
                          w.astype(np.float64).view(np.uint64))


def test_f16_conversion_is_the_nearest_binary16_by_brute_force():
    # every finite binary16 value; the nearest one to each weight, ties to
    # the even bit pattern (signed zeros compared by value)
    w = _float_w(1, 512, 2)[0]
    w = w[np.abs(w) < 65520.0]
    pats = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    vals = pats.view(np.float16).astype(np.float64)
    got = oracle.quantize(oracle.F16, np.pad(w, (0, (-w.size) % 32))[None, :]).view(np.uint16)[0][:w.size]
    for v, g in zip(w.astype(np.float64), got):
        dist = np.abs(vals - abs(v))
        best = np.flatnonzero(dist == dist.min())
        pick = best[0] if best.size == 1 else best[(pats[best] & 1) == 0][0]
        assert (g & 0x7FFF) == pats[pick]
        assert (g >> 15) == (1 if np.signbit(v) else 0)


@pytest.mark.parametrize("fmt", [oracle.F16, oracle.F32])
def test_float_qmv_uses_x_unquantized_exactly(fmt):
    from fractions import Fraction
    M, K, n = 3, 64, 2
    w = _float_w(M, K, 3)
    w[~np.isfinite(w.astype(np.float16))] = 1.0   # keep F16 rows finite
    # activations the activation rule would change (one large element per
    # block leaves the small ones a few codes wide)
    x = synth.activations(4, n, K)
    x[:, ::32] = 100.0
    x[:, 1] = 1e-3
    W = oracle.quantize(fmt, w)
    wh = oracle.dequant(fmt, W, K)
    y, sabs = oracle.qmv(fmt, W, x, K)
    for t in range(n):
        for m in range(M):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(wh[m], x[t]))
            assert abs(Fraction(float(y[t, m])) - exact) <= Fraction(2.0 ** -40) * abs(Fraction(float(sabs[t, m])))
            assert sabs[t, m] == pytest.approx(float(np.sum(np.abs(wh[m] * x[t].astype(np.float64)))), rel=1e-14)
    # the quantized-activation product is measurably different
    yq = _xhat(x) @ wh.T
    assert np.max(np.abs(yq - y)) > 1e-9 * np.max(sabs)


# --------------------------------------------------------------------------
# MoE
# --------------------------------------------------------------------------

E, H, F, TOPK = 6, 512, 512, 3


def _moe_pool(seed=5, identical=False):
    Wgu = np.stack([oracle.quantize(2, _rand_w(2 * F, H, seed=seed + (0 if identical else e)))
                    for e in range(E)])
    Wd = np.stack([oracle.quantize(1, _rand_w(H, F, seed=seed + 50 + (0 if identical else e)))
                   for e in range(E)])
    return Wgu, Wd


def test_synth_routing_properties():
    ids, g = synth.routing(9, 64, 128, 8)
    assert all(len(set(r)) == 8 for r in ids.tolist())
    assert ids.min() >= 0 and ids.max() < 128
    assert np.all(np.abs(g.sum(1, dtype=np.float64) - 1.0) <= 8 * 2.0 ** -24)
    assert np.all(g > 0)


def test_moe_top1_reduces_to_matvec_chain():
    Wgu, Wd = _moe_pool()
    x = synth.activations(1, 2, H)
    ids = np.array([[4], [1]], np.int32)
    gates = np.ones((2, 1), np.float32)
    out = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x)
    for t in range(2):
        e = ids[t, 0]
        gu, _ = oracle.qmv(2, Wgu[e], x[t:t + 1], H)
        g, u = gu[0, :F], gu[0, F:]
        h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
        assert np.array_equal(out["h32"][t], h)
        yd, _ = oracle.qmv(1, Wd[e], h[None, :], F)
        assert np.allclose(out["y"][t], yd[0], rtol=1e-13, atol=1e-15)


def test_moe_identical_experts_give_the_dense_ffn():
    Wgu, Wd = _moe_pool(identical=True)
    x = synth.activations(2, 3, H)
    ids, gates = synth.routing(4, 3, E, TOPK)
    out = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x)
    one = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids[:, :1], np.ones((3, 1), np.float32), x)
    gs = gates.astype(np.float64).sum(1, keepdims=True)
    assert np.allclose(out["y"], one["y"] * gs, rtol=1e-12, atol=1e-14)


def test_moe_expert_relabelling_is_bitwise_invariant():
    Wgu, Wd = _moe_pool()
    x = synth.activations(3, 4, H)
    ids, gates = synth.routing(6, 4, E, TOPK)
    perm = np.random.default_rng(0).permutation(E)       # new label of old expert e is perm[e]
    Wgu2 = np.empty_like(Wgu)
    Wd2 = np.empty_like(Wd)
    Wgu2[perm] = Wgu
    Wd2[perm] = Wd
    a = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x)["y"]
    b = oracle.moe(2, Wgu2, 1, Wd2, E, H, F, perm[ids].astype(np.int32), gates, x)["y"]
    assert np.array_equal(a, b)


def test_moe_invalid_slots_contribute_zero():
    Wgu, Wd = _moe_pool()
    x = synth.activations(4, 2, H)
    ids = np.array([[0, 9, 2], [3, 3, 1]], np.int32)      # out of range; duplicate
    gates = np.array([[0.5, 0.3, 0.2], [0.4, 0.35, 0.25]], np.float32)
    bad = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x)
    ok_ids = np.array([[0, 5, 2], [3, 4, 1]], np.int32)
    ok_g = gates.copy()
    ok_g[0, 1] = 0.0
    ok_g[1, 1] = 0.0
    ref = oracle.moe(2, Wgu, 1, Wd, E, H, F, ok_ids, ok_g, x)
    assert np.array_equal(bad["y"], ref["y"])
    assert not oracle.moe_slot_valid(ids, E, 0, 1) and not oracle.moe_slot_valid(ids, E, 1, 1)


def test_moe_thread_count_does_not_change_any_output():
    Wgu, Wd = _moe_pool()
    x = synth.activations(15, 5, H)
    ids, gates = synth.routing(16, 5, E, TOPK)
    a = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x, nthreads=1)
    for nt in (3, 0):
        b = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x, nthreads=nt)
        for k in a:
            assert np.array_equal(a[k], b[k]), k


def test_moe_slot_outputs_are_the_down_matvec_of_the_quantized_h():
    # o and its tolerance scale oabs, slot by slot, are the plain matvec of the
    # down weights with the slot's fp32 h (quantized by the activation rule)
    Wgu, Wd = _moe_pool()
    x = synth.activations(17, 3, H)
    ids, gates = synth.routing(18, 3, E, TOPK)
    out = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x, nthreads=2)
    for p, e in enumerate(ids.reshape(-1)):
        yo, so = oracle.qmv(1, Wd[e], out["h32"][p][None, :], F)
        assert np.array_equal(out["o"][p], yo[0]) and np.array_equal(out["oabs"][p], so[0])


def test_moe_given_h_reproduces_the_computed_path():
    Wgu, Wd = _moe_pool()
    x = synth.activations(5, 3, H)
    ids, gates = synth.routing(8, 3, E, TOPK)
    a = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x)
    b = oracle.moe(2, Wgu, 1, Wd, E, H, F, ids, gates, x, h_in=a["h32"])
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["hq"], b["hq"])


def test_q8_code_order_helper_follows_the_stated_rule():
    # the tests read the library's pre-quantized code order through this
    # helper; build a stored array from the rule element by element
    n, K = 2, 512
    nat = (np.arange(n * K).reshape(n, K) % 251).astype(np.int64)
    stored = np.zeros_like(nat)
    for t in range(n):
        for g in range(K // 256):
            for l in range(8):
                for p in range(32):
                    stored[t, g * 256 + (p // 16) * 128 + l * 16 + p % 16] = nat[t, g * 256 + l * 32 + p]
    assert np.array_equal(L.q8_codes_natural(stored), nat)


# --------------------------------------------------------------------------
# router: top-k selection and gate normalization
# --------------------------------------------------------------------------

@pytest.mark.parametrize("gating", [oracle.GATING_SOFTMAX, oracle.GATING_SIGMOID])
def test_route_select_matches_a_stable_sort(gating):
    # the picks are the first top_k of a lexicographic sort by (-logit,
    # index); logits drawn from few values so that ties are common
    r = np.random.default_rng(7 + gating)
    for E, k in [(8, 1), (8, 3), (64, 8), (300, 8)]:
        logits = r.integers(-3, 4, size=(20, E)).astype(np.float64) * 0.25
        ids, gates = oracle.route_select(logits, k, gating)
        for t in range(20):
            order = np.lexsort((np.arange(E), -logits[t]))
            assert np.array_equal(ids[t], order[:k])
            assert abs(gates[t].sum() - 1.0) < 1e-15 * k
            assert np.all(np.diff(gates[t]) <= 1e-15)  # gates follow the logits' order


def test_route_select_closed_forms():
    # softmax over the picked: logits ln 3, 0 -> 3/4, 1/4 (a third, smaller logit unpicked)
    ids, g = oracle.route_select(np.array([[np.log(3.0), 0.0, -5.0]]), 2, oracle.GATING_SOFTMAX)
    assert ids.tolist() == [[0, 1]] and np.allclose(g, [[0.75, 0.25]], rtol=0, atol=1e-15)
    # sigmoid: s(ln 3) = 3/4, s(0) = 1/2 -> 0.6, 0.4
    ids, g = oracle.route_select(np.array([[0.0, np.log(3.0), -np.log(3.0)]]), 2, oracle.GATING_SIGMOID)
    assert ids.tolist() == [[1, 0]] and np.allclose(g, [[0.6, 0.4]], rtol=0, atol=1e-15)
    # top-1 gives gate 1 and numpy's argmax (first maximum) in both modes
    r = np.random.default_rng(3)
    logits = r.standard_normal((50, 16))
    for gating in (0, 1):
        ids, g = oracle.route_select(logits, 1, gating)
        assert np.array_equal(ids[:, 0], logits.argmax(axis=1)) and np.all(g == 1.0)


def test_route_select_equals_renormalised_full_softmax():
    # the plain reading of "softmax gating, then normalise the picked weights"
    r = np.random.default_rng(11)
    logits = r.standard_normal((10, 128)) * 2
    ids, g = oracle.route_select(logits, 8, oracle.GATING_SOFTMAX)
    full = np.exp(logits - logits.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    pick = np.take_along_axis(full, ids.astype(np.int64), axis=1)
    assert np.allclose(g, pick / pick.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)


def test_route_relabelling_experts_permutes_the_picks():
    # permuting the router rows maps each pick through the permutation
    r = np.random.default_rng(5)
    E, H = 32, 512
    Wr = oracle.quantize(oracle.Q8_0, synth.weights(50, E, H))
    x = synth.activations(51, 6, H)
    perm = r.permutation(E)
    ids, g, _, _ = oracle.route(oracle.Q8_0, Wr, x, H, 4, oracle.GATING_SIGMOID)
    ids2, g2, _, _ = oracle.route(oracle.Q8_0, Wr[perm], x, H, 4, oracle.GATING_SIGMOID)
    inv = np.argsort(perm)
    assert np.array_equal(perm[ids2], ids) and np.array_equal(g, g2)
    assert np.array_equal(inv[ids], ids2)
