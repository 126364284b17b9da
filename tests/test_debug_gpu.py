"""The range-checked build (libqmv_debug.so: the same sources compiled with
QMV_DEBUG), a stand-in for a device memory checker.  Every global access of
its kernels is checked against the extent of its buffer as the host derives
it from the call's arguments, every shared-memory access against the CTA's
allocation; a failed check skips the access and sets QMV_DEVERR_RANGE.

  * Every kernel family, on tiny, ragged and tall shapes, runs through the
    debug library without a failed check, and its results are bitwise those
    of the release library (the checks change no arithmetic).
  * The checks are live: with the result buffers' extents handed to them a
    few elements short (qmv_debug_shrink_outputs), exactly the stores into
    those last elements are skipped and flagged, everything else is written
    as in the release build, and the next unshrunk call is clean again.  No
    access leaves its buffer in either case."""
import numpy as np
import pytest
import torch

from moe_matvec_gb300 import api, synth
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg(lib):
    return api.load_debug()


def flat(ts):
    if isinstance(ts, torch.Tensor):
        return [ts]
    out = []
    for t in ts:
        out += flat(t)
    return out


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def both(dbg, fn):
    """fn() through the release library, then through the debug one; returns
    (release results, debug results, the debug run's device error word)."""
    rel = flat(fn())
    torch.cuda.synchronize()
    with api.using(dbg):
        api.get_device_error()
        d = flat(fn())
        torch.cuda.synchronize()
        err = api.get_device_error()
    return rel, d, err


def check_same(dbg, fn, what, allowed=0):
    rel, d, err = both(dbg, fn)
    assert err & api.DEVERR_RANGE == 0, f"{what}: a range check failed in the debug build"
    assert err & ~allowed == 0, f"{what}: unexpected device error bits {err:#x}"
    for i, (a, b) in enumerate(zip(rel, d)):
        assert same_bits(a, b), f"{what}: result {i} differs between the release and debug builds"


def wq(fmt, M, K, seed):
    return api.quantize_weights(fmt, dev(synth.weights(seed, M, K)))


DENSE = [(0, 1, 256), (1, 2, 256), (2, 3, 512), (3, 5, 256), (4, 3, 256), (5, 2, 512), (6, 3, 1024),
         (7, 1, 32), (8, 2, 32), (0, 333, 1280), (1, 517, 2304), (2, 260, 1536), (7, 75, 1056),
         (8, 129, 544), (1, 7200, 512), (7, 4100, 512)]


@pytest.mark.parametrize("fmt,M,K", DENSE)
def test_matvec_in_range(dbg, fmt, M, K):
    W = wq(fmt, M, K, 200 + fmt + M)
    for n in (1, 2, 3, 5, 8, 16):
        x = dev(synth.activations(201 + n, n, K))
        check_same(dbg, lambda: api.run(fmt, W, x, M, K), f"qmv_run {fmt} {M}x{K} n{n}")


@pytest.mark.parametrize("fmt,M,K", [(0, 333, 1280), (1, 517, 2304), (2, 260, 1536), (1, 7200, 512),
                                     (7, 4100, 512)])
def test_splitk_residual_siblings_in_range(dbg, fmt, M, K):
    W = wq(fmt, M, K, 210 + fmt)
    groups = K // api.GROUP_WEIGHTS[fmt]
    for n in (1, 4, 16):
        x = dev(synth.activations(211 + n, n, K))
        r = dev(synth.activations(212 + n, n, M))
        for S in (1, 2, 3):
            if S > groups:
                continue
            check_same(dbg, lambda: api.splitk_run(fmt, W, x, M, K, n_split=S), f"splitk {fmt} n{n} S{S}")
            check_same(dbg, lambda: api.run_residual(fmt, W, x, r, M, K, n_split=S), f"residual {fmt} n{n} S{S}")
        check_same(dbg, lambda: api.run_siblings([(fmt, W, M), (fmt, W[: M // 2 + 1], M // 2 + 1)], x, K),
                   f"siblings {fmt} n{n}")


def test_static_splitk_in_range(dbg):
    M, K = 512, 8192
    W = wq(0, M, K, 220)
    for n in (1, 5):
        x = dev(synth.activations(221 + n, n, K))
        check_same(dbg, lambda: api.splitk_run_static(0, W, x, M, K, n_split=4), f"static n{n}")


def test_quantizers_in_range(dbg):
    for fmt, K in ((0, 256), (1, 512), (2, 512), (3, 256), (4, 256), (5, 512), (6, 1024), (7, 64), (8, 32)):
        w = dev(synth.weights(230 + fmt, 37, K))
        check_same(dbg, lambda: api.quantize_weights(fmt, w), f"quantize_weights {fmt}")
    for n, K in ((1, 256), (3, 1024), (64, 512)):
        x = dev(synth.activations(231 + n, n, K))
        check_same(dbg, lambda: api.quantize_act(x), f"quantize_act n{n}")


def test_router_in_range(dbg):
    E, H, top_k = 96, 1024, 6
    Wr = wq(0, E, H, 240)
    for n in (1, 7, 64):
        x = dev(synth.activations(241 + n, n, H))
        check_same(dbg, lambda: api.route_run(0, Wr, x, E, H, top_k), f"route n{n}")


def pool(fmt_gu, fmt_d, E, H, F, seed):
    Wgu = torch.stack([wq(fmt_gu, 2 * F, H, seed + 2 * e) for e in range(E)])
    Wd = torch.stack([wq(fmt_d, H, F, seed + 2 * e + 1) for e in range(E)])
    return api.moe_experts(E, H, F, fmt_gu, fmt_d, Wgu, Wd)


@pytest.mark.parametrize("fmt_gu,fmt_d,F", [(2, 1, 1536), (0, 2, 512), (1, 0, 768)])
def test_moe_in_range(dbg, fmt_gu, fmt_d, F):
    E, H, top_k = 16, 512, 4
    ex = pool(fmt_gu, fmt_d, E, H, F, 250 + F)
    for n in (1, 3, 4, 16, 64):
        ids, gates = synth.routing(251 + n, n, E, top_k)
        ids[-1, 0] = -1  # a slot that does not route (flagged, adds nothing)
        ids_d, gates_d, x = dev(ids), dev(gates), dev(synth.activations(252 + n, n, H))
        check_same(dbg, lambda: api.moe_run(ex, ids_d, gates_d, x), f"moe {fmt_gu}/{fmt_d} n{n}",
                   allowed=api.DEVERR_EXPERT_RANGE)
        api.get_device_error()


def test_moe_prefill_in_range(dbg):
    E, H, F, top_k = 8, 512, 256, 2
    ex = pool(2, 1, E, H, F, 260)
    for n in (70, 300):
        ids, gates = synth.routing(261 + n, n, E, top_k)
        ids_d, gates_d, x = dev(ids), dev(gates), dev(synth.activations(262 + n, n, H))
        check_same(dbg, lambda: api.moe_prefill_run(ex, ids_d, gates_d, x), f"prefill n{n}")


# ---- the checks are live: result extents handed to them a few elements short ----

def random_like(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    nb = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    return torch.randint(0, 256, (nb,), dtype=torch.uint8, generator=g).cuda().view(dtype).view(shape)


def check_tail_skipped(dbg, call, shape, dtype, cut, keep, what):
    """call(out) writes `out`; through the debug library with the extents
    `cut` elements (of the kernel's stores) short, the flat output's last
    `keep` elements (the stores that then fail their checks) keep their start
    bits, the rest is the release result, and the range bit is set; then an
    unshrunk call is clean."""
    ref = random_like(shape, dtype, 1)
    call(ref)
    torch.cuda.synchronize()
    out = random_like(shape, dtype, 2)
    start = out.clone()
    with api.using(dbg):
        api.get_device_error()
        api.debug_shrink_outputs(cut)
        try:
            call(out)
            torch.cuda.synchronize()
        finally:
            api.debug_shrink_outputs(0)
        err = api.get_device_error()
        assert err & api.DEVERR_RANGE, f"{what}: the shortened extent raised no range error"
        fo, fs, fr = out.reshape(-1), start.reshape(-1), ref.reshape(-1)
        assert same_bits(fo[-keep:], fs[-keep:]), f"{what}: a store past the checked extent was not skipped"
        assert same_bits(fo[:-keep], fr[:-keep]), f"{what}: stores inside the checked extent differ"
        again = random_like(shape, dtype, 3)
        call(again)
        torch.cuda.synchronize()
        assert api.get_device_error() == 0, f"{what}: the check still fails after the extent was restored"
        assert same_bits(again, ref)


@pytest.mark.parametrize("fmt,M,K,n,S", [(1, 300, 1024, 2, 1), (2, 260, 1536, 3, 1), (1, 7200, 512, 8, 1),
                                         (7, 4100, 512, 16, 1), (0, 333, 1280, 5, 3), (8, 129, 544, 16, 1)])
def test_dense_checks_are_live(dbg, fmt, M, K, n, S):
    W = wq(fmt, M, K, 270 + fmt)
    x = dev(synth.activations(271, n, K))
    check_tail_skipped(dbg, lambda out: api.splitk_run(fmt, W, x, M, K, n_split=S, out=out), (n, M),
                       torch.float32, 5, 5, f"matvec {fmt} {M}x{K} n{n} S{S}")


def test_moe_and_quantizer_checks_are_live(dbg):
    E, H, F, top_k, n = 16, 512, 1536, 4, 4
    ex = pool(2, 1, E, H, F, 280)
    ids, gates = synth.routing(281, n, E, top_k)
    ids_d, gates_d, x = dev(ids), dev(gates), dev(synth.activations(282, n, H))
    # the combine stores 4 outputs at a time: 3 short fails the last store
    check_tail_skipped(dbg, lambda out: api.moe_run(ex, ids_d, gates_d, x, out=out), (n, H), torch.float32, 3, 4,
                       "moe combine")
    w = dev(synth.weights(283, 9, 256))
    # F32 rows: one store per weight; Q4_K: one 144-byte group per store
    check_tail_skipped(dbg, lambda out: api.quantize_weights(8, w, out=out), (9, 256), torch.float32, 3, 3,
                       "F32 rows")
    check_tail_skipped(dbg, lambda out: api.quantize_weights(1, w, out=out), (9, 144), torch.uint8, 5, 144,
                       "Q4_K groups")
