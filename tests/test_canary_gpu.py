"""Canary bytes around every output and workspace buffer of every entry point
(a stand-in for a device memory checker).

Each result or workspace buffer is a view into a larger allocation whose
4 KiB guard bands on both sides hold seeded random bytes, and whose own bytes
start random too.  After each call: the guard bands are unchanged (no store
past either end), the result is bitwise equal to the same call into plain
buffers (every element was written: none still holds its random start), and
the inputs are unchanged (no stray store into them).  Shapes include the tiny
ones (1 to 3 rows, the smallest K of each format), ragged tails, and every
kernel family: fused and pre-quantized staging, split-K partials and their
reduction, the tensor-core Q4_K and F16 matvecs, siblings, the residual add,
the router, the MoE decode layer and the MoE prefill layer."""
import numpy as np
import pytest
import torch

from moe_matvec_gb300 import api, synth
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

GUARD = 4096


class Guarded:
    """A tensor of `shape` / `dtype` between two guard bands of random bytes."""

    def __init__(self, shape, dtype, seed):
        self.shape, self.dtype = tuple(shape), dtype
        self.nbytes = int(np.prod(self.shape)) * torch.empty((), dtype=dtype).element_size()
        g = torch.Generator().manual_seed(seed)
        host = torch.randint(0, 256, (2 * GUARD + self.nbytes,), dtype=torch.uint8, generator=g)
        self.buf = host.cuda()
        self.start = self.buf.clone()
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(self.shape)

    def check_guards(self, what):
        torch.cuda.synchronize()
        lo_ok = torch.equal(self.buf[:GUARD], self.start[:GUARD])
        hi_ok = torch.equal(self.buf[GUARD + self.nbytes:], self.start[GUARD + self.nbytes:])
        assert lo_ok and hi_ok, f"{what}: a store landed in the {'low' if not lo_ok else 'high'} guard band"


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def snapshot(*ts):
    return [t.clone() for t in ts]


def unchanged(before, *ts):
    torch.cuda.synchronize()
    return all(same_bits(a, b) for a, b in zip(before, ts))


def weights_dev(fmt, M, K, seed):
    return api.quantize_weights(fmt, dev(synth.weights(seed, M, K)))


# (format, M, K): tiny matrices at the smallest K of each format, ragged
# tiles, and tall ones that take the tensor-core kernels at 8 / 16 tokens
DENSE = [(0, 1, 256), (1, 2, 256), (2, 3, 512), (3, 1, 256), (4, 3, 256), (5, 2, 512), (6, 3, 1024),
         (7, 1, 32), (8, 2, 32), (0, 333, 1280), (1, 517, 2304), (2, 260, 1536), (7, 75, 1056),
         (8, 129, 544), (1, 7200, 512), (7, 4100, 512)]


@pytest.mark.parametrize("fmt,M,K", DENSE)
@pytest.mark.parametrize("n", [1, 3, 8, 16])
def test_matvec_writes_only_its_output(lib, fmt, M, K, n):
    W = weights_dev(fmt, M, K, 10 * fmt + M)
    x = dev(synth.activations(M + n, n, K))
    before = snapshot(W, x)
    ref = api.run(fmt, W, x, M, K)
    y = Guarded((n, M), torch.float32, seed=M * 31 + n)
    api.run(fmt, W, x, M, K, out=y.t)
    y.check_guards("qmv_run y")
    assert same_bits(y.t, ref), "qmv_run: the guarded output differs from a plain call's"
    assert unchanged(before, W, x), "qmv_run changed an input"


@pytest.mark.parametrize("fmt,M,K", [(0, 333, 1280), (1, 517, 2304), (2, 260, 1536), (1, 7200, 512)])
@pytest.mark.parametrize("n", [4, 9, 16])
@pytest.mark.parametrize("n_split", [1, 2, 3])
def test_splitk_writes_only_its_output_and_workspace(lib, fmt, M, K, n, n_split):
    groups = K // api.GROUP_WEIGHTS[fmt]
    if n_split > groups:
        pytest.skip("more splits than groups")
    W = weights_dev(fmt, M, K, 7 * fmt + M)
    x = dev(synth.activations(M + 3 * n, n, K))
    before = snapshot(W, x)
    wsb = api.splitk_workspace_fast_bytes(M, K, n, n_split)
    ref = api.splitk_run(fmt, W, x, M, K, n_split=n_split,
                         ws=torch.empty(max(16, wsb), dtype=torch.uint8, device="cuda"))
    y = Guarded((n, M), torch.float32, seed=1 + n_split)
    ws = Guarded((max(16, wsb),), torch.uint8, seed=2 + n_split)
    api.splitk_run(fmt, W, x, M, K, n_split=n_split, ws=ws.t, out=y.t)
    y.check_guards("qmv_splitk_run y")
    ws.check_guards("qmv_splitk_run workspace")
    assert same_bits(y.t, ref)
    assert unchanged(before, W, x)


@pytest.mark.parametrize("n", [1, 5])
def test_static_splitk_writes_only_its_output(lib, n):
    M, K = 512, 8192
    W = weights_dev(0, M, K, 44)
    x = dev(synth.activations(45, n, K))
    ref = api.splitk_run(0, W, x, M, K, n_split=4)
    y = Guarded((n, M), torch.float32, seed=46)
    api.splitk_run_static(0, W, x, M, K, n_split=4, out=y.t)
    y.check_guards("qmv_splitk_run_static y")
    assert same_bits(y.t, ref)


@pytest.mark.parametrize("n,n_split", [(1, 1), (3, 2), (6, 1), (6, 3)])
def test_residual_writes_only_its_output(lib, n, n_split):
    fmt, M, K = 1, 700, 2048
    W = weights_dev(fmt, M, K, 61)
    x = dev(synth.activations(62, n, K))
    r = dev(synth.activations(63, n, M))
    wsb = max(16, api.splitk_workspace_fast_bytes(M, K, n, n_split))
    ref = api.run_residual(fmt, W, x, r, M, K, n_split=n_split)
    before = snapshot(W, x, r)
    y = Guarded((n, M), torch.float32, seed=64)
    ws = Guarded((wsb,), torch.uint8, seed=65)
    api.run_residual(fmt, W, x, r, M, K, out=y.t, n_split=n_split, ws=ws.t)
    y.check_guards("qmv_run_residual y")
    ws.check_guards("qmv_run_residual workspace")
    assert same_bits(y.t, ref)
    assert unchanged(before, W, x, r)
    # in place: y += What Xhat in a guarded copy of r
    yi = Guarded((n, M), torch.float32, seed=66)
    yi.t.copy_(r)
    api.run_residual(fmt, W, x, yi.t, M, K, out=yi.t, n_split=n_split, ws=ws.t)
    yi.check_guards("qmv_run_residual in place")
    assert same_bits(yi.t, ref)


@pytest.mark.parametrize("n", [2, 5])
def test_siblings_write_only_their_outputs(lib, n):
    K = 1024
    mats = [(1, weights_dev(1, 300, K, 71), 300), (2, weights_dev(2, 64, K, 72), 64),
            (7, weights_dev(7, 40, K, 73), 40)]
    x = dev(synth.activations(74, n, K))
    refs = [api.run(f, W, x, M, K) for f, W, M in mats]
    outs = [Guarded((n, M), torch.float32, seed=75 + i) for i, (_, _, M) in enumerate(mats)]
    ws = Guarded((max(16, api.act_q8_bytes(K, n)),), torch.uint8, seed=79)
    api.run_siblings(mats, x, K, outs=[o.t for o in outs], ws=ws.t)
    for i, o in enumerate(outs):
        o.check_guards(f"qmv_run_siblings y{i}")
        assert same_bits(o.t, refs[i])
    ws.check_guards("qmv_run_siblings workspace")


def test_quantizers_write_only_their_outputs(lib):
    for fmt, K in ((0, 256), (1, 512), (2, 512), (3, 256), (4, 256), (5, 512), (6, 1024), (7, 64), (8, 32)):
        for M in (1, 3, 37):
            w = dev(synth.weights(90 + fmt, M, K))
            before = snapshot(w)
            ref = api.quantize_weights(fmt, w)
            out = Guarded(tuple(ref.shape), torch.uint8, seed=91 + fmt)
            api.quantize_weights(fmt, w, out=out.t)
            out.check_guards(f"qmv_quantize_weights format {fmt}")
            assert same_bits(out.t, ref)
            assert unchanged(before, w)
    # the activation quantizer, called through the C ABI with guarded outputs
    for n, K in ((1, 256), (3, 1024), (64, 512)):
        x = dev(synth.activations(95 + n, n, K))
        q0, d0, s0 = api.quantize_act(x)
        q = Guarded((n, K), torch.int8, seed=96)
        d = Guarded((n, K // 32), torch.float32, seed=97)
        s = Guarded((n, K // 32), torch.int32, seed=98)
        rc = api.load().qmv_quantize_act(x.data_ptr(), K, n, q.t.data_ptr(), d.t.data_ptr(), s.t.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        for g, ref, nm in ((q, q0, "q"), (d, d0, "d"), (s, s0, "s")):
            g.check_guards(f"qmv_quantize_act {nm}")
            assert same_bits(g.t, ref)


@pytest.mark.parametrize("n", [1, 7, 64])
def test_router_writes_only_its_outputs(lib, n):
    E, H, top_k = 96, 1024, 6
    Wr = weights_dev(0, E, H, 101)
    x = dev(synth.activations(102, n, H))
    ids0, gates0, logits0 = api.route_run(0, Wr, x, E, H, top_k)
    lg = Guarded((n, E), torch.float32, seed=103)
    ids = Guarded((n, top_k), torch.int32, seed=104)
    gates = Guarded((n, top_k), torch.float32, seed=105)
    api.route_run(0, Wr, x, E, H, top_k, logits=lg.t, ids=ids.t, gates=gates.t)
    for g, ref, nm in ((lg, logits0, "logits"), (ids, ids0, "ids"), (gates, gates0, "gates")):
        g.check_guards(f"moe_route_run {nm}")
        assert same_bits(g.t, ref)


def moe_pool(fmt_gu, fmt_d, E, H, F, seed):
    Wgu = torch.stack([weights_dev(fmt_gu, 2 * F, H, seed + 2 * e) for e in range(E)])
    Wd = torch.stack([weights_dev(fmt_d, H, F, seed + 2 * e + 1) for e in range(E)])
    return Wgu, Wd


@pytest.mark.parametrize("fmt_gu,fmt_d,F", [(2, 1, 1536), (0, 2, 512), (1, 0, 768)])
@pytest.mark.parametrize("n", [1, 3, 4, 16, 64])
def test_moe_writes_only_its_output_and_workspace(lib, fmt_gu, fmt_d, F, n):
    E, H, top_k = 16, 512, 4
    Wgu, Wd = moe_pool(fmt_gu, fmt_d, E, H, F, 110 + F)
    ex = api.moe_experts(E, H, F, fmt_gu, fmt_d, Wgu, Wd)
    ids_np, gates_np = synth.routing(120 + n, n, E, top_k)
    ids_np[0, -1] = E + 3  # an id out of range: its slot adds nothing (and flags the error word)
    ids, gates, x = dev(ids_np), dev(gates_np), dev(synth.activations(121 + n, n, H))
    before = snapshot(Wgu, Wd, ids, gates, x)
    wsb = api.moe_workspace_bytes(ex, n, top_k)
    ref = api.moe_run(ex, ids, gates, x, ws=torch.empty(wsb, dtype=torch.uint8, device="cuda"))
    y = Guarded((n, H), torch.float32, seed=122)
    ws = Guarded((wsb,), torch.uint8, seed=123)
    api.moe_run(ex, ids, gates, x, ws=ws.t, out=y.t)
    y.check_guards("moe_qmv_run y")
    ws.check_guards("moe_qmv_run workspace")
    assert same_bits(y.t, ref)
    assert unchanged(before, Wgu, Wd, ids, gates, x)
    api.get_device_error()  # clear the flag the bad id raised


@pytest.mark.parametrize("n", [70, 300])
def test_moe_prefill_writes_only_its_output_and_workspace(lib, n):
    E, H, F, top_k = 8, 512, 256, 2
    Wgu, Wd = moe_pool(2, 1, E, H, F, 130)
    ex = api.moe_experts(E, H, F, 2, 1, Wgu, Wd)
    ids_np, gates_np = synth.routing(131 + n, n, E, top_k)
    ids, gates, x = dev(ids_np), dev(gates_np), dev(synth.activations(132 + n, n, H))
    before = snapshot(Wgu, Wd, ids, gates, x)
    wsb = api.moe_prefill_workspace_bytes(ex, n, top_k)
    ref = api.moe_prefill_run(ex, ids, gates, x, ws=torch.empty(wsb, dtype=torch.uint8, device="cuda"))
    y = Guarded((n, H), torch.float32, seed=133)
    ws = Guarded((wsb,), torch.uint8, seed=134)
    api.moe_prefill_run(ex, ids, gates, x, ws=ws.t, out=y.t)
    y.check_guards("moe_qmv_prefill_run y")
    ws.check_guards("moe_qmv_prefill_run workspace")
    assert same_bits(y.t, ref)
    assert unchanged(before, Wgu, Wd, ids, gates, x)
