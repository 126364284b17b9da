"""GPU parity of the expert-grouped MoE decode layer against the oracle.

Graded stage by stage, because the requantization of h can flip a code when
the GPU's fp32 h differs from the oracle's in the last bits:
  (i)   h (SwiGLU output) within the propagated gate/up tolerance;
  (ii)  q8(h) bit-exact against the activation rule applied to the GPU's h;
  (iii) down projections and the combine against the oracle fed the GPU's h,
        within 1e-5 * sum |What x Hhat| (times the gates for y);
and end to end against the fully independent oracle within the matvec bound
plus the exact effect of those flips: sum_k |g_k| sum_i |What_i| |dHhat_i|,
dHhat the difference between the requantized h of the two paths."""
import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import api, synth
from tests.gpu_util import TOL, assert_within, dev

pytestmark = pytest.mark.gpu


def make_pool(fmt_gu, fmt_d, E, H, F, seed, experts=None):
    """Quantized pools; experts outside `experts` (if given) are left zero."""
    rb_gu, rb_d = oracle.row_bytes(fmt_gu, H), oracle.row_bytes(fmt_d, F)
    Wgu = np.zeros((E, 2 * F, rb_gu), np.uint8)
    Wd = np.zeros((E, H, rb_d), np.uint8)
    for e in (range(E) if experts is None else experts):
        Wgu[e] = oracle.quantize(fmt_gu, synth.weights(seed + 2 * e, 2 * F, H))
        Wd[e] = oracle.quantize(fmt_d, synth.weights(seed + 2 * e + 1, H, F))
    return Wgu, Wd


def run_gpu(fmt_gu, fmt_d, Wgu, Wd, E, H, F, ids, gates, x):
    n, top_k = ids.shape
    Wgu_d, Wd_d = dev(Wgu), dev(Wd)
    ex = api.moe_experts(E, H, F, fmt_gu, fmt_d, Wgu_d, Wd_d)
    ws = torch.zeros(api.moe_workspace_bytes(ex, n, top_k), dtype=torch.uint8, device="cuda")
    y = api.moe_run(ex, dev(ids), dev(gates), dev(x), ws=ws)
    torch.cuda.synchronize()
    off = api.moe_workspace_offsets(ex, n, top_k)
    S = n * top_k
    w = ws.cpu().numpy()
    out = dict(
        y=y.cpu().numpy(),
        h=w[off[0]:off[0] + S * F * 4].view(np.float32).reshape(S, F),
        hq=w[off[1]:off[1] + S * F].view(np.int8).reshape(S, F),
        hd=w[off[2]:off[2] + S * F // 32 * 4].view(np.float32).reshape(S, F // 32),
        hs=w[off[3]:off[3] + S * F // 32 * 4].view(np.int32).reshape(S, F // 32),
        o=w[off[4]:off[4] + S * H * 4].view(np.float32).reshape(S, H))
    return out, (Wgu_d, Wd_d, ex)


def valid_mask(ids, E):
    n, k = ids.shape
    return np.array([[oracle.moe_slot_valid(ids, E, t, j) for j in range(k)] for t in range(n)]).reshape(-1)


def flip_bound(fmt_d, Wd, F, ids_s, gates_s, valid, hq_g, hd_g, hq_r, hd_r):
    """Largest change of y that the requantized h of the GPU path (codes hq_g,
    scales hd_g: the activation rule on the GPU's h) can cause against the
    oracle's own (hq_r, hd_r): per token, sum_k |g_k| sum_i |Wdown_e[m][i]| *
    |Hhat_g[i] - Hhat_r[i]|.  Zero where the two requantizations agree; a
    code flipped by one adds d_h |What_i|, a changed block scale its whole
    block."""
    n, top_k = ids_s.shape
    H = Wd.shape[1]
    out = np.zeros((n, H))
    vslots = np.nonzero(valid)[0]
    for j, p in enumerate(vslots):
        hg = hq_g[j].astype(np.float64) * np.repeat(hd_g[j].astype(np.float64), 32)
        hr = hq_r[j].astype(np.float64) * np.repeat(hd_r[j].astype(np.float64), 32)
        dh = np.abs(hg - hr)
        cols = np.nonzero(dh)[0]
        if cols.size == 0:
            continue
        e = ids_s.reshape(-1)[p]
        What = np.abs(oracle.dequant(fmt_d, Wd[e], F))
        out[p // top_k] += abs(float(gates_s.reshape(-1)[p])) * (What[:, cols] @ dh[cols])
    return out


def check_stagewise(fmt_gu, fmt_d, Wgu, Wd, E, H, F, ids, gates, x, g, tokens=None):
    """Compare GPU outputs g (run on all tokens) for `tokens` (default all)."""
    n, top_k = ids.shape
    tokens = np.arange(n) if tokens is None else np.asarray(tokens)
    slots = (tokens[:, None] * top_k + np.arange(top_k)[None, :]).reshape(-1)
    ids_s, gates_s, x_s = ids[tokens], gates[tokens], x[tokens]
    valid = valid_mask(ids_s, E)
    ref = oracle.moe(fmt_gu, Wgu, fmt_d, Wd, E, H, F, ids_s, gates_s, x_s, nthreads=0)
    # (i) h within the propagated gate/up tolerance
    gr, ur = ref["g"][valid], ref["u"][valid]
    sig = 1.0 / (1.0 + np.exp(-gr))
    silu, dsilu = gr * sig, sig * (1.0 + gr * (1.0 - sig))
    h_gpu = g["h"][slots][valid].astype(np.float64)
    h_ref = silu * ur
    bound = (np.abs(dsilu * ur) * TOL * ref["gabs"][valid] + np.abs(silu) * TOL * ref["uabs"][valid]
             + 8 * np.spacing(np.abs(h_ref).astype(np.float32)).astype(np.float64) + 1e-30)
    bad = np.abs(h_gpu - h_ref) > bound
    assert not bad.any(), f"h: {bad.sum()} elements out of bound"
    # (ii) q8(h) bit-exact against the activation rule on the GPU's h
    q, d, s = oracle.act_quant(g["h"][slots][valid])
    assert np.array_equal(g["hq"][slots][valid], q)
    assert np.array_equal(g["hd"][slots][valid].view(np.uint32), d.view(np.uint32))
    assert np.array_equal(g["hs"][slots][valid], s)
    # (iii) down + combine against the oracle fed the GPU's h
    h_in = g["h"][slots].copy()
    h_in[~valid] = 0.0
    ref2 = oracle.moe(fmt_gu, Wgu, fmt_d, Wd, E, H, F, ids_s, gates_s, x_s, h_in=h_in, nthreads=0)
    assert_within(g["o"][slots][valid], ref2["o"][valid], ref2["oabs"][valid], what="o")
    assert_within(g["y"][tokens], ref2["y"], ref2["ybound"] * 1.1, what="y given h")
    # end to end against the independent oracle: the matvec bound plus the
    # exact effect of the codes (or scales) that the requantization of the
    # GPU's h decided differently from the oracle's own h
    fb = flip_bound(fmt_d, Wd, F, ids_s, gates_s, valid, q, d, ref["hq"][valid], ref["hd"][valid])
    slack = 1.1 * TOL * (ref["ybound"] + fb) + 1.001 * fb
    assert_within(g["y"][tokens], ref["y"], slack / TOL, what="y end to end")
    return int((q != ref["hq"][valid]).sum())


SMALL = [(2, 1, 8, 512, 512, 3, 1), (2, 1, 8, 512, 512, 3, 5), (2, 1, 6, 1024, 768, 2, 17),
         (1, 0, 5, 768, 512, 4, 9), (0, 2, 9, 512, 1024, 8, 64), (2, 1, 16, 512, 256, 1, 64),
         (1, 1, 3, 256, 256, 3, 64)]


@pytest.mark.parametrize("fmt_gu,fmt_d,E,H,F,top_k,n", SMALL)
def test_moe_small_stagewise(lib, fmt_gu, fmt_d, E, H, F, top_k, n):
    seed = 500 + E + H + F + n
    Wgu, Wd = make_pool(fmt_gu, fmt_d, E, H, F, seed)
    ids, gates = synth.routing(seed, n, E, top_k)
    x = synth.activations(seed, n, H)
    g, _ = run_gpu(fmt_gu, fmt_d, Wgu, Wd, E, H, F, ids, gates, x)
    check_stagewise(fmt_gu, fmt_d, Wgu, Wd, E, H, F, ids, gates, x, g)
    assert lib.get_device_error() == 0


@pytest.mark.parametrize("E,top_k,n", [(300, 4, 24), (512, 2, 20), (300, 4, 3), (512, 8, 2)])
def test_moe_many_experts(lib, E, top_k, n):
    # many experts; below 4 tokens more than one round of the routing scan
    # covers (32 per warp, 9 warps): the slot, group and work prefixes carry
    # across rounds
    H = F = 256
    ids, gates = synth.routing(900 + E, n, E, top_k)
    experts = sorted(set(ids.reshape(-1).tolist()))
    Wgu, Wd = make_pool(0, 1, E, H, F, 901 + E, experts=experts)
    x = synth.activations(902 + E, n, H)
    g, _ = run_gpu(0, 1, Wgu, Wd, E, H, F, ids, gates, x)
    check_stagewise(0, 1, Wgu, Wd, E, H, F, ids, gates, x, g)
    assert lib.get_device_error() == 0


def test_moe_all_tokens_on_the_same_experts(lib):
    # every token picks the same experts: one group per expert overflows the
    # per-group token count and is split into several groups
    E, H, F, top_k, n = 4, 512, 512, 2, 40
    Wgu, Wd = make_pool(2, 1, E, H, F, 77)
    ids = np.tile(np.array([[2, 0]], np.int32), (n, 1))
    gates = np.tile(np.array([[0.7, 0.3]], np.float32), (n, 1))
    x = synth.activations(78, n, H)
    g, _ = run_gpu(2, 1, Wgu, Wd, E, H, F, ids, gates, x)
    check_stagewise(2, 1, Wgu, Wd, E, H, F, ids, gates, x, g)


def test_moe_descriptor_keeps_its_weights_alive(lib):
    # the descriptor is built from temporary device tensors and other tensors
    # are allocated afterwards: the binding keeps the weights referenced, so
    # their memory is not recycled under the C struct's raw addresses
    E, H, F, top_k, n = 6, 512, 512, 2, 8
    Wgu, Wd = make_pool(2, 1, E, H, F, 95)
    ex = api.moe_experts(E, H, F, 2, 1, dev(Wgu), dev(Wd))
    filler = [torch.full((Wgu.size // 4,), 7.0, device="cuda") for _ in range(4)]
    ids, gates = synth.routing(96, n, E, top_k)
    x = synth.activations(97, n, H)
    ws = torch.zeros(api.moe_workspace_bytes(ex, n, top_k), dtype=torch.uint8, device="cuda")
    y = api.moe_run(ex, dev(ids), dev(gates), dev(x), ws=ws)
    torch.cuda.synchronize()
    off = api.moe_workspace_offsets(ex, n, top_k)
    S, w = n * top_k, ws.cpu().numpy()
    g = dict(y=y.cpu().numpy(),
             h=w[off[0]:off[0] + S * F * 4].view(np.float32).reshape(S, F),
             hq=w[off[1]:off[1] + S * F].view(np.int8).reshape(S, F),
             hd=w[off[2]:off[2] + S * F // 32 * 4].view(np.float32).reshape(S, F // 32),
             hs=w[off[3]:off[3] + S * F // 32 * 4].view(np.int32).reshape(S, F // 32),
             o=w[off[4]:off[4] + S * H * 4].view(np.float32).reshape(S, H))
    check_stagewise(2, 1, Wgu, Wd, E, H, F, ids, gates, x, g)
    del filler


def test_moe_relabelling_experts_is_bitwise_invariant(lib):
    E, H, F, top_k, n = 12, 512, 512, 4, 16
    Wgu, Wd = make_pool(2, 1, E, H, F, 90)
    ids, gates = synth.routing(91, n, E, top_k)
    x = synth.activations(92, n, H)
    a, _ = run_gpu(2, 1, Wgu, Wd, E, H, F, ids, gates, x)
    perm = np.random.default_rng(3).permutation(E)
    Wgu2, Wd2 = np.empty_like(Wgu), np.empty_like(Wd)
    Wgu2[perm], Wd2[perm] = Wgu, Wd
    b, _ = run_gpu(2, 1, Wgu2, Wd2, E, H, F, perm[ids].astype(np.int32), gates, x)
    assert np.array_equal(a["y"], b["y"])


def test_moe_invalid_ids_contribute_zero_and_flag(lib):
    E, H, F = 6, 512, 512
    Wgu, Wd = make_pool(2, 1, E, H, F, 60)
    ids = np.array([[0, 9, 2], [3, 3, 1], [-1, 4, 5]], np.int32)
    gates = np.array([[0.5, 0.3, 0.2], [0.4, 0.35, 0.25], [0.2, 0.3, 0.5]], np.float32)
    x = synth.activations(61, 3, H)
    assert lib.get_device_error() == 0
    g, _ = run_gpu(2, 1, Wgu, Wd, E, H, F, ids, gates, x)
    err = lib.get_device_error()
    assert err == (api.DEVERR_EXPERT_RANGE | api.DEVERR_EXPERT_DUP)
    assert lib.get_device_error() == 0          # read clears it
    check_stagewise(2, 1, Wgu, Wd, E, H, F, ids, gates, x, g)


_POOL = {}


def full_pool(seed=3000, n_base=4):
    """The full-size expert pool (128 experts, IQ4_XS gate/up 3072 x 4096,
    Q4_K down 4096 x 1536), every expert distinct: expert e holds the rows of
    base set e mod n_base (quantized by the oracle) in its own random order,
    gate and up rows permuted separately.  Cached with its device copy."""
    if "pool" not in _POOL:
        c = synth.MOE_CASE
        E, H, F = c.n_experts, c.hidden, c.ffn
        base_gu = [oracle.quantize(c.fmt_gate_up, synth.weights(seed + 2 * b, 2 * F, H)) for b in range(n_base)]
        base_d = [oracle.quantize(c.fmt_down, synth.weights(seed + 2 * b + 1, H, F)) for b in range(n_base)]
        r = np.random.default_rng(seed)
        Wgu = np.empty((E, 2 * F, base_gu[0].shape[1]), np.uint8)
        Wd = np.empty((E, H, base_d[0].shape[1]), np.uint8)
        for e in range(E):
            b = e % n_base
            Wgu[e, :F] = base_gu[b][r.permutation(F)]
            Wgu[e, F:] = base_gu[b][F + r.permutation(F)]
            Wd[e] = base_d[b][r.permutation(H)]
        _POOL["pool"] = (Wgu, Wd, dev(Wgu), dev(Wd))
    return _POOL["pool"]


@pytest.mark.parametrize("n_idx,n", list(enumerate(synth.MOE_CASE.n_toks)))
def test_moe_full_size_all_tokens(lib, n_idx, n):
    # every token of the full-size layer at each benchmarked batch, in the
    # launch configuration the benchmark times: at 64 tokens several experts
    # receive more tokens than a group holds, so their groups are split
    c = synth.MOE_CASE
    seed = synth.seed_for(c.index, 0, n_idx)
    ids, gates = synth.routing(seed, n, c.n_experts, c.top_k)
    x = synth.activations(seed, n, c.hidden)
    Wgu, Wd, Wgu_d, Wd_d = full_pool()
    ex = api.moe_experts(c.n_experts, c.hidden, c.ffn, c.fmt_gate_up, c.fmt_down, Wgu_d, Wd_d)
    ws = torch.zeros(api.moe_workspace_bytes(ex, n, c.top_k), dtype=torch.uint8, device="cuda")
    y = api.moe_run(ex, dev(ids), dev(gates), dev(x), ws=ws)
    torch.cuda.synchronize()
    off = api.moe_workspace_offsets(ex, n, c.top_k)
    S, F, H = n * c.top_k, c.ffn, c.hidden
    w = ws.cpu().numpy()
    g = dict(
        y=y.cpu().numpy(),
        h=w[off[0]:off[0] + S * F * 4].view(np.float32).reshape(S, F),
        hq=w[off[1]:off[1] + S * F].view(np.int8).reshape(S, F),
        hd=w[off[2]:off[2] + S * F // 32 * 4].view(np.float32).reshape(S, F // 32),
        hs=w[off[3]:off[3] + S * F // 32 * 4].view(np.int32).reshape(S, F // 32),
        o=w[off[4]:off[4] + S * H * 4].view(np.float32).reshape(S, H))
    counts = np.bincount(ids.reshape(-1), minlength=c.n_experts)
    if n == 64:
        assert (counts > 8).sum() >= 1     # split groups are exercised
    check_stagewise(c.fmt_gate_up, c.fmt_down, Wgu, Wd, c.n_experts, H, F, ids, gates, x, g)
    assert np.all(np.isfinite(g["y"]))
    assert lib.get_device_error() == 0
