"""GPU parity of the tensor-core MoE layer for large batches
(moe_qmv_prefill_run) against the oracle, graded stage by stage as the
decode layer is (tests/test_moe_gpu.py): h within the propagated gate/up
tolerance, q8(h) bit-exact by the activation rule on the GPU's h, o and y
against the oracle fed the GPU's h, and y end to end within the matvec bound
plus the exact effect of any requantization code that differs."""
import numpy as np
import pytest
import torch

from moe_matvec_gb300 import api, synth
from tests.gpu_util import dev
from tests.test_moe_gpu import check_stagewise, full_pool, make_pool

pytestmark = pytest.mark.gpu


def run_prefill(ex, ids, gates, x, F, H):
    n, top_k = ids.shape
    ws = torch.zeros(api.moe_prefill_workspace_bytes(ex, n, top_k), dtype=torch.uint8, device="cuda")
    y = api.moe_prefill_run(ex, dev(ids), dev(gates), dev(x), ws=ws)
    torch.cuda.synchronize()
    off = api.moe_prefill_workspace_offsets(ex, n, top_k)
    S = n * top_k
    w = ws.cpu().numpy()
    return dict(
        y=y.cpu().numpy(),
        h=w[off[0]:off[0] + S * F * 4].view(np.float32).reshape(S, F),
        hq=w[off[1]:off[1] + S * F].view(np.int8).reshape(S, F),
        hd=w[off[2]:off[2] + S * F // 32 * 4].view(np.float32).reshape(S, F // 32),
        hs=w[off[3]:off[3] + S * F // 32 * 4].view(np.int32).reshape(S, F // 32),
        o=w[off[4]:off[4] + S * H * 4].view(np.float32).reshape(S, H))


# (gate/up format, down format, experts, hidden, ffn, top_k, tokens): every
# decode format in both projections, experts with more slots than one tile
# holds (several slot tiles) and ragged counts
CASES = [(2, 1, 16, 1024, 512, 4, 256), (0, 2, 12, 512, 512, 3, 200), (1, 0, 8, 768, 256, 2, 333),
         (2, 1, 32, 512, 768, 8, 96), (1, 1, 4, 256, 256, 1, 70)]


@pytest.mark.parametrize("fmt_gu,fmt_d,E,H,F,top_k,n", CASES)
def test_prefill_stagewise(lib, fmt_gu, fmt_d, E, H, F, top_k, n):
    seed = 700 + E + H + F + n
    Wgu, Wd = make_pool(fmt_gu, fmt_d, E, H, F, seed)
    ids, gates = synth.routing(seed, n, E, top_k)
    x = synth.activations(seed, n, H)
    Wgu_d, Wd_d = dev(Wgu), dev(Wd)          # kept alive for the calls
    ex = api.moe_experts(E, H, F, fmt_gu, fmt_d, Wgu_d, Wd_d)
    g = run_prefill(ex, ids, gates, x, F, H)
    check_stagewise(fmt_gu, fmt_d, Wgu, Wd, E, H, F, ids, gates, x, g)
    assert lib.get_device_error() == 0


def test_prefill_invalid_ids_contribute_zero_and_flag(lib):
    E, H, F = 6, 512, 256
    Wgu, Wd = make_pool(2, 1, E, H, F, 61)
    ids, gates = synth.routing(62, 40, E, 3)
    ids[0, 1] = 9          # out of range
    ids[5, 2] = ids[5, 0]  # repeated within the token
    x = synth.activations(63, 40, H)
    assert lib.get_device_error() == 0
    Wgu_d, Wd_d = dev(Wgu), dev(Wd)          # kept alive for the calls
    ex = api.moe_experts(E, H, F, 2, 1, Wgu_d, Wd_d)
    g = run_prefill(ex, ids, gates, x, F, H)
    assert lib.get_device_error() == (api.DEVERR_EXPERT_RANGE | api.DEVERR_EXPERT_DUP)
    check_stagewise(2, 1, Wgu, Wd, E, H, F, ids, gates, x, g)


@pytest.mark.parametrize("n", [512, 2048])
def test_prefill_full_size_sampled_tokens(lib, n):
    # the full-size layer (128 experts, IQ4_XS gate/up 3072 x 4096, Q4_K down
    # 4096 x 1536) at a prompt-sized batch; 16 sampled tokens against the oracle
    c = synth.MOE_CASE
    ids, gates = synth.routing(7100 + n, n, c.n_experts, c.top_k)
    x = synth.activations(7101 + n, n, c.hidden)
    Wgu, Wd, Wgu_d, Wd_d = full_pool()
    ex = api.moe_experts(c.n_experts, c.hidden, c.ffn, c.fmt_gate_up, c.fmt_down, Wgu_d, Wd_d)
    g = run_prefill(ex, ids, gates, x, c.ffn, c.hidden)
    sample = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(n).integers(0, n, 14)]))
    check_stagewise(c.fmt_gate_up, c.fmt_down, Wgu, Wd, c.n_experts, c.hidden, c.ffn, ids, gates, x, g,
                    tokens=sample)
    assert np.all(np.isfinite(g["y"]))
    assert lib.get_device_error() == 0


def test_prefill_and_decode_layers_both_pass_on_one_batch(lib):
    # the two entry points on the same 64-token batch: each passes the full
    # stage-wise check (the oracle fixes one result; the two paths add their
    # fp32 block terms in different orders)
    E, H, F, top_k, n = 16, 1024, 512, 8, 64
    Wgu, Wd = make_pool(2, 1, E, H, F, 810)
    ids, gates = synth.routing(811, n, E, top_k)
    x = synth.activations(812, n, H)
    Wgu_d, Wd_d = dev(Wgu), dev(Wd)          # kept alive for the calls
    ex = api.moe_experts(E, H, F, 2, 1, Wgu_d, Wd_d)
    check_stagewise(2, 1, Wgu, Wd, E, H, F, ids, gates, x, run_prefill(ex, ids, gates, x, F, H))
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
