"""GPU parity of the router + top-k step against the oracle.

The picks are integers decided on floating-point logits, so they are graded
in the kernel's own precision: the GPU logits must match the oracle's fp64
logits within the matvec tolerance, and the picks must be exactly the
oracle's selection applied to the GPU's fp32 logits (comparisons are exact
in any precision).  The gates are the oracle's normalisation of those
logits within a few fp32 roundings.  Where the oracle's own fp64 logits
separate the k-th and (k+1)-th experts by more than the logits' tolerance,
the picks must also agree with the fully independent oracle."""
import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import api, synth
from tests.gpu_util import TOL, assert_within, dev

pytestmark = pytest.mark.gpu

CASES = [(0, 128, 4096, 1, 8, 0), (0, 128, 4096, 4, 8, 1), (0, 128, 4096, 64, 8, 0),
         (1, 64, 2048, 16, 6, 0), (2, 256, 1024, 33, 8, 1), (0, 512, 512, 5, 2, 0),
         (1, 8, 256, 3, 8, 1), (2, 37, 512, 7, 1, 0),
         (8, 128, 4096, 4, 8, 0), (7, 256, 2048, 16, 8, 1)]   # unquantized (F32 / F16) router rows


def route_gpu(fmt, Wr, x, E, H, top_k, gating):
    ids, gates, logits = api.route_run(fmt, dev(Wr), dev(x), E, H, top_k, gating)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), gates.cpu().numpy(), logits.cpu().numpy()


@pytest.mark.parametrize("fmt,E,H,n,top_k,gating", CASES)
def test_route_matches_oracle(lib, fmt, E, H, n, top_k, gating):
    seed = 700 + fmt + E + n + top_k
    Wr = oracle.quantize(fmt, synth.weights(seed, E, H))
    x = synth.activations(seed + 1, n, H)
    ids, gates, logits = route_gpu(fmt, Wr, x, E, H, top_k, gating)
    # (i) logits: the quantized matvec
    lr, sabs = oracle.qmv(fmt, Wr, x, H)
    assert_within(logits, lr, sabs, what="router logits")
    # (ii) picks exactly the oracle's selection on the GPU's own logits
    ids_own, gates_own = oracle.route_select(logits.astype(np.float64), top_k, gating)
    assert np.array_equal(ids, ids_own)
    assert np.allclose(gates, gates_own, rtol=4e-6, atol=1e-7)
    assert np.allclose(gates.sum(axis=1), 1.0, atol=4e-6)
    # (iii) against the independent oracle where its fp64 logits decide clearly
    ids_ref, _ = oracle.route_select(lr, top_k, gating)
    tol = TOL * sabs
    for t in range(n):
        srt = np.sort(lr[t])[::-1]
        gaps = srt[:top_k] - np.append(srt[1:top_k + 1], -np.inf)[:top_k]
        if np.all(gaps > 2 * tol[t].max()):
            assert np.array_equal(ids[t], ids_ref[t])


@pytest.mark.parametrize("gating", [0, 1])
def test_route_ties_go_to_the_lower_expert(lib, gating):
    # all-zero router rows: every logit is 0, the picks are 0..top_k-1 and
    # the gates uniform
    E, H, n, top_k = 96, 512, 5, 8
    Wr = oracle.quantize(0, np.zeros((E, H), np.float32))
    x = synth.activations(9, n, H)
    ids, gates, logits = route_gpu(0, Wr, x, E, H, top_k, gating)
    assert np.all(logits == 0)
    assert np.array_equal(ids, np.tile(np.arange(top_k, dtype=np.int32), (n, 1)))
    assert np.all(gates == np.float32(1 / top_k))


def test_route_feeds_the_moe_layer(lib):
    # ids / gates from the router are valid input of moe_qmv_run: no device
    # error, every id in range and distinct within a token
    E, H, F, n, top_k = 16, 512, 256, 12, 4
    Wr = oracle.quantize(0, synth.weights(31, E, H))
    x = synth.activations(32, n, H)
    ids, gates, _ = api.route_run(0, dev(Wr), dev(x), E, H, top_k, 0)
    i = ids.cpu().numpy()
    assert all(len(set(r)) == top_k and r.min() >= 0 and r.max() < E for r in i)
    wg = torch.from_numpy(np.stack([oracle.quantize(2, synth.weights(40 + e, 2 * F, H)) for e in range(E)])).cuda()
    wd = torch.from_numpy(np.stack([oracle.quantize(1, synth.weights(80 + e, H, F)) for e in range(E)])).cuda()
    ex = api.moe_experts(E, H, F, 2, 1, wg, wd)
    y = api.moe_run(ex, ids, gates, dev(x))
    torch.cuda.synchronize()
    assert np.all(np.isfinite(y.cpu().numpy()))
    assert lib.get_device_error() == 0
