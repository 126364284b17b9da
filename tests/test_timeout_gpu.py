"""The kernels' bounded waits, made to run out on purpose.

Every mbarrier wait in the library has a cycle limit after which the kernel
gives up, sets QMV_DEVERR_TIMEOUT in the device error word and returns, so a
stalled pipeline never hangs the GPU.  In the matvec and MoE kernels that limit
is a compile-time constant (about a second).  qmv_wait_probe runs the same
wait loop with a short limit on an mbarrier that nothing ever completes (a
flag that nothing sets): the wait must give up after its limit, the call must
return, the error must be reported, and the next matvec and MoE calls must be
correct and leave no error behind."""
import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import api, synth
from tests.gpu_util import assert_within, dev, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit", [1, 1 << 16, 1 << 22])
def test_wait_on_a_barrier_nothing_completes_gives_up_after_its_limit(lib, limit):
    assert lib.get_device_error() == 0
    cycles = lib.wait_probe(limit)                # synchronises: the kernel returned
    assert cycles >= limit
    assert cycles < limit + (1 << 26)             # one suspend (about a millisecond) past the limit at most
    assert lib.get_device_error() == api.DEVERR_TIMEOUT
    assert lib.get_device_error() == 0            # reading the word clears it


def test_wait_probe_rejects_limits_outside_its_range(lib):
    for bad in (0, -5, (1 << 31) + 1):
        with pytest.raises(api.QmvError):
            lib.wait_probe(bad)
    assert lib.get_device_error() == 0


def test_matvec_after_a_timeout_is_correct(lib):
    fmt, M, K, n = 0, 4096, 16384, 1
    Wn = oracle.quantize(fmt, synth.weights(1234, M, K))
    x = synth.activations(1235, n, K)
    Wd, xd = dev(Wn), dev(x)
    y0 = lib.run(fmt, Wd, xd, M, K)
    assert lib.get_device_error() == 0
    lib.wait_probe(1 << 20)
    assert lib.get_device_error() == api.DEVERR_TIMEOUT
    y1 = lib.run(fmt, Wd, xd, M, K)
    assert lib.get_device_error() == 0
    assert torch.equal(y0, y1)
    rows = sample_rows(M)
    yr, sabs = oracle.qmv(fmt, Wn[rows], x, K)
    assert_within(y1.cpu().numpy()[:, rows], yr, sabs, what="after the timeout")


def test_moe_after_a_timeout_is_correct(lib):
    E, H, F, top_k, n = 16, 2048, 1536, 4, 8
    Wgu = np.stack([oracle.quantize(2, synth.weights(1300 + 2 * e, 2 * F, H)) for e in range(E)])
    Wd = np.stack([oracle.quantize(1, synth.weights(1301 + 2 * e, H, F)) for e in range(E)])
    ids, gates = synth.routing(1302, n, E, top_k)
    x = synth.activations(1303, n, H)
    Wgu_d, Wd_d = dev(Wgu), dev(Wd)          # kept alive for the calls
    ex = api.moe_experts(E, H, F, 2, 1, Wgu_d, Wd_d)
    ws = torch.zeros(api.moe_workspace_bytes(ex, n, top_k), dtype=torch.uint8, device="cuda")
    idd, gd, xd = dev(ids), dev(gates), dev(x)
    y0 = api.moe_run(ex, idd, gd, xd, ws=ws).clone()
    assert lib.get_device_error() == 0
    lib.wait_probe(1 << 20)
    assert lib.get_device_error() == api.DEVERR_TIMEOUT
    y1 = api.moe_run(ex, idd, gd, xd, ws=ws)
    assert lib.get_device_error() == 0
    assert torch.equal(y0, y1)
