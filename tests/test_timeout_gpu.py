"""The kernels' bounded waits, made to run out on purpose.

Every wait in the library has a cycle limit after which the kernel gives up,
sets QMV_DEVERR_TIMEOUT in the device error word and returns, so a stalled
pipeline never hangs the GPU.  qmv_set_consumer_wait_limit shortens the limit
of the consumer warps' waits for weight stages; a bandwidth-bound matvec then
finds a stage that has not landed yet, gives up, and the next call (with the
default limit restored) must be correct and leave no error behind."""
import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import api, synth
from tests.gpu_util import assert_within, dev, sample_rows

pytestmark = pytest.mark.gpu


def test_short_consumer_wait_limit_times_out_and_the_next_call_is_correct(lib):
    # 71 MB of Q8_0 weights at one token: the consumers outrun HBM and wait
    # on most stages, so with a one-cycle limit some wait is late
    fmt, M, K, n = 0, 4096, 16384, 1
    Wn = oracle.quantize(fmt, synth.weights(1234, M, K))
    x = synth.activations(1235, n, K)
    Wd, xd = dev(Wn), dev(x)
    y0 = lib.run(fmt, Wd, xd, M, K)
    assert lib.get_device_error() == 0
    err = 0
    lib.set_consumer_wait_limit(1)
    try:
        for _ in range(3):
            lib.run(fmt, Wd, xd, M, K)
            err = lib.get_device_error()      # the call returned: the stream synchronised
            if err:
                break
    finally:
        lib.set_consumer_wait_limit(0)
    assert err == api.DEVERR_TIMEOUT
    y1 = lib.run(fmt, Wd, xd, M, K)
    assert lib.get_device_error() == 0
    assert torch.equal(y0, y1)
    rows = sample_rows(M)
    yr, sabs = oracle.qmv(fmt, Wn[rows], x, K)
    assert_within(y1.cpu().numpy()[:, rows], yr, sabs, what="after the timeout")


def test_moe_call_with_short_wait_limit_returns_and_the_next_call_is_correct(lib):
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
    lib.set_consumer_wait_limit(1)
    try:
        api.moe_run(ex, idd, gd, xd, ws=ws)
        err = lib.get_device_error()
    finally:
        lib.set_consumer_wait_limit(0)
    assert err in (0, api.DEVERR_TIMEOUT)     # whether a stage was late is timing; either way it returned
    y1 = api.moe_run(ex, idd, gd, xd, ws=ws)
    assert lib.get_device_error() == 0
    assert torch.equal(y0, y1)
