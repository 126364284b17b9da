"""The allocation-free split-K entry point, qmv_splitk_run_static.

It serves callers that may not call cudaMalloc themselves (for instance a
plugin that runs while its host framework captures a CUDA graph, or a host
that owns all of the device memory): the partial sums go to a static device
array inside the library instead of a caller workspace.  Two calls in a row
share that array; each must match qmv_splitk_run with a caller-allocated
workspace, within the tolerance of the other parity tests."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import api, synth
from tests.gpu_util import assert_within, dev

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_entry_point_on_two_calls(lib):
    cases = [(0, 512, 65536, 4, 16), (1, 300, 8192, 7, 0)]   # fmt, M, K, n_tok, n_split (0 = auto)
    for call, (fmt, M, K, n, S) in enumerate(cases):
        w = synth.weights(900 + call, M, K)
        x = synth.activations(901 + call, n, K)
        Wn = oracle.quantize(fmt, w)
        Wd, xd = dev(Wn), dev(x)
        y_static = lib.splitk_run_static(fmt, Wd, xd, M, K, n_split=S)
        y_ws = lib.splitk_run(fmt, Wd, xd, M, K, n_split=S)
        torch.cuda.synchronize()
        _, sabs = oracle.qmv(fmt, Wn, x, K)
        assert_within(y_static.cpu().numpy(), y_ws.cpu().numpy(), sabs, what=f"call {call}: static vs workspace")
    assert lib.get_device_error() == 0


def test_static_scratch_rejects_splits_that_do_not_fit(lib):
    L = api.load()
    small = torch.zeros(64, dtype=torch.float32, device="cuda")  # never read: the call is rejected first
    M, n, S = 151936, 16, 2
    assert api.splitk_workspace_bytes(M, n, S) > api.STATIC_SCRATCH_BYTES
    rc = L.qmv_splitk_run_static(0, small.data_ptr(), small.data_ptr(), small.data_ptr(), M, 5120, n, S,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -6   # QMV_ERR_WORKSPACE
