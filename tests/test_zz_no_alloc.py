"""The allocation-free split-K entry point, qmv_splitk_run_static.

It serves callers that may not call cudaMalloc themselves (for instance a
plugin that runs while its host framework captures a CUDA graph, or a host
that owns all of the device memory): the partial sums (and, above 4 tokens,
the once-quantized activations) go to a static device array inside the
library instead of a caller workspace.  Two calls in a row share that array;
each must give the same bits as qmv_splitk_run with a caller-allocated
workspace and the same split, and lie within the parity tolerance of the
oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_matvec_gb300 import api, synth
from tests.gpu_util import assert_within, dev

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_entry_point_on_two_calls(lib):
    # fmt, M, K, n_tok, n_split (0 = auto); 6 and 7 tokens quantize the activations into the array
    cases = [(0, 512, 65536, 4, 16), (0, 512, 65536, 6, 16), (1, 300, 8192, 7, 0)]
    # the automatic split of the last call is above one, so it uses the array
    assert lib.splitk_choose(1, 300, 8192, 7) > 1
    for call, (fmt, M, K, n, S) in enumerate(cases):
        w = synth.weights(900 + call, M, K)
        x = synth.activations(901 + call, n, K)
        Wn = oracle.quantize(fmt, w)
        Wd, xd = dev(Wn), dev(x)
        y_static = lib.splitk_run_static(fmt, Wd, xd, M, K, n_split=S)
        y_ws = lib.splitk_run(fmt, Wd, xd, M, K, n_split=S)
        torch.cuda.synchronize()
        a, b = y_static.cpu().numpy(), y_ws.cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"call {call}: static vs workspace bits"
        yr, sabs = oracle.qmv(fmt, Wn, x, K)
        assert_within(a, yr, sabs, what=f"call {call}: static vs oracle")
    assert lib.get_device_error() == 0


def test_static_scratch_rejects_splits_that_do_not_fit(lib):
    L = api.load()
    small = torch.zeros(64, dtype=torch.float32, device="cuda")  # never read: the call is rejected first
    M, n, S = 151936, 16, 2
    assert api.splitk_workspace_bytes(M, n, S) > api.STATIC_SCRATCH_BYTES
    rc = L.qmv_splitk_run_static(0, small.data_ptr(), small.data_ptr(), small.data_ptr(), M, 5120, n, S,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -6   # QMV_ERR_WORKSPACE
