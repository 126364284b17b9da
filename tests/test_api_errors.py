"""Host-side argument checking of the C ABI.  Every call here is invalid, so
the library returns its error code before touching any device (these run
with or without a GPU, and never launch)."""
import ctypes

import pytest

from moe_matvec_gb300 import api

A = 0x10000          # an aligned, never dereferenced address
MIS = 0x10004        # misaligned


@pytest.fixture(scope="module")
def L():
    return api.load()


def test_qmv_run_rejects_bad_arguments(L):
    assert L.qmv_run(9, A, A, A, 16, 256, 1, None) == -1
    assert L.qmv_run(3, A, A, A, 16, 100, 1, None) == -2        # Q5_K needs K % 256
    assert L.qmv_run(0, A, A, A, 0, 256, 1, None) == -2
    assert L.qmv_run(0, A, A, A, 16, 100, 1, None) == -2
    assert L.qmv_run(2, A, A, A, 16, 256, 1, None) == -2        # IQ4_XS needs K % 512
    assert L.qmv_run(0, A, A, A, 16, 256, 0, None) == -3
    assert L.qmv_run(0, A, A, A, 16, 256, 65, None) == -3
    assert L.qmv_run(0, None, A, A, 16, 256, 1, None) == -4
    assert L.qmv_run(0, A, MIS, A, 16, 256, 1, None) == -5
    assert L.qmv_run_q8(1, A, A, None, A, A, 16, 256, 1, None) == -4


def test_float_rows_shape_and_entry_points(L):
    # F16 / F32: K % 32, plain rows, fp32 activations only, no MoE pool (the
    # router takes them)
    assert L.qmv_row_bytes(7, 96) == 192 and L.qmv_row_bytes(8, 96) == 384
    assert L.qmv_row_bytes(7, 100) == -2
    assert L.qmv_run(8, A, A, A, 16, 100, 1, None) == -2
    assert L.qmv_run_q8(7, A, A, A, A, A, 16, 256, 1, None) == -1
    assert L.qmv_run_q8(8, A, A, A, A, A, 16, 256, 1, None) == -1
    assert L.qmv_quantize_weights(7, A, 4, 48, A, None) == -2
    ex = api.MoeExperts(128, 4096, 1536, 7, 1, 0, A, A)
    assert L.moe_qmv_workspace_bytes(ctypes.byref(ex), 4, 8) == 0
    assert L.moe_qmv_run(ctypes.byref(ex), A, A, A, A, 4, 8, A, 1 << 30, None) == -1


def test_splitk_rejects_bad_workspace(L):
    need = L.qmv_splitk_workspace_bytes(64, 2, 4)
    assert need == 4 * 2 * 64 * 4
    assert L.qmv_splitk_run(0, A, A, A, 64, 4096, 2, 4, A, need - 1, None) == -6
    assert L.qmv_splitk_run(0, A, A, A, 64, 4096, 2, 4, None, need, None) == -4
    assert L.qmv_splitk_run(0, A, A, A, 64, 4096, 2, 4, MIS, need, None) == -5
    assert L.qmv_splitk_run(0, A, A, A, 64, 4096, 2, 17, A, 1 << 30, None) == -2   # more splits than groups
    assert L.qmv_splitk_run(0, A, A, A, 64, 4096, 2, -1, A, need, None) == -2


def test_quantize_entry_points_reject_bad_arguments(L):
    assert L.qmv_quantize_act(A, 100, 1, A, A, A, None) == -2
    assert L.qmv_quantize_act(A, 256, 0, A, A, A, None) == -3
    assert L.qmv_quantize_act(A, 256, 1, A, None, A, None) == -4
    assert L.qmv_quantize_weights(9, A, 4, 256, A, None) == -1
    assert L.qmv_quantize_weights(1, A, 4, 128, A, None) == -2
    assert L.qmv_quantize_weights(1, A, 4, 256, MIS, None) == -5


def test_device_error_needs_an_output_pointer(L):
    assert L.qmv_get_device_error(None, None) == -4


def test_release_library_has_no_debug_switch(L):
    # the extent-shrinking switch of the range-checked build is not in the
    # release library: it answers QMV_ERR_UNAVAILABLE and changes nothing
    assert L.qmv_debug_shrink_outputs(1) == -9
    assert L.qmv_debug_shrink_outputs(0) == -9
    assert "not available" in api.strerror(-9)


def test_route_rejects_bad_arguments(L):
    # fmt, Wr, x, E, hidden, n_tok, top_k, gating, logits, ids, gates, stream
    assert L.moe_route_run(9, A, A, 128, 4096, 1, 8, 0, A, A, A, None) == -1
    assert L.moe_route_run(0, A, A, 128, 100, 1, 8, 0, A, A, A, None) == -2
    assert L.moe_route_run(0, A, A, 513, 4096, 1, 8, 0, A, A, A, None) == -2     # > 512 experts
    assert L.moe_route_run(0, A, A, 128, 4096, 1, 8, 2, A, A, A, None) == -2     # unknown gating
    assert L.moe_route_run(0, A, A, 128, 4096, 0, 8, 0, A, A, A, None) == -3
    assert L.moe_route_run(0, A, A, 128, 4096, 1, 9, 0, A, A, A, None) == -3     # top_k > 8
    assert L.moe_route_run(0, A, A, 4, 4096, 1, 5, 0, A, A, A, None) == -3       # top_k > experts
    assert L.moe_route_run(0, A, A, 128, 4096, 1, 8, 0, A, None, A, None) == -4
    assert L.moe_route_run(0, A, A, 128, 4096, 1, 8, 0, None, A, A, None) == -4
    assert L.moe_route_run(0, A, A, 128, 4096, 1, 8, 0, A, A, MIS, None) == -5


def test_residual_and_siblings_reject_bad_arguments(L):
    need = L.qmv_splitk_workspace_bytes(64, 2, 4)
    assert L.qmv_run_residual(0, A, A, None, A, 64, 4096, 2, 1, A, need, None) == -4
    assert L.qmv_run_residual(0, A, A, MIS, A, 64, 4096, 2, 1, A, need, None) == -5
    assert L.qmv_run_residual(0, A, A, A, A, 64, 4096, 2, 4, A, need - 1, None) == -6
    fm = (ctypes.c_int * 2)(0, 1)
    Wp = (ctypes.c_void_p * 2)(A, A)
    Mp = (ctypes.c_int64 * 2)(64, 64)
    yp = (ctypes.c_void_p * 2)(A, A)
    assert L.qmv_run_siblings(0, fm, Wp, Mp, yp, A, 4096, 2, A, 1 << 20, None) == -2
    assert L.qmv_run_siblings(9, fm, Wp, Mp, yp, A, 4096, 2, A, 1 << 20, None) == -2
    assert L.qmv_run_siblings(2, None, Wp, Mp, yp, A, 4096, 2, A, 1 << 20, None) == -4
    bad = (ctypes.c_int * 2)(0, 2)                                     # IQ4_XS needs K % 512
    assert L.qmv_run_siblings(2, bad, Wp, Mp, yp, A, 256 + 1024, 2, A, 1 << 20, None) == -2
    assert L.qmv_run_siblings(2, fm, Wp, Mp, yp, A, 4096, 8, A, 16, None) == -6    # workspace too small


def test_split_choice_fits_float_activations(L):
    # F16 / F32 rows: enough splits that one pass of up to 16 tokens' fp32
    # activations of a split range takes at most 96 KB (host logic only)
    assert L.qmv_splitk_choose(7, 17408, 5120, 16) == 5      # 5 chunks of 1024: 64 KB each
    assert L.qmv_splitk_choose(7, 17408, 5120, 1) == 1
    assert L.qmv_splitk_choose(8, 4096, 4096, 16) == 4       # 8 chunks of 512
    s = L.qmv_splitk_choose(8, 64, 65536, 2)
    assert s >= 6 and 128 % s == 0 and (65536 // s) * 2 * 4 <= 96 * 1024
    assert L.qmv_splitk_choose(1, 17408, 5120, 16) == 1      # quantized rows: the row count decides

