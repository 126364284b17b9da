"""The C-ABI library builds for sm_103a, loads, and exports every function
include/qmv.h declares (no GPU needed: nothing is called that touches a
device)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmv.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = src[src.index('extern "C" {'):]
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", body, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("qmv_run", "qmv_splitk_run", "moe_qmv_run", "moe_route_run", "qmv_quantize_act",
              "qmv_get_device_error"):
        assert n in names


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_library_builds_loads_and_exports_every_declared_symbol():
    from moe_matvec_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_strerror_and_row_bytes_need_no_device():
    from moe_matvec_gb300 import api
    lib = api.load()
    assert lib.qmv_row_bytes(0, 4096) == 4352
    assert lib.qmv_row_bytes(1, 5120) == 2880
    assert lib.qmv_row_bytes(2, 2048) == 1088
    assert lib.qmv_row_bytes(2, 256) == -2      # IQ4_XS needs K % 512 == 0
    assert lib.qmv_row_bytes(7, 256) == 512 and lib.qmv_row_bytes(8, 256) == 1024   # F16 / F32 rows
    assert lib.qmv_row_bytes(9, 256) == -1
    assert api.strerror(-6) == "workspace too small"
