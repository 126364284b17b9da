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


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_debug_library_builds_exports_every_symbol_and_takes_its_switch():
    # the range-checked build (QMV_DEBUG) of the same sources: the same
    # symbols, and its extent switch (host state only, no device touched)
    # accepts n >= 0 and rejects a negative n; the release library has no
    # switch (tests/test_api_errors.py)
    from moe_matvec_gb300 import api
    lib = api.load_debug()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.qmv_debug_shrink_outputs(-1) == -2
    assert lib.qmv_debug_shrink_outputs(7) == 0
    assert lib.qmv_debug_shrink_outputs(0) == 0
    assert lib.qmv_row_bytes(1, 5120) == 2880


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


C_CLIENT = r"""
#include <stdio.h>
#include "qmv.h"
int main(void) {
  moe_experts e = {0};
  long long a = (long long)qmv_row_bytes(QMV_Q4_K, 5120), b = (long long)qmv_row_bytes(QMV_F32, 96);
  int rc = qmv_run(QMV_Q8_0, (const void*)0, (const float*)0, (float*)0, 16, 256, 1, (cudaStream_t)0);
  printf("%lld %lld %d %d %s\n", a, b, rc, e.n_experts, qmv_strerror(QMV_ERR_WORKSPACE));
  return (a == 2880 && b == 384 && rc == QMV_ERR_NULL) ? 0 : 1;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_plain_c_client_compiles_links_and_calls(tmp_path):
    # the boundary is a C ABI: a C99 program includes the header, links the
    # library and calls host-only entry points
    import subprocess
    from moe_matvec_gb300 import build
    lib = build.build()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    if not os.path.exists(os.path.join(cuda, "include", "cuda_runtime_api.h")):
        pytest.skip("CUDA headers not found")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib)
    cudalib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d)), None)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(cuda, "include"), str(src), "-o", str(exe), "-L", libdir, "-lqmv", f"-Wl,-rpath,{libdir}"]
    if cudalib:
        cmd += ["-L", cudalib, f"-Wl,-rpath,{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split()[:4] == ["2880", "384", "-4", "0"]
