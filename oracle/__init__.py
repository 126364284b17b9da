"""CPU oracle of the quantized small-batch matvec / MoE decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library itself
never does.  The arithmetic lives in ``oracle.c`` (plain C, fp64 for the
dequantized products, the fp32 activation rule for integer codes), compiled
here with gcc on first use.  It shares no code with ``moe_matvec_gb300``.

Each function states what it computes; ``tests/test_oracle.py`` pins every one
of them against brute force, closed forms, library routines and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q8_0, Q4_K, IQ4_XS, Q5_K, Q6_K, Q8_G64, Q8_G128, F16, F32 = 0, 1, 2, 3, 4, 5, 6, 7, 8
FORMATS = (Q8_0, Q4_K, IQ4_XS, Q5_K, Q6_K, Q8_G64, Q8_G128)  # block-quantized
FLOAT_FORMATS = (F16, F32)  # unquantized rows; the activations stay fp32 (Xhat = x)
ALL_FORMATS = FORMATS + FLOAT_FORMATS
FORMAT_NAMES = {Q8_0: "Q8_0", Q4_K: "Q4_K", IQ4_XS: "IQ4_XS", Q5_K: "Q5_K", Q6_K: "Q6_K", Q8_G64: "Q8_G64",
                Q8_G128: "Q8_G128", F16: "F16", F32: "F32"}
GROUP_WEIGHTS = {Q8_0: 256, Q4_K: 256, IQ4_XS: 512, Q5_K: 256, Q6_K: 256, Q8_G64: 512, Q8_G128: 1024,
                 F16: 32, F32: 32}
GROUP_BYTES = {Q8_0: 272, Q4_K: 144, IQ4_XS: 272, Q5_K: 176, Q6_K: 208, Q8_G64: 528, Q8_G128: 1040,
               F16: 64, F32: 128}
# IQ4_XS codebook (int8), part of the format definition.
CODEBOOK = np.array([-127, -104, -83, -65, -49, -35, -22, -10,
                     1, 13, 25, 38, 53, 69, 89, 113], dtype=np.int64)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f64_to_f16.restype = ctypes.c_uint16
        lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.oracle_row_bytes.restype = _i64
        lib.oracle_row_bytes.argtypes = [ctypes.c_int, _i64]
        lib.oracle_act_quant.restype = None
        lib.oracle_act_quant.argtypes = [_ptr, _i64, _i64, _ptr, _ptr, _ptr]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_quantize.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr]
        lib.oracle_dequant.restype = ctypes.c_int
        lib.oracle_dequant.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr]
        lib.oracle_qmv.restype = ctypes.c_int
        lib.oracle_qmv.argtypes = [ctypes.c_int, _ptr, _i64, _i64, _ptr, _i64, _ptr, _ptr,
                                   ctypes.c_int]
        lib.oracle_moe_slot_valid.restype = ctypes.c_int
        lib.oracle_moe_slot_valid.argtypes = [_ptr, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int]
        lib.oracle_moe.restype = ctypes.c_int
        lib.oracle_moe.argtypes = ([ctypes.c_int, _ptr, ctypes.c_int, _ptr] + [ctypes.c_int] * 3
                                   + [_ptr, _ptr, _ptr, ctypes.c_int, ctypes.c_int, _ptr]
                                   + [_ptr] * 12 + [ctypes.c_int])
        lib.oracle_route_select.restype = ctypes.c_int
        lib.oracle_route_select.argtypes = [_ptr] + [ctypes.c_int] * 4 + [_ptr, _ptr]
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f64(h: int) -> float:
    """Value of the binary16 bit pattern h."""
    return _load().oracle_f16_to_f64(int(h) & 0xFFFF)


def f64_to_f16(v: float) -> int:
    """Bit pattern of v rounded to the nearest binary16 (ties to even)."""
    return int(_load().oracle_f64_to_f16(float(v)))


def row_bytes(fmt: int, K: int) -> int:
    """Bytes of one quantized row of K weights (negative if invalid)."""
    return int(_load().oracle_row_bytes(int(fmt), int(K)))


def act_quant(x: np.ndarray):
    """Activation rule on x fp32 [n][K]: returns (q int8 [n][K], d fp32
    [n][K/32], s int32 [n][K/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    n, K = x.shape
    assert K % 32 == 0
    q = np.empty((n, K), np.int8)
    d = np.empty((n, K // 32), np.float32)
    s = np.empty((n, K // 32), np.int32)
    _load().oracle_act_quant(_p(x), K, n, _p(q), _p(d), _p(s))
    return q, d, s


def quantize(fmt: int, w: np.ndarray) -> np.ndarray:
    """Quantize fp32 weights [M][K] into format fmt: uint8 [M][row_bytes]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    M, K = w.shape
    rb = row_bytes(fmt, K)
    assert rb > 0, "K not a multiple of the group size"
    out = np.zeros((M, rb), np.uint8)
    rc = _load().oracle_quantize(int(fmt), _p(w), M, K, _p(out))
    assert rc == 0
    return out


def dequant(fmt: int, W: np.ndarray, K: int) -> np.ndarray:
    """Dequantized weights What fp64 [M][K] of quantized rows W."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rb = row_bytes(fmt, K)
    M = W.size // rb
    out = np.empty((M, K), np.float64)
    rc = _load().oracle_dequant(int(fmt), _p(W), M, K, _p(out))
    assert rc == 0
    return out


def qmv(fmt: int, W: np.ndarray, x: np.ndarray, K: int, nthreads: int = 1):
    """y[t][m] = sum_k What[m][k] Xhat[t][k] (fp64) and the tolerance scale
    sabs[t][m] = sum_k |What[m][k] Xhat[t][k]|; x fp32 [n][K] (quantized by
    the activation rule, or used as it is for F16 / F32 weights)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    n = x.shape[0]
    assert x.shape[1] == K
    rb = row_bytes(fmt, K)
    M = W.size // rb
    y = np.empty((n, M), np.float64)
    sabs = np.empty((n, M), np.float64)
    rc = _load().oracle_qmv(int(fmt), _p(W), M, K, _p(x), n, _p(y), _p(sabs), int(nthreads))
    assert rc == 0
    return y, sabs


def moe_slot_valid(ids: np.ndarray, E: int, t: int, k: int) -> bool:
    """Whether slot (t, k) routes: id in [0, E) and not repeating an earlier
    id of the same token."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    return bool(_load().oracle_moe_slot_valid(_p(ids), ids.shape[1], int(E), int(t), int(k)))


def moe(fmt_gu: int, Wgu: np.ndarray, fmt_d: int, Wd: np.ndarray, E: int, H: int, F: int,
        ids: np.ndarray, gates: np.ndarray, x: np.ndarray, h_in: np.ndarray | None = None,
        nthreads: int = 1):
    """MoE decode layer (see oracle.c).  Wgu uint8 [E][2F][rb], Wd uint8
    [E][H][rb]; ids int32 [n][top_k]; gates fp32 [n][top_k]; x fp32 [n][H].
    Returns a dict of y, ybound, g, u, gabs, uabs, h32, hq, hd, hs, o, oabs
    (oabs[p][m] = sum_i |Wdown_e[m][i] Hhat_p[i]|, the tolerance scale of o).
    The per-slot projections run on nthreads threads (0: all host cores); the
    result does not depend on the thread count."""
    Wgu = np.ascontiguousarray(Wgu, dtype=np.uint8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, top_k = ids.shape
    S = n * top_k
    if nthreads <= 0:
        nthreads = os.cpu_count() or 1
    out = dict(
        y=np.empty((n, H)), ybound=np.empty((n, H)), g=np.empty((S, F)), u=np.empty((S, F)),
        gabs=np.empty((S, F)), uabs=np.empty((S, F)), h32=np.empty((S, F), np.float32),
        hq=np.empty((S, F), np.int8), hd=np.empty((S, F // 32), np.float32),
        hs=np.empty((S, F // 32), np.int32), o=np.empty((S, H)), oabs=np.empty((S, H)))
    if h_in is not None:
        h_in = np.ascontiguousarray(h_in, dtype=np.float32).reshape(S, F)
    rc = _load().oracle_moe(int(fmt_gu), _p(Wgu), int(fmt_d), _p(Wd), int(E), int(H), int(F),
                            _p(ids), _p(gates), _p(x), n, top_k, _p(h_in),
                            _p(out["y"]), _p(out["ybound"]), _p(out["g"]), _p(out["u"]),
                            _p(out["gabs"]), _p(out["uabs"]), _p(out["h32"]), _p(out["hq"]),
                            _p(out["hd"]), _p(out["hs"]), _p(out["o"]), _p(out["oabs"]),
                            int(nthreads))
    assert rc == 0
    return out


GATING_SOFTMAX, GATING_SIGMOID = 0, 1


def route_select(logits: np.ndarray, top_k: int, gating: int):
    """Top-k of router logits [n][E] (fp64; any fp32 logits are exact in it)
    and the normalised gates (see oracle.c): returns (ids int32 [n][top_k],
    gates fp64 [n][top_k])."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    if logits.ndim == 1:
        logits = logits[None, :]
    n, E = logits.shape
    ids = np.empty((n, top_k), np.int32)
    gates = np.empty((n, top_k), np.float64)
    rc = _load().oracle_route_select(_p(logits), n, E, int(top_k), int(gating), _p(ids), _p(gates))
    assert rc == 0
    return ids, gates


def route(fmt: int, Wr: np.ndarray, x: np.ndarray, H: int, top_k: int, gating: int):
    """Router: logits = What_r Xhat (the quantized matvec above, fp64), then
    route_select.  Wr uint8 [E][row_bytes]; x fp32 [n][H].  Returns (ids,
    gates, logits, sabs), sabs the logits' tolerance scale."""
    logits, sabs = qmv(fmt, Wr, x, H)
    ids, gates = route_select(logits, top_k, gating)
    return ids, gates, logits, sabs
