"""Python binding of the C-ABI library libqmv.so (see include/qmv.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory and
the current stream); results are returned as new tensors unless `out` is
given.  There is no CPU fallback: importing this module without a buildable
library raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from . import build as _build

Q8_0, Q4_K, IQ4_XS, Q5_K, Q6_K, Q8_G64, Q8_G128, F16, F32 = 0, 1, 2, 3, 4, 5, 6, 7, 8
FORMATS = {"Q8_0": Q8_0, "Q4_K": Q4_K, "IQ4_XS": IQ4_XS, "Q5_K": Q5_K, "Q6_K": Q6_K, "Q8_G64": Q8_G64,
           "Q8_G128": Q8_G128, "F16": F16, "F32": F32}
GROUP_WEIGHTS = {Q8_0: 256, Q4_K: 256, IQ4_XS: 512, Q5_K: 256, Q6_K: 256, Q8_G64: 512, Q8_G128: 1024,
                 F16: 32, F32: 32}
BYTES_PER_WEIGHT = {Q8_0: 272 / 256, Q4_K: 144 / 256, IQ4_XS: 272 / 512, Q5_K: 176 / 256, Q6_K: 208 / 256,
                    Q8_G64: 528 / 512, Q8_G128: 1040 / 1024, F16: 2.0, F32: 4.0}
MAX_TOKENS = 64
MAX_TOPK = 8

DEVERR_EXPERT_RANGE = 0x1
DEVERR_EXPERT_DUP = 0x2
DEVERR_TIMEOUT = 0x4
DEVERR_RANGE = 0x8


class QmvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class MoeExperts(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("hidden", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("fmt_gate_up", ctypes.c_int32), ("fmt_down", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


_i64, _vp, _int, _sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "qmv_row_bytes": (_i64, [_int, _i64]),
    "qmv_quantize_weights": (_int, [_int, _vp, _i64, _i64, _vp, _vp]),
    "qmv_quantize_act": (_int, [_vp, _i64, _int, _vp, _vp, _vp, _vp]),
    "qmv_run": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _int, _vp]),
    "qmv_run_q8": (_int, [_int, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp]),
    "qmv_splitk_choose": (_int, [_int, _i64, _i64, _int]),
    "qmv_splitk_workspace_bytes": (_sz, [_i64, _int, _int]),
    "qmv_act_q8_bytes": (_sz, [_i64, _int]),
    "qmv_splitk_run": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _int, _int, _vp, _sz, _vp]),
    "qmv_splitk_run_static": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _int, _int, _vp]),
    "moe_qmv_workspace_bytes": (_sz, [ctypes.POINTER(MoeExperts), _int, _int]),
    "moe_qmv_workspace_offsets": (_int, [ctypes.POINTER(MoeExperts), _int, _int, ctypes.POINTER(_sz * 5)]),
    "moe_qmv_run": (_int, [ctypes.POINTER(MoeExperts), _vp, _vp, _vp, _vp, _int, _int, _vp, _sz, _vp]),
    "moe_qmv_prefill_workspace_bytes": (_sz, [ctypes.POINTER(MoeExperts), _int, _int]),
    "moe_qmv_prefill_workspace_offsets": (_int, [ctypes.POINTER(MoeExperts), _int, _int, ctypes.POINTER(_sz * 5)]),
    "moe_qmv_prefill_run": (_int, [ctypes.POINTER(MoeExperts), _vp, _vp, _vp, _vp, _int, _int, _vp, _sz, _vp]),
    "moe_route_run": (_int, [_int, _vp, _vp, _int, _i64, _int, _int, _int, _vp, _vp, _vp, _vp]),
    "qmv_run_residual": (_int, [_int, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _vp, _sz, _vp]),
    "qmv_run_siblings": (_int, [_int, _vp, _vp, _vp, _vp, _vp, _i64, _int, _vp, _sz, _vp]),
    "qmv_get_device_error": (_int, [_vp, ctypes.POINTER(_int)]),
    "qmv_debug_shrink_outputs": (_int, [_i64]),
    "qmv_wait_probe": (_int, [ctypes.c_longlong, _vp, _vp]),
    "qmv_tc_probe": (_int, [_vp, _vp, _int, _vp, _vp]),
    "qmv_measure_pipes_scratch_bytes": (_sz, []),
    "qmv_measure_pipes": (_int, [ctypes.POINTER(ctypes.c_double), _int, _vp, _sz, _vp]),
    "qmv_check_rounding": (_int, [_vp, _vp]),
    "qmv_strerror": (ctypes.c_char_p, [_int]),
}

_lib = None


def _open(path: str):
    if not os.path.exists(path):
        raise ImportError(f"library not found at {path}")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name, None)
        if fn is None:
            continue
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None):
    """Load (building first if needed) libqmv.so and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _open(path or _build.build())
    return _lib


_debug_lib = None


def load_debug():
    """The QMV_DEBUG build of the library (libqmv_debug.so: every kernel access
    range-checked in software, see qmv_debug_shrink_outputs in qmv.h), built if
    needed.  It is not made the current library: run calls through it with
    `using(load_debug())`."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _open(_build.build(debug=True))
    return _debug_lib


@contextlib.contextmanager
def using(lib):
    """Within the block, every call of this module goes to `lib` (a library
    from load() or load_debug())."""
    global _lib
    prev = load()
    _lib = lib
    try:
        yield lib
    finally:
        _lib = prev


def debug_shrink_outputs(n: int) -> None:
    """Debug library only (inside `using(load_debug())`): later calls hand the
    range checks their result buffers' extents n elements short (0 restores)."""
    _check(load().qmv_debug_shrink_outputs(int(n)), "qmv_debug_shrink_outputs")


def strerror(code: int) -> str:
    return load().qmv_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise QmvError(rc, what)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def row_bytes(fmt: int, K: int) -> int:
    rb = load().qmv_row_bytes(int(fmt), int(K))
    _check(rb if rb < 0 else 0, "qmv_row_bytes")
    return int(rb)


def quantize_weights(fmt: int, w: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 weights [M][K] -> rows of format fmt, uint8 [M][row_bytes] (F16 / F32: the values
    converted, binary16 rounded to nearest even)."""
    M, K = w.shape
    rb = row_bytes(fmt, K)
    if out is None:
        out = torch.empty((M, rb), dtype=torch.uint8, device=w.device)
    _check(load().qmv_quantize_weights(int(fmt), _ptr(w), M, K, _ptr(out), _stream(stream)), "qmv_quantize_weights")
    return out


def quantize_act(x: torch.Tensor, stream=None):
    """Activation rule on x fp32 [n][K] -> (q int8 [n][K], d fp32 [n][K/32], s int32 [n][K/32]) in the
    library's Q8 activation layout (codes of each 256-element group halves first, see qmv.h)."""
    n, K = x.shape
    q = torch.empty((n, K), dtype=torch.int8, device=x.device)
    d = torch.empty((n, K // 32), dtype=torch.float32, device=x.device)
    s = torch.empty((n, K // 32), dtype=torch.int32, device=x.device)
    _check(load().qmv_quantize_act(_ptr(x), K, n, _ptr(q), _ptr(d), _ptr(s), _stream(stream)), "qmv_quantize_act")
    return q, d, s


def run(fmt: int, W: torch.Tensor, x: torch.Tensor, M: int, K: int, out: torch.Tensor | None = None,
        stream=None) -> torch.Tensor:
    """y [n][M] = What x Xhat (quantized matvec; F16 / F32 rows: Xhat = x), x fp32 [n][K]."""
    n = x.shape[0]
    if out is None:
        out = torch.empty((n, M), dtype=torch.float32, device=x.device)
    _check(load().qmv_run(int(fmt), _ptr(W), _ptr(x), _ptr(out), M, K, n, _stream(stream)), "qmv_run")
    return out


def run_q8(fmt: int, W: torch.Tensor, xq: torch.Tensor, xd: torch.Tensor, xs: torch.Tensor, M: int, K: int,
           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Matvec with activations already quantized by quantize_act (quantized formats only)."""
    n = xq.shape[0]
    if out is None:
        out = torch.empty((n, M), dtype=torch.float32, device=xq.device)
    _check(load().qmv_run_q8(int(fmt), _ptr(W), _ptr(xq), _ptr(xd), _ptr(xs), _ptr(out), M, K, n, _stream(stream)),
           "qmv_run_q8")
    return out


def splitk_choose(fmt: int, M: int, K: int, n_tok: int) -> int:
    s = load().qmv_splitk_choose(int(fmt), M, K, n_tok)
    _check(s if s < 0 else 0, "qmv_splitk_choose")
    return int(s)


def splitk_workspace_bytes(M: int, n_tok: int, n_split: int) -> int:
    return int(load().qmv_splitk_workspace_bytes(M, n_tok, n_split))


def act_q8_bytes(K: int, n_tok: int) -> int:
    return int(load().qmv_act_q8_bytes(K, n_tok))


def splitk_workspace_fast_bytes(M: int, K: int, n_tok: int, n_split: int) -> int:
    """Workspace that lets qmv_splitk_run quantize the activations once."""
    part = splitk_workspace_bytes(M, n_tok, n_split) if n_split > 1 else 0
    return ((part + 255) // 256) * 256 + act_q8_bytes(K, n_tok)


def splitk_run(fmt: int, W: torch.Tensor, x: torch.Tensor, M: int, K: int, n_split: int = 0,
               ws: torch.Tensor | None = None, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Split-K matvec; n_split = 0 picks the split from the shape.  Without a
    given workspace, one large enough for pre-quantized activations is made."""
    n = x.shape[0]
    if n_split == 0:
        n_split = splitk_choose(fmt, M, K, n)
    if out is None:
        out = torch.empty((n, M), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = torch.empty(max(16, splitk_workspace_fast_bytes(M, K, n, n_split)), dtype=torch.uint8, device=x.device)
    wsb = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().qmv_splitk_run(int(fmt), _ptr(W), _ptr(x), _ptr(out), M, K, n, n_split, _ptr(ws), wsb,
                                 _stream(stream)), "qmv_splitk_run")
    return out


def run_residual(fmt: int, W: torch.Tensor, x: torch.Tensor, r: torch.Tensor, M: int, K: int,
                 out: torch.Tensor | None = None, n_split: int = 0, ws: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """y = What Xhat + r (r fp32 [n][M]; out may be r for y += What Xhat)."""
    n = x.shape[0]
    if n_split == 0:
        n_split = splitk_choose(fmt, M, K, n)
    if out is None:
        out = torch.empty((n, M), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = torch.empty(max(16, splitk_workspace_fast_bytes(M, K, n, n_split)), dtype=torch.uint8, device=x.device)
    _check(load().qmv_run_residual(int(fmt), _ptr(W), _ptr(x), _ptr(r), _ptr(out), M, K, n, n_split, _ptr(ws),
                                   ws.numel(), _stream(stream)), "qmv_run_residual")
    return out


def run_siblings(mats, x: torch.Tensor, K: int, outs=None, ws: torch.Tensor | None = None, stream=None):
    """Sibling matvecs sharing x: mats is a list of (fmt, W, M); returns the
    list of y_i fp32 [n][M_i]."""
    n = x.shape[0]
    c = len(mats)
    if outs is None:
        outs = [torch.empty((n, M), dtype=torch.float32, device=x.device) for _, _, M in mats]
    if ws is None:
        ws = torch.empty(max(16, act_q8_bytes(K, n)), dtype=torch.uint8, device=x.device)
    fm = (ctypes.c_int * c)(*[int(f) for f, _, _ in mats])
    Wp = (ctypes.c_void_p * c)(*[W.data_ptr() for _, W, _ in mats])
    Mp = (ctypes.c_int64 * c)(*[int(M) for _, _, M in mats])
    yp = (ctypes.c_void_p * c)(*[o.data_ptr() for o in outs])
    _check(load().qmv_run_siblings(c, fm, Wp, Mp, yp, _ptr(x), K, n, _ptr(ws), ws.numel(), _stream(stream)),
           "qmv_run_siblings")
    return outs


STATIC_SCRATCH_BYTES = 8 << 20


def splitk_run_static(fmt: int, W: torch.Tensor, x: torch.Tensor, M: int, K: int, n_split: int = 0,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Split-K matvec for callers that cannot allocate: the partial sums use
    the library's static device array (see qmv_splitk_run_static)."""
    n = x.shape[0]
    if out is None:
        out = torch.empty((n, M), dtype=torch.float32, device=x.device)
    _check(load().qmv_splitk_run_static(int(fmt), _ptr(W), _ptr(x), _ptr(out), M, K, n, n_split, _stream(stream)),
           "qmv_splitk_run_static")
    return out


def moe_experts(n_experts: int, hidden: int, ffn: int, fmt_gate_up: int, fmt_down: int, w_gate_up: torch.Tensor,
                w_down: torch.Tensor) -> MoeExperts:
    """The expert pool descriptor.  It holds references to the two weight
    tensors, so their device memory stays allocated as long as the descriptor
    lives (the C struct itself keeps only their addresses)."""
    e = MoeExperts(n_experts, hidden, ffn, fmt_gate_up, fmt_down, 0, _ptr(w_gate_up), _ptr(w_down))
    e._tensors = (w_gate_up, w_down)
    return e


def moe_workspace_bytes(e: MoeExperts, n_tok: int, top_k: int) -> int:
    return int(load().moe_qmv_workspace_bytes(ctypes.byref(e), n_tok, top_k))


def moe_workspace_offsets(e: MoeExperts, n_tok: int, top_k: int):
    arr = (_sz * 5)()
    _check(load().moe_qmv_workspace_offsets(ctypes.byref(e), n_tok, top_k, ctypes.byref(arr)),
           "moe_qmv_workspace_offsets")
    return list(arr)


def moe_run(e: MoeExperts, ids: torch.Tensor, gates: torch.Tensor, x: torch.Tensor, ws: torch.Tensor | None = None,
            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Expert-grouped MoE decode layer; ids int32 [n][top_k], gates fp32 [n][top_k], x fp32 [n][hidden]."""
    n, top_k = ids.shape
    if out is None:
        out = torch.empty((n, e.hidden), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = torch.empty(moe_workspace_bytes(e, n, top_k), dtype=torch.uint8, device=x.device)
    _check(load().moe_qmv_run(ctypes.byref(e), _ptr(ids), _ptr(gates), _ptr(x), _ptr(out), n, top_k, _ptr(ws),
                              ws.numel(), _stream(stream)), "moe_qmv_run")
    return out


MAX_PREFILL_TOKENS = 16384


def moe_prefill_workspace_bytes(e: MoeExperts, n_tok: int, top_k: int) -> int:
    return int(load().moe_qmv_prefill_workspace_bytes(ctypes.byref(e), n_tok, top_k))


def moe_prefill_workspace_offsets(e: MoeExperts, n_tok: int, top_k: int):
    arr = (_sz * 5)()
    _check(load().moe_qmv_prefill_workspace_offsets(ctypes.byref(e), n_tok, top_k, ctypes.byref(arr)),
           "moe_qmv_prefill_workspace_offsets")
    return list(arr)


def moe_prefill_run(e: MoeExperts, ids: torch.Tensor, gates: torch.Tensor, x: torch.Tensor,
                    ws: torch.Tensor | None = None, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The MoE layer for large batches on the tensor cores (moe_qmv_prefill_run);
    arguments as moe_run, n up to MAX_PREFILL_TOKENS."""
    n, top_k = ids.shape
    if out is None:
        out = torch.empty((n, e.hidden), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = torch.empty(moe_prefill_workspace_bytes(e, n, top_k), dtype=torch.uint8, device=x.device)
    _check(load().moe_qmv_prefill_run(ctypes.byref(e), _ptr(ids), _ptr(gates), _ptr(x), _ptr(out), n, top_k,
                                      _ptr(ws), ws.numel(), _stream(stream)), "moe_qmv_prefill_run")
    return out


GATING_SOFTMAX, GATING_SIGMOID = 0, 1


def route_run(fmt: int, Wr: torch.Tensor, x: torch.Tensor, n_experts: int, hidden: int, top_k: int,
              gating: int = GATING_SOFTMAX, logits: torch.Tensor | None = None, ids: torch.Tensor | None = None,
              gates: torch.Tensor | None = None, stream=None):
    """Router and top-k: logits fp32 [n][E] = What_r Xhat, then per token the
    top_k experts by logit (ids int32 [n][top_k]) and their gates normalised
    over the picked ones (fp32 [n][top_k]).  Returns (ids, gates, logits)."""
    n = x.shape[0]
    dev = x.device
    if logits is None:
        logits = torch.empty((n, n_experts), dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty((n, top_k), dtype=torch.int32, device=dev)
    if gates is None:
        gates = torch.empty((n, top_k), dtype=torch.float32, device=dev)
    _check(load().moe_route_run(int(fmt), _ptr(Wr), _ptr(x), int(n_experts), int(hidden), n, int(top_k),
                                int(gating), _ptr(logits), _ptr(ids), _ptr(gates), _stream(stream)),
           "moe_route_run")
    return ids, gates, logits


def check_rounding(stream=None):
    """Mismatch counts (division, reciprocal) of the quantizer's branch-free
    arithmetic against IEEE round-to-nearest over every input of its range."""
    bad = torch.zeros(2, dtype=torch.int64, device="cuda")
    _check(load().qmv_check_rounding(_ptr(bad), _stream(stream)), "qmv_check_rounding")
    return [int(v) for v in bad.cpu()]


def tc_probe(A: torch.Tensor, B: torch.Tensor, stream=None) -> torch.Tensor:
    """A int8 [128][32], B int8 [N][32] -> A B^T fp32 [128][N] through the
    tcgen05 tensor cores (codes as f16, fp32 accumulator)."""
    N = B.shape[0]
    out = torch.empty((128, N), dtype=torch.float32, device=A.device)
    _check(load().qmv_tc_probe(_ptr(A), _ptr(B), N, _ptr(out), _stream(stream)), "qmv_tc_probe")
    return out


PIPE_NAMES = ("dp4a", "prmt", "ffma", "ffma2", "i2f", "mma_sync_s8_mac", "mma_sync_f16_mac",
              "tcgen05_f16_n256_mac", "tcgen05_f16_n64_mac", "tcgen05_f16_n32_mac")


def measure_pipes(stream=None) -> dict:
    """Measured per-SM per-clock rates (see qmv_measure_pipes), by name."""
    L = load()
    scratch = torch.empty(int(L.qmv_measure_pipes_scratch_bytes()), dtype=torch.uint8, device="cuda")
    arr = (ctypes.c_double * len(PIPE_NAMES))()
    n = L.qmv_measure_pipes(arr, len(PIPE_NAMES), _ptr(scratch), scratch.numel(), _stream(stream))
    _check(n if n < 0 else 0, "qmv_measure_pipes")
    return {PIPE_NAMES[i]: float(arr[i]) for i in range(n)}


def wait_probe(limit_cycles: int, stream=None) -> int:
    """Runs the kernels' bounded mbarrier wait with `limit_cycles` as its limit
    on a barrier that never completes (qmv_wait_probe); returns the SM cycles
    the wait lasted before it gave up.  Sets QMV_DEVERR_TIMEOUT."""
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(load().qmv_wait_probe(int(limit_cycles), _ptr(cyc), _stream(stream)), "qmv_wait_probe")
    return int(cyc.item())


def get_device_error(stream=None) -> int:
    v = _int(0)
    _check(load().qmv_get_device_error(_stream(stream), ctypes.byref(v)), "qmv_get_device_error")
    return int(v.value)
