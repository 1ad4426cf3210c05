"""GB300-native ragged-M grouped GEMM.

``Y_e = X_e . W_e`` for every expert e in one launch of a persistent,
warp-specialized tcgen05 kernel (see include/rgg.h for the full contract).

This module is a thin ctypes binding over ``librgg.so``: it turns torch
tensors into device pointers and the current CUDA stream into a handle, and
raises on a non-OK status.  Every step of the computation runs in the CUDA
library; there is no CPU or PyTorch fallback.  Build the library with
``python -c "import __graft_entry__ as g; g.build()"`` (or
``python ragged_grouped_gemm_02_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "RggError", "rgg_grouped_gemm", "rgg_grouped_gemm_swiglu", "rgg_grouped_gemm_fp8", "rgg_grouped_gemm_gather",
    "rgg_grouped_gemm_swiglu_gather", "rgg_grouped_gemm_noalloc", "rgg_export_tiles", "rgg_export_walk",
    "rgg_query_status",
    "rgg_plan", "rgg_status_string", "library_path", "load_library", "EXPORTED_SYMBOLS",
    "RGG_OK", "RGG_ERR_INVALID_ARG", "RGG_ERR_UNSUPPORTED", "RGG_ERR_CUDA", "RGG_ERR_BAD_OFFSETS",
    "RGG_ERR_DEVICE_TIMEOUT", "RGG_ERR_CAPACITY", "RGG_ERR_BAD_ROW_INDEX", "RGG_ERR_DEVICE_BOUNDS",
    "open_library", "debug_library_path",
]

RGG_OK = 0
RGG_ERR_INVALID_ARG = 1
RGG_ERR_UNSUPPORTED = 2
RGG_ERR_CUDA = 3
RGG_ERR_BAD_OFFSETS = 4
RGG_ERR_DEVICE_TIMEOUT = 5
RGG_ERR_CAPACITY = 6
RGG_ERR_BAD_ROW_INDEX = 7
RGG_ERR_DEVICE_BOUNDS = 8
RGG_DEBUG_PRODUCER_STALL = 1

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "librgg.so")
_DEBUG_LIB_PATH = os.path.join(_PKG, "librgg_debug.so")

# The C ABI entry points declared in include/rgg.h.
EXPORTED_SYMBOLS = (
    "rgg_create", "rgg_destroy", "rgg_grouped_gemm", "rgg_export_tiles", "rgg_query_status",
    "rgg_plan", "rgg_status_string", "rgg_last_cuda_error", "rgg_grouped_gemm_noalloc", "rgg_grouped_gemm_swiglu",
    "rgg_grouped_gemm_fp8", "rgg_grouped_gemm_gather", "rgg_grouped_gemm_swiglu_gather", "rgg_export_walk",
)


class RggError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


class _Options(ctypes.Structure):
    _fields_ = [("bm", ctypes.c_int), ("bn", ctypes.c_int), ("stages", ctypes.c_int),
                ("max_ctas", ctypes.c_int), ("timeout_ns", ctypes.c_uint64), ("host_counts", ctypes.c_void_p),
                ("debug_flags", ctypes.c_int), ("tail64", ctypes.c_int),
                ("op", ctypes.c_int), ("walk_order", ctypes.c_int), ("gather_mode", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_int64), ("mixed", ctypes.c_int),
                ("mixed_pair_sms", ctypes.c_int), ("pair_min_rows", ctypes.c_int)]


class _PlanInfo(ctypes.Structure):
    _fields_ = [("bm", ctypes.c_int), ("bn", ctypes.c_int), ("bk", ctypes.c_int), ("stages", ctypes.c_int),
                ("grid", ctypes.c_int), ("threads", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("tmem_cols", ctypes.c_int), ("max_tiles", ctypes.c_int64), ("tail64", ctypes.c_int),
                ("walk_order", ctypes.c_int), ("gather_mode", ctypes.c_int), ("workspace_bytes", ctypes.c_int64),
                ("mixed", ctypes.c_int), ("single_grid", ctypes.c_int), ("single_stages", ctypes.c_int),
                ("single_smem_bytes", ctypes.c_int), ("pair_min_rows", ctypes.c_int),
                ("device_split", ctypes.c_int)]


_lock = threading.Lock()
_lib = None
_handles: dict[int, ctypes.c_void_p] = {}


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load librgg.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = open_library(_LIB_PATH)
        return _lib


def open_library(path: str) -> ctypes.CDLL:
    """Open a build of the C ABI (librgg.so, or librgg_debug.so: the same
    entry points with every device access bounds-checked) and declare its
    entry points' argument types."""
    if not os.path.exists(path):
        raise RuntimeError("%s is not built: run __graft_entry__.build() first" % path)
    lib = ctypes.CDLL(path)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.rgg_create.argtypes = [ctypes.POINTER(ctypes.c_void_p), I]
    lib.rgg_create.restype = I
    lib.rgg_destroy.argtypes = [P]
    lib.rgg_destroy.restype = None
    lib.rgg_grouped_gemm.argtypes = [P, P, P, P, P, I, I64, I, I, P, ctypes.POINTER(_Options)]
    lib.rgg_grouped_gemm.restype = I
    lib.rgg_export_tiles.argtypes = [P, P, I, I64, I, I, I, P, I64, P, P]
    lib.rgg_export_tiles.restype = I
    lib.rgg_export_walk.argtypes = [P, P, I, I64, I, I, I, I, P, I64, P, P]
    lib.rgg_export_walk.restype = I
    lib.rgg_query_status.argtypes = [P, P]
    lib.rgg_query_status.restype = I
    lib.rgg_plan.argtypes = [I, I, I, I64, I, I, ctypes.POINTER(_Options), ctypes.POINTER(_PlanInfo)]
    lib.rgg_plan.restype = I
    lib.rgg_status_string.argtypes = [I]
    lib.rgg_status_string.restype = ctypes.c_char_p
    lib.rgg_last_cuda_error.argtypes = []
    lib.rgg_last_cuda_error.restype = ctypes.c_char_p
    lib.rgg_grouped_gemm_swiglu.argtypes = [P, P, P, P, P, I, I64, I, I, P, ctypes.POINTER(_Options)]
    lib.rgg_grouped_gemm_swiglu.restype = I
    lib.rgg_grouped_gemm_fp8.argtypes = [P, P, P, P, P, P, P, I, I64, I, I, P, ctypes.POINTER(_Options)]
    lib.rgg_grouped_gemm_fp8.restype = I
    for name in ("rgg_grouped_gemm_gather", "rgg_grouped_gemm_swiglu_gather"):
        fn = getattr(lib, name)
        fn.argtypes = [P, P, I64, P, P, P, P, I, I64, I, I, P, ctypes.POINTER(_Options)]
        fn.restype = I
    lib.rgg_grouped_gemm_noalloc.argtypes = [P, P, P, P, I, I64, I, I, P, P]
    lib.rgg_grouped_gemm_noalloc.restype = I
    return lib


def debug_library_path() -> str:
    return _DEBUG_LIB_PATH


def rgg_status_string(status: int) -> str:
    return load_library().rgg_status_string(int(status)).decode()


def _raise(status: int, call: str):
    lib = load_library()
    msg = "%s: %s" % (call, lib.rgg_status_string(status).decode())
    if status == RGG_ERR_CUDA:
        msg += " [%s]" % lib.rgg_last_cuda_error().decode()
    raise RggError(status, msg)


def _handle(device: int) -> ctypes.c_void_p:
    lib = load_library()
    with _lock:
        h = _handles.get(device)
        if h is None:
            h = ctypes.c_void_p()
            s = lib.rgg_create(ctypes.byref(h), int(device))
            if s != RGG_OK:
                _raise(s, "rgg_create(device=%d)" % device)
            _handles[device] = h
        return h


def _options(bm=0, bn=0, stages=0, max_ctas=0, timeout_ns=0, host_counts=None, debug_flags=0, tail64=0,
             op=0, walk_order=0, gather_mode=0, mixed=0, mixed_pair_sms=0, pair_min_rows=0):
    opt = _Options(int(bm), int(bn), int(stages), int(max_ctas), int(timeout_ns), None, int(debug_flags),
                   int(tail64), int(op), int(walk_order), int(gather_mode))
    opt.mixed = int(mixed)
    opt.mixed_pair_sms = int(mixed_pair_sms)
    opt.pair_min_rows = int(pair_min_rows)
    keep = None
    if host_counts is not None:
        import numpy as np
        keep = np.ascontiguousarray(np.asarray(host_counts, dtype=np.int32))
        opt.host_counts = keep.ctypes.data
    return opt, keep


def _set_workspace(opt, workspace):
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        opt.workspace = workspace.data_ptr()
        opt.workspace_bytes = workspace.numel() * workspace.element_size()


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def rgg_grouped_gemm(X, W, group_offsets, Y=None, *, bm=0, bn=0, stages=0, max_ctas=0, timeout_ns=0,
                     host_counts=None, debug_flags=0, tail64=0, walk_order=0, mixed=0, mixed_pair_sms=0,
                     pair_min_rows=0, stream=None, check=False):
    """Y_e = X_e . W_e for every expert (one kernel launch, asynchronous; the
    mixed launch, ``mixed=1``, runs a CTA-pair kernel and a 1-CTA kernel side
    by side).

    X: bf16 CUDA [M_tot, K]; W: bf16 CUDA [E, K, N]; group_offsets: int32
    CUDA [E+1]; Y: optional bf16 CUDA [M_tot, N] (allocated uninitialised when
    omitted: rows that belong to no expert are never written).  Keyword
    options map to ``rgg_options``.  ``check=True`` synchronises the stream
    and raises if the device reported bad offsets or a timeout.
    """
    import torch
    if not (X.is_cuda and W.is_cuda and group_offsets.is_cuda):
        raise ValueError("X, W and group_offsets must be CUDA tensors")
    if X.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or group_offsets.dtype != torch.int32:
        raise TypeError("X and W must be bf16 and group_offsets int32")
    if X.dim() != 2 or W.dim() != 3 or group_offsets.dim() != 1:
        raise ValueError("X must be [M_tot, K], W [E, K, N] and group_offsets [E+1]")
    if not (X.is_contiguous() and W.is_contiguous() and group_offsets.is_contiguous()):
        raise ValueError("X, W and group_offsets must be contiguous")
    M_tot, K = X.shape
    E, K2, N = W.shape
    if K2 != K or group_offsets.numel() != E + 1:
        raise ValueError("shape mismatch: X %s, W %s, offsets %d" % (tuple(X.shape), tuple(W.shape),
                                                                     group_offsets.numel()))
    device = X.device.index if X.device.index is not None else torch.cuda.current_device()
    if Y is None:
        Y = torch.empty(M_tot, N, dtype=torch.bfloat16, device=X.device)
    elif Y.shape != (M_tot, N) or Y.dtype != torch.bfloat16 or not Y.is_contiguous() or not Y.is_cuda:
        raise ValueError("Y must be a contiguous bf16 CUDA tensor of shape [M_tot, N]")
    lib = load_library()
    opt, keep = _options(bm, bn, stages, max_ctas, timeout_ns, host_counts, debug_flags, tail64, 0, walk_order,
                         mixed=mixed, mixed_pair_sms=mixed_pair_sms, pair_min_rows=pair_min_rows)
    st = _stream_ptr(stream, device)
    s = lib.rgg_grouped_gemm(_handle(device), X.data_ptr(), W.data_ptr(), group_offsets.data_ptr(), Y.data_ptr(),
                             E, M_tot, K, N, st, ctypes.byref(opt))
    del keep
    if s != RGG_OK:
        _raise(s, "rgg_grouped_gemm")
    if check:
        s = lib.rgg_query_status(_handle(device), st)
        if s != RGG_OK:
            _raise(s, "rgg_grouped_gemm (device status)")
    return Y


def rgg_grouped_gemm_swiglu(X, W13, group_offsets, H=None, *, bm=0, bn=0, stages=0, max_ctas=0, timeout_ns=0,
                            host_counts=None, debug_flags=0, tail64=0, walk_order=0, mixed=0, mixed_pair_sms=0,
                            pair_min_rows=0, stream=None, check=False):
    """H = silu(X_e . W13_e[:, :N]) * (X_e . W13_e[:, N:]) for every expert,
    one kernel launch (the fused gate-up projection with SiLU activation).

    X: bf16 CUDA [M_tot, K]; W13: bf16 CUDA [E, K, 2N] (gate columns first);
    group_offsets: int32 CUDA [E+1]; H: optional bf16 CUDA [M_tot, N]."""
    import torch
    if not (X.is_cuda and W13.is_cuda and group_offsets.is_cuda):
        raise ValueError("X, W13 and group_offsets must be CUDA tensors")
    if X.dtype != torch.bfloat16 or W13.dtype != torch.bfloat16 or group_offsets.dtype != torch.int32:
        raise TypeError("X and W13 must be bf16 and group_offsets int32")
    if not (X.is_contiguous() and W13.is_contiguous() and group_offsets.is_contiguous()):
        raise ValueError("X, W13 and group_offsets must be contiguous")
    M_tot, K = X.shape
    E, K2, N2 = W13.shape
    if K2 != K or N2 % 2 != 0 or group_offsets.numel() != E + 1:
        raise ValueError("shape mismatch: X %s, W13 %s, offsets %d" % (tuple(X.shape), tuple(W13.shape),
                                                                      group_offsets.numel()))
    N = N2 // 2
    device = X.device.index if X.device.index is not None else torch.cuda.current_device()
    if H is None:
        H = torch.empty(M_tot, N, dtype=torch.bfloat16, device=X.device)
    elif H.shape != (M_tot, N) or H.dtype != torch.bfloat16 or not H.is_contiguous() or not H.is_cuda:
        raise ValueError("H must be a contiguous bf16 CUDA tensor of shape [M_tot, N]")
    lib = load_library()
    opt, keep = _options(bm, bn, stages, max_ctas, timeout_ns, host_counts, debug_flags, tail64, 0, walk_order,
                         mixed=mixed, mixed_pair_sms=mixed_pair_sms, pair_min_rows=pair_min_rows)
    st = _stream_ptr(stream, device)
    s = lib.rgg_grouped_gemm_swiglu(_handle(device), X.data_ptr(), W13.data_ptr(), group_offsets.data_ptr(),
                                    H.data_ptr(), E, M_tot, K, N, st, ctypes.byref(opt))
    del keep
    if s != RGG_OK:
        _raise(s, "rgg_grouped_gemm_swiglu")
    if check:
        s = lib.rgg_query_status(_handle(device), st)
        if s != RGG_OK:
            _raise(s, "rgg_grouped_gemm_swiglu (device status)")
    return H


def rgg_grouped_gemm_fp8(X8, W8, sx, sw, group_offsets, Y=None, *, bm=0, bn=0, stages=0, max_ctas=0,
                         timeout_ns=0, host_counts=None, debug_flags=0, tail64=0, walk_order=0, stream=None,
                         check=False):
    """Y[i, j] = sx[i] * sw[e, j] * (X8_e . W8_e)[i, j] with FP8 E4M3 operands.

    X8: float8_e4m3fn CUDA [M_tot, K]; W8: float8_e4m3fn CUDA [E, K, N];
    sx: float32 CUDA [M_tot]; sw: float32 CUDA [E, N]; group_offsets: int32
    CUDA [E+1]; Y: optional bf16 CUDA [M_tot, N]."""
    import torch
    for t in (X8, W8, sx, sw, group_offsets):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("all operands must be contiguous CUDA tensors")
    if X8.dtype != torch.float8_e4m3fn or W8.dtype != torch.float8_e4m3fn:
        raise TypeError("X8 and W8 must be float8_e4m3fn")
    if sx.dtype != torch.float32 or sw.dtype != torch.float32 or group_offsets.dtype != torch.int32:
        raise TypeError("sx and sw must be float32 and group_offsets int32")
    M_tot, K = X8.shape
    E, K2, N = W8.shape
    if K2 != K or group_offsets.numel() != E + 1 or sx.shape != (M_tot,) or sw.shape != (E, N):
        raise ValueError("shape mismatch")
    device = X8.device.index if X8.device.index is not None else torch.cuda.current_device()
    if Y is None:
        Y = torch.empty(M_tot, N, dtype=torch.bfloat16, device=X8.device)
    elif Y.shape != (M_tot, N) or Y.dtype != torch.bfloat16 or not Y.is_contiguous() or not Y.is_cuda:
        raise ValueError("Y must be a contiguous bf16 CUDA tensor of shape [M_tot, N]")
    lib = load_library()
    opt, keep = _options(bm, bn, stages, max_ctas, timeout_ns, host_counts, debug_flags, tail64, 0, walk_order)
    st = _stream_ptr(stream, device)
    s = lib.rgg_grouped_gemm_fp8(_handle(device), X8.data_ptr(), W8.data_ptr(), sx.data_ptr(), sw.data_ptr(),
                                 group_offsets.data_ptr(), Y.data_ptr(), E, M_tot, K, N, st, ctypes.byref(opt))
    del keep
    if s != RGG_OK:
        _raise(s, "rgg_grouped_gemm_fp8")
    if check:
        s = lib.rgg_query_status(_handle(device), st)
        if s != RGG_OK:
            _raise(s, "rgg_grouped_gemm_fp8 (device status)")
    return Y


def rgg_grouped_gemm_noalloc(X, W, group_offsets, Y=None, status_out=None, stream=None):
    """The same product through the entry point that allocates nothing (no
    handle; the kernel's status word lives in a fixed device array inside
    librgg.so).  For callers that cannot allocate device memory where they run
    the GEMM.  ``status_out``: optional int32 CUDA tensor [1] that receives the
    device status once the stream reaches it.  Y, if omitted, is allocated
    here by torch -- pass it in to allocate nothing."""
    import torch
    M_tot, K = X.shape
    E, _, N = W.shape
    if Y is None:
        Y = torch.empty(M_tot, N, dtype=torch.bfloat16, device=X.device)
    device = X.device.index if X.device.index is not None else torch.cuda.current_device()
    st = _stream_ptr(stream, device)
    s = load_library().rgg_grouped_gemm_noalloc(X.data_ptr(), W.data_ptr(), group_offsets.data_ptr(), Y.data_ptr(),
                                                E, M_tot, K, N,
                                                status_out.data_ptr() if status_out is not None else None, st)
    if s != RGG_OK:
        _raise(s, "rgg_grouped_gemm_noalloc")
    return Y


def _gather_call(name, X_tok, row_index, W, group_offsets, out, swiglu, bm, bn, stages, max_ctas, timeout_ns,
                 host_counts, debug_flags, tail64, walk_order, gather_mode, workspace, stream, check):
    import torch
    if not (X_tok.is_cuda and row_index.is_cuda and W.is_cuda and group_offsets.is_cuda):
        raise ValueError("X_tok, row_index, W and group_offsets must be CUDA tensors")
    if (X_tok.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or row_index.dtype != torch.int32
            or group_offsets.dtype != torch.int32):
        raise TypeError("X_tok and W must be bf16, row_index and group_offsets int32")
    if not all(t.is_contiguous() for t in (X_tok, row_index, W, group_offsets)):
        raise ValueError("X_tok, row_index, W and group_offsets must be contiguous")
    T, K = X_tok.shape
    E, K2, NW = W.shape
    M_tot = row_index.numel()
    if K2 != K or group_offsets.numel() != E + 1 or row_index.dim() != 1 or (swiglu and NW % 2 != 0):
        raise ValueError("shape mismatch: X_tok %s, row_index %s, W %s, offsets %d" % (
            tuple(X_tok.shape), tuple(row_index.shape), tuple(W.shape), group_offsets.numel()))
    N = NW // 2 if swiglu else NW
    device = X_tok.device.index if X_tok.device.index is not None else torch.cuda.current_device()
    if out is None:
        out = torch.empty(M_tot, N, dtype=torch.bfloat16, device=X_tok.device)
    elif out.shape != (M_tot, N) or out.dtype != torch.bfloat16 or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("the output must be a contiguous bf16 CUDA tensor of shape [M_tot, N]")
    lib = load_library()
    opt, keep = _options(bm, bn, stages, max_ctas, timeout_ns, host_counts, debug_flags, tail64, 0, walk_order,
                         gather_mode)
    _set_workspace(opt, workspace)
    st = _stream_ptr(stream, device)
    s = getattr(lib, name)(_handle(device), X_tok.data_ptr(), T, row_index.data_ptr(), W.data_ptr(),
                           group_offsets.data_ptr(), out.data_ptr(), E, M_tot, K, N, st, ctypes.byref(opt))
    del keep
    if s != RGG_OK:
        _raise(s, name)
    if check:
        s = lib.rgg_query_status(_handle(device), st)
        if s != RGG_OK:
            _raise(s, name + " (device status)")
    return out


def rgg_grouped_gemm_gather(X_tok, row_index, W, group_offsets, Y=None, *, bm=0, bn=0, stages=0, max_ctas=0,
                            timeout_ns=0, host_counts=None, debug_flags=0, tail64=0, walk_order=0, gather_mode=0,
                            workspace=None, stream=None, check=False):
    """Y[i] = X_tok[row_index[i]] . W_e for every routed row i of expert e,
    the token gather fused into the kernel's activation loads.

    X_tok: bf16 CUDA [T, K]; row_index: int32 CUDA [M_tot]; W: bf16 CUDA
    [E, K, N]; group_offsets: int32 CUDA [E+1]; Y: optional bf16 CUDA
    [M_tot, N] (routed row order).  gather_mode: 0 auto, 1 fused (TMA
    tile::gather4 in the GEMM), 2 two-pass (row gather into a workspace, then
    the grouped GEMM); workspace: CUDA tensor of at least M_tot*K*2 bytes,
    needed by the two-pass mode (the library allocates nothing: without one
    the automatic mode runs the fused gather)."""
    return _gather_call("rgg_grouped_gemm_gather", X_tok, row_index, W, group_offsets, Y, False, bm, bn, stages,
                        max_ctas, timeout_ns, host_counts, debug_flags, tail64, walk_order, gather_mode, workspace,
                        stream, check)


def rgg_grouped_gemm_swiglu_gather(X_tok, row_index, W13, group_offsets, H=None, *, bm=0, bn=0, stages=0,
                                   max_ctas=0, timeout_ns=0, host_counts=None, debug_flags=0, tail64=0,
                                   walk_order=0, gather_mode=0, workspace=None, stream=None, check=False):
    """H[i] = silu(x W13_e[:, :N]) * (x W13_e[:, N:]) with x = X_tok[row_index[i]]:
    the fused gate-up projection reading its tokens through the gather.

    W13: bf16 CUDA [E, K, 2N] (gate columns first); H: optional bf16 CUDA [M_tot, N]."""
    return _gather_call("rgg_grouped_gemm_swiglu_gather", X_tok, row_index, W13, group_offsets, H, True, bm, bn,
                        stages, max_ctas, timeout_ns, host_counts, debug_flags, tail64, walk_order, gather_mode,
                        workspace, stream, check)


def rgg_export_tiles(group_offsets, M_tot: int, N: int, bm: int, bn: int, cap: int | None = None, stream=None):
    """The flat tile list the kernel walks, built on the device by the same
    code: returns (int32 CPU tensor [min(T, cap), 4] of (expert, row0, rows,
    col0), T).  Raises if the device rejects the offsets."""
    return _export("rgg_export_tiles", group_offsets, M_tot, N, bm, bn, None, cap, stream)


def rgg_export_walk(group_offsets, M_tot: int, N: int, bm: int, bn: int, walk_order: int, cap: int | None = None,
                    stream=None):
    """The same tile list in the order walk order ``walk_order`` (0..4)
    visits it: row p is the tile at walk position p.  Returns (descriptors, T)
    as rgg_export_tiles."""
    return _export("rgg_export_walk", group_offsets, M_tot, N, bm, bn, int(walk_order), cap, stream)


def _export(name, group_offsets, M_tot, N, bm, bn, walk_order, cap, stream):
    import torch
    E = group_offsets.numel() - 1
    device = group_offsets.device.index if group_offsets.device.index is not None else torch.cuda.current_device()
    if cap is None:
        cap = (M_tot // bm + E) * (-(-N // bn))
    desc = torch.empty(max(cap, 1) * 4, dtype=torch.int32, device=group_offsets.device)
    n = torch.empty(1, dtype=torch.int32, device=group_offsets.device)
    lib = load_library()
    st = _stream_ptr(stream, device)
    args = [_handle(device), group_offsets.data_ptr(), E, int(M_tot), int(N), int(bm), int(bn)]
    if walk_order is not None:
        args.append(walk_order)
    s = getattr(lib, name)(*args, desc.data_ptr(), int(cap), n.data_ptr(), st)
    if s != RGG_OK:
        _raise(s, name)
    s = lib.rgg_query_status(_handle(device), st)
    T = int(n.item())
    if s not in (RGG_OK, RGG_ERR_CAPACITY):
        _raise(s, name + " (device status)")
    return desc[: 4 * min(T, cap)].view(-1, 4).cpu(), T


def rgg_query_status(device: int | None = None, stream=None) -> int:
    """Synchronise the stream, return and clear the device status word."""
    import torch
    if device is None:
        device = torch.cuda.current_device()
    return int(load_library().rgg_query_status(_handle(device), _stream_ptr(stream, device)))


def rgg_plan(E: int, M_tot: int, K: int, N: int, *, num_sms: int = 0, smem_optin: int = 0, bm=0, bn=0,
             stages=0, max_ctas=0, host_counts=None, tail64=0, op: str = "gemm",
             walk_order=0, gather_mode=0, workspace=None, mixed=0, mixed_pair_sms=0, pair_min_rows=0) -> dict:
    """The launch configuration rgg_grouped_gemm (op="gemm") or
    rgg_grouped_gemm_swiglu (op="swiglu", N = output width) would use (host-only).
    For the gather ops, ``workspace`` (the tensor the call would get, True
    for "a workspace will be given", or None) decides whether the two-pass
    mode can run; the planner only looks at whether there is one."""
    lib = load_library()
    opt, keep = _options(bm, bn, stages, max_ctas, 0, host_counts, 0, tail64,
                         {"gemm": 0, "swiglu": 1, "fp8": 2, "gather": 3, "swiglu_gather": 4}[op], walk_order,
                         gather_mode, mixed=mixed, mixed_pair_sms=mixed_pair_sms, pair_min_rows=pair_min_rows)
    if workspace is True:
        opt.workspace = 16  # never dereferenced: rgg_plan reads only whether a workspace is given
        opt.workspace_bytes = 1 << 62
    else:
        _set_workspace(opt, workspace)
    info = _PlanInfo()
    s = lib.rgg_plan(int(num_sms), int(smem_optin), int(E), int(M_tot), int(K), int(N), ctypes.byref(opt),
                     ctypes.byref(info))
    del keep
    if s != RGG_OK:
        _raise(s, "rgg_plan")
    return {f: getattr(info, f) for f, _ in _PlanInfo._fields_}
