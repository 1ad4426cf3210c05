"""The fp64 CPU oracle for the ragged-M grouped GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline``
and ``--impl reference`` legs may import this package.  The CUDA library never
imports, links or calls it, and it imports nothing from the CUDA library: the
two sides share only the seeded input generators in
``ragged_grouped_gemm_02_gb300.workloads``, which hold none of the method's
arithmetic.

The arithmetic lives in ``rgg_oracle.c`` (plain C, fp64, OpenMP); this module
compiles it with gcc on first use and wraps it with numpy.  Every function
cites the page passage it follows; see the header of ``rgg_oracle.c``.

Inputs are numpy arrays of bf16 *bit patterns* (``uint16``), so the oracle sees
exactly the bf16-rounded values the GPU receives.

Parity status: every function here is pinned by ``tests/test_oracle.py``
against the pages' printed figures, exact rational arithmetic, a library
special case, integer-exact cases and the invariants the pages fix.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rgg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "librgg_oracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_OK = 0
ORACLE_ERR_INVALID_ARG = 1
ORACLE_ERR_BAD_OFFSETS = 4
ORACLE_ERR_BAD_ROW_INDEX = 7


def build(force: bool = False) -> str:
    """Compile ``rgg_oracle.c`` into ``librgg_oracle.so`` next to it."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-std=c11",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.rgg_oracle_check_offsets.argtypes = [P, ctypes.c_int, i64]
        lib.rgg_oracle_check_offsets.restype = ctypes.c_int
        lib.rgg_oracle_grouped_gemm.argtypes = [P, P, P, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int, P, ctypes.c_int]
        lib.rgg_oracle_grouped_gemm.restype = ctypes.c_int
        lib.rgg_oracle_grouped_gemm_points.argtypes = [P, P, P, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int,
                                                       P, P, i64, P, ctypes.c_int]
        lib.rgg_oracle_grouped_gemm_points.restype = ctypes.c_int
        lib.rgg_oracle_tile_list.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, i64]
        lib.rgg_oracle_tile_list.restype = i64
        lib.rgg_oracle_row_utilisation.argtypes = [P, ctypes.c_int, ctypes.c_int]
        lib.rgg_oracle_row_utilisation.restype = ctypes.c_double
        lib.rgg_oracle_grouped_swiglu.argtypes = [P, P, P, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int, P,
                                                  ctypes.c_int]
        lib.rgg_oracle_grouped_swiglu.restype = ctypes.c_int
        lib.rgg_oracle_silu.argtypes = [ctypes.c_double]
        lib.rgg_oracle_silu.restype = ctypes.c_double
        lib.rgg_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.rgg_oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.rgg_oracle_grouped_gemm_fp8.argtypes = [P, P, P, P, P, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int,
                                                    P, ctypes.c_int]
        lib.rgg_oracle_grouped_gemm_fp8.restype = ctypes.c_int
        lib.rgg_oracle_gather_rows.argtypes = [P, i64, ctypes.c_int, P, i64, i64, P]
        lib.rgg_oracle_gather_rows.restype = ctypes.c_int
        lib.rgg_oracle_max_threads.argtypes = []
        lib.rgg_oracle_max_threads.restype = ctypes.c_int
        del i32
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _as_offsets(off) -> np.ndarray:
    off = np.ascontiguousarray(np.asarray(off, dtype=np.int64))
    if off.ndim != 1 or off.size < 2:
        raise ValueError("group offsets must be a 1-D array of E+1 entries")
    if off.min() < -(2 ** 31) or off.max() >= 2 ** 31:
        raise ValueError("group offsets must fit int32")
    return off.astype(np.int32)


def max_threads() -> int:
    return int(_load().rgg_oracle_max_threads())


def check_offsets(off, M_tot: int) -> int:
    """0 when the offsets are valid (0 <= off[0] <= ... <= off[E] <= M_tot), else 4."""
    off = _as_offsets(off)
    return int(_load().rgg_oracle_check_offsets(_ptr(off), off.size - 1, int(M_tot)))


def grouped_gemm(X_bits: np.ndarray, W_bits: np.ndarray, off, nthreads: int = 0,
                 out: np.ndarray | None = None) -> np.ndarray:
    """Y = X_e . W_e for every expert, in fp64 (worklog, "What I am measuring").

    X_bits: uint16 [M_tot, K]; W_bits: uint16 [E, K, N]; off: int [E+1].
    Rows that belong to no expert keep the value they had in ``out`` (NaN
    when ``out`` is not given), so tests can see that nothing wrote them.
    """
    X_bits, W_bits, off = _as_bits(X_bits), _as_bits(W_bits), _as_offsets(off)
    if X_bits.ndim != 2 or W_bits.ndim != 3:
        raise ValueError("X must be [M_tot, K] and W [E, K, N]")
    M_tot, K = X_bits.shape
    E, K2, N = W_bits.shape
    if K2 != K or off.size != E + 1:
        raise ValueError("shape mismatch: X %s, W %s, offsets %d" % (X_bits.shape, W_bits.shape, off.size))
    if out is None:
        out = np.full((M_tot, N), np.nan, dtype=np.float64)
    if out.shape != (M_tot, N) or out.dtype != np.float64 or not out.flags.c_contiguous:
        raise ValueError("out must be a C-contiguous float64 [M_tot, N] array")
    rc = _load().rgg_oracle_grouped_gemm(_ptr(X_bits), _ptr(W_bits), _ptr(off), E, M_tot, K, N,
                                         _ptr(out), int(nthreads))
    if rc != ORACLE_OK:
        raise OracleError("oracle rejected the arguments (code %d)" % rc)
    return out


def grouped_gemm_points(X_bits: np.ndarray, W_bits: np.ndarray, off, rows, cols,
                        nthreads: int = 0) -> np.ndarray:
    """The same definition at chosen outputs (rows[p], cols[p]) only; NaN where
    the row belongs to no expert."""
    X_bits, W_bits, off = _as_bits(X_bits), _as_bits(W_bits), _as_offsets(off)
    M_tot, K = X_bits.shape
    E, _, N = W_bits.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int32))
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    out = np.empty(rows.size, dtype=np.float64)
    rc = _load().rgg_oracle_grouped_gemm_points(_ptr(X_bits), _ptr(W_bits), _ptr(off), E, M_tot, K, N,
                                                _ptr(rows), _ptr(cols), rows.size, _ptr(out), int(nthreads))
    if rc != ORACLE_OK:
        raise OracleError("oracle rejected the arguments (code %d)" % rc)
    return out


def silu(z: float) -> float:
    """silu(z) = z / (1 + exp(-z)) in fp64, as the fused oracle applies it."""
    return float(_load().rgg_oracle_silu(float(z)))


def grouped_swiglu(X_bits: np.ndarray, W13_bits: np.ndarray, off, nthreads: int = 0,
                   out: np.ndarray | None = None) -> np.ndarray:
    """H = silu(X_e . W13_e[:, :N]) * (X_e . W13_e[:, N:]) per expert, fp64.

    W13_bits: uint16 [E, K, 2N] (gate columns first, then up columns).
    Rows of no expert keep their value in ``out`` (NaN when not given)."""
    X_bits, W13_bits, off = _as_bits(X_bits), _as_bits(W13_bits), _as_offsets(off)
    M_tot, K = X_bits.shape
    E, K2, N2 = W13_bits.shape
    if K2 != K or off.size != E + 1 or N2 % 2 != 0:
        raise ValueError("shape mismatch: X %s, W13 %s, offsets %d" % (X_bits.shape, W13_bits.shape, off.size))
    N = N2 // 2
    if out is None:
        out = np.full((M_tot, N), np.nan, dtype=np.float64)
    rc = _load().rgg_oracle_grouped_swiglu(_ptr(X_bits), _ptr(W13_bits), _ptr(off), E, M_tot, K, N, _ptr(out),
                                           int(nthreads))
    if rc != ORACLE_OK:
        raise OracleError("oracle rejected the arguments (code %d)" % rc)
    return out


def e4m3_to_f64(code: int) -> float:
    """The value of one FP8 E4M3 code (sign, 4-bit exponent with bias 7, 3-bit mantissa)."""
    return float(_load().rgg_oracle_e4m3_to_f64(int(code) & 0xFF))


def grouped_gemm_fp8(X8: np.ndarray, W8: np.ndarray, sx: np.ndarray, sw: np.ndarray, off, nthreads: int = 0,
                     out: np.ndarray | None = None) -> np.ndarray:
    """Y[i, j] = sx[i] * sw[e, j] * sum_k x8[i, k] w8[e, k, j] in fp64.

    X8: uint8 E4M3 codes [M_tot, K]; W8: uint8 E4M3 codes [E, K, N];
    sx: float32 [M_tot]; sw: float32 [E, N]; off: int [E+1]."""
    X8 = np.ascontiguousarray(X8)
    W8 = np.ascontiguousarray(W8)
    if X8.dtype != np.uint8 or W8.dtype != np.uint8:
        raise TypeError("FP8 operands are passed as uint8 codes")
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    off = _as_offsets(off)
    M_tot, K = X8.shape
    E, K2, N = W8.shape
    if K2 != K or off.size != E + 1 or sx.shape != (M_tot,) or sw.shape != (E, N):
        raise ValueError("shape mismatch")
    if out is None:
        out = np.full((M_tot, N), np.nan, dtype=np.float64)
    rc = _load().rgg_oracle_grouped_gemm_fp8(_ptr(X8), _ptr(W8), _ptr(sx), _ptr(sw), _ptr(off), E, M_tot, K, N,
                                             _ptr(out), int(nthreads))
    if rc != ORACLE_OK:
        raise OracleError("oracle rejected the arguments (code %d)" % rc)
    return out


def gather_rows(Xtok_bits: np.ndarray, row_index, begin: int = 0, end: int | None = None,
                out: np.ndarray | None = None) -> np.ndarray:
    """Xg[i] = X_tok[row_index[i]] for begin <= i < end (the token gather the
    worklog's "Scope of these results" leaves out).  Xtok_bits: uint16 [T, K];
    row_index: int [M_tot].  Rows outside [begin, end) keep their value in
    ``out`` (zero when not given).  An index outside [0, T) raises."""
    Xtok_bits = _as_bits(Xtok_bits)
    if Xtok_bits.ndim != 2:
        raise ValueError("X_tok must be [T, K]")
    T, K = Xtok_bits.shape
    idx = np.ascontiguousarray(np.asarray(row_index, dtype=np.int64))
    if idx.ndim != 1:
        raise ValueError("row_index must be 1-D")
    if idx.size and (idx.min() < -(2 ** 31) or idx.max() >= 2 ** 31):
        raise ValueError("row_index must fit int32")
    idx = idx.astype(np.int32)
    M_tot = idx.size
    end = M_tot if end is None else int(end)
    if out is None:
        out = np.zeros((M_tot, K), dtype=np.uint16)
    if out.shape != (M_tot, K) or out.dtype != np.uint16 or not out.flags.c_contiguous:
        raise ValueError("out must be a C-contiguous uint16 [M_tot, K] array")
    if not 0 <= begin <= end <= M_tot:
        raise ValueError("need 0 <= begin <= end <= M_tot")
    rc = _load().rgg_oracle_gather_rows(_ptr(Xtok_bits), T, K, _ptr(idx), int(begin), int(end), _ptr(out))
    if rc != ORACLE_OK:
        raise OracleError("oracle rejected the gather (code %d)" % rc)
    return out


def grouped_gemm_gather(Xtok_bits: np.ndarray, row_index, W_bits: np.ndarray, off, nthreads: int = 0,
                        out: np.ndarray | None = None) -> np.ndarray:
    """Y[i] = X_tok[row_index[i]] . W_e for every row i of every expert e:
    the grouped product of the gathered rows, fp64."""
    off = _as_offsets(off)
    Xg = gather_rows(Xtok_bits, row_index, int(off[0]), int(off[-1]))
    return grouped_gemm(Xg, W_bits, off, nthreads=nthreads, out=out)


def grouped_swiglu_gather(Xtok_bits: np.ndarray, row_index, W13_bits: np.ndarray, off, nthreads: int = 0,
                          out: np.ndarray | None = None) -> np.ndarray:
    """The fused gate-up projection with SiLU of the gathered rows, fp64."""
    off = _as_offsets(off)
    Xg = gather_rows(Xtok_bits, row_index, int(off[0]), int(off[-1]))
    return grouped_swiglu(Xg, W13_bits, off, nthreads=nthreads, out=out)


def tile_list(off, N: int, BM: int, BN: int) -> np.ndarray:
    """The worklog's flat tile list (section 2): int32 [T, 4] rows of
    (expert, row0, rows, col0), expert-major, then M tile, then N tile."""
    off = _as_offsets(off)
    lib = _load()
    T = lib.rgg_oracle_tile_list(_ptr(off), off.size - 1, int(N), int(BM), int(BN), None, 0)
    if T < 0:
        raise OracleError("oracle rejected the tile-list arguments")
    desc = np.zeros((max(T, 1), 4), dtype=np.int32)
    T2 = lib.rgg_oracle_tile_list(_ptr(off), off.size - 1, int(N), int(BM), int(BN), _ptr(desc), T)
    assert T2 == T
    return desc[:T]


def tile_count(off, N: int, BM: int, BN: int) -> int:
    off = _as_offsets(off)
    T = _load().rgg_oracle_tile_list(_ptr(off), off.size - 1, int(N), int(BM), int(BN), None, 0)
    if T < 0:
        raise OracleError("oracle rejected the tile-list arguments")
    return int(T)


def row_utilisation(off, BM: int) -> float:
    """eta of worklog section 2.1: sum m_e / (BM * sum ceil(m_e / BM))."""
    off = _as_offsets(off)
    v = _load().rgg_oracle_row_utilisation(_ptr(off), off.size - 1, int(BM))
    if v < 0:
        raise OracleError("oracle rejected the row-utilisation arguments")
    return float(v)
