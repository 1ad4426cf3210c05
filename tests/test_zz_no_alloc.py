"""rgg_grouped_gemm_noalloc: the entry point for callers that cannot allocate
device memory (an engine plugin that may not allocate in its execute step,
code under CUDA-graph capture in global mode, a process whose memory belongs
to a pool allocator).  It takes no handle and keeps the kernel's status word
in a fixed device array inside librgg.so.

These tests call it through the C ABI and compare its output with the
handle-based rgg_grouped_gemm on the same inputs, on two calls in a row, with
the tolerance the other GPU tests use.  The file is named so that pytest
collects it last; it also passes alone in a fresh process (its first call sets
the device up).
"""
import ctypes

import numpy as np
import pytest
import torch

import ragged_grouped_gemm_02_gb300 as rgg
from ragged_grouped_gemm_02_gb300 import _build
from ragged_grouped_gemm_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RTOL = 1e-2
CANARY = 0x7FC1


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    lib = rgg.load_library()
    P = ctypes.c_void_p
    lib.rgg_grouped_gemm_noalloc.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                             ctypes.c_int, P, P]
    lib.rgg_grouped_gemm_noalloc.restype = ctypes.c_int
    return lib


def _call(lib, X, W, off, Y, status):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.rgg_grouped_gemm_noalloc(X.data_ptr(), W.data_ptr(), off.data_ptr(), Y.data_ptr(),
                                        W.shape[0], X.shape[0], X.shape[1], W.shape[2],
                                        status.data_ptr() if status is not None else None, stream)


@pytest.mark.parametrize("counts,K,N,spare", [([37, 0, 64, 155], 256, 512, 0),
                                              ([500, 3, 0, 257, 1024, 77, 129, 2], 512, 520, 9),
                                              ([16] * 32, 1024, 2048, 0)])
def test_noalloc_matches_handle_entry_point_twice(lib, counts, K, N, spare):
    inp = wl.make_custom(counts, K=K, N=N, seed=51, spare_rows=spare)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    ref = rgg.rgg_grouped_gemm(X, W, off, check=True).double().cpu().numpy()
    M_used = int(inp.offsets[-1])
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        Y = torch.full((X.shape[0], N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        assert _call(lib, X, W, off, Y, status) == rgg.RGG_OK
        torch.cuda.synchronize()
        assert int(status.item()) == rgg.RGG_OK
        got = Y.double().cpu().numpy()
        err = np.abs(got[:M_used] - ref[:M_used])
        assert (err <= RTOL * np.maximum(1.0, np.abs(ref[:M_used]))).all()
        assert bool((Y.view(torch.int16)[M_used:] == CANARY).all())


def test_noalloc_reports_bad_offsets_then_recovers(lib):
    inp = wl.make_custom([50, 10, 40], K=64, N=128, seed=52)
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = torch.zeros(100, 128, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 50, 40, 100], dtype=torch.int32, device="cuda")
    assert _call(lib, X, W, bad, Y, status) == rgg.RGG_OK
    torch.cuda.synchronize()
    assert int(status.item()) == rgg.RGG_ERR_BAD_OFFSETS
    good = torch.from_numpy(inp.offsets).cuda()
    assert _call(lib, X, W, good, Y, status) == rgg.RGG_OK  # the call clears the shared status word
    torch.cuda.synchronize()
    assert int(status.item()) == rgg.RGG_OK


def test_noalloc_rejects_sizes_it_cannot_take(lib):
    P = ctypes.c_void_p
    buf = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.rgg_grouped_gemm_noalloc(P(p), P(p), P(p), P(p), 4097, 64, 64, 64, None, st) == \
        rgg.RGG_ERR_UNSUPPORTED
    assert lib.rgg_grouped_gemm_noalloc(P(p), P(p), P(p), P(p), 4, 64, 60, 64, None, st) == \
        rgg.RGG_ERR_INVALID_ARG
    assert lib.rgg_grouped_gemm_noalloc(P(p), P(p), P(p), P(p), 4, 1 << 31, 64, 64, None, st) == \
        rgg.RGG_ERR_INVALID_ARG
    assert lib.rgg_grouped_gemm_noalloc(P(p + 2), P(p), P(p), P(p), 4, 64, 64, 64, None, st) == \
        rgg.RGG_ERR_INVALID_ARG
