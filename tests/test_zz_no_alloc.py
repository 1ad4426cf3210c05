"""rgg_grouped_gemm_noalloc: the entry point for callers that cannot allocate
device memory where they run the GEMM (an inference-engine plugin that may not
allocate in its execute step, a process whose device memory all belongs to a
pool allocator).  It takes no handle and keeps the kernel's status word in a
fixed device array inside librgg.so.

These tests call it through the C ABI and compare its output, on two calls in
a row, with the handle-based rgg_grouped_gemm on the same inputs and with the
fp64 oracle, within the tolerance the other GPU tests use
(|gpu - oracle| <= 1e-2 * max(1, |oracle|)).  The file is named so that pytest
collects it last; it also passes alone in a fresh process (its first call sets
the device up).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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
    oracle.build()
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


# The second case is planned as the mixed launch with fixed walks whose SM split is taken on the
# device (no host counts), the last as the mixed launch with device-side tile claims, whose claim
# counters also live in the fixed device array: two calls in a row check that the first leaves
# them ready for the second.
@pytest.mark.parametrize("counts,K,N,spare,mixed", [([37, 0, 64, 155], 256, 512, 0, 0),
                                                    ([500, 3, 0, 257, 1024, 77, 129, 2], 512, 520, 9, 2),
                                                    ([16] * 32, 1024, 2048, 0, 0),
                                                    ([1000, 1100, 900, 1100, 1050, 990, 1010, 1042], 256, 4096,
                                                     4, 1)])
def test_noalloc_matches_handle_entry_point_and_oracle_twice(lib, counts, K, N, spare, mixed):
    inp = wl.make_custom(counts, K=K, N=N, seed=51, spare_rows=spare)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    plan = rgg.rgg_plan(len(counts), X.shape[0], K, N)
    assert plan["mixed"] == mixed
    handle = rgg.rgg_grouped_gemm(X, W, off, check=True).double().cpu().numpy()
    exact = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M_used = int(inp.offsets[-1])
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        Y = torch.full((X.shape[0], N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        assert _call(lib, X, W, off, Y, status) == rgg.RGG_OK
        torch.cuda.synchronize()
        assert int(status.item()) == rgg.RGG_OK
        got = Y.double().cpu().numpy()
        for ref in (handle, exact):
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


def test_noalloc_with_no_rows_checks_the_offsets(lib):
    # M_tot = 0: nothing to multiply, but the offsets are still checked on the device
    X = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(3, 64, 128, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(0, 128, dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for offs, want in (([0, 0, 0, 0], rgg.RGG_OK), ([0, 1, 0, 0], rgg.RGG_ERR_BAD_OFFSETS),
                       ([0, 0, 0, 0], rgg.RGG_OK)):
        off = torch.tensor(offs, dtype=torch.int32, device="cuda")
        assert _call(lib, X, W, off, Y, status) == rgg.RGG_OK
        torch.cuda.synchronize()
        assert int(status.item()) == want


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
