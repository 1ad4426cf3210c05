"""Parity of the FP8 (E4M3) grouped GEMM (rgg_grouped_gemm_fp8) with the fp64
oracle, on a GB300.

Y[i, j] = sx[i] * sw[e, j] * sum_k x8[i, k] w8[e, k, j]; the GPU accumulates in
fp32 and rounds once to bf16, so the same elementwise bar as the bf16 path
applies: |gpu - oracle| <= 1e-2 * max(1, |oracle|).  Integer codes with unit
scales are exact in fp32 and bf16 (bit-exact comparison), which pins the FP8
operand layouts, the K = 32 MMA steps and the 128-column weight panels.
"""

import numpy as np
import pytest
import torch

import oracle
import ragged_grouped_gemm_02_gb300 as rgg
from ragged_grouped_gemm_02_gb300 import _build
from ragged_grouped_gemm_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CANARY = 0x7FC1
RTOL = 1e-2
SHAPES = [(64, 128), (64, 256), (128, 128), (128, 256)]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()


def _run(f, **opts):
    X8, W8 = f.X8.cuda(), f.W8.cuda()
    sx, sw = f.sx.cuda(), f.sw.cuda()
    off = torch.from_numpy(f.offsets).cuda()
    Y = torch.full((X8.shape[0], W8.shape[2]), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    rgg.rgg_grouped_gemm_fp8(X8, W8, sx, sw, off, Y, check=True, **opts)
    torch.cuda.synchronize()
    return Y.cpu()


def _ref(f):
    return oracle.grouped_gemm_fp8(wl.fp8_codes(f.X8), wl.fp8_codes(f.W8), f.sx.numpy(), f.sw.numpy(), f.offsets)


def _check(f, Y):
    ref = _ref(f)
    M_used = int(f.offsets[-1])
    got = Y[:M_used].double().numpy()
    err = np.abs(got - ref[:M_used])
    bound = RTOL * np.maximum(1.0, np.abs(ref[:M_used]))
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, "%d outputs out of tolerance, first %s gpu %r oracle %r" % (
        bad.shape[0], bad[0].tolist(), got[tuple(bad[0])], ref[:M_used][tuple(bad[0])])
    assert bool((Y.view(torch.int16)[M_used:] == CANARY).all())


@pytest.mark.parametrize("bm,bn", SHAPES)
def test_integer_codes_bit_exact(bm, bn):
    # K = 128 = one FP8 stage; K = 384 three stages; ragged counts with an empty expert
    for K in (128, 384):
        f = wl.make_fp8_custom([3, 0, 130, 64, 1, 200, 65], K=K, N=256, seed=91, integer_valued=True,
                               spare_rows=4)
        Y = _run(f, bm=bm, bn=bn)
        ref = _ref(f)
        M_used = int(f.offsets[-1])
        assert np.array_equal(Y[:M_used].double().numpy(), ref[:M_used])
        assert bool((Y.view(torch.int16)[M_used:] == CANARY).all())


@pytest.mark.parametrize("bm,bn", SHAPES)
def test_scaled_random_with_k_and_n_tails(bm, bn):
    # K = 272 (a 16-wide K tail past two 128-wide stages), N = 400 (not a multiple of 128)
    counts = [0, 1, 63, 64, 65, 127, 128, 129, 300, 17]
    f = wl.make_fp8_custom(counts, K=272, N=400, seed=92)
    _check(f, _run(f, bm=bm, bn=bn))


def test_auto_plan_and_tail_tiles():
    f = wl.make_fp8_custom([500, 3, 0, 257, 1024, 77, 129, 2, 640, 64], K=512, N=512, seed=93)
    _check(f, _run(f))
    _check(f, _run(f, tail64=-1))


def test_bad_offsets_rejected():
    f = wl.make_fp8_custom([50, 10, 40], K=64, N=128, seed=94)
    X8, W8, sx, sw = f.X8.cuda(), f.W8.cuda(), f.sx.cuda(), f.sw.cuda()
    Y = torch.full((100, 128), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm_fp8(X8, W8, sx, sw, torch.tensor([0, 50, 40, 100], dtype=torch.int32, device="cuda"),
                                 Y, check=True)
    assert ei.value.status == rgg.RGG_ERR_BAD_OFFSETS
    assert bool((Y.view(torch.int16) == CANARY).all())


@pytest.mark.parametrize("name", ["decode", "uniform", "skew16k", "prefill"])
def test_full_size(name):
    # every routed output against the whole fp64 oracle product, in the benchmark's launch configuration
    f = wl.make_fp8_inputs(name)
    X8, W8, sx, sw = f.X8.cuda(), f.W8.cuda(), f.sx.cuda(), f.sw.cuda()
    off = torch.from_numpy(f.offsets).cuda()
    Y = rgg.rgg_grouped_gemm_fp8(X8, W8, sx, sw, off, check=True, host_counts=f.counts)
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm_fp8(wl.fp8_codes(f.X8), wl.fp8_codes(f.W8), f.sx.numpy(), f.sw.numpy(), f.offsets)
    lo, hi = int(f.offsets[0]), int(f.offsets[-1])
    got = Y[lo:hi].double().cpu().numpy()
    err = np.abs(got - ref[lo:hi])
    bad = ~(err <= RTOL * np.maximum(1.0, np.abs(ref[lo:hi])))
    assert not bad.any(), "%s: %d outputs out of tolerance, max err %.4g" % (name, int(bad.sum()), err.max())
