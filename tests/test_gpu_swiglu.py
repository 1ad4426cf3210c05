"""Parity of the fused gate-up projection + SiLU (rgg_grouped_gemm_swiglu)
with the fp64 oracle, on a GB300.

Same bar as the plain GEMM: |gpu - oracle| <= 1e-2 * max(1, |oracle|)
elementwise, rows of no expert untouched.  At full size the oracle value of a
sampled output is silu(g) * u with g and u from the oracle's pinned grouped
GEMM at the gate column j and the up column N + j.
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
SHAPES = [(64, 128), (64, 256), (128, 128), (128, 256),
          pytest.param(256, 128, marks=pytest.mark.pair), pytest.param(256, 256, marks=pytest.mark.pair)]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()


def _run(inp, **opts):
    X, W13 = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    N = W13.shape[2] // 2
    H = torch.full((X.shape[0], N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    rgg.rgg_grouped_gemm_swiglu(X, W13, off, H, check=True, **opts)
    torch.cuda.synchronize()
    return H.cpu()


def _check(inp, H):
    ref = oracle.grouped_swiglu(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M_used = int(inp.offsets[-1])
    got = H[:M_used].double().numpy()
    err = np.abs(got - ref[:M_used])
    bound = RTOL * np.maximum(1.0, np.abs(ref[:M_used]))
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, "%d outputs out of tolerance, first %s gpu %r oracle %r" % (
        bad.shape[0], bad[0].tolist(), got[tuple(bad[0])], ref[:M_used][tuple(bad[0])])
    assert bool((H.view(torch.int16)[M_used:] == CANARY).all())


@pytest.mark.parametrize("bm,bn", SHAPES)
def test_tiny_every_tile_shape(bm, bn):
    inp = wl.make_custom([37, 0, 64, 155], K=256, N=2 * 256, seed=71, spare_rows=4)
    _check(inp, _run(inp, bm=bm, bn=bn))


@pytest.mark.parametrize("bm,bn", SHAPES)
def test_ragged_k_and_n_tails(bm, bn):
    # output N = 520: a half 16-column chunk at the end, and gate panels that
    # run past column N into the up half (masked); K = 264
    counts = [0, 1, 63, 64, 65, 127, 128, 129, 300, 17]
    inp = wl.make_custom(counts, K=264, N=2 * 520, seed=72)
    _check(inp, _run(inp, bm=bm, bn=bn))


def test_auto_plan_and_tail_tiles():
    counts = [500, 3, 0, 257, 1024, 77, 129, 2, 640, 64]
    inp = wl.make_custom(counts, K=512, N=2 * 384, seed=73)
    _check(inp, _run(inp))
    _check(inp, _run(inp, tail64=-1))


def test_bad_offsets_rejected():
    inp = wl.make_custom([50, 10, 40], K=64, N=2 * 128, seed=74)
    X, W13 = inp.X.cuda(), inp.W.cuda()
    H = torch.full((100, 128), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm_swiglu(X, W13, torch.tensor([0, 50, 40, 100], dtype=torch.int32, device="cuda"), H,
                                    check=True)
    assert ei.value.status == rgg.RGG_ERR_BAD_OFFSETS
    assert bool((H.view(torch.int16) == CANARY).all())


@pytest.mark.parametrize("name", ["decode", "uniform", "skew16k", "prefill"])
def test_full_size(name):
    # the workload's weights read as W13 = [gate | up] with N/2 output columns; every routed
    # output against the whole fp64 oracle product, in the benchmark's launch configuration
    inp = wl.make_inputs(name)
    X, W13 = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    H = rgg.rgg_grouped_gemm_swiglu(X, W13, off, check=True, host_counts=inp.counts)
    torch.cuda.synchronize()
    ref = oracle.grouped_swiglu(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    lo, hi = int(inp.offsets[0]), int(inp.offsets[-1])
    got = H[lo:hi].double().cpu().numpy()
    err = np.abs(got - ref[lo:hi])
    bad = ~(err <= RTOL * np.maximum(1.0, np.abs(ref[lo:hi])))
    assert not bad.any(), "%s: %d outputs out of tolerance, max err %.4g" % (name, int(bad.sum()), err.max())


# the mixed launch with the fused epilogue: large experts on CTA pairs (256-row tiles, gate on the
# first CTA and up on the second), small ones on single CTAs, claimed (1) or walked in a fixed
# order (2); integer inputs with K = 64 are exact
MIXED_COUNTS = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 384, 385, 511, 700, 3, 0, 1000]


@pytest.mark.parametrize("mode", [1, 2], ids=["claims", "fixed-walks"])
@pytest.mark.parametrize("opts", [dict(), dict(mixed_pair_sms=-1), dict(mixed_pair_sms=2), dict(mixed_pair_sms=76),
                                  dict(max_ctas=5)], ids=["auto", "no-pairs", "pairs-2", "pairs-76", "5-ctas"])
def test_mixed_launch_bit_exact(mode, opts):
    inp = wl.make_custom(MIXED_COUNTS, K=64, N=2 * 264, seed=75, integer_valued=True, spare_rows=3)
    X, W13 = inp.X.cuda(), inp.W.cuda()
    H = torch.full((X.shape[0], 264), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    rgg.rgg_grouped_gemm_swiglu(X, W13, torch.from_numpy(inp.offsets).cuda(), H, check=True, mixed=mode,
                                host_counts=inp.counts, **opts)
    torch.cuda.synchronize()
    ref = oracle.grouped_swiglu(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M = int(inp.offsets[-1])
    # integer gate and up products are exact; silu(g) * u is then computed in fp32 and rounded to bf16
    got = H.cpu()[:M].double().numpy()
    err = np.abs(got - ref[:M])
    assert (err <= RTOL * np.maximum(1.0, np.abs(ref[:M]))).all(), "max err %.4g" % err.max()
    assert bool((H.view(torch.int16)[M:] == CANARY).all())
