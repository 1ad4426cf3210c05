"""Parity of the cluster-multicast kernel (rgg_options.multicast = 1) with the
fp64 oracle, on a GB300.

The kernel runs 128-row 1-CTA tiles on clusters of two CTAs; the two tiles of
each unit share the weight panel (consecutive M tiles of one expert), the X
rows (neighbouring N tiles of an expert's last M tile) or nothing (leftover
tiles of two experts, the second CTA repeating the first's tile when their
count is odd).  The counts below produce every kind: experts with one, two,
three and five M tiles, tails of <= 64 and of 65-128 rows in either CTA,
N tile counts odd and even, odd and even leftover counts, an empty expert and
rows that belong to no expert.  Integer-valued inputs with K <= 64 are exact,
so there the result must equal the oracle bit for bit; otherwise the bar is
|gpu - oracle| <= 1e-2 * max(1, |oracle|).
"""
import zlib

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
# nine experts with an odd M tile count (an odd leftover count when N tiles are odd)
COUNTS_ODD = [3, 0, 130, 64, 1, 200, 65, 127, 129, 300, 257, 513, 40]
# the same without the last expert: eight leftovers
COUNTS_EVEN = COUNTS_ODD[:-1]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()


def _canary(M, N):
    return torch.full((M, N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def _run(inp, offsets=None, **opts):
    off = inp.offsets if offsets is None else np.asarray(offsets, dtype=np.int32)
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = _canary(X.shape[0], W.shape[2])
    rgg.rgg_grouped_gemm(X, W, torch.from_numpy(off).cuda(), Y, check=True, multicast=1, **opts)
    torch.cuda.synchronize()
    return Y.cpu()


def _bit_exact(inp, Y, off=None):
    off = inp.offsets if off is None else off
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), off)
    covered = np.zeros(inp.X.shape[0], dtype=bool)
    covered[off[0]:off[-1]] = True
    assert np.array_equal(Y[covered].double().numpy(), ref[covered]), "integer case not bit-exact"
    assert bool((Y.view(torch.int16)[torch.from_numpy(~covered)] == CANARY).all()), "rows of no expert written"


def _close(got, ref):
    err = np.abs(got - ref)
    bound = RTOL * np.maximum(1.0, np.abs(ref))
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, "%d outputs out of tolerance; first %s: gpu %r oracle %r" % (
        bad.shape[0], bad[0].tolist(), got[tuple(bad[0])], ref[tuple(bad[0])])


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("N", [384, 512, 520])
@pytest.mark.parametrize("counts", [COUNTS_ODD, COUNTS_EVEN], ids=["odd_leftovers", "even_leftovers"])
def test_integer_inputs_bit_exact(bn, N, counts):
    inp = wl.make_custom(counts, K=64, N=N, seed=141, integer_valued=True, spare_rows=5)
    _bit_exact(inp, _run(inp, bn=bn))


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("tail64", [1, -1])
@pytest.mark.parametrize("walk_order", [0, 1, 2])
def test_integer_inputs_walk_orders_and_tails(bn, tail64, walk_order):
    inp = wl.make_custom(COUNTS_ODD, K=64, N=384, seed=142, integer_valued=True, spare_rows=3)
    _bit_exact(inp, _run(inp, bn=bn, tail64=tail64, walk_order=walk_order))


@pytest.mark.parametrize("max_ctas", [2, 6, 38])
def test_few_clusters_walk_every_unit(max_ctas):
    inp = wl.make_custom(COUNTS_ODD, K=64, N=520, seed=143, integer_valued=True, spare_rows=2)
    _bit_exact(inp, _run(inp, bn=256, max_ctas=max_ctas))


@pytest.mark.parametrize("counts,N", [([1], 128), ([1], 256), ([64], 128), ([129], 128), ([0, 5, 0], 384),
                                      ([700], 136)])
def test_single_unit_and_degenerate_cases(counts, N):
    # one tile (the second CTA repeats it without storing), one expert, narrow N
    inp = wl.make_custom(counts, K=64, N=N, seed=144, integer_valued=True, spare_rows=4)
    _bit_exact(inp, _run(inp, bn=128))


def test_all_experts_empty_writes_nothing():
    inp = wl.make_custom([0, 0, 0], K=64, N=256, seed=145, spare_rows=40)
    Y = _run(inp)
    assert bool((Y.view(torch.int16) == CANARY).all())


def test_offsets_need_not_cover_all_rows():
    inp = wl.make_custom([40, 60, 50], K=64, N=256, seed=146, integer_valued=True, spare_rows=20)
    off = np.array([7, 47, 107, 157], dtype=np.int32)
    _bit_exact(inp, _run(inp, offsets=off, bn=256), off)


@pytest.mark.parametrize("bn", [128, 256])
def test_random_values_with_k_and_n_tails(bn):
    counts = [0, 1, 63, 64, 65, 127, 128, 129, 300, 0, 17, 1000]
    inp = wl.make_custom(counts, K=264, N=640, seed=147)
    Y = _run(inp, bn=bn)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    _close(Y.double().numpy(), ref)


def test_bounded_wait_reports_timeout_and_context_survives():
    inp = wl.make_inputs("tiny")
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    Y = _canary(256, 512)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm(X, W, off, Y, check=True, timeout_ns=20_000_000, multicast=1,
                             debug_flags=rgg.RGG_DEBUG_PRODUCER_STALL)
    assert ei.value.status == rgg.RGG_ERR_DEVICE_TIMEOUT
    assert rgg.rgg_query_status() == rgg.RGG_OK
    _bit_exact_tiny = _run(inp)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    _close(_bit_exact_tiny.double().numpy(), ref)


def test_same_result_as_the_1cta_kernel():
    # the same tiles and the same K order per tile: bit-identical to the 128-row 1-CTA kernel
    inp = wl.make_custom(COUNTS_ODD, K=512, N=1024, seed=148)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    Y1 = rgg.rgg_grouped_gemm(X, W, off, check=True, bm=128, bn=256)
    Y2 = rgg.rgg_grouped_gemm(X, W, off, check=True, bn=256, multicast=1)
    M = int(inp.offsets[-1])
    assert torch.equal(Y1[:M].view(torch.int16), Y2[:M].view(torch.int16))


def test_fused_gate_up():
    inp = wl.make_custom([37, 0, 64, 155, 300, 1, 129], K=256, N=2 * 384, seed=149, spare_rows=4)
    X, W13 = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    H = _canary(X.shape[0], 384)
    rgg.rgg_grouped_gemm_swiglu(X, W13, off, H, check=True, multicast=1)
    torch.cuda.synchronize()
    ref = oracle.grouped_swiglu(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M = int(inp.offsets[-1])
    _close(H[:M].double().cpu().numpy(), ref[:M])
    assert bool((H.view(torch.int16)[M:] == CANARY).all())


@pytest.mark.parametrize("K", [128, 384])
def test_fp8_integer_codes_bit_exact(K):
    f = wl.make_fp8_custom(COUNTS_ODD, K=K, N=512, seed=150, integer_valued=True, spare_rows=4)
    X8, W8 = f.X8.cuda(), f.W8.cuda()
    Y = _canary(X8.shape[0], 512)
    rgg.rgg_grouped_gemm_fp8(X8, W8, f.sx.cuda(), f.sw.cuda(), torch.from_numpy(f.offsets).cuda(), Y,
                             check=True, multicast=1)
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm_fp8(wl.fp8_codes(f.X8), wl.fp8_codes(f.W8), f.sx.numpy(), f.sw.numpy(), f.offsets)
    M = int(f.offsets[-1])
    assert np.array_equal(Y[:M].double().cpu().numpy(), ref[:M])
    assert bool((Y.view(torch.int16)[M:].cpu() == CANARY).all())


def _sample_points(off, N, rng, extra=3000):
    rows, cols = [], []
    for e in range(off.size - 1):
        if off[e + 1] > off[e]:
            for r in (off[e], off[e + 1] - 1):
                rows += [r] * 3
                cols += list(rng.integers(0, N, 2)) + [N - 1]
    rows += list(rng.integers(off[0], off[-1], extra))
    cols += list(rng.integers(0, N, extra))
    return np.asarray(rows, dtype=np.int64), np.asarray(cols, dtype=np.int64)


@pytest.mark.parametrize("name", ["skew16k", "skew2k", "uniform", "decode"])
def test_full_size_sampled(name):
    inp = wl.make_inputs(name)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    Y = rgg.rgg_grouped_gemm(X, W, off, check=True, host_counts=inp.counts, multicast=1)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(Y).all())
    rng = np.random.default_rng(zlib.crc32(name.encode()) + 11)
    rows, cols = _sample_points(inp.offsets, inp.W.shape[2], rng)
    ref = oracle.grouped_gemm_points(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets, rows, cols)
    got = Y[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    _close(got, ref)
