"""Parity of the mixed launch (rgg_options.mixed = 1) with the fp64 oracle, on a GB300.

The mixed launch runs the experts of at least pair_min_rows rows as 256 x 256
tiles on CTA pairs and the other experts as 128 x 256 tiles on single CTAs:
two kernels that share the GPU and either claim tiles from two device
counters, each taking the other class's tiles once its own runs out
(mixed = 1), or walk their own class in a fixed order (mixed = 2; a kernel
whose partner has no SMs walks both classes).  Whatever the split of the SMs
(all to pairs, all to single CTAs, or anything between), whether the kernels
overlap, whichever kernel ends up running a tile, and whatever the host
counts claim, every tile must be computed exactly once:

* integer-valued inputs with K <= 64 are exact in fp32 and bf16, so the result
  must equal the oracle bit for bit (this also pins the 128-row pair tail
  layout and the narrowed last N tile of both kernels);
* random inputs within |gpu - oracle| <= 1e-2 * max(1, |oracle|);
* rows of no expert keep their NaN canary.
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


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()


def _run(inp, offsets=None, mixed=1, **opts):
    off = inp.offsets if offsets is None else np.asarray(offsets, dtype=np.int32)
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = torch.full((X.shape[0], W.shape[2]), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    rgg.rgg_grouped_gemm(X, W, torch.from_numpy(off).cuda(), Y, check=True, mixed=mixed, **opts)
    torch.cuda.synchronize()
    return Y.cpu()


def _check(inp, Y, exact):
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    lo, hi = int(inp.offsets[0]), int(inp.offsets[-1])
    got = Y[lo:hi].double().numpy()
    if exact:
        assert np.array_equal(got, ref[lo:hi])
    else:
        err = np.abs(got - ref[lo:hi])
        bad = ~(err <= RTOL * np.maximum(1.0, np.abs(ref[lo:hi])))
        assert not bad.any(), "%d outputs out of tolerance, max err %.4g" % (int(bad.sum()), err.max())
    v = Y.view(torch.int16)
    assert bool((v[:lo] == CANARY).all()) and bool((v[hi:] == CANARY).all())


# experts of every size class: empty, tiny, <= 64, <= 128, < 256, = 256, pair tiles
# with tails of <= 128 and > 128 rows
COUNTS = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 384, 385, 511, 700, 3, 0, 1000]
SPLITS = [dict(), dict(mixed_pair_sms=-1), dict(mixed_pair_sms=2), dict(mixed_pair_sms=76),
          dict(mixed_pair_sms=146), dict(max_ctas=3), dict(max_ctas=9, mixed_pair_sms=4)]
SPLIT_IDS = ["auto", "no-pairs", "pairs-2", "pairs-76", "pairs-146", "3-ctas", "9-ctas-4-pairs"]


@pytest.mark.parametrize("mode", [1, 2], ids=["claims", "fixed-walks"])
@pytest.mark.parametrize("opts", SPLITS, ids=SPLIT_IDS)
@pytest.mark.parametrize("N", [512, 520, 136])
def test_integer_inputs_bit_exact(opts, N, mode):
    inp = wl.make_custom(COUNTS, K=64, N=N, seed=161, integer_valued=True, spare_rows=5)
    _check(inp, _run(inp, mixed=mode, host_counts=inp.counts, **opts), exact=True)


@pytest.mark.parametrize("mode", [1, 2], ids=["claims", "fixed-walks"])
@pytest.mark.parametrize("wrong", [[1000] * 19, [10] * 19, list(range(19)), [0] * 18 + [10000]],
                         ids=["all-large", "all-small", "ramp", "one-large"])
def test_host_counts_that_disagree_with_the_device_offsets(mode, wrong):
    # the host counts only size the split: the classes come from the device offsets, and a
    # kernel whose partner got no SMs runs both classes
    inp = wl.make_custom(COUNTS, K=64, N=264, seed=169, integer_valued=True, spare_rows=1)
    _check(inp, _run(inp, mixed=mode, host_counts=np.asarray(wrong)), exact=True)


@pytest.mark.parametrize("pmin", [1, 64, 129, 256, 1000, 1 << 20])
def test_class_threshold_moves_experts_between_kernels(pmin):
    inp = wl.make_custom(COUNTS, K=64, N=264, seed=162, integer_valued=True, spare_rows=2)
    for mode in (1, 2):
        _check(inp, _run(inp, mixed=mode, pair_min_rows=pmin), exact=True)
        _check(inp, _run(inp, mixed=mode, pair_min_rows=pmin, host_counts=inp.counts), exact=True)


@pytest.mark.parametrize("opts", [dict(), dict(mixed_pair_sms=-1), dict(mixed_pair_sms=76), dict(mixed=2),
                                  dict(mixed=2, mixed_pair_sms=76)])
def test_random_inputs_with_k_and_n_tails(opts):
    inp = wl.make_custom(COUNTS, K=264, N=520, seed=163, spare_rows=3)
    _check(inp, _run(inp, host_counts=inp.counts, **opts), exact=False)


def test_offsets_that_leave_rows_uncovered():
    counts = [300, 0, 40, 600, 37]
    inp = wl.make_custom(counts, K=64, N=256, seed=164, integer_valued=True, spare_rows=0)
    off = inp.offsets.copy()
    M = int(off[-1])
    shifted = np.concatenate([[50], off[1:-1], [M - 20]]).astype(np.int32)  # rows [0,50) and [M-20, M) uncovered
    Y = _run(inp, offsets=shifted)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), shifted)
    assert np.array_equal(Y[50:M - 20].double().numpy(), ref[50:M - 20])
    v = Y.view(torch.int16)
    assert bool((v[:50] == CANARY).all()) and bool((v[M - 20:] == CANARY).all())


def test_no_rows_and_bad_offsets():
    inp = wl.make_custom([50, 10, 40], K=64, N=128, seed=165)
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = torch.full((100, 128), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    empty = torch.zeros(4, dtype=torch.int32, device="cuda")
    rgg.rgg_grouped_gemm(X, W, empty, Y, check=True, mixed=1)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm(X, W, torch.tensor([0, 50, 40, 100], dtype=torch.int32, device="cuda"), Y,
                             check=True, mixed=1)
    assert ei.value.status == rgg.RGG_ERR_BAD_OFFSETS
    assert bool((Y.view(torch.int16) == CANARY).all())


@pytest.mark.parametrize("opts", [dict(), dict(mixed_pair_sms=-1), dict(mixed_pair_sms=76), dict(mixed=2)])
def test_bounded_wait_reports_timeout_and_context_survives(opts):
    inp = wl.make_custom([300, 37, 0, 64], K=256, N=512, seed=166)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    mode = opts.pop("mixed", 1)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm(X, W, off, check=True, mixed=mode, timeout_ns=20_000_000,
                             debug_flags=rgg.RGG_DEBUG_PRODUCER_STALL, host_counts=inp.counts, **opts)
    assert ei.value.status == rgg.RGG_ERR_DEVICE_TIMEOUT
    assert rgg.rgg_query_status() == rgg.RGG_OK
    _check(inp, _run(inp, mixed=mode, host_counts=inp.counts, **opts), exact=False)


# the split of the SMs taken on the device from the offsets (fixed walks, no host counts): both
# kernels launched over all the SMs, the CTAs past their kernel's share leave at once
SPLIT_COUNTS = [COUNTS, [256] * 19, [16] * 19, [0] * 18 + [3000], [2000, 1] * 9 + [0], [0] * 19]


@pytest.mark.parametrize("counts", SPLIT_COUNTS, ids=["mixed", "all-pairs", "all-single", "one", "alternating",
                                                      "empty"])
@pytest.mark.parametrize("max_ctas", [0, 2, 3, 9])
def test_split_from_device_offsets(counts, max_ctas):
    inp = wl.make_custom(counts, K=64, N=520, seed=169, integer_valued=True, spare_rows=5)
    E, M = len(counts), int(inp.offsets[-1])
    if M == 0:
        pytest.skip("no rows: nothing to plan")
    p = rgg.rgg_plan(E, M, 64, 520, mixed=2, max_ctas=max_ctas)
    assert p["device_split"] == 1
    _check(inp, _run(inp, mixed=2, max_ctas=max_ctas), exact=True)
    # the same offsets again: the graph of a replayed step sees the split it planned
    _check(inp, _run(inp, mixed=2, max_ctas=max_ctas), exact=True)


def test_split_from_device_offsets_follows_new_routing_in_a_graph():
    # one captured launch planned without counts, replayed on offsets of other shapes
    K, N = 128, 392
    shapes = [COUNTS, [16] * 19, [1500] + [10] * 18, [256] * 19]
    inps = [wl.make_custom(c, K=K, N=N, seed=170 + i, spare_rows=0) for i, c in enumerate(shapes)]
    M = max(int(i.offsets[-1]) for i in inps)
    X = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    W = inps[0].W.cuda()
    off = torch.zeros(len(COUNTS) + 1, dtype=torch.int32, device="cuda")
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    off.copy_(torch.from_numpy(inps[0].offsets))
    rgg.rgg_grouped_gemm(X, W, off, Y, check=True, mixed=2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rgg.rgg_grouped_gemm(X, W, off, Y, mixed=2)
    for inp in inps + inps[::-1]:
        m = int(inp.offsets[-1])
        X.zero_()
        X[:m].copy_(inp.X[:m].cuda())
        W.copy_(inp.W.cuda())
        off.copy_(torch.from_numpy(inp.offsets))
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert rgg.rgg_query_status() == rgg.RGG_OK
        ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
        got = Y[:m].double().cpu().numpy()
        err = np.abs(got - ref[:m])
        assert (err <= RTOL * np.maximum(1.0, np.abs(ref[:m]))).all()


def test_repeated_calls_and_graph_replay():
    # the counters are zeroed per call; a captured call (memset + pair kernel +
    # 1-CTA kernel launched after it) replays on new data
    a = wl.make_custom(COUNTS, K=128, N=392, seed=167)
    b = wl.make_custom(COUNTS, K=128, N=392, seed=168)
    X, W = a.X.cuda(), a.W.cuda()
    off = torch.from_numpy(a.offsets).cuda()
    Y = torch.empty(X.shape[0], 392, dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        rgg.rgg_grouped_gemm(X, W, off, Y, check=True, mixed=1, host_counts=a.counts)
    _check(a, Y.cpu(), exact=False)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rgg.rgg_grouped_gemm(X, W, off, Y, mixed=1, host_counts=a.counts)
    for inp in (b, a, b):
        X.copy_(inp.X.cuda())
        W.copy_(inp.W.cuda())
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert rgg.rgg_query_status() == rgg.RGG_OK
        _check(inp, Y.cpu(), exact=False)


@pytest.mark.parametrize("name", ["uniform", "skew16k", "skew2k", "prefill"])
def test_full_size(name):
    # every routed output of the full workload against the whole oracle product, with the
    # split planned from the counts and from the device offsets alone
    inp = wl.make_inputs(name)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    for opts in (dict(host_counts=inp.counts, mixed=1), dict(mixed=1), dict(host_counts=inp.counts, mixed=2),
                 dict(mixed=2)):
        Y = torch.empty(X.shape[0], W.shape[2], dtype=torch.bfloat16, device="cuda")
        rgg.rgg_grouped_gemm(X, W, off, Y, check=True, **opts)
        torch.cuda.synchronize()
        got = Y.double().cpu().numpy()
        err = np.abs(got - ref)
        bad = ~(err <= RTOL * np.maximum(1.0, np.abs(ref)))
        assert not bad.any(), "%s: %d outputs out of tolerance" % (name, int(bad.sum()))
        del Y
