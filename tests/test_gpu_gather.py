"""Parity of the token-gather grouped GEMM (rgg_grouped_gemm_gather and
rgg_grouped_gemm_swiglu_gather) with the fp64 oracle, on a GB300.

The oracle is the pinned gather (routed row i reads token row_index[i]) followed
by the pinned grouped product.  Same bar as the plain GEMM: integer-valued
inputs bit-exact, random inputs |gpu - oracle| <= 1e-2 * max(1, |oracle|),
rows of no expert untouched, index entries of rows of no expert never read.
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
SHAPES = [(64, 128), (64, 192), (64, 256), (128, 128), (128, 192), (128, 256)]
SWIGLU_SHAPES = [(64, 128), (64, 256), (128, 128), (128, 256)]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()


def _canary(rows, cols):
    return torch.full((rows, cols), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def _workspace(mode, M_tot, K):
    """The caller's workspace for the two-pass mode (None for the fused mode)."""
    return torch.empty(M_tot, K, dtype=torch.bfloat16, device="cuda") if mode == 2 else None


def _run(g, swiglu=False, **opts):
    Xtok, W = g.Xtok.cuda(), g.W.cuda()
    idx = torch.from_numpy(g.row_index).cuda()
    off = torch.from_numpy(g.offsets).cuda()
    N = W.shape[2] // 2 if swiglu else W.shape[2]
    Y = _canary(idx.numel(), N)
    if opts.get("gather_mode") == 2 and "workspace" not in opts:  # the two-pass mode runs on a caller workspace
        opts["workspace"] = torch.empty(idx.numel(), Xtok.shape[1], dtype=torch.bfloat16, device="cuda")
    fn = rgg.rgg_grouped_gemm_swiglu_gather if swiglu else rgg.rgg_grouped_gemm_gather
    fn(Xtok, idx, W, off, Y, check=True, **opts)
    torch.cuda.synchronize()
    return Y.cpu()


def _ref(g, swiglu=False):
    f = oracle.grouped_swiglu_gather if swiglu else oracle.grouped_gemm_gather
    return f(wl.bf16_bits(g.Xtok), g.row_index, wl.bf16_bits(g.W), g.offsets)


def _assert_untouched(Y, lo, hi):
    v = Y.view(torch.int16)
    assert bool((v[:lo] == CANARY).all()) and bool((v[hi:] == CANARY).all())


def _check_close(g, Y, swiglu=False):
    ref = _ref(g, swiglu)
    lo, hi = int(g.offsets[0]), int(g.offsets[-1])
    got = Y[lo:hi].double().numpy()
    err = np.abs(got - ref[lo:hi])
    bound = RTOL * np.maximum(1.0, np.abs(ref[lo:hi]))
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, "%d outputs out of tolerance, first %s gpu %r oracle %r" % (
        bad.shape[0], bad[0].tolist(), got[tuple(bad[0])], ref[lo:hi][tuple(bad[0])])
    _assert_untouched(Y, lo, hi)


MODES = [1, 2]  # fused (TMA tile::gather4 in the GEMM), two-pass (row gather, then the grouped GEMM)


@pytest.mark.parametrize("bm,bn", SHAPES)
@pytest.mark.parametrize("tail64", [0, -1])
@pytest.mark.parametrize("mode", MODES)
def test_integer_inputs_bit_exact(bm, bn, tail64, mode):
    # tokens shared between experts (T < M_tot), an empty expert, groups of
    # four cut by the expert's end, and spare rows whose index is -1
    counts = [3, 0, 130, 64, 1, 200, 65, 127, 129]
    g = wl.make_gather_custom(counts, T=256, K=64, N=384, seed=91, integer_valued=True, spare_rows=3)
    Y = _run(g, bm=bm, bn=bn, tail64=tail64, gather_mode=mode)
    ref = _ref(g)
    M_used = int(g.offsets[-1])
    assert np.array_equal(Y[:M_used].double().numpy(), ref[:M_used])
    _assert_untouched(Y, 0, M_used)


@pytest.mark.parametrize("bm,bn", [(64, 256), (128, 192), (128, 128)])
@pytest.mark.parametrize("mode", MODES)
def test_ragged_random_k_and_n_tails(bm, bn, mode):
    # K = 264: the last K block holds one 8-column chunk, the rest zero-filled
    counts = [0, 1, 63, 64, 65, 127, 128, 129, 300, 0, 17]
    g = wl.make_gather_custom(counts, T=400, K=264, N=640, seed=92)
    _check_close(g, _run(g, bm=bm, bn=bn, gather_mode=mode))


@pytest.mark.parametrize("mode", MODES)
def test_auto_plan_many_tiles_and_walk_orders(mode):
    counts = [500, 3, 0, 257, 1024, 77, 129, 2, 640, 64]
    g = wl.make_gather_custom(counts, T=1100, K=512, N=1024, seed=93)
    for walk in (0, 1, 3, 4):
        _check_close(g, _run(g, walk_order=walk, gather_mode=mode))


def test_rows_before_the_first_expert_are_not_read():
    # offsets start at 6: rows [0, 6) belong to no expert and their index is garbage
    g = wl.make_gather_custom([0, 20, 9], T=64, K=128, N=256, seed=94, integer_valued=True, spare_rows=2)
    idx = np.concatenate([np.full(6, 1 << 30, dtype=np.int32), g.row_index])
    off = (g.offsets + 6).astype(np.int32)
    g2 = wl.GatherInputs(g.Xtok, idx, g.W, off, g.counts)
    Y = _run(g2)
    ref = _ref(g2)
    assert np.array_equal(Y[6:35].double().numpy(), ref[6:35])
    _assert_untouched(Y, 6, 35)


@pytest.mark.parametrize("mode", MODES)
def test_identity_index_matches_the_grouped_kernel_bitwise(mode):
    # with row_index = arange the gathered operand is X itself: same tiles,
    # same MMA order, so the two kernels agree bit for bit
    inp = wl.make_custom([100, 0, 37, 300, 5], K=256, N=384, seed=95, spare_rows=3)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    idx = torch.arange(X.shape[0], dtype=torch.int32, device="cuda")
    M_used = int(inp.offsets[-1])
    for bm, bn in [(64, 256), (128, 192)]:
        Y1 = rgg.rgg_grouped_gemm(X, W, off, bm=bm, bn=bn, check=True)
        Y2 = rgg.rgg_grouped_gemm_gather(X, idx, W, off, bm=bm, bn=bn, gather_mode=mode, check=True,
                                         workspace=_workspace(mode, idx.numel(), X.shape[1]))
        assert torch.equal(Y1[:M_used].view(torch.int16), Y2[:M_used].view(torch.int16))


@pytest.mark.parametrize("mode", MODES)
def test_bad_row_index_is_reported_and_other_rows_are_right(mode):
    g = wl.make_gather_custom([40, 0, 70], T=96, K=64, N=256, seed=96, integer_valued=True)
    idx = g.row_index.copy()
    idx[5], idx[77] = 96, -7                     # one past the end, and negative
    Xtok, W = g.Xtok.cuda(), g.W.cuda()
    off = torch.from_numpy(g.offsets).cuda()
    Y = _canary(idx.size, 256)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm_gather(Xtok, torch.from_numpy(idx).cuda(), W, off, Y, gather_mode=mode, check=True,
                                    workspace=_workspace(mode, idx.size, Xtok.shape[1]))
    assert ei.value.status == rgg.RGG_ERR_BAD_ROW_INDEX
    assert rgg.rgg_query_status() == rgg.RGG_OK  # the status word was read and cleared
    ref = _ref(g)
    good = np.ones(idx.size, dtype=bool)
    good[[5, 77]] = False
    assert np.array_equal(Y.cpu()[good].double().numpy(), ref[good])


@pytest.mark.parametrize("mode", MODES)
def test_bounded_wait_reports_timeout_and_context_survives(mode):
    g = wl.make_gather_custom([37, 0, 64, 155], T=200, K=256, N=512, seed=97)
    Xtok, W = g.Xtok.cuda(), g.W.cuda()
    idx, off = torch.from_numpy(g.row_index).cuda(), torch.from_numpy(g.offsets).cuda()
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm_gather(Xtok, idx, W, off, check=True, timeout_ns=20_000_000, gather_mode=mode,
                                    workspace=_workspace(mode, idx.numel(), Xtok.shape[1]),
                                    debug_flags=rgg.RGG_DEBUG_PRODUCER_STALL)
    assert ei.value.status == rgg.RGG_ERR_DEVICE_TIMEOUT
    assert rgg.rgg_query_status() == rgg.RGG_OK
    _check_close(g, _run(g, gather_mode=mode))


def test_caller_workspace_and_its_size_check():
    # K = 64 with integer inputs: every output is an exact integer of at most 256 in magnitude
    g = wl.make_gather_custom([37, 0, 64, 155], T=200, K=64, N=512, seed=99, integer_valued=True)
    M, K = g.row_index.size, 64
    ws = torch.empty(M * K * 2 + 64, dtype=torch.uint8, device="cuda")
    Y = _run(g, gather_mode=2, workspace=ws)
    assert np.array_equal(Y.double().numpy(), _ref(g))
    Xtok, W = g.Xtok.cuda(), g.W.cuda()
    idx, off = torch.from_numpy(g.row_index).cuda(), torch.from_numpy(g.offsets).cuda()
    for bad in (ws[:M * K * 2 - 16], ws[8:8 + M * K * 2]):  # too small; not 16-byte aligned
        with pytest.raises(rgg.RggError) as ei:
            rgg.rgg_grouped_gemm_gather(Xtok, idx, W, off, gather_mode=2, workspace=bad)
        assert ei.value.status == rgg.RGG_ERR_INVALID_ARG


def test_no_workspace_means_no_two_pass_call():
    # the library allocates nothing: two passes need the caller's workspace, and without one
    # the automatic choice runs the fused gather even where two passes would be faster
    g = wl.make_gather_custom([3000, 7000, 9000], T=9500, K=64, N=256, seed=102, integer_valued=True)
    Xtok, W = g.Xtok.cuda(), g.W.cuda()
    idx, off = torch.from_numpy(g.row_index).cuda(), torch.from_numpy(g.offsets).cuda()
    for kw in (dict(gather_mode=2), dict(bm=256)):
        with pytest.raises(rgg.RggError) as ei:
            rgg.rgg_grouped_gemm_gather(Xtok, idx, W, off, **kw)
        assert ei.value.status == rgg.RGG_ERR_INVALID_ARG
    assert rgg.rgg_plan(3, idx.numel(), 64, 256, op="gather", host_counts=g.counts)["gather_mode"] == 1
    assert np.array_equal(_run(g, host_counts=g.counts).double().numpy(), _ref(g))
    ws = torch.empty(idx.numel(), 64, dtype=torch.bfloat16, device="cuda")
    assert rgg.rgg_plan(3, idx.numel(), 64, 256, op="gather", host_counts=g.counts, workspace=ws)["gather_mode"] == 2
    assert np.array_equal(_run(g, host_counts=g.counts, workspace=ws).double().numpy(), _ref(g))


def test_no_routed_rows():
    Xtok = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(3, 64, 128, dtype=torch.bfloat16, device="cuda")
    off = torch.zeros(4, dtype=torch.int32, device="cuda")
    idx = torch.zeros(0, dtype=torch.int32, device="cuda")
    Y = rgg.rgg_grouped_gemm_gather(Xtok, idx, W, off, check=True)
    assert Y.shape == (0, 128)


@pytest.mark.parametrize("bm,bn", SWIGLU_SHAPES)
@pytest.mark.parametrize("mode", MODES)
def test_swiglu_gather(bm, bn, mode):
    counts = [37, 0, 64, 155, 1, 66]
    g = wl.make_gather_custom(counts, T=180, K=256, N=2 * 256, seed=98, spare_rows=4)
    _check_close(g, _run(g, swiglu=True, bm=bm, bn=bn, gather_mode=mode), swiglu=True)


@pytest.mark.parametrize("name,swiglu", [("decode", False), ("skew16k", False), ("uniform", False),
                                         ("prefill", False), ("decode", True), ("uniform", True)])
def test_full_size(name, swiglu):
    # every routed output against the oracle's gather followed by its whole product, in the
    # launch configuration the benchmark times (tile shape planned from the counts, a caller
    # workspace) and with no workspace (the fused gather)
    g = wl.make_gather_inputs(name)
    ref = _ref(g, swiglu)
    Xtok, W = g.Xtok.cuda(), g.W.cuda()
    idx, off = torch.from_numpy(g.row_index).cuda(), torch.from_numpy(g.offsets).cuda()
    fn = rgg.rgg_grouped_gemm_swiglu_gather if swiglu else rgg.rgg_grouped_gemm_gather
    ws = torch.empty(idx.numel(), Xtok.shape[1], dtype=torch.bfloat16, device="cuda")
    lo, hi = int(g.offsets[0]), int(g.offsets[-1])
    for opts in (dict(workspace=ws), dict()):
        Y = fn(Xtok, idx, W, off, check=True, host_counts=g.counts, **opts)
        torch.cuda.synchronize()
        got = Y[lo:hi].double().cpu().numpy()
        err = np.abs(got - ref[lo:hi])
        bad = ~(err <= RTOL * np.maximum(1.0, np.abs(ref[lo:hi])))
        assert not bad.any(), "%s: %d outputs out of tolerance, max err %.4g" % (name, int(bad.sum()), err.max())
        del Y
