"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on a GB300.

Tolerance (the contract the method states): |gpu - oracle| <= 1e-2 * max(1, |oracle|)
elementwise, the oracle in fp64 and not rounded to bf16.  Integer-valued
inputs with K <= 64 are exact in fp32 and in bf16, so there the GPU must
equal the oracle bit for bit; that also pins the TMEM lane-to-row mapping,
the swizzled operand layouts and the row/column masks.  The flat tile list
must match the oracle's enumeration exactly.

Rows that belong to no expert are pre-filled with a NaN canary bit pattern
and must still hold it afterwards.
"""

import numpy as np
import pytest
import torch

import oracle
import ragged_grouped_gemm_02_gb300 as rgg
from ragged_grouped_gemm_02_gb300 import _build
from ragged_grouped_gemm_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CANARY = 0x7FC1  # a bf16 NaN the kernel never produces
RTOL = 1e-2
SHAPES = [(64, 128), (64, 192), (64, 256), (128, 128), (128, 192), (128, 256)]
# 256-row tiles computed by a CTA pair (tcgen05 cta_group::2)
PAIR_SHAPES = [pytest.param(256, 128, marks=pytest.mark.pair), pytest.param(256, 256, marks=pytest.mark.pair)]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()
    assert rgg.load_library() is not None
    return torch.device("cuda:0")


def _canary(M, N):
    return torch.full((M, N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def _run(inp, offsets=None, **opts):
    off = inp.offsets if offsets is None else np.asarray(offsets, dtype=np.int32)
    X = inp.X.cuda()
    W = inp.W.cuda()
    d_off = torch.from_numpy(off).cuda()
    Y = _canary(X.shape[0], W.shape[2])
    rgg.rgg_grouped_gemm(X, W, d_off, Y, check=True, **opts)
    torch.cuda.synchronize()
    return Y.cpu()


def _assert_untouched(Y, rows):
    bits = Y.view(torch.int16)[rows]
    assert bool((bits == CANARY).all()), "rows that belong to no expert were written"


def _assert_close(Y, ref, rows):
    y = Y[rows].double().numpy()
    r = ref[rows]
    err = np.abs(y - r)
    bound = RTOL * np.maximum(1.0, np.abs(r))
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, "%d outputs out of tolerance; first %s: gpu %r oracle %r" % (
        bad.shape[0], bad[0].tolist(), y[tuple(bad[0])], r[tuple(bad[0])])


def _full_parity(inp, offsets=None, **opts):
    off = inp.offsets if offsets is None else np.asarray(offsets, dtype=np.int32)
    Y = _run(inp, off, **opts)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), off)
    M = inp.X.shape[0]
    covered = np.zeros(M, dtype=bool)
    covered[off[0]:off[-1]] = True
    _assert_close(Y, ref, covered)
    if (~covered).any():
        _assert_untouched(Y, torch.from_numpy(~covered))
    return Y, ref


# ---------------------------------------------------------------- small cases

@pytest.mark.parametrize("bm,bn", SHAPES + PAIR_SHAPES)
def test_tiny_config_every_tile_shape(bm, bn):
    _full_parity(wl.make_inputs("tiny"), bm=bm, bn=bn)


def test_tiny_config_auto_plan():
    _full_parity(wl.make_inputs("tiny"))


@pytest.mark.parametrize("bm,bn", SHAPES + PAIR_SHAPES)
@pytest.mark.parametrize("N", [512, 520])
def test_integer_inputs_bit_exact(bm, bn, N):
    # ragged counts around the tile sizes, an empty expert, spare rows at the end;
    # N = 520 leaves a half 16-column chunk (128-bit store path)
    counts = [3, 0, 130, 64, 1, 200, 65, 127]
    inp = wl.make_custom(counts, K=64, N=N, seed=31, integer_valued=True, spare_rows=5)
    Y = _run(inp, bm=bm, bn=bn)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M_used = int(inp.offsets[-1])
    assert np.array_equal(Y[:M_used].double().numpy(), ref[:M_used]), "integer case not bit-exact"
    _assert_untouched(Y, slice(M_used, None))


@pytest.mark.parametrize("bm,bn", SHAPES + PAIR_SHAPES)
@pytest.mark.parametrize("tail64", [0, -1, 1])
def test_integer_inputs_bit_exact_modes(bm, bn, tail64):
    # 64-row tail tiles automatic, off and on
    counts = [3, 0, 130, 64, 1, 200, 65, 127, 129]
    inp = wl.make_custom(counts, K=64, N=384, seed=38, integer_valued=True, spare_rows=3)
    Y = _run(inp, bm=bm, bn=bn, tail64=tail64)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M_used = int(inp.offsets[-1])
    assert np.array_equal(Y[:M_used].double().numpy(), ref[:M_used])
    _assert_untouched(Y, slice(M_used, None))


@pytest.mark.parametrize("bm,bn", SHAPES + PAIR_SHAPES)
@pytest.mark.parametrize("walk_order", [1, 2, 3, 4])
def test_integer_inputs_bit_exact_walk_orders(bm, bn, walk_order):
    # any walk over the tile list visits every tile exactly once
    counts = [3, 0, 130, 64, 1, 200, 65, 127, 129, 500]
    inp = wl.make_custom(counts, K=64, N=384, seed=39, integer_valued=True, spare_rows=3)
    Y = _run(inp, bm=bm, bn=bn, walk_order=walk_order)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M_used = int(inp.offsets[-1])
    assert np.array_equal(Y[:M_used].double().numpy(), ref[:M_used])
    _assert_untouched(Y, slice(M_used, None))


@pytest.mark.parametrize("bm,bn", [(64, 256), (128, 192), (128, 128)] + PAIR_SHAPES)
def test_ragged_random_k_and_n_tails(bm, bn):
    # K = 264 (a 8-wide K tail), N = 640 (not a multiple of 192 or 256), sizes around 64/128
    counts = [0, 1, 63, 64, 65, 127, 128, 129, 300, 0, 17]
    inp = wl.make_custom(counts, K=264, N=640, seed=32)
    _full_parity(inp, bm=bm, bn=bn)


def test_ragged_random_auto_plan_many_tiles():
    counts = [500, 3, 0, 257, 1024, 77, 129, 2, 640, 64]
    inp = wl.make_custom(counts, K=512, N=1024, seed=33)
    _full_parity(inp)


def test_offsets_need_not_cover_all_rows():
    # experts own rows [7, 7 + 150); rows before and after belong to nobody
    inp = wl.make_custom([40, 60, 50], K=128, N=256, seed=34, spare_rows=20)
    off = np.array([7, 47, 107, 157], dtype=np.int32)
    _full_parity(inp, offsets=off, bm=128, bn=128)
    _full_parity(inp, offsets=off, bm=64, bn=256)


@pytest.mark.pair
def test_offsets_need_not_cover_all_rows_pair():
    inp = wl.make_custom([40, 60, 50], K=128, N=256, seed=34, spare_rows=20)
    off = np.array([7, 47, 107, 157], dtype=np.int32)
    _full_parity(inp, offsets=off, bm=256, bn=256)


def test_all_experts_empty_writes_nothing():
    inp = wl.make_custom([0, 0, 0], K=64, N=128, seed=35, spare_rows=50)
    Y = _run(inp)
    _assert_untouched(Y, slice(None))


def test_zero_rows():
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(2, 64, 128, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    rgg.rgg_grouped_gemm(X, W, torch.zeros(3, dtype=torch.int32, device="cuda"), Y, check=True)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm(X, W, torch.tensor([0, 1, 1], dtype=torch.int32, device="cuda"), Y, check=True)
    assert ei.value.status == rgg.RGG_ERR_BAD_OFFSETS


@pytest.mark.parametrize("off", [[0, 50, 40, 100], [0, 50, 60, 101], [-1, 50, 60, 100]])
def test_bad_offsets_rejected_and_nothing_written(off):
    inp = wl.make_custom([50, 10, 40], K=64, N=128, seed=36)
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = _canary(100, 128)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm(X, W, torch.tensor(off, dtype=torch.int32, device="cuda"), Y, check=True)
    assert ei.value.status == rgg.RGG_ERR_BAD_OFFSETS
    _assert_untouched(Y.cpu(), slice(None))
    # the context is still usable and the status word was cleared
    _full_parity(inp)


@pytest.mark.parametrize("bm", [64, 128, pytest.param(256, marks=pytest.mark.pair)])
def test_bounded_wait_reports_timeout_and_context_survives(bm):
    # the producer issues nothing, so the first MMA wait can only end by its limit
    inp = wl.make_inputs("tiny")
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    Y = _canary(256, 512)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_grouped_gemm(X, W, off, Y, check=True, timeout_ns=20_000_000, bm=bm,
                             debug_flags=rgg.RGG_DEBUG_PRODUCER_STALL)
    assert ei.value.status == rgg.RGG_ERR_DEVICE_TIMEOUT
    assert rgg.rgg_query_status() == rgg.RGG_OK
    _full_parity(inp, bm=bm)


def test_non_default_stream_and_determinism():
    inp = wl.make_custom([100, 0, 37, 300], K=256, N=384, seed=37)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Y1 = rgg.rgg_grouped_gemm(X, W, off)
        Y2 = rgg.rgg_grouped_gemm(X, W, off)
    s.synchronize()
    assert rgg.rgg_query_status(stream=s) == rgg.RGG_OK
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    _assert_close(Y1.cpu(), ref, slice(None))


# --------------------------------------------------------------- tile list

def _export_matches_oracle(off, M_tot, N, bm, bn):
    d_off = torch.from_numpy(np.asarray(off, dtype=np.int32)).cuda()
    desc, T = rgg.rgg_export_tiles(d_off, M_tot, N, bm, bn)
    ref = oracle.tile_list(off, N, bm, bn)
    assert T == ref.shape[0]
    assert np.array_equal(desc.numpy(), ref)


@pytest.mark.parametrize("bm,bn", SHAPES + PAIR_SHAPES)
@pytest.mark.parametrize("name", ["tiny", "decode", "uniform", "skew16k", "skew2k", "prefill",
                                  "worklog_skew16k", "decode_sweep_m1", "decode_sweep_m256"])
def test_tile_list_bit_exact(name, bm, bn):
    w = wl.WORKLOADS[name]
    counts = wl.workload_counts(w)
    _export_matches_oracle(wl.offsets_from_counts(counts), int(counts.sum()), w.N, bm, bn)


def test_tile_list_edge_cases():
    _export_matches_oracle([0, 0, 0], 10, 512, 128, 128)
    _export_matches_oracle([3, 3, 10, 10, 11], 20, 520, 64, 256)
    off = wl.offsets_from_counts(np.random.default_rng(5).integers(0, 300, 4096))
    _export_matches_oracle(off, int(off[-1]), 4096, 128, 256)


def test_tile_list_capacity():
    off = np.array([0, 37, 37, 101, 256], dtype=np.int32)
    d_off = torch.from_numpy(off).cuda()
    desc, T = rgg.rgg_export_tiles(d_off, 256, 512, 128, 128, cap=5)
    ref = oracle.tile_list(off, 512, 128, 128)
    assert T == 16 and desc.shape == (5, 4)
    assert np.array_equal(desc.numpy(), ref[:5])


def _walk_reference(off, N, bm, bn, walk_order):
    """The visit order of each walk, restated from its definition on top of
    the oracle's list-order enumeration."""
    ref = oracle.tile_list(off, N, bm, bn)
    T = ref.shape[0]
    if walk_order == 0:
        return ref
    if walk_order == 1:
        return ref[[(T - 1 - (p >> 1)) if (p & 1) else (p >> 1) for p in range(T)]]
    if walk_order == 2:
        stride = next((q for q in (7919, 6841, 5009, 1009) if T % q), 1)
        return ref[[(p * stride) % T for p in range(T)]]
    counts = np.diff(np.asarray(off, dtype=np.int64))
    first = {}
    for i, e in enumerate(ref[:, 0]):
        first.setdefault(int(e), i)
    if walk_order == 4:  # each expert's tiles by (N tile, M tile)
        out = []
        for e in sorted(first):
            block = ref[ref[:, 0] == e]
            out.append(block[np.lexsort((block[:, 1], block[:, 3]))])
        return np.concatenate(out) if out else ref
    # 3: experts by decreasing row count (ties by index), their tiles in list order, then front/back
    order = sorted(range(counts.size), key=lambda e: (-counts[e], e))
    seq = np.concatenate([ref[ref[:, 0] == e] for e in order if e in first])
    return seq[[(T - 1 - (p >> 1)) if (p & 1) else (p >> 1) for p in range(T)]]


@pytest.mark.parametrize("bm,bn", [(64, 128), (128, 256), pytest.param(256, 256, marks=pytest.mark.pair)])
@pytest.mark.parametrize("name", ["tiny", "decode", "uniform", "skew16k", "skew2k", "prefill", "worklog_skew16k"])
@pytest.mark.parametrize("walk_order", [0, 1, 2, 3, 4])
def test_walk_export_bit_exact(name, bm, bn, walk_order):
    # the order in which the persistent CTAs visit the tiles, written out by the kernels' own decode
    w = wl.WORKLOADS[name]
    counts = wl.workload_counts(w)
    off = wl.offsets_from_counts(counts)
    M = int(counts.sum())
    d_off = torch.from_numpy(np.asarray(off, dtype=np.int32)).cuda()
    desc, T = rgg.rgg_export_walk(d_off, M, w.N, bm, bn, walk_order)
    canon = oracle.tile_list(off, w.N, bm, bn)
    assert T == canon.shape[0]
    got = desc.numpy()
    # a permutation of the list: every tile exactly once
    key = lambda a: a[np.lexsort(a.T[::-1])]  # noqa: E731
    assert np.array_equal(key(got), key(canon))
    assert np.array_equal(got, _walk_reference(off, w.N, bm, bn, walk_order))


# --------------------------------------------------------- full-size configs

FULL = ["decode", "uniform", "skew16k", "skew2k", "prefill"] + [
    "decode_sweep_m%d" % m for m in (1, 4, 8, 32, 64, 128, 256)]


def _compare_routed(Y, ref, off, what):
    """Every output of every routed row against the whole oracle product."""
    lo, hi = int(off[0]), int(off[-1])
    got = Y[lo:hi].double().cpu().numpy()
    r = ref[lo:hi]
    err = np.abs(got - r)
    bad = ~(err <= RTOL * np.maximum(1.0, np.abs(r)))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d of %d outputs out of tolerance; first (row %d, col %d): gpu %r oracle %r" % (
            what, int(bad.sum()), bad.size, lo + i[0], i[1], got[tuple(i)], r[tuple(i)]))


@pytest.mark.parametrize("name", FULL)
def test_full_size_config(name):
    # The whole fp64 product (about 30 s for prefill on the host cores), compared with
    # every routed output of the launch configuration the benchmark times (tile shape
    # planned from the counts), of the plan made from the device offsets alone, and,
    # on the large-group workloads, of the CTA-pair tiles.
    inp = wl.make_inputs(name)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    modes = [("bench plan", dict(host_counts=inp.counts)), ("device-offsets plan", dict())]
    if name in ("uniform", "skew16k", "prefill"):
        modes.append(("pair 256x256", dict(bm=256, bn=256)))
    for what, opts in modes:
        Y = torch.empty(X.shape[0], W.shape[2], dtype=torch.bfloat16, device="cuda")
        rgg.rgg_grouped_gemm(X, W, off, Y, check=True, **opts)
        torch.cuda.synchronize()
        _compare_routed(Y, ref, inp.offsets, "%s, %s" % (name, what))
        del Y
