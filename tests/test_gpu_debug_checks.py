"""The bounds-checked debug build (librgg_debug.so) on the ragged edge cases, on a GB300.

librgg_debug.so is the same C ABI built with -DRGG_DEBUG_CHECKS: before every
TMA copy, global store and TMEM load its kernels check the coordinates or the
address against the bounds of what they touch (and every tile descriptor
against its expert's rows), record RGG_ERR_DEVICE_BOUNDS and skip the access
if a check fails, so nothing is issued out of bounds.  It stands in for a
memory checker.  On the edge cases of the method -- experts of 0, 1, 63, 64,
65, 127, 128, 129 rows and beyond, K = 264 and N = 520 tails, every tile shape
and kernel family -- no check may fire (status RGG_OK) and the results must
match the fp64 oracle as the release build's do.
"""
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
EDGE = [0, 1, 63, 64, 65, 127, 128, 129]
EDGE_PAIRS = EDGE + [255, 256, 257, 300, 385]


@pytest.fixture(scope="module", autouse=True)
def debug_lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()
    lib = rgg.open_library(rgg.debug_library_path())
    saved_lib, saved_handles = rgg._lib, rgg._handles
    rgg._lib, rgg._handles = lib, {}
    yield lib
    for h in rgg._handles.values():
        lib.rgg_destroy(h)
    rgg._lib, rgg._handles = saved_lib, saved_handles


def _check(got, ref, lo, hi, exact):
    g = got[lo:hi].double().numpy()
    r = ref[lo:hi]
    if exact:
        assert np.array_equal(g, r)
    else:
        err = np.abs(g - r)
        assert (err <= RTOL * np.maximum(1.0, np.abs(r))).all(), "max err %.4g" % err.max()
    v = got.view(torch.int16)
    assert bool((v[:lo] == CANARY).all()) and bool((v[hi:] == CANARY).all())


def _canary(M, N):
    return torch.full((M, N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)


GEMM_OPTS = [dict(bm=64, bn=128), dict(bm=64, bn=256), dict(bm=128, bn=192), dict(bm=128, bn=256),
             dict(bm=128, bn=256, tail64=-1), dict(bm=256, bn=128), dict(bm=256, bn=256), dict(walk_order=3),
             dict(walk_order=4, bm=256), dict(mixed=1), dict(mixed=1, mixed_pair_sms=-1),
             dict(mixed=1, mixed_pair_sms=2), dict(mixed=1, max_ctas=5), dict(mixed=2), dict(mixed=2, mixed_pair_sms=-1),
             dict(mixed=2, mixed_pair_sms=4, max_ctas=7), dict(mixed=2, host_counts=None),
             dict(mixed=2, host_counts=None, max_ctas=7)]


@pytest.mark.parametrize("opts", GEMM_OPTS, ids=[str(o) for o in GEMM_OPTS])
@pytest.mark.parametrize("K,integer", [(264, False), (64, True)])
def test_grouped_gemm_edges(opts, K, integer):
    inp = wl.make_custom(EDGE_PAIRS, K=K, N=520, seed=171, integer_valued=integer, spare_rows=3)
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = _canary(X.shape[0], 520)
    kw = dict(host_counts=inp.counts)
    kw.update(opts)  # host_counts=None: the split of a mixed launch from the device offsets
    rgg.rgg_grouped_gemm(X, W, torch.from_numpy(inp.offsets).cuda(), Y, check=True, **kw)
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    _check(Y.cpu(), ref, 0, int(inp.offsets[-1]), integer)


@pytest.mark.parametrize("opts", [dict(bm=64, bn=128), dict(bm=128, bn=256), dict(bm=256, bn=256), dict(mixed=1),
                                  dict(mixed=2, host_counts=True), dict(mixed=1, mixed_pair_sms=-1), dict(mixed=2)])
def test_swiglu_edges(opts):
    inp = wl.make_custom(EDGE_PAIRS, K=264, N=2 * 520, seed=172, spare_rows=2)
    X, W = inp.X.cuda(), inp.W.cuda()
    H = _canary(X.shape[0], 520)
    opts = dict(opts)
    if opts.pop("host_counts", False):
        opts["host_counts"] = inp.counts
    rgg.rgg_grouped_gemm_swiglu(X, W, torch.from_numpy(inp.offsets).cuda(), H, check=True, **opts)
    torch.cuda.synchronize()
    ref = oracle.grouped_swiglu(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    _check(H.cpu(), ref, 0, int(inp.offsets[-1]), False)


@pytest.mark.parametrize("opts", [dict(bm=64, bn=128), dict(bm=128, bn=256)])
def test_fp8_edges(opts):
    f = wl.make_fp8_custom(EDGE, K=272, N=528, seed=173, spare_rows=2)
    Y = _canary(f.X8.shape[0], 528)
    rgg.rgg_grouped_gemm_fp8(f.X8.cuda(), f.W8.cuda(), f.sx.cuda(), f.sw.cuda(), torch.from_numpy(f.offsets).cuda(),
                             Y, check=True, **opts)
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm_fp8(wl.fp8_codes(f.X8), wl.fp8_codes(f.W8), f.sx.numpy(), f.sw.numpy(), f.offsets)
    _check(Y.cpu(), ref, 0, int(f.offsets[-1]), False)


@pytest.mark.parametrize("mode", [1, 2])
def test_gather_edges(mode):
    g = wl.make_gather_custom(EDGE, T=300, K=264, N=520, seed=174, spare_rows=2)
    Xtok, W = g.Xtok.cuda(), g.W.cuda()
    idx = torch.from_numpy(g.row_index).cuda()
    Y = _canary(idx.numel(), 520)
    ws = torch.empty(idx.numel(), 264, dtype=torch.bfloat16, device="cuda") if mode == 2 else None
    rgg.rgg_grouped_gemm_gather(Xtok, idx, W, torch.from_numpy(g.offsets).cuda(), Y, check=True, gather_mode=mode,
                                workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm_gather(wl.bf16_bits(g.Xtok), g.row_index, wl.bf16_bits(g.W), g.offsets)
    _check(Y.cpu(), ref, 0, int(g.offsets[-1]), False)
