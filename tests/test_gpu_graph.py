"""The library's launches can be captured in a CUDA graph and replayed (GB300).

Each call reads the routed counts on the device and allocates nothing (the
handle's status word exists from rgg_create; the two-pass gather's workspace
is the caller's), so a captured launch replays on new data in the same
buffers.  Checked against the fp64 oracle with the usual tolerance.
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


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()


def _close(got, ref):
    err = np.abs(got - ref)
    assert (err <= RTOL * np.maximum(1.0, np.abs(ref))).all(), "max err %.4g" % err.max()


@pytest.mark.parametrize("bm,bn", [(64, 256), (128, 192), pytest.param(256, 256, marks=pytest.mark.pair)])
def test_grouped_gemm_replays_on_new_data(bm, bn):
    counts = [100, 0, 37, 300, 9]
    a = wl.make_custom(counts, K=256, N=512, seed=121)
    b = wl.make_custom(counts, K=256, N=512, seed=122)
    X, W = a.X.cuda(), a.W.cuda()
    off = torch.from_numpy(a.offsets).cuda()
    Y = torch.empty(X.shape[0], 512, dtype=torch.bfloat16, device="cuda")
    rgg.rgg_grouped_gemm(X, W, off, Y, bm=bm, bn=bn, check=True)  # first call outside the capture
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rgg.rgg_grouped_gemm(X, W, off, Y, bm=bm, bn=bn)
    for inp in (b, a):
        X.copy_(inp.X.cuda())
        W.copy_(inp.W.cuda())
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert rgg.rgg_query_status() == rgg.RGG_OK
        ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
        _close(Y.double().cpu().numpy(), ref)


def test_two_pass_gather_replays_on_new_indices():
    counts = [300, 0, 700, 200]
    a = wl.make_gather_custom(counts, T=900, K=128, N=256, seed=123)
    b = wl.make_gather_custom(counts, T=900, K=128, N=256, seed=124)
    Xtok, W = a.Xtok.cuda(), a.W.cuda()
    idx, off = torch.from_numpy(a.row_index).cuda(), torch.from_numpy(a.offsets).cuda()
    Y = torch.empty(idx.numel(), 256, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(idx.numel(), 128, dtype=torch.bfloat16, device="cuda")
    rgg.rgg_grouped_gemm_gather(Xtok, idx, W, off, Y, gather_mode=2, workspace=ws, check=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rgg.rgg_grouped_gemm_gather(Xtok, idx, W, off, Y, gather_mode=2, workspace=ws)
    for inp in (b, a):
        Xtok.copy_(inp.Xtok.cuda())
        W.copy_(inp.W.cuda())
        idx.copy_(torch.from_numpy(inp.row_index).cuda())
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert rgg.rgg_query_status() == rgg.RGG_OK
        ref = oracle.grouped_gemm_gather(wl.bf16_bits(inp.Xtok), inp.row_index, wl.bf16_bits(inp.W), inp.offsets)
        _close(Y.double().cpu().numpy(), ref)
