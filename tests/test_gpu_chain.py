"""Back-to-back launches on one stream, on a GB300.

Every GEMM kernel is launched with programmatic stream serialisation: it may
become resident while the kernel ahead of it on the stream is still running,
and it waits on the device before its first global memory access (the mixed
launch's 1-CTA kernel relies on its pair kernel having waited).  These tests
chain launches whose data depend on each other, with no host synchronisation
in between, and check both directions of the dependency:

* read after write: Y1 = X W1, then Y2 = Y1 W2.  Y1 starts as NaN canaries,
  so a second launch that read it early shows up; Y2 must match the fp64
  oracle's product of the finished Y1;
* write after read: Y = X W, then a GEMM whose output is X.  Y must match the
  oracle on the original X;
* the same chains captured in a CUDA graph and replayed, with the canaries
  written again by a torch kernel between the launches;

for every kernel family: 64- and 128-row tiles, CTA pairs, and the mixed
launch with claims and with fixed walks (with and without its pair kernel).
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
COUNTS = [1500, 40, 700, 300, 129, 64, 900, 2000]
K1, N1, N2 = 2048, 1024, 512

PLANS = [dict(bm=64, bn=256), dict(bm=128, bn=256), dict(bm=256, bn=256), dict(mixed=1), dict(mixed=2),
         dict(mixed=2, mixed_pair_sms=-1), dict(mixed=1, mixed_pair_sms=-1)]
PLAN_IDS = ["64x256", "128x256", "pairs", "mixed-claims", "mixed-fixed", "mixed-no-pairs", "claims-no-pairs"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()
    oracle.build()


@pytest.fixture(scope="module")
def data():
    a = wl.make_custom(COUNTS, K=K1, N=N1, seed=191, spare_rows=40)
    b = wl.make_custom(COUNTS, K=N1, N=N2, seed=192, spare_rows=40)
    return a, b


def _canary(M, N):
    return torch.full((M, N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def _assert_close(got, ref, lo, hi):
    g = got[lo:hi].double().numpy()
    r = ref[lo:hi]
    err = np.abs(g - r)
    bad = ~(err <= RTOL * np.maximum(1.0, np.abs(r)))
    assert not bad.any(), "%d outputs out of tolerance, max err %.4g" % (int(bad.sum()), np.nanmax(err))


@pytest.mark.parametrize("opts", PLANS, ids=PLAN_IDS)
def test_read_after_write(data, opts):
    a, b = data
    X, W1, W2 = a.X.cuda(), a.W.cuda(), b.W.cuda()
    off = torch.from_numpy(a.offsets).cuda()
    M = X.shape[0]
    Y1, Y2 = _canary(M, N1), _canary(M, N2)
    torch.cuda.synchronize()
    rgg.rgg_grouped_gemm(X, W1, off, Y1, host_counts=a.counts, **opts)
    rgg.rgg_grouped_gemm(Y1, W2, off, Y2, host_counts=a.counts, **opts)
    torch.cuda.synchronize()
    assert rgg.rgg_query_status() == rgg.RGG_OK
    y1 = Y1.cpu()
    lo, hi = int(a.offsets[0]), int(a.offsets[-1])
    assert not torch.isnan(y1[lo:hi].float()).any()
    ref = oracle.grouped_gemm(wl.bf16_bits(y1), wl.bf16_bits(b.W), a.offsets)
    _assert_close(Y2.cpu(), ref, lo, hi)


@pytest.mark.parametrize("opts", PLANS, ids=PLAN_IDS)
def test_write_after_read(data, opts):
    a, b = data
    X, W1 = a.X.cuda(), a.W.cuda()
    off = torch.from_numpy(a.offsets).cuda()
    M = X.shape[0]
    # Z V has the shape of X: the second launch overwrites the first one's input
    z = wl.make_custom(COUNTS, K=256, N=K1, seed=193, spare_rows=40)
    Z, V = z.X.cuda(), z.W.cuda()
    Y = _canary(M, N1)
    torch.cuda.synchronize()
    rgg.rgg_grouped_gemm(X, W1, off, Y, host_counts=a.counts, **opts)
    rgg.rgg_grouped_gemm(Z, V, off, X, host_counts=a.counts, **opts)
    torch.cuda.synchronize()
    assert rgg.rgg_query_status() == rgg.RGG_OK
    lo, hi = int(a.offsets[0]), int(a.offsets[-1])
    ref = oracle.grouped_gemm(wl.bf16_bits(a.X), wl.bf16_bits(a.W), a.offsets)
    _assert_close(Y.cpu(), ref, lo, hi)


@pytest.mark.parametrize("opts", [dict(bm=128, bn=256), dict(mixed=1), dict(mixed=2)],
                         ids=["128x256", "mixed-claims", "mixed-fixed"])
def test_chain_in_cuda_graph(data, opts):
    a, b = data
    X, W1, W2 = a.X.cuda(), a.W.cuda(), b.W.cuda()
    off = torch.from_numpy(a.offsets).cuda()
    M = X.shape[0]
    Y1, Y2 = _canary(M, N1), _canary(M, N2)
    nan16 = torch.tensor(CANARY, dtype=torch.int16, device="cuda")

    def step():
        Y1.view(torch.int16).fill_(nan16)
        Y2.view(torch.int16).fill_(nan16)
        rgg.rgg_grouped_gemm(X, W1, off, Y1, host_counts=a.counts, **opts)
        rgg.rgg_grouped_gemm(Y1, W2, off, Y2, host_counts=a.counts, **opts)
        rgg.rgg_grouped_gemm(Y1, W2, off, Y2, host_counts=a.counts, **opts)

    step()  # plans and tensor maps before the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert rgg.rgg_query_status() == rgg.RGG_OK
    lo, hi = int(a.offsets[0]), int(a.offsets[-1])
    y1 = Y1.cpu()
    ref1 = oracle.grouped_gemm(wl.bf16_bits(a.X), wl.bf16_bits(a.W), a.offsets)
    _assert_close(y1, ref1, lo, hi)
    ref2 = oracle.grouped_gemm(wl.bf16_bits(y1), wl.bf16_bits(b.W), a.offsets)
    _assert_close(Y2.cpu(), ref2, lo, hi)
