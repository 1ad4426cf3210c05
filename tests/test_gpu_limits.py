"""Limits and randomized configurations of the grouped GEMM against the fp64
oracle, on a GB300.

* The largest expert count the library takes (E = 4096), with most experts
  holding a handful of rows or none, on every kernel family: the per-CTA
  offsets and tile prefix then fill 32 KB of shared memory and the ring
  gets fewer stages.  Integer-valued inputs with K <= 64 are exact, so the
  result must equal the oracle bit for bit.
* Seeded random configurations over expert counts, row counts (with empty
  and single-row experts), K and N tails, tile shapes, walk orders, tail-tile
  modes, against the tolerance
  |gpu - oracle| <= 1e-2 * max(1, |oracle|), rows of no expert untouched.
* Four million routed rows, every output checked.
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


def _canary(M, N):
    return torch.full((M, N), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)


def _run(inp, **opts):
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = _canary(X.shape[0], W.shape[2])
    rgg.rgg_grouped_gemm(X, W, torch.from_numpy(inp.offsets).cuda(), Y, check=True, **opts)
    torch.cuda.synchronize()
    return Y.cpu()


def _close(got, ref):
    err = np.abs(got - ref)
    bound = RTOL * np.maximum(1.0, np.abs(ref))
    bad = np.argwhere(~(err <= bound))
    assert bad.size == 0, "%d outputs out of tolerance; first %s: gpu %r oracle %r" % (
        bad.shape[0], bad[0].tolist(), got[tuple(bad[0])], ref[tuple(bad[0])])


@pytest.mark.parametrize("opts", [dict(), dict(bm=64, bn=128), dict(bm=128, bn=256), dict(bm=256, bn=256),
                                  dict(mixed=1), dict(mixed=2)],
                         ids=["auto", "64x128", "128x256", "pair", "mixed-claims", "mixed-device-split"])
def test_max_experts_bit_exact(opts):
    rng = np.random.default_rng(4096)
    counts = rng.integers(0, 6, 4096) * (rng.random(4096) < 0.6)
    counts[17] = 300  # one expert of several M tiles among thousands of tiny ones
    inp = wl.make_custom(counts, K=64, N=136, seed=151, integer_valued=True, spare_rows=7)
    plan = rgg.rgg_plan(4096, inp.X.shape[0], 64, 136, **opts)
    assert plan["stages"] >= 2
    Y = _run(inp, **opts)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M = int(inp.offsets[-1])
    assert np.array_equal(Y[:M].double().numpy(), ref[:M])
    assert bool((Y.view(torch.int16)[M:] == CANARY).all())


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.integers(1, 300))
    kind = seed % 4
    if kind == 0:    # small groups
        counts = rng.integers(0, 40, E)
    elif kind == 1:  # power-law skew over a random permutation
        counts = rng.permutation((600.0 * (np.arange(E) + 1.0) ** -1.1).astype(np.int64))
    elif kind == 2:  # balanced around a random size
        counts = rng.integers(1, 2 * int(rng.integers(8, 400)), E)
    else:            # mostly empty with a few large experts
        counts = np.where(rng.random(E) < 0.8, 0, rng.integers(1, 900, E))
    counts = counts * (rng.random(E) < 0.9)
    if counts.sum() > 6000:  # keep the fp64 oracle's share of the test time small
        counts = counts * 6000 // counts.sum()
    K = int(rng.choice([64, 128, 200, 264, 512]))
    N = 8 * int(rng.integers(2, 96))
    choices = [dict(), dict(bm=64), dict(bm=128), dict(bm=256), dict(bm=128, bn=192), dict(bm=64, bn=128),
               dict(bm=256, bn=128), dict(bm=128, tail64=-1), dict(bm=256, tail64=-1), dict(mixed=1),
               dict(mixed=2), dict(mixed=2, no_counts=True)]
    opts = dict(choices[int(rng.integers(len(choices)))])
    if not opts.get("mixed"):
        walks = [0, 1, 2, 3, 4] if E <= 256 else [0, 1, 2, 4]
        opts["walk_order"] = int(rng.choice(walks))
    no_counts = opts.pop("no_counts", False)  # the mixed launch's SM split from the device offsets
    if rng.random() < 0.5 and not no_counts:
        opts["host_counts"] = counts
    return counts, K, N, opts


@pytest.mark.parametrize("seed", range(32))
def test_random_configurations(seed):
    counts, K, N, opts = _random_case(seed)
    inp = wl.make_custom(counts, K=K, N=N, seed=2000 + seed, spare_rows=int(seed % 3) * 5)
    Y = _run(inp, **opts)
    M = int(inp.offsets[-1])
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    if 2.0 * M * K * N <= 4e8:
        ref = oracle.grouped_gemm(xb, wb, inp.offsets)
        _close(Y[:M].double().numpy(), ref[:M])
    else:  # larger cases: every expert's first and last row, the last column, and random outputs
        rng = np.random.default_rng(seed)
        edge = np.concatenate([inp.offsets[:-1][counts > 0], inp.offsets[1:][counts > 0] - 1])
        edge_cols = np.stack([np.zeros(edge.size), np.full(edge.size, N - 1), rng.integers(0, N, edge.size)], 1)
        rows = np.concatenate([np.repeat(edge, 3), rng.integers(0, M, 3000)]).astype(np.int64)
        cols = np.concatenate([edge_cols.reshape(-1), rng.integers(0, N, 3000)]).astype(np.int64)
        ref = oracle.grouped_gemm_points(xb, wb, inp.offsets, rows, cols)
        _close(Y.double().numpy()[rows, cols], ref)
    assert bool((Y.view(torch.int16)[M:] == CANARY).all())


def test_four_million_rows():
    # 4 194 304 routed rows over 16 experts, every output checked: the oracle runs expert by
    # expert (each expert's product is independent) so that its fp64 result stays ~0.5 GB
    rng = np.random.default_rng(77)
    counts = rng.multinomial(1 << 22, np.full(16, 1.0 / 16))
    inp = wl.make_custom(counts, K=64, N=256, seed=152)
    X, W = inp.X.cuda(), inp.W.cuda()
    Y = rgg.rgg_grouped_gemm(X, W, torch.from_numpy(inp.offsets).cuda(), check=True, host_counts=counts)
    torch.cuda.synchronize()
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    off = inp.offsets
    for e in range(counts.size):
        r0, r1 = int(off[e]), int(off[e + 1])
        ref = oracle.grouped_gemm(np.ascontiguousarray(xb[r0:r1]), np.ascontiguousarray(wb[e:e + 1]), [0, r1 - r0])
        _close(Y[r0:r1].double().cpu().numpy(), ref)


@pytest.mark.parametrize("opts", [dict(bm=64, bn=256), dict(bm=128, bn=256), dict(bm=256, bn=256),
                                  dict(bm=128, bn=192, walk_order=3), dict(bm=256, bn=256, walk_order=4)],
                         ids=["64x256", "128x256", "pair", "128x192-sorted", "pair-nmajor"])
@pytest.mark.parametrize("max_ctas", [1, 2, 3, 37])
def test_few_persistent_ctas_walk_every_tile(opts, max_ctas):
    # a grid far smaller than the tile count: each CTA (or pair) walks many tiles, rings wrap many times
    counts = [3, 0, 130, 64, 1, 200, 65, 127, 129, 500]
    inp = wl.make_custom(counts, K=128, N=392, seed=153, integer_valued=True, spare_rows=2)
    K64 = wl.make_custom(counts, K=64, N=392, seed=153, integer_valued=True, spare_rows=2)
    for case in (inp, K64):
        Y = _run(case, max_ctas=max_ctas, **opts)
        ref = oracle.grouped_gemm(wl.bf16_bits(case.X), wl.bf16_bits(case.W), case.offsets)
        M = int(case.offsets[-1])
        if case is K64:
            assert np.array_equal(Y[:M].double().numpy(), ref[:M])
        else:
            _close(Y[:M].double().numpy(), ref[:M])
        assert bool((Y.view(torch.int16)[M:] == CANARY).all())


def test_host_counts_that_disagree_with_the_device_offsets():
    # host counts only steer the plan; the kernels read the offsets on the device
    counts = np.array([700, 0, 3, 260, 1, 90])
    inp = wl.make_custom(counts, K=64, N=264, seed=154, integer_valued=True, spare_rows=3)
    ref = oracle.grouped_gemm(wl.bf16_bits(inp.X), wl.bf16_bits(inp.W), inp.offsets)
    M = int(inp.offsets[-1])
    for wrong in ([16] * 6, [1000, 1000, 1000, 1000, 1000, 1000], [0, 0, 0, 0, 0, 1054], counts[::-1]):
        Y = _run(inp, host_counts=np.asarray(wrong))
        assert np.array_equal(Y[:M].double().numpy(), ref[:M]), wrong
        assert bool((Y.view(torch.int16)[M:] == CANARY).all())
