"""The seeded input generators (no GPU).  They hold no arithmetic of the
method; these tests only check that each workload has the shape, the row
counts and the routing rule it is meant to have."""
import numpy as np
import pytest
import torch

from ragged_grouped_gemm_02_gb300 import workloads as wl


def test_offsets_from_counts():
    assert wl.offsets_from_counts([37, 0, 64, 155]).tolist() == [0, 37, 37, 101, 256]
    assert wl.offsets_from_counts([0]).tolist() == [0, 0]
    with pytest.raises(ValueError):
        wl.offsets_from_counts([3, -1])


@pytest.mark.parametrize("name,E,M", [("tiny", 4, 256), ("decode", 32, 512), ("uniform", 64, 16384),
                                      ("skew16k", 64, 16384), ("skew2k", 64, 2048), ("prefill", 32, 32768),
                                      ("worklog_skew16k", 64, 16384), ("decode_sweep_m1", 32, 32),
                                      ("decode_sweep_m256", 32, 8192)])
def test_counts_sum_and_size(name, E, M):
    c = wl.workload_counts(name)
    assert c.size == E and int(c.sum()) == M and (c >= 0).all()
    assert wl.total_rows(wl.WORKLOADS[name]) == M


def test_tiny_counts_have_an_empty_expert():
    assert wl.workload_counts("tiny").tolist() == [37, 0, 64, 155]


def test_largest_remainder_is_a_permuted_power_law():
    # sorted descending, the seeded split must be the rank^-1.2 largest-remainder split
    for name, M, top, bottom in [("skew16k", 16384, 4793, 33), ("skew2k", 2048, 599, 4)]:
        c = np.sort(wl.workload_counts(name))[::-1]
        assert c[0] == top and c[-1] == bottom
        w = np.array([(r + 1.0) ** -1.2 for r in range(64)])
        share = w / w.sum() * M
        assert np.all(np.abs(c - share) < 1.0)
    # the permutation is seeded and not the identity
    c = wl.workload_counts("skew16k")
    assert not (np.diff(c) <= 0).all()
    assert np.array_equal(c, wl.workload_counts("skew16k"))


def test_multinomial_routing_is_plausible():
    c = wl.workload_counts("prefill")
    # 32,768 tokens over 32 experts: mean 1024, binomial sd ~31.5
    assert abs(c.mean() - 1024) < 1e-9 and c.min() > 850 and c.max() < 1200


def test_make_inputs_tiny():
    inp = wl.make_inputs("tiny")
    assert inp.X.shape == (256, 256) and inp.X.dtype == torch.bfloat16
    assert inp.W.shape == (4, 256, 512) and inp.W.dtype == torch.bfloat16
    assert inp.offsets.tolist() == [0, 37, 37, 101, 256]
    # W ~ N(0, 1/K): sample sd close to 1/16
    assert abs(inp.W.float().std().item() - 1.0 / 16) < 0.005
    again = wl.make_inputs("tiny")
    assert torch.equal(inp.X, again.X) and torch.equal(inp.W, again.W)


def test_integer_valued_custom_inputs():
    inp = wl.make_custom([3, 4], K=16, N=8, seed=0, integer_valued=True, spare_rows=1)
    assert inp.X.shape == (8, 16)
    v = torch.cat([inp.X.flatten().float(), inp.W.flatten().float()])
    assert v.min() >= -2 and v.max() <= 2 and torch.equal(v, v.round())


def test_bf16_bits_roundtrip():
    t = torch.tensor([1.0, -2.5, 0.0078125], dtype=torch.bfloat16)
    b = wl.bf16_bits(t)
    back = (b.astype(np.uint32) << 16).view(np.float32)
    assert back.tolist() == [1.0, -2.5, 0.0078125]
