"""Expert-parallel sharding emulated on one GB300: the experts split into G
contiguous ranges (ragged_grouped_gemm_02_gb300.sharding, the layout each of
G GPUs would hold), one grouped-GEMM call per range on its own rows, its own
slice of W and offsets rebased to its first row, all writing into one Y.  The
shards need no exchange, so the assembled Y must equal the single call over
all experts bit for bit (same tile shape, same K order per output)."""
import numpy as np
import pytest
import torch

import ragged_grouped_gemm_02_gb300 as rgg
from ragged_grouped_gemm_02_gb300 import _build, sharding
from ragged_grouped_gemm_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    _build.build()


@pytest.mark.parametrize("name", ["decode", "skew16k", "prefill"])
@pytest.mark.parametrize("world", [2, 8])
def test_shards_assemble_the_full_result(name, world):
    inp = wl.make_inputs(name)
    X, W = inp.X.cuda(), inp.W.cuda()
    off = torch.from_numpy(inp.offsets).cuda()
    plan = rgg.rgg_plan(W.shape[0], X.shape[0], X.shape[1], W.shape[2], host_counts=inp.counts)
    shape = dict(bm=plan["bm"], bn=plan["bn"])
    full = rgg.rgg_grouped_gemm(X, W, off, check=True, **shape)
    Y = torch.full_like(full, float("nan"))
    for rank in range(world):
        s = sharding.expert_shard(inp.offsets, world, rank)
        if s.row_end == s.row_begin:
            continue
        rgg.rgg_grouped_gemm(X[s.row_begin:s.row_end], W[s.expert_begin:s.expert_end].contiguous(),
                             torch.from_numpy(s.local_offsets).cuda(), Y[s.row_begin:s.row_end], check=True,
                             host_counts=inp.counts[s.expert_begin:s.expert_end], **shape)
    torch.cuda.synchronize()
    M = int(inp.offsets[-1])
    assert torch.equal(Y[:M].view(torch.int16), full[:M].view(torch.int16))
