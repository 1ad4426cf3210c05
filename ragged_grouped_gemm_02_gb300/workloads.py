"""Seeded synthetic inputs for the ragged-M grouped GEMM.

This module is the one piece shared by the CUDA path's tests/bench and by the
CPU oracle's tests.  It holds no arithmetic of the method itself: it only
draws X, W and the per-expert row counts m_e, and turns counts into the
group-offset prefix that both sides read.

Recipe (the pages give shapes and routing rules but no value distribution):

* X ~ N(0, 1) and W ~ N(0, 1/K), drawn in fp32 from one CPU
  ``torch.Generator`` seeded per workload -- routing draws first (if the rule
  has any), then X, then W -- and rounded to bf16 (round-to-nearest-even).
  Outputs are then O(1).
* Routing rules:
    - ``power_law_counts_first_experts``: the worklog's skew generator
      ("Grouped GEMM for Imbalanced Experts on Blackwell: A WIP Worklog",
      section 2.1 "Skew and tile efficiency"): expert e gets rows in
      proportion to (e+1)^-s.  The page does not say how fractions are
      rounded; flooring and then handing the leftover rows one each to the
      first (largest) experts reproduces the page's printed extremes (4,793
      and 32 rows at s=1.2, M=16,384, E=64) and its descriptor counts.
    - ``power_law_counts_largest_remainder``: the same power law over a
      seeded random permutation of the experts, rounded by largest remainder
      (ties to the lower rank), the skewed-routing workload.
    - ``multinomial_counts``: each token picks one expert uniformly at
      random (prefill-scale routing).
    - uniform: every expert gets the same count (the worklog's balanced runs
      and the Pearl article's decode example, "Why MoE needs a grouped GEMM":
      32 experts x ~16 tokens, 16x6144 . 6144x4096).

The random streams of ``torch.Generator`` are only guaranteed equal on one
machine; nothing stored in the repository depends on them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


def offsets_from_counts(counts) -> np.ndarray:
    """int32 [E+1] exclusive prefix of the per-expert row counts."""
    counts = np.asarray(counts, dtype=np.int64)
    if counts.ndim != 1 or (counts < 0).any():
        raise ValueError("counts must be a 1-D array of non-negative integers")
    off = np.zeros(counts.size + 1, dtype=np.int64)
    np.cumsum(counts, out=off[1:])
    if off[-1] >= 2 ** 31:
        raise ValueError("total rows must fit int32")
    return off.astype(np.int32)


def power_law_counts_first_experts(M: int, E: int, s: float) -> np.ndarray:
    """Worklog section 2.1 skew: rows of expert e proportional to (e+1)^-s,
    floored, leftover rows given one each to experts 0, 1, 2, ..."""
    w = np.array([(e + 1.0) ** (-s) for e in range(E)], dtype=np.float64)
    share = w / w.sum() * M
    counts = np.floor(share).astype(np.int64)
    left = int(M - counts.sum())
    for i in range(left):
        counts[i % E] += 1
    return counts


def power_law_counts_largest_remainder(M: int, E: int, s: float, gen: torch.Generator) -> np.ndarray:
    """Power law rank^-s over a seeded random permutation of the experts,
    rounded by largest remainder (ties to the lower rank) so the sum is M."""
    perm = torch.randperm(E, generator=gen).numpy()
    w = np.array([(r + 1.0) ** (-s) for r in range(E)], dtype=np.float64)
    share = w / w.sum() * M
    by_rank = np.floor(share).astype(np.int64)
    left = int(M - by_rank.sum())
    order = np.argsort(-(share - by_rank), kind="stable")
    by_rank[order[:left]] += 1
    counts = np.zeros(E, dtype=np.int64)
    counts[perm] = by_rank  # the expert at rank r is perm[r]
    return counts


def multinomial_counts(M: int, E: int, gen: torch.Generator) -> np.ndarray:
    """Each of M tokens assigned to one of E experts uniformly at random."""
    expert_of_token = torch.randint(0, E, (M,), generator=gen)
    return np.bincount(expert_of_token.numpy(), minlength=E).astype(np.int64)


@dataclass
class Workload:
    name: str
    E: int
    K: int
    N: int
    seed: int
    routing: str                      # "explicit", "uniform", "powerlaw_lr", "powerlaw_first", "multinomial"
    counts: list | None = None        # for "explicit"
    m_per_expert: int | None = None   # for "uniform"
    M_tot: int | None = None          # for the routed rules
    s: float = 0.0
    note: str = ""
    meta: dict = field(default_factory=dict)


def _decode_sweep():
    return {"decode_sweep_m%d" % m: Workload("decode_sweep_m%d" % m, 32, 6144, 4096, 4, "uniform",
                                             m_per_expert=m,
                                             note="decode sweep point, %d rows per expert" % m)
            for m in (1, 4, 8, 32, 64, 128, 256)}


WORKLOADS = {
    "tiny": Workload("tiny", 4, 256, 512, 0, "explicit", counts=[37, 0, 64, 155],
                     note="oracle-sized case with an empty expert and ragged tails"),
    "decode": Workload("decode", 32, 6144, 4096, 1, "uniform", m_per_expert=16,
                       note="small-decode, weight-bound: 32 experts x 16 rows, 16x6144 . 6144x4096"),
    "uniform": Workload("uniform", 64, 1024, 2688, 2, "uniform", m_per_expert=256,
                        note="worklog default shape, uniform routing, 16,384 rows"),
    "skew16k": Workload("skew16k", 64, 1024, 2688, 3, "powerlaw_lr", M_tot=16384, s=1.2,
                        note="rank^-1.2 over a seeded expert permutation, largest remainder"),
    "skew2k": Workload("skew2k", 64, 1024, 2688, 3, "powerlaw_lr", M_tot=2048, s=1.2,
                       note="the skewed rule at 2,048 rows"),
    "prefill": Workload("prefill", 32, 6144, 4096, 4, "multinomial", M_tot=32768,
                        note="prefill-scale: 32,768 tokens, one uniformly random expert each"),
    "worklog_skew16k": Workload("worklog_skew16k", 64, 1024, 2688, 5, "powerlaw_first", M_tot=16384, s=1.2,
                                note="the worklog's own s=1.2 split (first-experts remainder)"),
}
WORKLOADS.update(_decode_sweep())


def counts_for(w: Workload, gen: torch.Generator | None = None) -> np.ndarray:
    if w.routing == "explicit":
        return np.asarray(w.counts, dtype=np.int64)
    if w.routing == "uniform":
        return np.full(w.E, w.m_per_expert, dtype=np.int64)
    if w.routing == "powerlaw_first":
        return power_law_counts_first_experts(w.M_tot, w.E, w.s)
    if gen is None:
        raise ValueError("routing %r draws from the generator" % w.routing)
    if w.routing == "powerlaw_lr":
        return power_law_counts_largest_remainder(w.M_tot, w.E, w.s, gen)
    if w.routing == "multinomial":
        return multinomial_counts(w.M_tot, w.E, gen)
    raise ValueError("unknown routing %r" % w.routing)


def total_rows(w: Workload) -> int:
    if w.routing == "explicit":
        return int(sum(w.counts))
    if w.routing == "uniform":
        return int(w.E * w.m_per_expert)
    return int(w.M_tot)


@dataclass
class Inputs:
    X: torch.Tensor          # bf16 [M_tot, K], CPU
    W: torch.Tensor          # bf16 [E, K, N], CPU
    offsets: np.ndarray      # int32 [E+1]
    counts: np.ndarray       # int64 [E]
    workload: Workload


def draw_matrices(M_tot: int, E: int, K: int, N: int, gen: torch.Generator):
    """X ~ N(0,1) [M_tot,K] then W ~ N(0,1/K) [E,K,N], fp32 draws rounded to bf16."""
    X = torch.randn(M_tot, K, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn(E, K, N, generator=gen, dtype=torch.float32) * (1.0 / math.sqrt(K))).to(torch.bfloat16)
    return X, W


def workload_counts(w: Workload | str) -> np.ndarray:
    """The per-expert row counts of a workload (the routing draws come first
    from the workload's generator, so this needs no matrix draws)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    gen = torch.Generator().manual_seed(w.seed)
    return counts_for(w, gen)


def make_inputs(w: Workload | str) -> Inputs:
    """Draw a workload's inputs on the CPU: routing first, then X, then W."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    gen = torch.Generator().manual_seed(w.seed)
    counts = counts_for(w, gen)
    M_tot = total_rows(w)
    if int(counts.sum()) != M_tot:
        raise AssertionError("routing produced %d rows, expected %d" % (counts.sum(), M_tot))
    X, W = draw_matrices(M_tot, w.E, w.K, w.N, gen)
    return Inputs(X, W, offsets_from_counts(counts), counts, w)


def make_custom(counts, K: int, N: int, seed: int, integer_valued: bool = False,
                spare_rows: int = 0) -> Inputs:
    """Inputs for explicit counts (tests).  ``integer_valued`` draws X and W
    uniformly from {-2,...,2} so that every partial sum is an exact integer;
    ``spare_rows`` adds rows after the last expert that belong to no expert."""
    counts = np.asarray(counts, dtype=np.int64)
    E = counts.size
    M_tot = int(counts.sum()) + int(spare_rows)
    gen = torch.Generator().manual_seed(seed)
    if integer_valued:
        X = torch.randint(-2, 3, (M_tot, K), generator=gen).to(torch.bfloat16)
        W = torch.randint(-2, 3, (E, K, N), generator=gen).to(torch.bfloat16)
    else:
        X, W = draw_matrices(M_tot, E, K, N, gen)
    w = Workload("custom", E, K, N, seed, "explicit", counts=[int(c) for c in counts])
    return Inputs(X, W, offsets_from_counts(counts), counts, w)


@dataclass
class Fp8Inputs:
    X8: torch.Tensor         # float8_e4m3fn [M_tot, K], CPU
    W8: torch.Tensor         # float8_e4m3fn [E, K, N], CPU
    sx: torch.Tensor         # float32 [M_tot]: row i of X is X8[i] * sx[i]
    sw: torch.Tensor         # float32 [E, N]: column j of W[e] is W8[e][:, j] * sw[e, j]
    offsets: np.ndarray
    counts: np.ndarray


E4M3_MAX = 448.0


def quantize_fp8(X: torch.Tensor, W: torch.Tensor):
    """Per-row (X) and per-(expert, column) (W) amax scaling into FP8 E4M3
    codes with torch's round-to-nearest conversion.  Input preparation only:
    the grouped GEMM receives the codes and the scales."""
    Xf, Wf = X.float(), W.float()
    sx = (Xf.abs().amax(dim=1) / E4M3_MAX).clamp_min(1e-12)
    sw = (Wf.abs().amax(dim=1) / E4M3_MAX).clamp_min(1e-12)            # [E, N]
    X8 = (Xf / sx[:, None]).to(torch.float8_e4m3fn)
    W8 = (Wf / sw[:, None, :]).to(torch.float8_e4m3fn)
    return X8, W8, sx.float(), sw.float()


def make_fp8_inputs(w: Workload | str) -> Fp8Inputs:
    """A workload's inputs drawn as for the bf16 path (same seed and routing),
    then quantised to E4M3 with per-row / per-column scales."""
    inp = make_inputs(w)
    X8, W8, sx, sw = quantize_fp8(inp.X, inp.W)
    return Fp8Inputs(X8, W8, sx, sw, inp.offsets, inp.counts)


def make_fp8_custom(counts, K: int, N: int, seed: int, integer_valued: bool = False, spare_rows: int = 0):
    """Explicit-count FP8 inputs; ``integer_valued`` gives codes of {-2..2}
    with every scale 1, so every partial sum is an exact integer."""
    inp = make_custom(counts, K, N, seed, integer_valued=integer_valued, spare_rows=spare_rows)
    if integer_valued:
        X8 = inp.X.float().to(torch.float8_e4m3fn)
        W8 = inp.W.float().to(torch.float8_e4m3fn)
        sx = torch.ones(inp.X.shape[0], dtype=torch.float32)
        sw = torch.ones(inp.W.shape[0], inp.W.shape[2], dtype=torch.float32)
    else:
        X8, W8, sx, sw = quantize_fp8(inp.X, inp.W)
    return Fp8Inputs(X8, W8, sx, sw, inp.offsets, inp.counts)


def fp8_codes(t: torch.Tensor) -> np.ndarray:
    """The uint8 codes of a float8_e4m3fn CPU tensor (what the oracle reads)."""
    if t.dtype != torch.float8_e4m3fn:
        raise TypeError("expected a float8_e4m3fn tensor")
    return t.contiguous().view(torch.uint8).numpy()


@dataclass
class GatherInputs:
    Xtok: torch.Tensor        # bf16 [T, K], CPU: the tokens in their own order
    row_index: np.ndarray     # int32 [M_tot]: routed row i reads token row_index[i]
    W: torch.Tensor           # bf16 [E, K, N], CPU
    offsets: np.ndarray       # int32 [E+1]
    counts: np.ndarray        # int64 [E]


def routed_row_index(counts, T: int, gen: torch.Generator, spare_rows: int = 0) -> np.ndarray:
    """Token index of every routed row: expert e's m_e rows are m_e distinct
    tokens drawn without replacement from [0, T), in increasing token order
    (the order a stable sort of the (token, expert) pairs by expert leaves
    them in).  Rows after the last expert (``spare_rows``) get -1: they belong
    to no expert and must never be read."""
    counts = np.asarray(counts, dtype=np.int64)
    if counts.size and counts.max() > T:
        raise ValueError("an expert cannot receive more distinct tokens than there are (m_e <= T)")
    parts = [torch.randperm(T, generator=gen)[:int(m)].sort().values.numpy() for m in counts]
    parts.append(np.full(int(spare_rows), -1, dtype=np.int64))
    return np.concatenate(parts).astype(np.int32)


def make_gather_custom(counts, T: int, K: int, N: int, seed: int, integer_valued: bool = False,
                       spare_rows: int = 0) -> GatherInputs:
    """Token matrix, weights and routed token indices for explicit counts:
    X_tok [T, K] first, then W, then the index draws, from one seeded
    generator (integer_valued: entries uniform in {-2..2})."""
    counts = np.asarray(counts, dtype=np.int64)
    E = counts.size
    gen = torch.Generator().manual_seed(seed)
    if integer_valued:
        Xtok = torch.randint(-2, 3, (T, K), generator=gen).to(torch.bfloat16)
        W = torch.randint(-2, 3, (E, K, N), generator=gen).to(torch.bfloat16)
    else:
        Xtok, W = draw_matrices(T, E, K, N, gen)
    idx = routed_row_index(counts, T, gen, spare_rows)
    return GatherInputs(Xtok, idx, W, offsets_from_counts(counts), counts)


def make_gather_inputs(w: Workload | str, T: int | None = None) -> GatherInputs:
    """A workload's routed counts and matrices, with the activations held as
    T tokens (default T = M_tot) that the routed rows index into."""
    w = WORKLOADS[w] if isinstance(w, str) else w
    counts = workload_counts(w)
    M_tot = int(counts.sum())
    T = M_tot if T is None else int(T)
    gen = torch.Generator().manual_seed(w.seed + 1000)
    Xtok, W = draw_matrices(T, w.E, w.K, w.N, gen)
    idx = routed_row_index(counts, T, gen)
    return GatherInputs(Xtok, idx, W, offsets_from_counts(counts), counts)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a bf16 CPU tensor (what the oracle reads)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
