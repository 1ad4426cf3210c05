"""Pins for the fp64 CPU oracle (no GPU).

The oracle is only trusted because these tests tie it to things other than
itself:

* figures the worklog prints ("Grouped GEMM for Imbalanced Experts on
  Blackwell: A WIP Worklog"): descriptor counts, the s=1.2 skew extremes,
  eta waste percentages, eta-scaled estimates (tests/golden/worklog_figures.json);
* a hand-worked tile list for the 4-expert case, written out below from the
  enumeration rule of the worklog's section 2;
* exact rational arithmetic on tiny inputs (the fp64 sum must sit within the
  textbook error bound of the exact value);
* a library special case (one expert is a plain GEMM: numpy float64 matmul);
* integer-valued inputs, where every partial sum is an exact integer and the
  result must equal numpy's int64 product bit for bit;
* the invariants the pages fix: experts are independent GEMMs, rows of no
  expert are untouched, permuting the experts permutes the output blocks.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from ragged_grouped_gemm_02_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worklog_figures.json")


def _figures():
    with open(GOLDEN) as f:
        return json.load(f)


def _counts(routing, M, E=64):
    if routing == "uniform":
        return np.full(E, M // E, dtype=np.int64)
    if routing == "worklog_skew":
        return wl.power_law_counts_first_experts(M, E, 1.2)
    raise ValueError(routing)


# ----------------------------------------------------------------- tile list

@pytest.mark.parametrize("entry", _figures()["tile_counts"], ids=lambda e: "%s-%d-%dx%d" % (
    e["routing"], e["M"], e["BM"], e["BN"]))
def test_tile_counts_match_worklog(oracle_mod, entry):
    off = wl.offsets_from_counts(_counts(entry["routing"], entry["M"], entry["E"]))
    assert oracle_mod.tile_count(off, entry["N"], entry["BM"], entry["BN"]) == entry["tiles"], entry["cite"]
    assert oracle_mod.tile_list(off, entry["N"], entry["BM"], entry["BN"]).shape[0] == entry["tiles"]


def test_skew_split_extremes_match_worklog():
    f = _figures()["skew_extremes"]
    c = wl.power_law_counts_first_experts(f["M"], f["E"], f["s"])
    assert c.sum() == f["M"]
    assert c.max() == f["max_rows"] and c.min() == f["min_rows"], f["cite"]
    # the skew is monotone in the expert index
    assert (np.diff(c) <= 0).all()


def test_tiny_tile_list_worked_by_hand(oracle_mod):
    # m = [37, 0, 64, 155], N = 512, BM = BN = 128 -> offsets [0, 37, 37, 101, 256].
    # Worklog section 2: for e, for mt < ceil(m_e/BM), for nt < ceil(N/BN):
    #   {e, off[e] + mt*BM, min(BM, m_e - mt*BM), nt*BN}
    # expert 0: one M tile of 37 rows; expert 1: nothing; expert 2: one tile of
    # 64 rows starting at row 37; expert 3: rows 101..228 (128) then 229..255 (27).
    expected = []
    for e, row0, rows in [(0, 0, 37), (2, 37, 64), (3, 101, 128), (3, 229, 27)]:
        for col0 in (0, 128, 256, 384):
            expected.append((e, row0, rows, col0))
    got = oracle_mod.tile_list([0, 37, 37, 101, 256], 512, 128, 128)
    assert [tuple(r) for r in got.tolist()] == expected
    # the same experts with BM = 64, BN = 256: expert 3 now splits into rows
    # 101..164, 165..228 and 229..255 (27), each over the N tiles at 0 and 256
    expected = []
    for e, row0, rows in [(0, 0, 37), (2, 37, 64), (3, 101, 64), (3, 165, 64), (3, 229, 27)]:
        for col0 in (0, 256):
            expected.append((e, row0, rows, col0))
    got = oracle_mod.tile_list([0, 37, 37, 101, 256], 512, 64, 256)
    assert [tuple(r) for r in got.tolist()] == expected


def test_tile_list_edge_cases(oracle_mod):
    # all experts empty: no tiles at all
    assert oracle_mod.tile_count([0, 0, 0, 0], 512, 128, 128) == 0
    assert oracle_mod.tile_list([0, 0, 0], 512, 64, 128).shape == (0, 4)
    # N not a multiple of BN: the last N tile is partial but still one tile
    t = oracle_mod.tile_list([0, 1], 520, 128, 256)
    assert [tuple(r) for r in t.tolist()] == [(0, 0, 1, 0), (0, 0, 1, 256), (0, 0, 1, 512)]
    # exact multiples produce no empty trailing tile
    t = oracle_mod.tile_list([0, 128, 384], 128, 128, 128)
    assert [tuple(r) for r in t.tolist()] == [(0, 0, 128, 0), (1, 128, 128, 0), (1, 256, 128, 0)]
    # rows beyond off[E] (spare rows) are never tiled
    assert oracle_mod.tile_count([5, 10], 64, 64, 64) == 1
    assert oracle_mod.tile_list([5, 10], 64, 64, 64).tolist() == [[0, 5, 5, 0]]


def test_tile_list_rejects_bad_offsets(oracle_mod):
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.tile_list([0, 10, 5], 64, 64, 64)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.tile_list([-1, 10], 64, 64, 64)


# --------------------------------------------------------- row utilisation

@pytest.mark.parametrize("entry", _figures()["eta_waste_percent"], ids=lambda e: "%s-%d-BM%d" % (
    e["routing"], e["M"], e["BM"]))
def test_eta_waste_matches_worklog(oracle_mod, entry):
    off = wl.offsets_from_counts(_counts(entry["routing"], entry["M"]))
    eta = oracle_mod.row_utilisation(off, entry["BM"])
    assert round(100.0 * (1.0 - eta), 1) == entry["waste"], entry["cite"]


@pytest.mark.parametrize("entry", _figures()["eta_estimates"], ids=lambda e: "%s-%d" % (e["routing"], e["M"]))
def test_eta_scaled_estimate_matches_worklog(oracle_mod, entry):
    off = wl.offsets_from_counts(_counts(entry["routing"], entry["M"]))
    eta = oracle_mod.row_utilisation(off, entry["BM"])
    assert round(eta, 3) == entry["eta_3dp"], entry["cite"]
    assert round(entry["balanced_tflops"] * round(eta, 3), 1) == entry["estimate"], entry["cite"]


def test_eta_edge_cases(oracle_mod):
    assert oracle_mod.row_utilisation([0, 0, 0], 128) == 1.0
    assert oracle_mod.row_utilisation([0, 128, 256], 128) == 1.0
    assert oracle_mod.row_utilisation([0, 1], 128) == 1.0 / 128


# ------------------------------------------------------------- the product

def _exact(x_bits, w_bits, off):
    """Exact rational Y for tiny inputs, the definition with Fractions."""
    M, K = x_bits.shape
    E, _, N = w_bits.shape
    xf = x_bits.astype(np.uint32) << 16
    wf = w_bits.astype(np.uint32) << 16
    xv = xf.view(np.float32)
    wv = wf.view(np.float32)
    out = {}
    absum = {}
    for e in range(E):
        for i in range(off[e], off[e + 1]):
            for j in range(N):
                terms = [Fraction(float(xv[i, k])) * Fraction(float(wv[e, k, j])) for k in range(K)]
                out[(i, j)] = sum(terms, Fraction(0))
                absum[(i, j)] = sum(abs(t) for t in terms)
    return out, absum


def test_matches_exact_rational_arithmetic(oracle_mod):
    inp = wl.make_custom([2, 0, 3, 1], K=24, N=10, seed=11, spare_rows=2)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = oracle_mod.grouped_gemm(xb, wb, inp.offsets)
    exact, absum = _exact(xb, wb, inp.offsets)
    K = xb.shape[1]
    for (i, j), v in exact.items():
        bound = K * 2.0 ** -52 * float(absum[(i, j)]) + 1e-300
        assert abs(Y[i, j] - float(v)) <= bound, (i, j, Y[i, j], float(v))
    # the two spare rows belong to no expert and keep the NaN canary
    assert np.isnan(Y[6:]).all()


def test_single_expert_is_plain_gemm(oracle_mod):
    inp = wl.make_custom([77], K=96, N=40, seed=12)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = oracle_mod.grouped_gemm(xb, wb, inp.offsets)
    ref = inp.X.double().numpy() @ inp.W[0].double().numpy()
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_integer_inputs_are_exact(oracle_mod):
    # entries in {-2..2}, K = 64: every partial sum is an integer of magnitude <= 256
    counts = [3, 0, 9, 1, 5]
    inp = wl.make_custom(counts, K=64, N=24, seed=13, integer_valued=True)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = oracle_mod.grouped_gemm(xb, wb, inp.offsets)
    Xi = inp.X.to(torch.int64).numpy()
    Wi = inp.W.to(torch.int64).numpy()
    off = inp.offsets
    for e in range(len(counts)):
        ref = Xi[off[e]:off[e + 1]] @ Wi[e]
        assert np.array_equal(Y[off[e]:off[e + 1]], ref.astype(np.float64))


def test_experts_are_independent_gemms(oracle_mod):
    counts = [5, 0, 17, 3]
    inp = wl.make_custom(counts, K=40, N=32, seed=14)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = oracle_mod.grouped_gemm(xb, wb, inp.offsets)
    off = inp.offsets
    for e in range(len(counts)):
        if counts[e] == 0:
            continue
        Ye = oracle_mod.grouped_gemm(np.ascontiguousarray(xb[off[e]:off[e + 1]]),
                                     np.ascontiguousarray(wb[e:e + 1]), [0, counts[e]])
        assert np.array_equal(Y[off[e]:off[e + 1]], Ye)


def test_permuting_experts_permutes_blocks(oracle_mod):
    counts = np.array([4, 9, 0, 6, 2])
    inp = wl.make_custom(counts, K=32, N=16, seed=15)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = oracle_mod.grouped_gemm(xb, wb, inp.offsets)
    perm = np.array([3, 0, 4, 2, 1])
    off = inp.offsets
    xp = np.concatenate([xb[off[p]:off[p + 1]] for p in perm])
    wp = np.ascontiguousarray(wb[perm])
    offp = wl.offsets_from_counts(counts[perm])
    Yp = oracle_mod.grouped_gemm(xp, wp, offp)
    for new_e, old_e in enumerate(perm):
        assert np.array_equal(Yp[offp[new_e]:offp[new_e + 1]], Y[off[old_e]:off[old_e + 1]])


def test_rows_of_no_expert_untouched(oracle_mod):
    # offsets may start after row 0 and end before M_tot; those rows are nobody's
    inp = wl.make_custom([4, 3], K=16, N=8, seed=16, spare_rows=5)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    off = np.array([2, 6, 9], dtype=np.int32)
    Y = oracle_mod.grouped_gemm(xb, wb, off)
    assert np.isnan(Y[:2]).all() and np.isnan(Y[9:]).all()
    assert not np.isnan(Y[2:9]).any()
    # a preset output keeps its values outside the experts
    out = np.full(Y.shape, -7.0)
    oracle_mod.grouped_gemm(xb, wb, off, out=out)
    assert (out[:2] == -7.0).all() and (out[9:] == -7.0).all()


def test_points_equal_full_product(oracle_mod):
    counts = [6, 0, 11, 2]
    inp = wl.make_custom(counts, K=48, N=20, seed=17, spare_rows=3)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = oracle_mod.grouped_gemm(xb, wb, inp.offsets)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, xb.shape[0], 200)
    cols = rng.integers(0, 20, 200)
    P = oracle_mod.grouped_gemm_points(xb, wb, inp.offsets, rows, cols)
    ref = Y[rows, cols]
    assert np.array_equal(np.isnan(P), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(P[ok], ref[ok])


@pytest.mark.parametrize("off,M", [([0, 5, 3], 8), ([0, 4, 9], 8), ([-1, 2, 3], 8)])
def test_bad_offsets_rejected(oracle_mod, off, M):
    inp = wl.make_custom([1, 1], K=8, N=8, seed=18, spare_rows=M - 2)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    assert oracle_mod.check_offsets(off, M) == oracle_mod.ORACLE_ERR_BAD_OFFSETS
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.grouped_gemm(xb, wb, off)


def test_k_not_multiple_of_tile_and_odd_n(oracle_mod):
    # shapes the pages never use (K=264, N=520) still follow the definition
    inp = wl.make_custom([3, 2], K=264, N=520, seed=19)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = oracle_mod.grouped_gemm(xb, wb, inp.offsets)
    Xd, Wd = inp.X.double().numpy(), inp.W.double().numpy()
    np.testing.assert_allclose(Y[:3], Xd[:3] @ Wd[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Y[3:], Xd[3:] @ Wd[1], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ FP8 (E4M3)

def test_e4m3_decoder_matches_library_for_every_code(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).float().double().numpy()
    mine = np.array([oracle_mod.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(mine)) and nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(mine[~nan], lib[~nan])
    # format landmarks: largest finite 448, smallest subnormal 2^-9, one = 0x38
    assert oracle_mod.e4m3_to_f64(0x7E) == 448.0 and oracle_mod.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle_mod.e4m3_to_f64(0x38) == 1.0 and oracle_mod.e4m3_to_f64(0xB8) == -1.0


def test_fp8_integer_codes_are_exact(oracle_mod):
    counts = [3, 0, 9, 1, 5]
    f = wl.make_fp8_custom(counts, K=64, N=24, seed=81, integer_valued=True)
    Y = oracle_mod.grouped_gemm_fp8(wl.fp8_codes(f.X8), wl.fp8_codes(f.W8), f.sx.numpy(), f.sw.numpy(), f.offsets)
    Xi = f.X8.float().to(torch.int64).numpy()
    Wi = f.W8.float().to(torch.int64).numpy()
    off = f.offsets
    for e in range(len(counts)):
        assert np.array_equal(Y[off[e]:off[e + 1]], (Xi[off[e]:off[e + 1]] @ Wi[e]).astype(np.float64))


def test_fp8_single_expert_is_scaled_plain_gemm(oracle_mod):
    f = wl.make_fp8_custom([33], K=96, N=40, seed=82)
    Y = oracle_mod.grouped_gemm_fp8(wl.fp8_codes(f.X8), wl.fp8_codes(f.W8), f.sx.numpy(), f.sw.numpy(), f.offsets)
    ref = (f.X8.double().numpy() @ f.W8[0].double().numpy()) * np.outer(f.sx.double().numpy(),
                                                                         f.sw[0].double().numpy())
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_fp8_scales_factor_per_row_and_per_expert_column(oracle_mod):
    counts = [4, 0, 6, 2]
    f = wl.make_fp8_custom(counts, K=32, N=16, seed=83)
    X8, W8 = wl.fp8_codes(f.X8), wl.fp8_codes(f.W8)
    sx, sw = f.sx.numpy().copy(), f.sw.numpy().copy()
    Y = oracle_mod.grouped_gemm_fp8(X8, W8, sx, sw, f.offsets)
    sx2, sw2 = sx.copy(), sw.copy()
    sx2[5] *= 2.0                 # row 5 belongs to expert 2
    sw2[2, 3] *= 4.0              # column 3 of expert 2 only
    Y2 = oracle_mod.grouped_gemm_fp8(X8, W8, sx2, sw2, f.offsets)
    expect = Y.copy()
    expect[5] *= 2.0
    expect[4:10, 3] *= 4.0
    np.testing.assert_allclose(Y2, expect, rtol=1e-15, atol=0)


# ------------------------------------------- fused gate-up + SiLU activation

def test_silu_closed_forms(oracle_mod):
    # silu(0) = 0; the logistic function at 1 is 1 / (1 + 1/e) = 0.7310585786300049
    assert oracle_mod.silu(0.0) == 0.0
    assert abs(oracle_mod.silu(1.0) - 0.7310585786300049) < 1e-15
    # sigma(z) + sigma(-z) = 1, hence silu(z) - silu(-z) = z (catches sign slips)
    for z in (-7.5, -1.25, 0.3, 2.0, 11.0):
        assert abs((oracle_mod.silu(z) - oracle_mod.silu(-z)) - z) < 1e-12 * max(1.0, abs(z))
    # far tails: silu(z) -> z for large z, -> 0 for very negative z
    assert abs(oracle_mod.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle_mod.silu(-40.0)) < 1e-15


def test_swiglu_equals_gated_product_of_the_grouped_gemm(oracle_mod):
    # the fused result is silu(gate) * up, each being the (pinned) grouped GEMM
    # of the gate and up halves of W13
    counts = [4, 0, 9, 3]
    N = 24
    inp = wl.make_custom(counts, K=40, N=2 * N, seed=61, spare_rows=2)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    H = oracle_mod.grouped_swiglu(xb, wb, inp.offsets)
    G = oracle_mod.grouped_gemm(xb, np.ascontiguousarray(wb[:, :, :N]), inp.offsets)
    U = oracle_mod.grouped_gemm(xb, np.ascontiguousarray(wb[:, :, N:]), inp.offsets)
    M_used = int(inp.offsets[-1])
    silu = np.vectorize(oracle_mod.silu)
    np.testing.assert_allclose(H[:M_used], silu(G[:M_used]) * U[:M_used], rtol=1e-14, atol=1e-14)
    assert np.isnan(H[M_used:]).all()


def test_swiglu_integer_inputs_against_exact_products(oracle_mod):
    # integer-valued inputs: gate and up are exact integers (numpy int64), so
    # H must equal silu(g) * u computed from them to fp64 rounding
    counts = [2, 5, 0, 1]
    N = 16
    inp = wl.make_custom(counts, K=32, N=2 * N, seed=62, integer_valued=True)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    H = oracle_mod.grouped_swiglu(xb, wb, inp.offsets)
    Xi, Wi, off = inp.X.to(torch.int64).numpy(), inp.W.to(torch.int64).numpy(), inp.offsets
    for e in range(len(counts)):
        g = (Xi[off[e]:off[e + 1]] @ Wi[e][:, :N]).astype(np.float64)
        u = (Xi[off[e]:off[e + 1]] @ Wi[e][:, N:]).astype(np.float64)
        ref = g / (1.0 + np.exp(-g)) * u
        np.testing.assert_allclose(H[off[e]:off[e + 1]], ref, rtol=1e-14, atol=1e-12)


# ------------------------------------------------------------ token gather

def test_gather_worked_by_hand(oracle_mod):
    # three tokens with distinct rows; routed rows read tokens 2, 0, 2, 1
    Xtok = np.array([[1, 2, 3], [4, 5, 6], [7, 8, 9]], dtype=np.uint16)
    Xg = oracle_mod.gather_rows(Xtok, [2, 0, 2, 1])
    assert Xg.tolist() == [[7, 8, 9], [1, 2, 3], [7, 8, 9], [4, 5, 6]]


def test_gather_equals_library_indexing(oracle_mod):
    gen = np.random.default_rng(71)
    Xtok = gen.integers(0, 1 << 16, size=(50, 24), dtype=np.uint16)
    idx = gen.integers(0, 50, size=300)
    np.testing.assert_array_equal(oracle_mod.gather_rows(Xtok, idx), Xtok[idx])


def test_gather_by_permutation_and_its_inverse_is_identity(oracle_mod):
    gen = np.random.default_rng(72)
    Xtok = gen.integers(0, 1 << 16, size=(40, 16), dtype=np.uint16)
    p = gen.permutation(40)
    back = oracle_mod.gather_rows(oracle_mod.gather_rows(Xtok, p), np.argsort(p))
    np.testing.assert_array_equal(back, Xtok)


def test_gather_only_the_given_range_and_rejects_bad_indices(oracle_mod):
    Xtok = np.arange(12, dtype=np.uint16).reshape(4, 3)
    # rows outside [begin, end) are neither read nor written: their index may be anything
    Xg = oracle_mod.gather_rows(Xtok, [-5, 3, 0, 99], begin=1, end=3)
    assert Xg.tolist() == [[0, 0, 0], [9, 10, 11], [0, 1, 2], [0, 0, 0]]
    oracle_mod.gather_rows(Xtok, [3])                       # T - 1 is the last valid token
    for bad in ([4], [-1], [0, 2**31 - 1]):
        with pytest.raises(oracle_mod.OracleError):
            oracle_mod.gather_rows(Xtok, bad)


def test_gathered_single_expert_is_plain_gemm_of_indexed_rows(oracle_mod):
    g = wl.make_gather_custom([37], T=50, K=48, N=24, seed=73)
    Y = oracle_mod.grouped_gemm_gather(wl.bf16_bits(g.Xtok), g.row_index, wl.bf16_bits(g.W), g.offsets)
    ref = g.Xtok.double().numpy()[g.row_index] @ g.W[0].double().numpy()
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_gathered_integer_inputs_are_exact(oracle_mod):
    # tokens shared between experts (T < M_tot), an empty expert and spare rows
    counts = [5, 0, 7, 3]
    g = wl.make_gather_custom(counts, T=9, K=32, N=16, seed=74, integer_valued=True, spare_rows=2)
    Y = oracle_mod.grouped_gemm_gather(wl.bf16_bits(g.Xtok), g.row_index, wl.bf16_bits(g.W), g.offsets)
    Xi, Wi, off = g.Xtok.to(torch.int64).numpy(), g.W.to(torch.int64).numpy(), g.offsets
    for e in range(len(counts)):
        rows = g.row_index[off[e]:off[e + 1]]
        np.testing.assert_array_equal(Y[off[e]:off[e + 1]], (Xi[rows] @ Wi[e]).astype(np.float64))
    assert np.isnan(Y[off[-1]:]).all()


def test_gathered_identity_index_is_the_grouped_gemm(oracle_mod):
    inp = wl.make_custom([6, 0, 11, 2], K=40, N=24, seed=75)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    idx = np.arange(inp.X.shape[0])
    np.testing.assert_array_equal(oracle_mod.grouped_gemm_gather(xb, idx, wb, inp.offsets),
                                  oracle_mod.grouped_gemm(xb, wb, inp.offsets))


def test_gathered_swiglu_is_swiglu_of_gathered_rows(oracle_mod):
    N = 16
    g = wl.make_gather_custom([4, 9, 0, 3], T=12, K=32, N=2 * N, seed=76, integer_valued=True)
    H = oracle_mod.grouped_swiglu_gather(wl.bf16_bits(g.Xtok), g.row_index, wl.bf16_bits(g.W), g.offsets)
    Xi, Wi, off = g.Xtok.to(torch.int64).numpy(), g.W.to(torch.int64).numpy(), g.offsets
    for e in range(4):
        rows = g.row_index[off[e]:off[e + 1]]
        gate = (Xi[rows] @ Wi[e][:, :N]).astype(np.float64)
        up = (Xi[rows] @ Wi[e][:, N:]).astype(np.float64)
        np.testing.assert_allclose(H[off[e]:off[e + 1]], gate / (1.0 + np.exp(-gate)) * up, rtol=1e-14,
                                   atol=1e-12)


def test_routed_row_index_recipe():
    counts = [5, 0, 7, 3]
    idx = wl.routed_row_index(counts, 9, torch.Generator().manual_seed(1), spare_rows=2)
    off = wl.offsets_from_counts(counts)
    assert idx.dtype == np.int32 and idx.size == 17
    for e in range(4):
        part = idx[off[e]:off[e + 1]]
        assert np.all(np.diff(part) > 0) and part.min(initial=0) >= 0 and part.max(initial=0) < 9
    assert idx[15:].tolist() == [-1, -1]
    with pytest.raises(ValueError):
        wl.routed_row_index([10], 9, torch.Generator().manual_seed(1))
