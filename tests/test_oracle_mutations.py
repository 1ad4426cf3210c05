"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each case edits one line of a private copy of oracle/rgg_oracle.c (a dropped
term, a transposed operand, a wrong expert, a flipped sign, a shifted row
range, a wrong tile rule, a wrong rounding in eta), compiles the copy with gcc
into a temporary directory and runs the same kinds of checks that
tests/test_oracle.py applies to the real oracle.  Every mutant must fail at
least one of them, and the unmutated copy must pass all of them.  All of this
runs on the CPU.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest
import torch

from ragged_grouped_gemm_02_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rgg_oracle.c")
GOLDEN = os.path.join(ROOT, "tests", "golden", "worklog_figures.json")

MUTANTS = {
    "dropped_last_k": ("for (int k = 0; k < K; ++k) {", "for (int k = 0; k < K - 1; ++k) {"),
    "transposed_w": ("acc[j] += x * bf16_bits_to_f64(wrow[j]);",
                     "acc[j] += x * bf16_bits_to_f64(We[(int64_t)j * K + k]);"),
    "wrong_expert": ("const uint16_t* We = W + (int64_t)e * K * N;\n        #pragma omp parallel",
                     "const uint16_t* We = W + (int64_t)((e + 1) % E) * K * N;\n        #pragma omp parallel"),
    "flipped_sign": ("acc[j] += x * bf16_bits_to_f64(wrow[j]);", "acc[j] -= x * bf16_bits_to_f64(wrow[j]);"),
    "skipped_first_row": ("const int64_t row_begin = off[e], row_end = off[e + 1];",
                          "const int64_t row_begin = off[e] + (off[e + 1] > off[e] ? 1 : 0), row_end = off[e + 1];"),
    "x_row_of_next_expert": ("const double x = bf16_bits_to_f64(X[i * K + k]);",
                             "const double x = bf16_bits_to_f64(X[((i + 1) % M_tot) * K + k]);"),
    "tile_rows_not_clipped": ("desc[4 * count + 2] = (int32_t)(left < BM ? left : BM);",
                              "desc[4 * count + 2] = (int32_t)BM;"),
    "tile_row0_off_by_tile": ("desc[4 * count + 1] = (int32_t)(off[e] + mt * BM);",
                              "desc[4 * count + 1] = (int32_t)(off[e] + mt * BN);"),
    "tile_count_floor": ("const int64_t m_tiles = ceil_div64(m_e, BM);", "const int64_t m_tiles = m_e / BM;"),
    "eta_floor": ("scheduled_tiles += ceil_div64(m_e, BM);", "scheduled_tiles += m_e / BM + 1;"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "gate_up_swapped": ("H[i * N + j] = silu_f64(acc[j]) * acc[N + j];",
                        "H[i * N + j] = silu_f64(acc[N + j]) * acc[j];"),
    "swiglu_plain_product": ("H[i * N + j] = silu_f64(acc[j]) * acc[N + j];",
                             "H[i * N + j] = acc[j] * acc[N + j];"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "fp8_scale_ignores_expert": ("const float* swe = sw + (int64_t)e * N;", "const float* swe = sw;"),
    "gather_ignores_index": ("for (int k = 0; k < K; ++k) Xg[i * K + k] = Xtok[r * K + k];",
                             "for (int k = 0; k < K; ++k) Xg[i * K + k] = Xtok[(i % T) * K + k];"),
    "gather_next_rows_index": ("const int64_t r = row_index[i];",
                               "const int64_t r = row_index[i + 1 < end ? i + 1 : i];"),
    "gather_accepts_t": ("(int64_t)row_index[i] >= T) return ORACLE_ERR_BAD_ROW_INDEX;",
                         "(int64_t)row_index[i] > T) return ORACLE_ERR_BAD_ROW_INDEX;"),
}


def _build(tmp_path, name, mutation):
    src = open(SRC).read()
    if mutation is not None:
        # the same slip everywhere the line occurs (the fused function repeats
        # the GEMM's inner loop)
        old, new = mutation
        assert src.count(old) >= 1, "mutation anchor for %s not found" % name
        src = src.replace(old, new)
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("lib%s.so" % name)
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                    "-o", str(so), str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    P = ctypes.c_void_p
    lib.rgg_oracle_grouped_gemm.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P,
                                            ctypes.c_int]
    lib.rgg_oracle_grouped_gemm.restype = ctypes.c_int
    lib.rgg_oracle_tile_list.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                         ctypes.c_int64]
    lib.rgg_oracle_tile_list.restype = ctypes.c_int64
    lib.rgg_oracle_row_utilisation.argtypes = [P, ctypes.c_int, ctypes.c_int]
    lib.rgg_oracle_row_utilisation.restype = ctypes.c_double
    lib.rgg_oracle_grouped_swiglu.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P,
                                              ctypes.c_int]
    lib.rgg_oracle_grouped_swiglu.restype = ctypes.c_int
    lib.rgg_oracle_silu.argtypes = [ctypes.c_double]
    lib.rgg_oracle_silu.restype = ctypes.c_double
    return lib


def _gemm(lib, xb, wb, off):
    M, K = xb.shape
    E, _, N = wb.shape
    off = np.ascontiguousarray(off, dtype=np.int32)
    Y = np.full((M, N), np.nan)
    rc = lib.rgg_oracle_grouped_gemm(xb.ctypes.data, wb.ctypes.data, off.ctypes.data, E, M, K, N,
                                     Y.ctypes.data, 1)
    assert rc == 0
    return Y


def _tiles(lib, off, N, BM, BN):
    off = np.ascontiguousarray(off, dtype=np.int32)
    T = lib.rgg_oracle_tile_list(off.ctypes.data, off.size - 1, N, BM, BN, None, 0)
    d = np.zeros((max(T, 1), 4), dtype=np.int32)
    lib.rgg_oracle_tile_list(off.ctypes.data, off.size - 1, N, BM, BN, d.ctypes.data, T)
    return [tuple(r) for r in d[:T].tolist()]


def _product_checks_pass(lib):
    # library special case: one expert
    inp = wl.make_custom([9], K=40, N=24, seed=21)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = _gemm(lib, xb, wb, inp.offsets)
    if not np.allclose(Y, inp.X.double().numpy() @ inp.W[0].double().numpy(), rtol=1e-12, atol=1e-12):
        return False
    # integer-exact, several experts with an empty one and spare rows
    counts = [3, 0, 5, 2]
    inp = wl.make_custom(counts, K=32, N=16, seed=22, integer_valued=True, spare_rows=2)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    Y = _gemm(lib, xb, wb, inp.offsets)
    Xi, Wi, off = inp.X.to(torch.int64).numpy(), inp.W.to(torch.int64).numpy(), inp.offsets
    for e in range(len(counts)):
        if not np.array_equal(Y[off[e]:off[e + 1]], (Xi[off[e]:off[e + 1]] @ Wi[e]).astype(np.float64)):
            return False
    return bool(np.isnan(Y[off[-1]:]).all())


def _tile_checks_pass(lib):
    expected = []
    for e, row0, rows in [(0, 0, 37), (2, 37, 64), (3, 101, 128), (3, 229, 27)]:
        for col0 in (0, 128, 256, 384):
            expected.append((e, row0, rows, col0))
    if _tiles(lib, [0, 37, 37, 101, 256], 512, 128, 128) != expected:
        return False
    expected = []
    for e, row0, rows in [(0, 0, 37), (2, 37, 64), (3, 101, 64), (3, 165, 64), (3, 229, 27)]:
        for col0 in (0, 256):
            expected.append((e, row0, rows, col0))
    if _tiles(lib, [0, 37, 37, 101, 256], 512, 64, 256) != expected:
        return False
    figs = json.load(open(GOLDEN))
    for entry in figs["tile_counts"]:
        c = (np.full(64, entry["M"] // 64) if entry["routing"] == "uniform"
             else wl.power_law_counts_first_experts(entry["M"], 64, 1.2))
        if len(_tiles(lib, wl.offsets_from_counts(c), entry["N"], entry["BM"], entry["BN"])) != entry["tiles"]:
            return False
    return True


def _eta_checks_pass(lib):
    figs = json.load(open(GOLDEN))
    for entry in figs["eta_waste_percent"]:
        c = (np.full(64, entry["M"] // 64) if entry["routing"] == "uniform"
             else wl.power_law_counts_first_experts(entry["M"], 64, 1.2))
        off = np.ascontiguousarray(wl.offsets_from_counts(c))
        eta = lib.rgg_oracle_row_utilisation(off.ctypes.data, 64, entry["BM"])
        if round(100.0 * (1.0 - eta), 1) != entry["waste"]:
            return False
    return True


def _swiglu_checks_pass(lib):
    # closed forms of the activation, then integer inputs against exact gate / up products
    if lib.rgg_oracle_silu(0.0) != 0.0 or abs(lib.rgg_oracle_silu(1.0) - 0.7310585786300049) > 1e-15:
        return False
    if abs((lib.rgg_oracle_silu(2.0) - lib.rgg_oracle_silu(-2.0)) - 2.0) > 1e-12:
        return False
    counts, N = [2, 0, 3], 8
    inp = wl.make_custom(counts, K=16, N=2 * N, seed=63, integer_valued=True)
    xb, wb = wl.bf16_bits(inp.X), wl.bf16_bits(inp.W)
    off = np.ascontiguousarray(inp.offsets, dtype=np.int32)
    H = np.full((xb.shape[0], N), np.nan)
    if lib.rgg_oracle_grouped_swiglu(xb.ctypes.data, wb.ctypes.data, off.ctypes.data, len(counts), xb.shape[0],
                                     16, N, H.ctypes.data, 1) != 0:
        return False
    Xi, Wi = inp.X.to(torch.int64).numpy(), inp.W.to(torch.int64).numpy()
    for e in range(len(counts)):
        g = (Xi[off[e]:off[e + 1]] @ Wi[e][:, :N]).astype(np.float64)
        u = (Xi[off[e]:off[e + 1]] @ Wi[e][:, N:]).astype(np.float64)
        if not np.allclose(H[off[e]:off[e + 1]], g / (1.0 + np.exp(-g)) * u, rtol=1e-13, atol=1e-12):
            return False
    return True


def _fp8_checks_pass(lib):
    lib.rgg_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.rgg_oracle_e4m3_to_f64.restype = ctypes.c_double
    P = ctypes.c_void_p
    lib.rgg_oracle_grouped_gemm_fp8.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                ctypes.c_int, P, ctypes.c_int]
    lib.rgg_oracle_grouped_gemm_fp8.restype = ctypes.c_int
    # every code against the library's own E4M3 conversion
    lib_vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([lib.rgg_oracle_e4m3_to_f64(c) for c in range(256)])
    ok = ~np.isnan(lib_vals)
    if not np.array_equal(mine[ok], lib_vals[ok]):
        return False
    # two experts with distinct column scales against the scaled plain product
    f = wl.make_fp8_custom([3, 4], K=16, N=8, seed=84)
    X8, W8 = wl.fp8_codes(f.X8), wl.fp8_codes(f.W8)
    sx, sw = f.sx.numpy(), f.sw.numpy()
    off = np.ascontiguousarray(f.offsets, dtype=np.int32)
    Y = np.full((7, 8), np.nan)
    if lib.rgg_oracle_grouped_gemm_fp8(X8.ctypes.data, W8.ctypes.data, sx.ctypes.data, sw.ctypes.data,
                                       off.ctypes.data, 2, 7, 16, 8, Y.ctypes.data, 1) != 0:
        return False
    Xd, Wd = f.X8.double().numpy(), f.W8.double().numpy()
    for e in range(2):
        ref = (Xd[off[e]:off[e + 1]] @ Wd[e]) * np.outer(sx[off[e]:off[e + 1]].astype(np.float64),
                                                         sw[e].astype(np.float64))
        if not np.allclose(Y[off[e]:off[e + 1]], ref, rtol=1e-12, atol=1e-12):
            return False
    return True


def _gather_checks_pass(lib):
    P = ctypes.c_void_p
    lib.rgg_oracle_gather_rows.argtypes = [P, ctypes.c_int64, ctypes.c_int, P, ctypes.c_int64, ctypes.c_int64, P]
    lib.rgg_oracle_gather_rows.restype = ctypes.c_int

    def gather(Xtok, idx, begin, end):
        Xtok = np.ascontiguousarray(Xtok, dtype=np.uint16)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        out = np.zeros((idx.size, Xtok.shape[1]), dtype=np.uint16)
        rc = lib.rgg_oracle_gather_rows(Xtok.ctypes.data, Xtok.shape[0], Xtok.shape[1], idx.ctypes.data, begin,
                                        end, out.ctypes.data)
        return rc, out

    # the hand-worked case, then the library's fancy indexing, then the range rule
    rc, Xg = gather([[1, 2, 3], [4, 5, 6], [7, 8, 9]], [2, 0, 2, 1], 0, 4)
    if rc != 0 or Xg.tolist() != [[7, 8, 9], [1, 2, 3], [7, 8, 9], [4, 5, 6]]:
        return False
    gen = np.random.default_rng(71)
    Xtok = gen.integers(0, 1 << 16, size=(50, 24), dtype=np.uint16)
    idx = gen.integers(0, 50, size=300)
    rc, Xg = gather(Xtok, idx, 0, 300)
    if rc != 0 or not np.array_equal(Xg, Xtok[idx]):
        return False
    for bad in ([4], [-1]):
        if gather(np.zeros((4, 3)), bad, 0, 1)[0] == 0:
            return False
    return True


def _all_pass(lib):
    return (_product_checks_pass(lib) and _tile_checks_pass(lib) and _eta_checks_pass(lib)
            and _swiglu_checks_pass(lib) and _fp8_checks_pass(lib) and _gather_checks_pass(lib))


def test_unmutated_copy_passes(tmp_path):
    assert _all_pass(_build(tmp_path, "clean", None))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert not _all_pass(_build(tmp_path, name, MUTANTS[name])), "pins missed mutant %s" % name
