"""The C ABI without a GPU: the library builds, loads, exports every entry
point include/rgg.h declares, and its host-only logic (the planner, argument
checks, status strings) behaves as documented.  No compute call is made."""
import ctypes
import os
import re

import pytest

import ragged_grouped_gemm_02_gb300 as rgg
from ragged_grouped_gemm_02_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return rgg.load_library()


def _declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(rgg_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_abi():
    names = _declared_functions()
    assert set(rgg.EXPORTED_SYMBOLS) <= names
    assert "rgg_grouped_gemm" in names and "rgg_export_tiles" in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), "librgg.so does not export %s" % name


def test_debug_library_exports_every_declared_symbol(lib):
    # librgg_debug.so: the same ABI with every device access bounds-checked
    dbg = rgg.open_library(rgg.debug_library_path())
    for name in _declared_functions():
        assert hasattr(dbg, name), "librgg_debug.so does not export %s" % name
    assert dbg.rgg_status_string(rgg.RGG_ERR_DEVICE_BOUNDS).decode().startswith("RGG_ERR_DEVICE_BOUNDS")


CHECKS_PROGRAM = r"""
#include <cstdio>
#include "rgg_checks.cuh"
using namespace rgg;
#define EXPECT(c) do { if (!(c)) { std::printf("failed: %s (line %d)\n", #c, __LINE__); return 1; } } while (0)
int main() {
    // X box: K coordinate inside [0, K) on a 16-byte boundary, first row inside [0, rows)
    EXPECT(x_box_ok(0, 0, 264, 10, 2));
    EXPECT(x_box_ok(256, 9, 264, 10, 2));
    EXPECT(!x_box_ok(264, 0, 264, 10, 2));
    EXPECT(!x_box_ok(4, 0, 264, 10, 2));      // 8 bytes: not a 16-byte boundary
    EXPECT(x_box_ok(16, 0, 272, 10, 1));      // FP8: 16 elements
    EXPECT(!x_box_ok(8, 0, 272, 10, 1));
    EXPECT(!x_box_ok(0, 10, 264, 10, 2));
    EXPECT(!x_box_ok(0, -1, 264, 10, 2));
    // W box: column, K coordinate, expert
    EXPECT(w_box_ok(512, 192, 3, 520, 264, 4, 2));
    EXPECT(!w_box_ok(520, 0, 0, 520, 264, 4, 2));
    EXPECT(!w_box_ok(4, 0, 0, 520, 264, 4, 2));
    EXPECT(!w_box_ok(0, 0, 4, 520, 264, 4, 2));
    EXPECT(!w_box_ok(0, 0, -1, 520, 264, 4, 2));
    EXPECT(w_box_ok(576, 0, 0, 520, 264, 4, 2, 64));   // a pair's second half past the last column
    EXPECT(!w_box_ok(584, 0, 0, 520, 264, 4, 2, 64));
    // stores: the expert's rows, columns inside [0, N)
    EXPECT(store_ok(37, 504, 16, 37, 38, 520));
    EXPECT(!store_ok(37, 512, 16, 37, 38, 520));
    EXPECT(store_ok(37, 512, 8, 37, 38, 520));
    EXPECT(!store_ok(38, 0, 8, 37, 38, 520));
    EXPECT(!store_ok(36, 0, 8, 37, 38, 520));
    EXPECT(!store_ok(37, -16, 16, 37, 38, 520));
    // TMEM columns
    EXPECT(tmem_cols_ok(480, 32, 512));
    EXPECT(!tmem_cols_ok(481, 32, 512));
    // tile descriptors against the offsets {0, 0, 37, 101}
    const int32_t off[4] = {0, 0, 37, 101};
    EXPECT(tile_ok(1, 0, 37, 0, off, 3, 520));
    EXPECT(tile_ok(2, 37, 64, 512, off, 3, 520));
    EXPECT(!tile_ok(0, 0, 1, 0, off, 3, 520));    // an empty expert has no rows
    EXPECT(!tile_ok(2, 37, 65, 0, off, 3, 520));  // past the expert's last row
    EXPECT(!tile_ok(2, 36, 1, 0, off, 3, 520));   // before its first
    EXPECT(!tile_ok(2, 37, 1, 520, off, 3, 520));
    EXPECT(!tile_ok(3, 0, 1, 0, off, 3, 520));
    EXPECT(!tile_ok(-1, 0, 1, 0, off, 3, 520));
    std::printf("ok\n");
    return 0;
}
"""


def test_bounds_check_predicates_on_the_host(tmp_path):
    # the debug build's predicates are plain host/device functions: their arithmetic is checked here
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    (tmp_path / "checks.cc").write_text(CHECKS_PROGRAM)
    csrc = os.path.join(ROOT, "ragged_grouped_gemm_02_gb300", "csrc")
    r = subprocess.run([gxx, "-std=c++17", "-Wall", "-Werror", "-I", csrc, str(tmp_path / "checks.cc"), "-o",
                        str(tmp_path / "checks")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(tmp_path / "checks")], capture_output=True, text=True, timeout=30)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout


def test_library_has_no_runtime_cuda_dependency():
    # the CUDA runtime is linked statically; the library loads on a machine
    # without a GPU or a driver and reaches the driver only when called
    import subprocess
    out = subprocess.run(["ldd", rgg.library_path()], capture_output=True, text=True).stdout
    assert "libcudart" not in out and "libcuda.so" not in out


def test_status_strings(lib):
    for code in range(9):
        s = rgg.rgg_status_string(code)
        assert s.startswith("RGG_")
    assert rgg.rgg_status_string(99) == "unknown rgg_status"


def test_null_handle_is_rejected_without_touching_cuda(lib):
    P = ctypes.c_void_p
    s = lib.rgg_grouped_gemm(None, P(16), P(16), P(16), P(16), 4, 256, 256, 512, None, None)
    assert s == rgg.RGG_ERR_INVALID_ARG
    assert lib.rgg_query_status(None, None) == rgg.RGG_ERR_INVALID_ARG
    assert lib.rgg_export_tiles(None, P(16), 4, 256, 512, 128, 128, None, 0, P(16), None) == rgg.RGG_ERR_INVALID_ARG


def test_create_without_a_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    s = lib.rgg_create(ctypes.byref(h), 0)
    assert s in (rgg.RGG_ERR_CUDA, rgg.RGG_ERR_INVALID_ARG)
    assert not h.value


# ------------------------------------------------------------------ planner

def test_plan_small_decode_uses_64_row_tiles(lib):
    # 16 rows per expert: the Pearl article's 64-row tiles where experts average <= 64 rows
    p = rgg.rgg_plan(32, 512, 6144, 4096)
    assert p["bm"] == 64 and p["bk"] == 64 and p["threads"] == 192
    assert p["grid"] == 152 and 2 <= p["stages"] <= 16
    assert p["smem_bytes"] <= 232448


def test_plan_large_balanced_groups_use_cta_pairs(lib):
    # 256 rows per expert, balanced: one 256-row pair tile per expert
    p = rgg.rgg_plan(64, 16384, 1024, 2688)
    assert p["bm"] == 256 and p["bn"] == 256 and p["tmem_cols"] == 512 and p["grid"] % 2 == 0


def test_plan_skewed_counts_prefer_128_row_tiles(lib):
    # the same total under rank^-1.2 skew: 256-row tiles on every expert would be 40 % padding,
    # so the static plan takes 128-row tiles with the size-sorted walk; the automatic plan runs the
    # large experts on CTA pairs beside them instead (the mixed launch with fixed walks)
    from ragged_grouped_gemm_02_gb300 import workloads as wl
    counts = wl.workload_counts("skew16k")
    p = rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=counts, mixed=-1)
    assert p["bm"] == 128 and p["bn"] == 256 and p["tail64"] == 1 and p["walk_order"] == 3
    p = rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=counts)
    assert p["mixed"] == 2 and p["bm"] == 256 and p["bn"] == 256 and p["grid"] == 88 and p["single_grid"] == 64
    # experts of 128 rows: a pair tile would be half empty
    p = rgg.rgg_plan(32, 4096, 6144, 4096, host_counts=[128] * 32)
    assert p["bm"] == 128


def test_plan_wave_cost_prefers_exact_n_tiling(lib):
    # N = 2688 = 14 x 192: with 1-CTA 128-row tiles forced, BN = 192 leaves no padded columns
    p = rgg.rgg_plan(64, 16384, 1024, 2688, bm=128)
    assert p["bn"] == 192 and p["tmem_cols"] == 512


def test_plan_stages_fill_shared_memory(lib):
    for bm, bn in [(64, 128), (64, 256), (128, 128), (128, 192), (128, 256)]:
        p = rgg.rgg_plan(64, 16384, 1024, 2688, bm=bm, bn=bn)
        stage = (bm + bn) * 128
        assert p["bm"] == bm and p["bn"] == bn
        # one more stage would not fit
        assert p["stages"] == 16 or (p["stages"] + 1) * stage + 1024 > 232448 - 8 * 65 - 200
        # more than half the SM's shared memory: one CTA (one TMEM allocation) per SM
        assert p["smem_bytes"] > 232448 // 2


def test_plan_host_counts_guide_bm(lib):
    # most experts tiny, but the routed rows average > 64 over busy experts
    counts = [0] * 60 + [1000, 1000, 1000, 1000]
    assert rgg.rgg_plan(64, 4000, 1024, 2688, host_counts=counts)["bm"] == 128
    counts = [16] * 32
    assert rgg.rgg_plan(32, 512, 6144, 4096, host_counts=counts)["bm"] == 64


def test_plan_grid_never_exceeds_tiles_or_sms(lib):
    p = rgg.rgg_plan(4, 256, 256, 512)
    assert p["max_tiles"] == (256 // p["bm"] + 4) * (-(-512 // p["bn"]))
    assert p["grid"] <= min(152, p["max_tiles"])
    assert rgg.rgg_plan(4, 256, 256, 512, max_ctas=3)["grid"] == 3
    assert rgg.rgg_plan(64, 16384, 1024, 2688, num_sms=148)["grid"] == 148


def test_plan_walk_order_choice(lib):
    from ragged_grouped_gemm_02_gb300 import workloads as wl
    # experts of three M tiles or more on CTA pairs: the mixed launch's claims in list order, each
    # expert N-major (the static walk order 4 when the mixed launch is off or cannot run)
    p = rgg.rgg_plan(32, 32768, 6144, 4096, host_counts=wl.workload_counts("prefill"))
    assert p["mixed"] == 1 and (p["grid"], p["single_grid"]) == (152, 0)
    assert rgg.rgg_plan(32, 32768, 6144, 4096)["mixed"] == 1  # balanced estimate without counts
    for kw in (dict(mixed=-1), dict(stages=6), dict(tail64=-1)):
        p = rgg.rgg_plan(32, 32768, 6144, 4096, host_counts=wl.workload_counts("prefill"), **kw)
        assert p["mixed"] == 0 and p["walk_order"] == 4, kw
    assert rgg.rgg_plan(32, 32768, 6144, 4096, host_counts=wl.workload_counts("prefill"), op="fp8")["walk_order"] == 4
    # one or two M tiles per expert: list order
    assert rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=wl.workload_counts("uniform"))["walk_order"] == 0
    assert rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=wl.workload_counts("uniform"), op="fp8")["walk_order"] == 0
    assert rgg.rgg_plan(32, 512, 6144, 4096, host_counts=wl.workload_counts("decode"))["walk_order"] == 0
    # strong skew: the size-sorted interleave (when the mixed launch is off)
    assert rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=wl.workload_counts("skew16k"),
                        mixed=-1)["walk_order"] == 3
    # an explicit order is kept; -1 asks for list order
    assert rgg.rgg_plan(32, 32768, 6144, 4096, walk_order=1)["walk_order"] == 1
    assert rgg.rgg_plan(32, 32768, 6144, 4096, walk_order=-1)["walk_order"] == 0
    assert rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=wl.workload_counts("skew16k"),
                        walk_order=-1)["walk_order"] == 0


@pytest.mark.parametrize("kw", [dict(E=0), dict(K=12), dict(N=100), dict(K=4), dict(M_tot=-1),
                                dict(M_tot=2 ** 31)])
def test_plan_rejects_bad_sizes(lib, kw):
    args = dict(E=4, M_tot=256, K=256, N=512)
    args.update(kw)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_plan(args["E"], args["M_tot"], args["K"], args["N"])
    assert ei.value.status == rgg.RGG_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(bm=32), dict(bn=64), dict(stages=1), dict(stages=17), dict(max_ctas=-1),
                                dict(walk_order=5), dict(walk_order=-2)])
def test_plan_rejects_bad_options(lib, kw):
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_plan(4, 256, 256, 512, **kw)
    assert ei.value.status == rgg.RGG_ERR_INVALID_ARG


def test_plan_rejects_too_many_experts(lib):
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_plan(4097, 4097, 256, 512)
    assert ei.value.status == rgg.RGG_ERR_UNSUPPORTED


def test_plan_too_many_stages_for_shared_memory(lib):
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_plan(64, 16384, 1024, 2688, bm=128, bn=256, stages=16)
    assert ei.value.status == rgg.RGG_ERR_UNSUPPORTED


def test_plan_cta_pair_mode(lib):
    p = rgg.rgg_plan(64, 16384, 1024, 2688, bm=256, bn=256)
    assert p["bm"] == 256 and p["bn"] == 256 and p["tmem_cols"] == 512
    assert p["grid"] % 2 == 0 and p["grid"] <= 152
    # each CTA holds 128 rows of X and half of the weight tile per stage
    stage = (128 + 128) * 128
    assert p["stages"] == 16 or (p["stages"] + 1) * stage + 1024 > 232448 - 8 * 65 - 200
    p = rgg.rgg_plan(4, 256, 256, 512, bm=256, bn=128)
    assert p["grid"] == 2 * min(76, (256 // 256 + 4) * 4)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_plan(64, 16384, 1024, 2688, bm=256, bn=192)
    assert ei.value.status == rgg.RGG_ERR_INVALID_ARG


def test_plan_gather_modes(lib):
    # small expert groups (64-row tiles): the gather is fused into the GEMM
    p = rgg.rgg_plan(32, 512, 6144, 4096, op="gather", workspace=True)
    assert p["gather_mode"] == 1 and p["bm"] == 64 and p["workspace_bytes"] == 0
    p = rgg.rgg_plan(32, 512, 6144, 2048, op="swiglu_gather")
    assert p["gather_mode"] == 1 and p["bm"] == 64 and p["bn"] in (128, 256)
    # large groups with a caller workspace: two passes, the second being the plain plan (CTA pairs included)
    plain = rgg.rgg_plan(64, 16384, 1024, 2688)
    p = rgg.rgg_plan(64, 16384, 1024, 2688, op="gather", workspace=True)
    assert p["gather_mode"] == 2 and p["workspace_bytes"] == 16384 * 1024 * 2
    assert (p["bm"], p["bn"], p["stages"]) == (plain["bm"], plain["bn"], plain["stages"])
    assert plain["gather_mode"] == 0 and plain["workspace_bytes"] == 0
    # without one the call allocates nothing and runs the fused gather; the plan still
    # reports the workspace the preferred two-pass mode would need
    p = rgg.rgg_plan(64, 16384, 1024, 2688, op="gather")
    assert p["gather_mode"] == 1 and p["bm"] in (64, 128) and p["workspace_bytes"] == 16384 * 1024 * 2
    # 32 rows per expert: 64-row tiles, but already two-pass; 16 or fewer: fused
    assert rgg.rgg_plan(32, 1024, 6144, 4096, op="gather", workspace=True)["gather_mode"] == 2
    assert rgg.rgg_plan(32, 512, 6144, 4096, op="gather", workspace=True)["gather_mode"] == 1
    assert rgg.rgg_plan(4, 1024, 256, 256, op="gather", host_counts=[1000, 8, 8, 8],
                        workspace=True)["gather_mode"] == 2
    assert rgg.rgg_plan(4, 1024, 256, 256, op="gather", host_counts=[20, 0, 0, 0],
                        workspace=True)["gather_mode"] == 1
    # the fused mode on request: 1-CTA tiles only
    p = rgg.rgg_plan(64, 16384, 1024, 2688, op="gather", gather_mode=1, workspace=True)
    assert p["gather_mode"] == 1 and p["bm"] == 128 and p["workspace_bytes"] == 0
    assert rgg.rgg_plan(64, 16384, 1024, 2688, op="gather", bm=256, workspace=True)["gather_mode"] == 2
    # the two-pass mode on request reports its workspace (the call itself needs one)
    p = rgg.rgg_plan(64, 16384, 1024, 2688, op="gather", gather_mode=2)
    assert p["gather_mode"] == 2 and p["workspace_bytes"] == 16384 * 1024 * 2
    for kw in ({"op": "gather", "bm": 256, "gather_mode": 1}, {"op": "swiglu_gather", "bn": 192},
               {"op": "gather", "gather_mode": 3}, {"op": "gather", "bm": 256}):
        with pytest.raises(rgg.RggError) as ei:
            rgg.rgg_plan(64, 16384, 1024, 2688, **kw)
        assert ei.value.status == rgg.RGG_ERR_INVALID_ARG


def test_gather_null_handle_is_rejected_without_touching_cuda(lib):
    P = ctypes.c_void_p
    for fn in (lib.rgg_grouped_gemm_gather, lib.rgg_grouped_gemm_swiglu_gather):
        s = fn(None, P(16), 100, P(16), P(16), P(16), P(16), 4, 256, 256, 512, None, None)
        assert s == rgg.RGG_ERR_INVALID_ARG


def test_plan_fused_gate_up_pair_tails(lib):
    # balanced large groups: CTA pairs; 256-column pair tiles run tails of <= 128 rows as M = 128
    # pair MMAs (each CTA loads 64 gate columns and their up columns), 128-column ones keep
    # 256-row tails (a 64-column panel cannot hold both); BN = 192 is refused
    p = rgg.rgg_plan(32, 32768, 6144, 2048, op="swiglu")
    assert p["bm"] == 256 and p["bn"] == 256 and p["tail64"] == 1
    assert rgg.rgg_plan(32, 32768, 6144, 2048, op="swiglu", bm=256, bn=128)["tail64"] == 0
    assert rgg.rgg_plan(64, 16384, 1024, 1344, op="swiglu")["bm"] == 256
    assert rgg.rgg_plan(64, 16384, 1024, 2688, op="gemm", bm=256)["tail64"] == 1
    assert rgg.rgg_plan(32, 512, 6144, 2048, op="swiglu")["bm"] == 64
    with pytest.raises(rgg.RggError):
        rgg.rgg_plan(64, 16384, 1024, 1344, op="swiglu", bn=192)
    # FP8 runs on 1-CTA tiles only (64 or 128 rows; BN 128 or 256)
    assert rgg.rgg_plan(64, 16384, 1024, 2688, op="fp8")["bm"] == 128
    for kw in (dict(bm=256), dict(bn=192)):
        with pytest.raises(rgg.RggError) as ei:
            rgg.rgg_plan(64, 16384, 1024, 2688, op="fp8", **kw)
        assert ei.value.status == rgg.RGG_ERR_INVALID_ARG


def test_plan_reports_the_launch_block_size(lib):
    # plain bf16 and CTA pairs: 6 warps; FP8 and the fused gate-up op on 1-CTA tiles: 10
    assert rgg.rgg_plan(64, 16384, 1024, 2688, bm=128)["threads"] == 192
    assert rgg.rgg_plan(64, 16384, 1024, 2688, op="fp8")["threads"] == 320
    assert rgg.rgg_plan(64, 16384, 1024, 1344, op="swiglu", bm=128)["threads"] == 320
    assert rgg.rgg_plan(32, 32768, 6144, 2048, op="swiglu")["threads"] == 320  # pairs, per CTA


def test_plan_mixed_launch(lib):
    # the mixed launch: pairs for the experts of >= pair_min_rows rows, single CTAs for the rest
    from ragged_grouped_gemm_02_gb300 import workloads as wl
    skew = wl.workload_counts("skew16k")
    p = rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=skew, mixed=1)
    assert p["mixed"] == 1 and p["bm"] == 256 and p["bn"] == 256 and p["tail64"] == 1
    assert p["grid"] % 2 == 0 and 0 < p["grid"] < 152 and p["grid"] + p["single_grid"] == 152
    assert p["stages"] >= 4 and p["single_stages"] >= 3 and p["pair_min_rows"] == 256
    assert p["smem_bytes"] <= 232448 and p["single_smem_bytes"] <= 232448 and p["tmem_cols"] == 512
    # every expert large: all SMs to the pairs; every expert small: all to single CTAs
    assert (rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=[256] * 64, mixed=1)["grid"],
            rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=[256] * 64, mixed=1)["single_grid"]) == (152, 0)
    q = rgg.rgg_plan(32, 512, 6144, 4096, host_counts=[16] * 32, mixed=1)
    assert (q["grid"], q["single_grid"]) == (0, 152)
    # without host counts the experts are taken as balanced
    assert rgg.rgg_plan(64, 16384, 1024, 2688, mixed=1)["grid"] == 152
    assert rgg.rgg_plan(64, 2048, 1024, 2688, mixed=1)["single_grid"] == 152
    # an explicit split, a threshold, a grid cap
    p = rgg.rgg_plan(64, 16384, 1024, 2688, mixed=1, mixed_pair_sms=76, pair_min_rows=1000)
    assert (p["grid"], p["single_grid"], p["pair_min_rows"]) == (76, 76, 1000)
    p = rgg.rgg_plan(64, 16384, 1024, 2688, mixed=1, mixed_pair_sms=-1)
    assert (p["grid"], p["single_grid"]) == (0, 152)
    p = rgg.rgg_plan(4, 256, 256, 512, host_counts=[100, 0, 300, 1], mixed=1, max_ctas=3)
    assert p["grid"] == 2 and p["single_grid"] == 1
    # chosen by the planner: fixed walks for a strong skew over 128-row tiles (host counts), claims
    # for experts of three or more 256-row tiles; off for balanced mid-size experts and small groups.
    # Without counts, experts of one to three 256-row tiles on average take the fixed walks with the
    # split from the device offsets (both kernels over all the SMs)
    assert rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=skew)["mixed"] == 2
    assert rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=skew)["device_split"] == 0
    p = rgg.rgg_plan(64, 16384, 1024, 2688)
    assert (p["mixed"], p["device_split"], p["grid"], p["single_grid"]) == (2, 1, 152, 152)
    p = rgg.rgg_plan(64, 16384, 1024, 2688, max_ctas=9)
    assert (p["mixed"], p["device_split"], p["grid"], p["single_grid"]) == (2, 1, 8, 9)
    assert rgg.rgg_plan(64, 4096, 1024, 2688)["mixed"] == 0          # 64 rows per expert
    assert rgg.rgg_plan(64, 16384, 1024, 2688, op="swiglu")["mixed"] == 0
    assert rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=[256] * 64)["mixed"] == 0
    assert rgg.rgg_plan(64, 2048, 1024, 2688, host_counts=wl.workload_counts("skew2k"))["mixed"] == 0
    assert rgg.rgg_plan(32, 32768, 6144, 4096)["mixed"] == 1
    # the fused gate-up op: claims for the large experts, but no fixed walks for a skew
    assert rgg.rgg_plan(32, 32768, 6144, 2048, op="swiglu")["mixed"] == 1
    assert rgg.rgg_plan(64, 16384, 1024, 1344, host_counts=skew, op="swiglu")["mixed"] == 0
    p = rgg.rgg_plan(64, 16384, 1024, 1344, host_counts=skew, op="swiglu", mixed=2)
    assert p["mixed"] == 2 and p["grid"] > 0 and p["single_grid"] > 0
    # the fixed walks on request; an explicit split or claims keep the launched grids as the split
    p = rgg.rgg_plan(64, 16384, 1024, 2688, host_counts=skew, mixed=2, mixed_pair_sms=76)
    assert (p["mixed"], p["grid"], p["single_grid"]) == (2, 76, 76)
    p = rgg.rgg_plan(64, 16384, 1024, 2688, mixed=2, mixed_pair_sms=76)
    assert (p["mixed"], p["grid"], p["single_grid"], p["device_split"]) == (2, 76, 76, 0)
    assert rgg.rgg_plan(64, 16384, 1024, 2688, mixed=1)["device_split"] == 0


def _mixed_split(counts, N, pmin, sms):
    # The SM split of the mixed launch restated: per 256-column tile, 2 (128 + c/2) for a 256-row
    # pair tile (c rounded up to 128; 2 (64 + c/2) for a pair tile of <= 128 rows), 128 + c for a
    # 128-row 1-CTA tile (c rounded up to 64; 64 + c for <= 64 rows); pair work weighted 112/100;
    # the pair share of the SMs rounded up to an even count within [2, sms - 1].
    cp = cs = 0
    for m in counts:
        for c0 in range(0, N, 256):
            cols = min(256, N - c0)
            pc, sc = -(-cols // 128) * 128, -(-cols // 64) * 64
            if m >= pmin:
                r = m % 256
                cp += (m // 256) * 2 * (128 + pc // 2) + (2 * (128 + pc // 2) if r > 128 else
                                                          2 * (64 + pc // 2) if r > 0 else 0)
            elif m > 0:
                r = m % 128
                cs += (m // 128) * (128 + sc) + ((128 + sc) if r > 64 else (64 + sc) if r > 0 else 0)
    if cp == 0:
        return 0
    if cs == 0:
        return sms & ~1
    wp, ws = 112 * cp, 100 * cs
    pair = ((sms * wp + wp + ws) // (wp + ws)) & ~1
    return min(max(pair, 2), (sms - 1) & ~1)


@pytest.mark.parametrize("counts,N,pmin", [("skew16k", 2688, 256), ("worklog_skew16k", 2688, 256),
                                           ("skew16k", 2688, 512), ([300, 5, 70, 129, 1000, 0], 520, 256),
                                           ([256] * 8 + [16] * 8, 4096, 256), ([16] * 32, 4096, 256),
                                           ([1000] * 4, 136, 256)])
@pytest.mark.parametrize("sms", [152, 9, 3])
def test_plan_mixed_split_matches_its_cost_model(lib, counts, N, pmin, sms):
    from ragged_grouped_gemm_02_gb300 import workloads as wl
    c = [int(x) for x in (wl.workload_counts(counts) if isinstance(counts, str) else counts)]
    p = rgg.rgg_plan(len(c), sum(c), 1024, N, host_counts=c, mixed=2, max_ctas=sms, pair_min_rows=pmin)
    pair = min(_mixed_split(c, N, pmin, sms), sms & ~1)
    assert (p["grid"], p["single_grid"], p["device_split"]) == (pair, sms - pair, 0)


@pytest.mark.parametrize("kw,status", [(dict(bm=128), "INVALID_ARG"), (dict(bn=128), "INVALID_ARG"),
                                       (dict(tail64=-1), "INVALID_ARG"), (dict(mixed_pair_sms=3), "INVALID_ARG"),
                                       (dict(mixed_pair_sms=154), "INVALID_ARG"),
                                       (dict(mixed_pair_sms=-2), "INVALID_ARG"),
                                       (dict(pair_min_rows=-1), "INVALID_ARG"), (dict(mixed=3), "INVALID_ARG"),
                                       (dict(op="gather", gather_mode=1), "UNSUPPORTED"), (dict(op="fp8"), "UNSUPPORTED")])
def test_plan_mixed_rejects(lib, kw, status):
    args = dict(mixed=1)
    args.update(kw)
    with pytest.raises(rgg.RggError) as ei:
        rgg.rgg_plan(64, 16384, 1024, 2688, **args)
    assert ei.value.status == getattr(rgg, "RGG_ERR_" + status)
