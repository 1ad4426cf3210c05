"""The C ABI from C (no GPU needed): a C11 program that includes only
include/rgg.h, compiled with warnings as errors and linked against
librgg.so, calls the host-only planner and the status strings.  Its output
must equal what the Python binding (ctypes) reads through the same calls, so
the header is valid C and the struct layouts on both sides agree."""
import os
import shutil
import subprocess

import pytest

import ragged_grouped_gemm_02_gb300 as rgg
from ragged_grouped_gemm_02_gb300 import _build
from ragged_grouped_gemm_02_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "rgg.h"

static char ws_marker[16]; /* rgg_plan only reads whether a gather workspace is given */

static void plan(int E, int64_t M, int K, int N, const int32_t* counts, int op, int bm, int walk, int ws,
                 int mixed) {
    rgg_options o;
    memset(&o, 0, sizeof(o));
    o.host_counts = counts;
    o.op = op;
    o.bm = bm;
    o.walk_order = walk;
    o.mixed = mixed;
    if (ws) {
        o.workspace = ws_marker;
        o.workspace_bytes = (int64_t)1 << 62;
    }
    rgg_plan_info p;
    memset(&p, 0, sizeof(p));
    rgg_status s = rgg_plan(0, 0, E, M, K, N, &o, &p);
    printf("%d %d %d %d %d %d %d %d %lld %d %d %d %lld %d %d %d %d %d %d\n", (int)s, p.bm, p.bn, p.bk, p.stages,
           p.grid, p.threads, p.smem_bytes, (long long)p.max_tiles, p.tail64, p.walk_order, p.gather_mode,
           (long long)p.workspace_bytes, p.mixed, p.single_grid, p.single_stages, p.single_smem_bytes,
           p.pair_min_rows, p.device_split);
}

int main(void) {
    static int32_t skew[64];
    FILE* f = fopen("counts.txt", "r");
    for (int e = 0; e < 64; ++e)
        if (fscanf(f, "%d", &skew[e]) != 1) return 2;
    fclose(f);
    plan(32, 512, 6144, 4096, NULL, 0, 0, 0, 0, 0);
    plan(64, 16384, 1024, 2688, NULL, 0, 0, 0, 0, 0);
    plan(64, 16384, 1024, 2688, skew, 0, 0, 0, 0, 0);
    plan(64, 16384, 1024, 2688, skew, 2, 0, 0, 0, 0);
    plan(64, 16384, 1024, 1344, skew, 1, 0, 0, 0, 0);
    plan(64, 16384, 1024, 2688, skew, 3, 0, 0, 0, 0);
    plan(64, 16384, 1024, 2688, skew, 3, 0, 0, 1, 0);
    plan(32, 32768, 6144, 4096, NULL, 0, 0, 0, 0, 0);
    plan(4, 256, 256, 512, NULL, 0, 64, 5, 0, 0);
    plan(64, 16384, 1024, 2688, skew, 0, 0, 0, 0, 1);
    plan(64, 16384, 1024, 2688, skew, 2, 0, 0, 0, 1);
    printf("%s|%s\n", rgg_status_string(RGG_ERR_BAD_OFFSETS), rgg_status_string(RGG_OK));
    return 0;
}
"""

CASES = [
    dict(E=32, M=512, K=6144, N=4096),
    dict(E=64, M=16384, K=1024, N=2688),
    dict(E=64, M=16384, K=1024, N=2688, counts=True),
    dict(E=64, M=16384, K=1024, N=2688, counts=True, op="fp8"),
    dict(E=64, M=16384, K=1024, N=1344, counts=True, op="swiglu"),
    dict(E=64, M=16384, K=1024, N=2688, counts=True, op="gather"),
    dict(E=64, M=16384, K=1024, N=2688, counts=True, op="gather", ws=True),
    dict(E=32, M=32768, K=6144, N=4096),
    dict(E=4, M=256, K=256, N=512, bm=64, walk_order=5),
    dict(E=64, M=16384, K=1024, N=2688, counts=True, mixed=1),
    dict(E=64, M=16384, K=1024, N=2688, counts=True, op="fp8", mixed=1),
]


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = _build.build()
    d = tmp_path_factory.mktemp("c_abi")
    (d / "prog.c").write_text(PROGRAM)
    counts = wl.workload_counts("skew16k")
    (d / "counts.txt").write_text(" ".join(str(int(c)) for c in counts))
    libdir = os.path.dirname(lib)
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(d / "prog.c"), "-o", str(d / "prog"), "-L", libdir, "-lrgg", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(d / "prog")], cwd=d, capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    return r.stdout.strip().splitlines(), counts


def test_c_program_sees_the_same_plans_as_python(c_output):
    lines, counts = c_output
    assert len(lines) == len(CASES) + 1
    for line, case in zip(lines, CASES):
        vals = [int(v) for v in line.split()]
        kw = dict(op=case.get("op", "gemm"), bm=case.get("bm", 0), walk_order=case.get("walk_order", 0),
                  workspace=True if case.get("ws") else None, mixed=case.get("mixed", 0))
        if case.get("counts"):
            kw["host_counts"] = counts
        if vals[0] != rgg.RGG_OK:
            with pytest.raises(rgg.RggError) as ei:
                rgg.rgg_plan(case["E"], case["M"], case["K"], case["N"], **kw)
            assert ei.value.status == vals[0]
            continue
        p = rgg.rgg_plan(case["E"], case["M"], case["K"], case["N"], **kw)
        fields = ["bm", "bn", "bk", "stages", "grid", "threads", "smem_bytes", "max_tiles", "tail64", "walk_order",
                  "gather_mode", "workspace_bytes", "mixed", "single_grid", "single_stages", "single_smem_bytes",
                  "pair_min_rows", "device_split"]
        assert vals[1:] == [p[f] for f in fields], (case, vals, p)


def test_c_program_status_strings(c_output):
    lines, _ = c_output
    bad, ok = lines[-1].split("|")
    assert bad == rgg.rgg_status_string(rgg.RGG_ERR_BAD_OFFSETS)
    assert ok == rgg.rgg_status_string(rgg.RGG_OK)
