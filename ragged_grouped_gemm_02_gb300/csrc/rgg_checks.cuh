// rgg_checks.cuh -- the bounds checks of the debug build (-DRGG_DEBUG_CHECKS,
// librgg_debug.so).
//
// Every TMA copy, global store, TMEM load and claimed tile descriptor of the
// kernels is checked against the bounds of what it touches before it is
// issued.  A check that fails records RGG_ERR_DEVICE_BOUNDS in the status word
// and the access is skipped, so nothing is ever issued out of bounds: a
// skipped copy leaves its stage's byte count short, the waits on it run out
// (bounded) and the launch ends with the bounds error, which is recorded
// first.  The accesses guarded are the ones a partial tile makes near the
// edges of an expert ("Grouped GEMM for Imbalanced Experts on Blackwell: A WIP
// Worklog", section 5.4: rows past the expert are read, never stored).  The
// release build compiles every check to `true`.
//
// The predicates are plain host/device functions so that their arithmetic is
// tested on the host as well.
#pragma once

#include <cstdint>

#ifndef __CUDACC__
#define __host__
#define __device__
#define __forceinline__ inline
#endif

namespace rgg {

constexpr int kStatusDeviceBounds = 8;

// A box of X (or of the token matrix) at K coordinate k and row `row`:
// k inside [0, K) on a 16-byte boundary (`elem_bytes` per element), the box's
// first row inside [0, rows).  Rows of the box past the end are zero-filled by
// the copy itself.
__host__ __device__ __forceinline__ bool x_box_ok(int64_t k, int64_t row, int64_t K, int64_t rows, int elem_bytes) {
    return k >= 0 && k < K && (k * elem_bytes) % 16 == 0 && row >= 0 && row < rows;
}

// A box of W [E, K, Nw] at column `col`, K coordinate k, expert e.  The box
// may start up to `overhang` columns past the last one: the second CTA of a
// pair tile whose columns end inside the first CTA's half loads a box that
// lies wholly past column Nw, which the copy zero-fills.
__host__ __device__ __forceinline__ bool w_box_ok(int64_t col, int64_t k, int64_t e, int64_t Nw, int64_t K, int64_t E,
                                                  int elem_bytes, int64_t overhang = 0) {
    return col >= 0 && col < Nw + overhang && (col * elem_bytes) % 16 == 0 && k >= 0 && k < K &&
           (k * elem_bytes) % 16 == 0 && e >= 0 && e < E;
}

// A store of `width` elements of row `row` at column `col`: the row inside the
// expert's rows [row_lo, row_hi), the columns inside [0, N).
__host__ __device__ __forceinline__ bool store_ok(int64_t row, int64_t col, int64_t width, int64_t row_lo,
                                                  int64_t row_hi, int64_t N) {
    return row >= row_lo && row < row_hi && col >= 0 && col + width <= N;
}

// A TMEM load of `width` columns from column `col` of an allocation of `ncols`.
__host__ __device__ __forceinline__ bool tmem_cols_ok(uint32_t col, uint32_t width, uint32_t ncols) {
    return col + width <= ncols;
}

// A tile descriptor: a real expert, rows inside that expert, a column tile
// inside [0, N).
__host__ __device__ __forceinline__ bool tile_ok(int32_t expert, int32_t row0, int32_t rows, int32_t col0,
                                                 const int32_t* off, int E, int64_t N) {
    if (expert < 0 || expert >= E || rows < 1 || col0 < 0 || col0 >= N) return false;
    return row0 >= off[expert] && static_cast<int64_t>(row0) + rows <= off[expert + 1];
}

#if defined(__CUDACC__) && defined(RGG_DEBUG_CHECKS)
__device__ __forceinline__ bool bounds_ok(bool cond, int32_t* status) {
    if (!cond) atomicCAS(status, 0, kStatusDeviceBounds);
    return cond;
}
#define RGG_BOUNDS_OK(cond, status) ::rgg::bounds_ok((cond), (status))
#else
#define RGG_BOUNDS_OK(cond, status) true
#endif

}  // namespace rgg
