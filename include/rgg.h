/*
 * rgg.h -- C ABI of the GB300 (sm_103a) ragged-M grouped GEMM library (librgg.so).
 *
 * The operation (sources cited by page title and section):
 *
 *   "Grouped GEMM for Imbalanced Experts on Blackwell: A WIP Worklog",
 *   "What I am measuring" and section 2 "The Grouped Problem and the flat tile
 *   list": after routing, the rows of X are grouped by expert and one launch
 *   computes E independent products  Y_e = X_e . W_e,  [m_e, K] x [K, N],
 *   where m_e is known only at run time and may be zero.  "Grouped GEMM"
 *   (InferenceX glossary), "Technical definition": independent matrix
 *   multiplications with different row counts in one launch.
 *
 * Data layout (all row-major, all device memory, all owned by the caller):
 *   X             bf16 [M_tot, K]      rows grouped by expert
 *   W             bf16 [E, K, N]       expert e's weight is W[e], N contiguous
 *   group_offsets int32 [E + 1]        expert e owns rows [off[e], off[e+1])
 *   Y             bf16 [M_tot, N]      written only on rows some expert owns
 * Accumulation is fp32; each output is rounded once to bf16 (nearest even).
 *
 * Offsets are valid when 0 <= off[0] <= off[1] <= ... <= off[E] <= M_tot.
 * Rows outside [off[0], off[E]) belong to no expert and are never written.
 * The library reads the offsets on the device only, so the routed row counts
 * never have to reach the host.
 *
 * Errors: arguments the host can check are checked before anything is
 * launched and reported by the return value.  What only the device can see
 * (invalid offsets, a pipeline wait that ran past its time limit) is recorded
 * in a status word owned by the handle and reported by rgg_query_status();
 * a launch that finds invalid offsets writes nothing to Y.  Nothing traps.
 *
 * Streams: every launching call is asynchronous on the given stream (a
 * cudaStream_t passed as void*; NULL is the legacy default stream).
 * rgg_grouped_gemm allocates nothing per call.  The GEMM kernels are
 * launched with programmatic stream serialisation: one may become resident
 * while the kernel ahead of it on the stream still runs, and waits on the
 * device for that kernel to complete before touching any memory, so the
 * usual stream order holds for its inputs and outputs.  Each lets the next
 * launch on the stream start early in turn: a caller's kernel launched after
 * it with programmatic serialisation must wait on the device
 * (cudaGridDependencySynchronize) before reading the output, as that launch
 * mode requires anyway; copies and kernels launched the usual way follow
 * completion as always.
 */
#ifndef RGG_H
#define RGG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rgg_status {
    RGG_OK = 0,
    RGG_ERR_INVALID_ARG = 1,     /* null pointer, bad size, misaligned pointer, unsupported option value */
    RGG_ERR_UNSUPPORTED = 2,     /* a valid request this build cannot run (no sm_103 device, E too large, ...) */
    RGG_ERR_CUDA = 3,            /* a CUDA runtime / driver call failed; see rgg_last_cuda_error() */
    RGG_ERR_BAD_OFFSETS = 4,     /* device-detected: group offsets not valid; nothing was written */
    RGG_ERR_DEVICE_TIMEOUT = 5,  /* device-detected: a pipeline wait exceeded the time limit; Y is incomplete */
    RGG_ERR_CAPACITY = 6,        /* rgg_export_tiles: more tiles than the output capacity (count still exact) */
    RGG_ERR_BAD_ROW_INDEX = 7,   /* device-detected (gather calls): a token index read was outside [0, T); the
                                    rows with such an index hold unspecified values, all other rows are right */
    RGG_ERR_DEVICE_BOUNDS = 8    /* device-detected, debug build (librgg_debug.so) only: a copy, store, TMEM load
                                    or tile descriptor failed its bounds check and was not issued; Y is
                                    incomplete.  The release build never reports it. */
} rgg_status;

typedef struct rgg_handle rgg_handle;

/* Tuning overrides; a zeroed struct (or a NULL pointer) means "choose automatically". */
typedef struct rgg_options {
    int bm;                      /* rows per tile: 0 = auto, or 64, 128, or 256 = a CTA pair on two SMs
                                    (tcgen05 cta_group::2, 128 rows per CTA; BN must then be 128 or 256) */
    int bn;                      /* columns per tile: 0 = auto, or 128, 192, 256 */
    int stages;                  /* shared-memory ring depth: 0 = as many as fit, else 2..16 */
    int max_ctas;                /* persistent CTAs: 0 = one per SM, else an upper bound */
    uint64_t timeout_ns;         /* limit of any single pipeline wait: 0 = 2 s */
    const int32_t* host_counts;  /* optional HOST copy of m_e[E] to guide the tile shape; NULL = use M_tot/E */
    int debug_flags;             /* 0 in normal use.  RGG_DEBUG_PRODUCER_STALL makes the load pipeline issue
                                    nothing, so the first MMA wait can only end by its time limit: a test of the
                                    bounded waits, which then report RGG_ERR_DEVICE_TIMEOUT */
    int tail64;                  /* tail tiles: 0 = auto (on), 1 = on, -1 = off.  With 128-row tiles a tile
                                    that holds the last <= 64 rows of its expert runs as a 64-row MMA
                                    with a 64-row X box; with CTA-pair (256-row) tiles one that holds
                                    the last <= 128 rows runs as a 128-row pair MMA, 64 rows per CTA */
    int op;                      /* for rgg_plan only: 0 = plan rgg_grouped_gemm, 1 = plan
                                    rgg_grouped_gemm_swiglu (then N is the output width), 2 = plan
                                    rgg_grouped_gemm_fp8, 3 = plan rgg_grouped_gemm_gather, 4 = plan
                                    rgg_grouped_gemm_swiglu_gather (N is the output width) */
    int walk_order;              /* order of the persistent CTAs' walk over the tile list (any order gives the
                                    same result): 0 = automatic (list order, or 3 when host_counts show a
                                    strong skew, or 4 when experts average three M tiles or more),
                                    1 = front/back interleave, 2 = strided scatter,
                                    3 = front/back interleave over the experts sorted by row count (E <= 256;
                                    chosen automatically when the largest expert holds over four times the
                                    mean), 4 = list order with each expert's tiles taken N tile by N tile
                                    (the M tiles that read one weight panel run side by side), -1 = list
                                    order, never replaced. */
    int gather_mode;             /* gather calls only: how the routed rows are fetched (same result either
                                    way).  1 = fused: the GEMM's producer loads them with TMA
                                    tile::gather4, four rows per copy, once per N tile; 2 = two-pass: a
                                    row-gather kernel writes them once, in routed order, into a workspace
                                    and the grouped GEMM reads that with whole-tile TMA boxes.  0 = auto:
                                    two-pass when the experts that have rows average more than 24 rows and
                                    the caller passes a workspace, else fused. */
    void* workspace;             /* two-pass gather only: caller-owned device memory of at least
                                    M_tot * K * 2 bytes, 16-byte aligned (rgg_plan reports the size in
                                    rgg_plan_info.workspace_bytes).  The library never allocates inside a
                                    call: without a workspace the automatic mode runs the fused gather,
                                    and gather_mode = 2 (or bm = 256, which only the two-pass mode can
                                    run) is RGG_ERR_INVALID_ARG. */
    int64_t workspace_bytes;     /* size of `workspace` in bytes */
    int mixed;                   /* rgg_grouped_gemm only: the mixed launch.  1 = on: experts of at least
                                    pair_min_rows rows run 256 x 256 tiles on CTA pairs (tcgen05
                                    cta_group::2; an expert's last tile of <= 128 rows as a 128-row pair
                                    MMA) and the other experts 128 x 256 tiles on single CTAs (<= 64-row
                                    tails as 64-row MMAs), as two kernels on disjoint SMs that claim tiles
                                    from two device counters and take each other's tiles when their own
                                    class runs out.  The classes are formed on the device from the offsets.
                                    2 = the same two kernels without claims: each walks its own class in a
                                    fixed order (and the other class too when the other kernel has no
                                    SMs), so the split of the SMs decides the balance.  0 = auto (the
                                    planner's choice), -1 = off.  On: bm and bn must be 0 or 256, tail64
                                    must not be -1, walk_order is not used. */
    int mixed_pair_sms;          /* mixed launch: SMs given to the pair kernel (even; the 1-CTA kernel gets
                                    the rest).  0 = split by the estimated work of each class: from
                                    host_counts when given; else, with fixed walks, from the device offsets
                                    (see rgg_plan_info.device_split), and with claims from balanced
                                    experts.  -1 = no pair kernel. */
    int pair_min_rows;           /* mixed launch: smallest expert (rows) that runs on CTA pairs; 0 = 256 */
} rgg_options;

#define RGG_DEBUG_PRODUCER_STALL 1

/* The configuration a call would use (see rgg_plan). */
typedef struct rgg_plan_info {
    int bm, bn, bk;              /* tile rows, tile columns, K per pipeline stage */
    int stages;                  /* ring depth */
    int grid;                    /* persistent CTAs launched */
    int threads;                 /* threads per CTA */
    int smem_bytes;              /* dynamic shared memory per CTA */
    int tmem_cols;               /* TMEM columns allocated per CTA (two accumulator buffers) */
    int64_t max_tiles;           /* upper bound on the flat tile count for these sizes */
    int tail64;                  /* 1 when tail tiles run as shorter MMAs (see rgg_options.tail64) */
    int walk_order;              /* walk order (see rgg_options) */
    int gather_mode;             /* gather ops: the mode the call runs with these options (1 = fused
                                    tile::gather4, 2 = two-pass); else 0 */
    int64_t workspace_bytes;     /* gather ops: the workspace the two-pass mode needs when it is asked
                                    for, or when the automatic choice prefers it (it runs only with a
                                    caller workspace); else 0 */
    int mixed;                   /* 1 (claims) or 2 (fixed walks) for the mixed launch: then bm, bn, stages,
                                    grid, smem_bytes describe its pair kernel (grid 0: none) and the next
                                    three its 1-CTA kernel */
    int single_grid;             /* mixed launch: CTAs of the 1-CTA kernel (0: none) */
    int single_stages;           /* mixed launch: ring depth of the 1-CTA kernel */
    int single_smem_bytes;       /* mixed launch: dynamic shared memory per CTA of the 1-CTA kernel */
    int pair_min_rows;           /* mixed launch: smallest expert on CTA pairs */
    int device_split;            /* mixed launch with fixed walks: 1 when the split of the SMs between the
                                    two kernels is taken on the device from the offsets (no host_counts,
                                    mixed_pair_sms 0): both kernels are launched over all the SMs (grid and
                                    single_grid above), every CTA computes the same split, and the CTAs past
                                    their kernel's share leave at once; else 0 */
} rgg_plan_info;

/*
 * Create a handle bound to CUDA device `device`: queries the SM count and the
 * shared-memory limit, checks for compute capability 10.3 (sm_103), and
 * allocates the handle's 256-byte device word, zeroed (once per handle; no
 * call allocates device memory after this).  Its first int32 is the status
 * word; three int32 at byte 64 are the mixed launch's tile counters, which
 * each mixed launch leaves at zero again when its last CTA ends.  On success
 * *out owns the handle; release it with rgg_destroy.  Returns
 * RGG_ERR_UNSUPPORTED on any other GPU.
 *
 * Concurrency: calls on one handle may run on any streams, but they share the
 * handle's status word (rgg_query_status returns the first error any of them
 * recorded); mixed launches (rgg_options.mixed) on one handle must not overlap
 * on the GPU, since they share the tile counters: order them on one stream.
 * Use a handle from several host threads only under the caller's own lock.
 */
rgg_status rgg_create(rgg_handle** out, int device);

/* Free the handle and its status word.  NULL is ignored. */
void rgg_destroy(rgg_handle* h);

/*
 * Y_e = X_e . W_e for every expert e, in one kernel launch on `stream`
 * (Worklog section 2 and section 7 "Next: tcgen05 and adaptive BM"): a
 * persistent, warp-specialized tcgen05 kernel walks the flat tile list it
 * builds from group_offsets.
 *
 * X, W, Y: device pointers, 16-byte aligned.  group_offsets: device int32
 * [E+1].  Requirements: 1 <= E <= 4096, 0 <= M_tot < 2^31, K >= 8 and
 * N >= 8 with K % 8 == 0 and N % 8 == 0 (the 16-byte row-stride rule of the
 * tensor-memory accelerator).  `opt` may be NULL.
 *
 * Returns RGG_OK once the launch is queued.  Invalid offsets or a device
 * timeout are reported later by rgg_query_status.  The call allocates
 * nothing and only reads the offsets on the device.
 */
rgg_status rgg_grouped_gemm(rgg_handle* h, const void* X, const void* W, const int32_t* group_offsets,
                            void* Y, int E, int64_t M_tot, int K, int N, void* stream,
                            const rgg_options* opt);

/*
 * The fused gate-up projection of an expert FFN with its activation, in one
 * launch: for every expert e and every row i it owns,
 *     H[i, j] = silu(g) * u,  g = X[i,:] . W13[e][:, j],  u = X[i,:] . W13[e][:, N + j],
 * silu(z) = z / (1 + exp(-z)), for 0 <= j < N.  The Worklog ("What I am
 * measuring", section 7 "Scope of these results") leaves this activation out
 * of its measured GEMM; the Pearl article ("What the 15% measures") times the
 * gate and up projections.  The pages do not name the activation; SiLU
 * gating (SwiGLU) is the reading taken.
 *
 * W13: bf16 [E, K, 2N] (gate columns [0, N), up columns [N, 2N)); H: bf16
 * [M_tot, N].  Each tile loads BN/2 gate and the matching BN/2 up columns,
 * one MMA of width BN puts both in TMEM, and the epilogue forms silu(g) * u in
 * fp32 before rounding once to bf16.  Tiles are 64 or 128 rows on one CTA
 * or 256 rows on a CTA pair (rgg_options.bm 0, 64, 128 or 256; bn 0, 128 or
 * 256, the MMA width).  Other arguments, requirements
 * (N % 8 == 0 here is the output width) and errors as for rgg_grouped_gemm.
 */
rgg_status rgg_grouped_gemm_swiglu(rgg_handle* h, const void* X, const void* W13, const int32_t* group_offsets,
                                   void* H, int E, int64_t M_tot, int K, int N, void* stream,
                                   const rgg_options* opt);

/*
 * FP8 grouped GEMM: for every row i of expert e and every column j,
 *     Y[i, j] = sx[i] * sw[e, j] * sum_k x8[i, k] * w8[e, k, j]
 * with X8 and W8 holding FP8 E4M3 codes (the OCP "E4M3FN" format).  The Pearl
 * article ("What the 15% measures") refers to Pearl's FP8 scheme without
 * describing it; the reading taken keeps the K loop free of scales: one fp32
 * scale per row of X and one per (expert, output column) of W, applied to the
 * fp32 accumulator in the epilogue, the result rounded once to bf16.  The MMA
 * is tcgen05.mma kind::f8f6f4 (K = 32 per instruction); a shared-memory stage
 * holds 128 K elements (one 128-byte swizzle row), so X and W stream at half
 * the bytes of the bf16 path.
 *
 * X8: uint8 codes [M_tot, K]; W8: uint8 codes [E, K, N]; sx: fp32 [M_tot];
 * sw: fp32 [E, N] (16-byte aligned); Y: bf16 [M_tot, N].  K and N are
 * multiples of 16 (the 16-byte row-stride rule for one-byte elements).  Tiles
 * are 1-CTA (rgg_options.bm 0, 64 or 128; bn 0, 128 or 256).  Other
 * arguments and errors as for rgg_grouped_gemm.
 */
rgg_status rgg_grouped_gemm_fp8(rgg_handle* h, const void* X8, const void* W8, const float* sx, const float* sw,
                                const int32_t* group_offsets, void* Y, int E, int64_t M_tot, int K, int N,
                                void* stream, const rgg_options* opt);

/*
 * The flat tile list the kernel walks, written out for checking (Worklog
 * section 2, "Source -- k1/common.cuh . k1/harness.cu"): descriptors
 * {expert, row0, rows, col0} in expert-major, M-tile, N-tile order, built on
 * the device by the same code the GEMM kernel uses.
 *
 * desc_out: device int32 [4 * cap] (may be NULL when cap == 0).
 * n_tiles_out: device int32 [1], receives the total tile count T (also when
 * T > cap, in which case only the first cap descriptors are written and the
 * status word records RGG_ERR_CAPACITY).  bm in {64, 128, 256}, bn in
 * {128, 192, 256}.  Asynchronous on `stream`; invalid offsets are reported by
 * rgg_query_status (T is then written as -1).
 */
rgg_status rgg_export_tiles(rgg_handle* h, const int32_t* group_offsets, int E, int64_t M_tot, int N,
                            int bm, int bn, int32_t* desc_out, int64_t cap, int32_t* n_tiles_out,
                            void* stream);

/*
 * The same tile list in the order the persistent walk visits it: entry p is
 * the tile at walk position p, which persistent CTA (or CTA pair) c of a grid
 * of G visits in its (p / G)-th step when p % G == c.  walk_order as in
 * rgg_options (0..4; 3 needs E <= 256, else RGG_ERR_UNSUPPORTED): 0 is the
 * list order of rgg_export_tiles, 1 the front/back interleave, 2 the strided
 * scatter, 3 the interleave over the experts sorted by row count, 4 each
 * expert's tiles N tile by N tile.  Every order lists each tile exactly once.
 * Decoded on the device by the code the GEMM kernels use; arguments, capacity
 * and status as for rgg_export_tiles.
 */
rgg_status rgg_export_walk(rgg_handle* h, const int32_t* group_offsets, int E, int64_t M_tot, int N, int bm,
                           int bn, int walk_order, int32_t* desc_out, int64_t cap, int32_t* n_tiles_out,
                           void* stream);

/*
 * Synchronize `stream`, read the device status word, reset it to RGG_OK and
 * return what it held (RGG_OK when no launch reported a problem).  Host-side
 * CUDA failures return RGG_ERR_CUDA.
 */
rgg_status rgg_query_status(rgg_handle* h, void* stream);

/*
 * The configuration rgg_grouped_gemm would choose for these sizes on a GPU
 * with `num_sms` SMs and `smem_optin` bytes of opt-in shared memory per block
 * (pass 0 for both to use GB300's 152 and 232448).  Pure host code: needs no
 * GPU.  The tile shape follows the Worklog's section 6 and section 7 point
 * that BM must be chosen from the expert sizes, and the Pearl article's
 * 64-row tiles where experts average 64 rows or fewer ("Four changes").
 */
rgg_status rgg_plan(int num_sms, int smem_optin, int E, int64_t M_tot, int K, int N,
                    const rgg_options* opt, rgg_plan_info* out);

/* A static, human-readable name for a status code. */
const char* rgg_status_string(rgg_status s);

/* The text of the last CUDA error seen by this library on this thread ("" if none). */
const char* rgg_last_cuda_error(void);

/*
 * rgg_grouped_gemm_noalloc -- the same product as rgg_grouped_gemm (default
 * options, same plan, kernels and launch code) for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry point.
 *
 * Who needs it: code that must not call cudaMalloc where it runs the GEMM --
 * an inference-engine plugin whose execute step runs inside the engine's
 * memory budget and may not allocate, or a process whose device memory all
 * belongs to a pool allocator that other code may not go around.
 * rgg_grouped_gemm needs a handle, and rgg_create allocates the handle's status
 * word.  This call takes no handle and allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Scratch: the kernels' only scratch -- the 4-byte status word and, when the
 * plan is the mixed launch, three int32 tile counters that the launch leaves
 * at zero when it ends -- lives in a file-scope device array of 256 bytes that
 * every GPU which loads librgg.so holds until the process exits.  The scratch
 * need does not grow with the problem, so only the kernel's own limits bound
 * a call (1 <= E <= 4096, 0 <= M_tot < 2^31, K and N multiples of 8): other
 * sizes are rejected with RGG_ERR_INVALID_ARG or RGG_ERR_UNSUPPORTED before
 * anything is launched.
 *
 * The call runs on the current CUDA device.  Its first call on a device sets
 * up that device (it looks up the array's device address with
 * cudaGetSymbolAddress and reads the SM count); make that first call before
 * any stream capture.  The address is kept for the life of the process: do not
 * use this entry point on a device after cudaDeviceReset() on that device.
 * Each call clears the status word, launches the kernel
 * and, when status_out is not NULL, copies the final status word into
 * *status_out (device memory or pinned host memory, int32): RGG_OK,
 * RGG_ERR_BAD_OFFSETS or RGG_ERR_DEVICE_TIMEOUT, valid once the stream has
 * reached that point.  All calls share the one array, so calls that overlap
 * on the GPU (other streams, other threads) race on it.
 *
 * Arguments, layouts and ownership as for rgg_grouped_gemm; asynchronous on
 * `stream` (a cudaStream_t, NULL = legacy default stream).
 */
rgg_status rgg_grouped_gemm_noalloc(const void* X, const void* W, const int32_t* group_offsets, void* Y,
                                    int E, int64_t M_tot, int K, int N, int32_t* status_out, void* stream);

/*
 * rgg_grouped_gemm_gather -- the grouped product with the token gather fused
 * into the activation loads:
 *
 *     Y[i, :] = X_tok[row_index[i], :] . W[e]      for every row i of expert e
 *
 * The Worklog starts after routing with the rows already grouped ("What I am
 * measuring") and names the permutation of rows and the scatter/gather of
 * tokens among the work it leaves out ("Scope of these results"); the
 * InferenceX glossary entry "Grouped GEMM" ("Engineering details") describes
 * that permutation.  Two ways to fetch the rows (rgg_options.gather_mode):
 * fused, where each tile reads its rows straight from the token matrix, four
 * rows per TMA tile::gather4 copy, only the groups of four that hold rows of
 * the tile's expert; or two-pass, where one kernel copies each routed row
 * once into a workspace and the grouped GEMM (CTA pairs included) reads it.
 * The automatic choice is fused for small expert groups, two-pass otherwise.
 *
 * X_tok      device bf16 [T, K], row-major: the tokens in their own order;
 *            16-byte aligned.  1 <= T < 2^31 (T may be 0 only when M_tot is 0).
 * row_index  device int32 [M_tot], 4-byte aligned: the token of each routed
 *            row.  Only the entries of rows [off[0], off[E]) are read; each
 *            must lie in [0, T), else the status word records
 *            RGG_ERR_BAD_ROW_INDEX, that row is computed from token 0 and the
 *            others are unaffected.  A token may appear in several experts.
 * W, group_offsets, Y, E, M_tot, K, N: as for rgg_grouped_gemm; Y is in
 *            routed (grouped) row order.
 * Options as for rgg_grouped_gemm, plus gather_mode and workspace; fused
 * tiles are 64 or 128 rows (no CTA pair).  The two-pass mode runs only with a
 * caller workspace (rgg_options.workspace; the call allocates nothing): calls
 * that share one workspace must be ordered on one stream.
 * Errors: as for rgg_grouped_gemm, plus RGG_ERR_BAD_ROW_INDEX (device-detected,
 * read with rgg_query_status) and RGG_ERR_INVALID_ARG for a workspace that is
 * missing (gather_mode = 2 or bm = 256), too small or misaligned.
 * Asynchronous on `stream`.
 */
rgg_status rgg_grouped_gemm_gather(rgg_handle* h, const void* X_tok, int64_t T, const int32_t* row_index,
                                   const void* W, const int32_t* group_offsets, void* Y, int E, int64_t M_tot,
                                   int K, int N, void* stream, const rgg_options* opt);

/*
 * rgg_grouped_gemm_swiglu_gather -- rgg_grouped_gemm_swiglu on gathered rows:
 * H[i, :] = silu(X_tok[row_index[i]] . W13[e][:, :N]) * (X_tok[row_index[i]] .
 * W13[e][:, N:]).  W13 is bf16 [E, K, 2N] (gate columns first), H is bf16
 * [M_tot, N]; everything else as for rgg_grouped_gemm_gather.  The gate-up
 * projection is the MoE op that reads tokens, so this is where the gather
 * belongs in a layer.
 */
rgg_status rgg_grouped_gemm_swiglu_gather(rgg_handle* h, const void* X_tok, int64_t T, const int32_t* row_index,
                                          const void* W13, const int32_t* group_offsets, void* H, int E,
                                          int64_t M_tot, int K, int N, void* stream, const rgg_options* opt);

#ifdef __cplusplus
}
#endif

#endif /* RGG_H */
