/*
 * mbtile.h -- C ABI of the multi-stage mbarrier / bulk-tensor tile pipeline
 * for NVIDIA GB300 (sm_103a).
 *
 * The library streams a 2-D row-major matrix from device memory through a ring
 * of shared-memory stages.  One elected thread of a producer warp loads each
 * tile with a single bulk tensor copy (TMA) into a 128-byte-swizzled stage and
 * registers the expected bytes on the stage's "full" mbarrier; consumer warps
 * wait on that barrier, use the tile, and arrive on the stage's "empty"
 * mbarrier so the producer may refill it.  The consumers either write the tile
 * back out (tile_copy) or reduce it to fp32 row sums (tile_rowsum).
 *
 * Where the operations are defined:
 *   - "cute(11) Hopper TMA copy": §1 and §3 (a single thread issues one bulk
 *     tensor load of a whole tile; the mbarrier expects the tile's bytes; the
 *     tile is written back and must equal the input, §4); §2.2 (128-byte
 *     swizzle atom, 16-byte units); §6 (proxy visibility: a load by the copy
 *     engine followed by an mbarrier wait needs no extra fence).
 *   - "cute(12) async_pipeline": §1 (a full/empty barrier pair per stage, the
 *     producer at most S tiles ahead), §2 (the (index, phase, count) cursor,
 *     producer start phase 1), §3 and §6.6-6.10 (acquire, wait, release, tail).
 *   - "异步协作：mbarrier" (Async coordination: mbarrier): a phase completes
 *     when both the owed arrivals and the tx-count reach zero; waits use the
 *     phase parity and must be retried.
 *   - "CUDA features 10: Pipelines" (§4.10.4-4.10.5): warp-uniform control of
 *     the pipeline and completing every acquired stage before exit.
 *   The row sum is not on the pages (their consumer only "uses" the tile); it
 *   is the plain definition out[i] = sum_j src[i][j].
 *
 * Conventions common to every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller, except in
 *     the host-buffer forms (tile_copy_host, tile_rowsum_host).  The library
 *     allocates device memory in two places only: the host-buffer forms'
 *     staging pool, and the sum workspace it keeps per (device, stream) for
 *     row and column sums called without a workspace of the caller's (see
 *     tile_rowsum; allocated in stream order with cudaMallocAsync on the
 *     first such call on a stream, freed by tile_workspace_release).  Besides
 *     those it keeps per-device caches (SM count, shared-memory limit, the
 *     driver's tensor-map encoder) and a small per-device status word (see
 *     tile_status).  tile_rowsum_noalloc allocates nothing.
 *   - Matrices are row-major: element (i, j) is at ptr[i * ld + j], with the
 *     row pitch ld in elements.  The logical shape is M rows by N columns.
 *     Base pointers must be 16-byte aligned.  When ld * element size is a
 *     multiple of 16 bytes the tiles are moved by 2-D bulk tensor copies into
 *     128-byte-swizzled stages.  Otherwise (a bulk tensor copy needs 16-byte
 *     global strides) the stages are filled by 1-D bulk copies of 16-byte-
 *     aligned windows of the matrix's bytes: supported for tile_rowsum at any
 *     pitch and for tile_copy when src and dst are both dense (ld = N); other
 *     cases return MBT_ERR_ALIGN.  Row sums of rows of at most 64 bytes take
 *     the 1-D path whatever the pitch (one thread sums a whole row), unless
 *     more than 8 consumer warps are asked for.  A copy's stage then holds tile_m x tile_n
 *     elements' worth of bytes.  A row sum's window, whatever the tile, holds
 *     whole rows -- at most 32 KB while 8 rows fit in that, else at most 64
 *     KB -- or one of equal pieces (at most 64 KB) of a longer row, within
 *     what `stages` stages leave of the shared memory.  A longer row is cut
 *     into the fewest pieces that fit, or into the count that puts the most
 *     bytes of stages in flight on an SM (CTAs that fit, at most four, x
 *     stages x stage bytes) where that is at least 5 % more.
 *   - A tile is tile_m rows by tile_n columns.  tile_n * element size must be
 *     128, 256, 512 or 1024 bytes (1, 2, 4 or 8 side-by-side 128-byte boxes,
 *     each one bulk copy with the 128-byte swizzle); 1 <= tile_m <= 256;
 *     1 <= stages <= 8.  Tiles that run past row M or column N are loaded
 *     with zero fill and never written past the logical shape.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream) of the
 *     current device.  Calls are asynchronous on it, like any CUDA library.
 *     The pipeline kernels are launched with programmatic stream
 *     serialization: one may be launched, and set up its shared memory, while
 *     the previous kernel of the stream completes, but it reads and writes
 *     global memory only after that kernel has completed and its writes are
 *     visible.  Stream order is therefore what it would be without it: a call
 *     may read what the call before it wrote.
 *   - Return value: MBT_OK, or a negative mbt_status.  Argument errors are
 *     detected on the host before anything is launched.  A pipeline wait that
 *     runs past its time budget on the device does not hang: the kernel
 *     records MBT_ERR_TIMEOUT in the per-device status word (or in the call's
 *     own buffer, mbt_opts.status) and returns; tile_status reports the
 *     word.
 *   - Thread safety: entry points may be called from several host threads.
 *     Concurrent calls must not share a workspace.
 */
#ifndef MBTILE_H
#define MBTILE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  Copies move raw bits; row sums widen exactly to fp32. */
typedef enum mbt_dtype { MBT_F16 = 0, MBT_BF16 = 1, MBT_F32 = 2 } mbt_dtype;

typedef enum mbt_status {
    MBT_OK = 0,
    MBT_ERR_ARG = -1,          /* null pointer, bad size, shape or enum */
    MBT_ERR_ALIGN = -2,        /* base or row pitch not 16-byte aligned */
    MBT_ERR_UNSUPPORTED = -3,  /* tile shape / warp count outside the supported set */
    MBT_ERR_SMEM = -4,         /* stages x tile exceed the shared memory of one CTA */
    MBT_ERR_CUDA = -5,         /* a CUDA runtime call or the launch failed */
    MBT_ERR_TIMEOUT = -6,      /* a pipeline wait ran out of its time budget */
    MBT_ERR_DRIVER = -7,       /* tensor-map encoder unavailable or it refused */
    MBT_ERR_WORKSPACE = -8     /* workspace given but smaller than required, or
                                  the library's own would have to be allocated
                                  or grown during a stream capture */
} mbt_status;

/* Optional settings.  A zero-filled struct (or a NULL pointer) selects every
 * default. */
typedef struct mbt_opts {
    int64_t ld_src;          /* row pitch of src in elements; 0 => N */
    int64_t ld_dst;          /* row pitch of dst in elements (copy); 0 => N */
    int32_t max_ctas;        /* upper bound on the grid; 0 => no bound */
    int32_t ctas_per_sm;     /* CTAs per SM of the persistent grid (capped
                                at what fits); 0 => at least 2, and enough
                                that the stages on one SM hold ~64 KB (copy)
                                or ~128 KB (row sum) */
    int32_t consumer_warps;  /* consumer warps per CTA, 1..8 (up to 16 for
                                tile_rowsum and tile_colsum, see the
                                conventions above); 0 => tile_copy 4 (1 with
                                bulk stores); tile_rowsum 8, or 4 when the
                                default grid puts 3+ CTAs on an SM and
                                tile_m <= 128, or (with a 2-D tensor map) 2
                                CTAs at 3+ stages and tile_m <= 128, or 16
                                where one CTA per SM runs; tile_colsum 2
                                where 4+ CTAs per SM are wanted, else 8, or
                                4 at 3 CTAs per SM and tile_m <= 128;
                                tile_copy_rowsum 4 for tiles of one 128-byte
                                box and at most 128 rows, else 8, or 4 at 3+
                                CTAs per SM and tile_m <= 128.  The CTA has
                                one more warp, the
                                producer, and the warps mbt_plan.threads
                                lists. */
    int32_t store_mode;      /* tile_copy only (same result in every mode).
                                1: one consumer thread writes each landed
                                stage back with bulk tensor stores (same
                                swizzled box layout; the store map ends at the
                                last whole 16-byte chunk of a row, and a
                                row's partial last chunk is stored by the
                                warp's lanes); the CTA has one consumer warp
                                and consumer_warps is ignored.  2: the
                                consumer warps store with 16-byte st.global.
                                0 (default): 1 when rows end inside a 16-byte
                                chunk (LSU stores would leave a partly written
                                last sector per row), else 2; always 2 with
                                the unified pipeline.  mbt_plan.bulk_stores
                                tells which.  Source of the store recipe:
                                "cute(11) Hopper TMA copy" §6.3-6.4. */
    uint64_t wait_budget_ns; /* time bound of every mbarrier wait; 0 => 1 s */
    int32_t *log;            /* optional device buffer of int32 records, see
                                below; NULL => no log */
    int64_t log_capacity;    /* records per role in `log` */
    void *workspace;         /* row and column sums: device scratch that lets
                                several CTAs share one row band (column
                                strip); NULL => the library's own workspace
                                for (device, stream), unless no_split */
    size_t workspace_bytes;  /* size of `workspace` */
    int32_t fault;           /* test hook, 0 = none.  1: the producer starts at
                                phase 0; 2: consumers never release a stage.
                                Both make the pipeline stall by design, so the
                                call ends with MBT_ERR_TIMEOUT after about
                                (stages + 2) x wait_budget_ns; no bulk copy is
                                in flight when the kernel returns. */
    int32_t pipeline;        /* tile_copy only.  0: warp-specialised (a
                                producer warp and consumer warps, full/empty
                                barrier pair per stage; default).  1: unified
                                -- every warp consumes; one elected thread
                                issues each tile S-1 tiles ahead; a CTA-wide
                                barrier releases a stage ("CUDA features 10:
                                Pipelines" §4.10.7 prologue / steady state /
                                epilogue).  Kept as a measured comparison
                                point; consumer_warps counts all warps.
                                tile_rowsum only (same sums, bit for bit):
                                2: one full/empty pair per stage;
                                3: a pair per 128-byte box of a stage
                                wherever the tile allows it (see
                                mbt_plan.box_barriers); 0 chooses 3 for at
                                most 2 stages, else 2 (per-box pairs gain at
                                2 stages and lose at 3 on the bf16 64 x 256
                                row sum). */
    int32_t host_slab_rows;  /* tile_copy_host / tile_rowsum_host only: rows
                                per slab; 0 => whole row bands of about
                                MBT_HOST_SLAB_BYTES.  Must be 0 for the
                                device calls. */
    int32_t reserved0;       /* must be 0 */
    int32_t *status;         /* optional device int32[4], zero on entry: a
                                pipeline wait of this call that runs out of
                                its budget is recorded here ({code, block,
                                stage, role * 2 + parity}, as tile_status
                                reports it) instead of in the per-device
                                status word, so that calls on concurrent
                                streams can tell whose wait stalled.  The
                                caller reads it after the stream has
                                finished and clears it before reuse.  NULL =>
                                the per-device word.  Must be 4-byte
                                aligned. */
    int32_t no_split;        /* row and column sums: 1 => every row band
                                (column strip) is reduced by a single CTA and
                                no workspace is used (workspace must be NULL);
                                0 => bands (strips) may be split over several
                                CTAs of a persistent grid.  Must be 0 for
                                tile_copy. */
    int32_t reserved1;       /* must be 0 */
} mbt_opts;

/* Launch plan, as computed by tile_plan (host only, no CUDA calls). */
typedef struct mbt_plan {
    int32_t grid;            /* CTAs launched */
    int32_t threads;         /* threads per CTA = 32 x (1 + consumer_warps),
                                plus the flush warp of the tiled row sums
                                (the fused operation's too) and of the column
                                sum (which finishes each band's / strip's
                                sums while the consumers go on), plus the
                                fused operation's store warp; none without a
                                producer warp (unified copy) */
    int32_t consumer_warps;
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t boxes;           /* 128-byte boxes per tile row */
    int32_t box_inner;       /* elements per box row (128 / element size) */
    int32_t box_rows;        /* rows per box (= tile_m) */
    int32_t tx_bytes;        /* bytes registered on a full barrier per tile */
    int32_t stage_bytes;     /* shared-memory bytes of one stage */
    int32_t split;           /* row sum: 1 if a band may span several CTAs */
    int32_t kmax;            /* row sum: most CTAs contributing to one band */
    int32_t flat;            /* 1: row pitch not a multiple of 16 bytes; the
                                1-D bulk-copy kernels run, num_tiles counts
                                their windows */
    int32_t box_barriers;    /* row sum: 1 if every 128-byte box of a stage
                                has its own full/empty barrier pair, so the
                                consumer warps of one box start on it, and
                                release it, independently of the other boxes.
                                Possible when each consumer warp reads a
                                single box: 32 x consumer_warps = tile_m x
                                tpr with tpr a multiple of boxes and tile_m x
                                tpr / boxes a multiple of 32; see
                                mbt_opts.pipeline for when it is chosen */
    int32_t col_group;       /* column sum: adjacent column strips taken
                                together, band by band (2 where strips are
                                split over CTAs and the tile row is 128
                                bytes, or up to 512 bytes with one CTA per
                                SM, and the pair's threads per 16-byte chunk
                                column, 32 x consumer_warps / (8 x boxes),
                                are a multiple of 8; else 1); 0 for the other
                                operations */
    int32_t bulk_stores;     /* copy: 1 if stages are written back with bulk
                                tensor stores (see mbt_opts.store_mode; always
                                1 for tile_copy_rowsum) */
    int32_t phase_shift;     /* flat row sum with whole rows per window: the
                                lane groups of one 8-lane shared-memory phase
                                sum rows 2^phase_shift apart, which spreads
                                their 16-byte reads over the bank groups; 0
                                otherwise */
    int64_t tiles_m;         /* tiles down the rows (row bands) */
    int64_t tiles_n;         /* tiles across the columns */
    int64_t num_tiles;
    size_t workspace_bytes;  /* row sum: workspace bytes this plan needs */
} mbt_plan;

enum { MBT_OP_COPY = 0, MBT_OP_ROWSUM = 1, MBT_OP_COPY_ROWSUM = 2, MBT_OP_COLSUM = 3 };

/*
 * tile_copy -- dst[i][j] = src[i][j], bit for bit, for 0 <= i < M, 0 <= j < N.
 *
 * Defined by "cute(11) Hopper TMA copy" §4 and "cute(12) async_pipeline" §3:
 * every tile is loaded by one bulk tensor copy into a swizzled stage and the
 * consumer warps store it back with 16-byte coalesced stores.
 *   src, dst   device pointers, dense (ld = N) or pitched (see opts);
 *              src and dst must not overlap unless equal.
 *   M, N       logical shape, >= 0 (M == 0 or N == 0: nothing to do).
 *   tile_m, tile_n, stages, dtype: see the conventions above.
 * Elements of dst outside the logical shape (pad columns) are not written.
 */
int tile_copy(const void *src, void *dst, int64_t M, int64_t N, int tile_m,
              int tile_n, int stages, int dtype, void *stream);
int tile_copy_ex(const void *src, void *dst, int64_t M, int64_t N, int tile_m,
                 int tile_n, int stages, int dtype, void *stream,
                 const mbt_opts *opts);

/*
 * tile_rowsum -- out[i] = sum over j < N of src[i][j], for 0 <= i < M.
 *
 * Elements are widened exactly to fp32 and summed in fp32 in a fixed order
 * (per thread: the 16-byte chunks of a tile in column order; then the tiles
 * of a band in column order; then the threads of a row; then, with a
 * workspace, the CTAs of a band in CTA order), so repeated calls with the same
 * plan give identical bits.
 *   src        device pointer, dense or pitched (opts->ld_src).
 *   out        device pointer to M floats (dense).
 *   M, N       >= 0.  N == 0 writes zeros; M == 0 does nothing.
 * The bands' tiles are split evenly over a persistent grid and the last CTA
 * to finish its part of a band adds the band's partial sums in CTA order.
 * That needs a workspace (band tickets and partial sums).  tile_rowsum, and
 * tile_rowsum_ex with opts->workspace NULL, use the library's own workspace
 * for (current device, stream): allocated in stream order (cudaMallocAsync,
 * then zero-filled) on the first such call on the stream, grown the same way
 * when a larger plan needs more, and reused by every later call on that
 * stream -- make the first call on a stream, for the largest shape, before
 * any stream capture on it (an allocation during a capture would break the
 * capture, so it returns MBT_ERR_WORKSPACE instead).  Calls on one stream are
 * ordered, so they may share it; calls on different streams have their own.
 * Free it with tile_workspace_release before destroying a stream whose
 * handle a new stream could take while the old one's work is still running.
 * A call that stops on a timed-out wait may leave band tickets set; the
 * next call on the stream clears them (the workspace alternates two ticket
 * sets, and each call zeroes the one it does not use).
 * With a caller's workspace (opts->workspace; size from
 * tile_rowsum_workspace_bytes, zero-filled before its first use, and left
 * zero-filled by every call that completes without a timeout) the plan and
 * the sums are the same, bit for bit.  opts->no_split = 1: each row band
 * (tile_m rows) is reduced by one CTA, no workspace.
 */
int tile_rowsum(const void *src, float *out, int64_t M, int64_t N, int tile_m,
                int tile_n, int stages, int dtype, void *stream);
int tile_rowsum_ex(const void *src, float *out, int64_t M, int64_t N,
                   int tile_m, int tile_n, int stages, int dtype, void *stream,
                   const mbt_opts *opts);

/*
 * tile_copy_rowsum -- both results in one pass over src:
 *   dst[i][j] = src[i][j] (bit for bit) and out[i] = sum over j < N of src[i][j].
 *
 * The fused form of the two consumers the pages' pipeline feeds ("cute(12)
 * async_pipeline" §3: the consumer uses each landed tile): each tile is read
 * from device memory once; one consumer thread writes the landed stage back
 * with bulk tensor stores ("cute(11) Hopper TMA copy" §6.3-6.4) while the
 * consumer warps reduce it.  The CTA has a producer warp, a store warp (bulk
 * tensor stores of each row's whole 16-byte chunks; its lanes store a row's
 * partial chunk at column N), a flush warp (each band's sums, as in
 * tile_rowsum) and the row-sum warps; each stage is released
 * when both the store and the row-sum warps are done with it.  Row sums are
 * bit-identical to tile_rowsum's with the same plan.  Workspace: as for
 * tile_rowsum (the library's own unless opts->workspace is given; size for a
 * caller's from tile_copy_rowsum_workspace_bytes).
 *   src, dst   as in tile_copy (opts->ld_src, opts->ld_dst; must not overlap
 *              unless equal); out as in tile_rowsum.
 * opts->store_mode must be 0.
 */
int tile_copy_rowsum(const void *src, void *dst, float *out, int64_t M, int64_t N,
                     int tile_m, int tile_n, int stages, int dtype, void *stream);
int tile_copy_rowsum_ex(const void *src, void *dst, float *out, int64_t M, int64_t N,
                        int tile_m, int tile_n, int stages, int dtype, void *stream,
                        const mbt_opts *opts);

/*
 * tile_colsum -- out[j] = sum over i < M of src[i][j] in fp32, 0 <= j < N.
 *
 * A second reduction of the same pipeline's tiles ("cute(12) async_pipeline"
 * §3: the consumer uses each landed tile; the pages name no reduction, this is
 * the plain definition).  The producer takes the tiles in strip-major order --
 * down each column strip of tile_n columns -- so the consumer threads keep
 * their columns' sums in registers across a strip; 32 x consumer_warps
 * threads are split over the tile row's 16-byte chunks (at least one thread
 * per chunk: tile_n * element size <= 32 x consumer_warps x 16 bytes, else
 * MBT_ERR_UNSUPPORTED).  out: device fp32[N], 4-byte aligned.  Elements are
 * widened exactly; each thread adds its rows in order, the threads of a
 * column and the CTAs sharing a strip are combined in a fixed order, so
 * repeated calls with the same plan give bit-identical sums.  The row pitch
 * must be a multiple of 16 bytes (MBT_ERR_ALIGN otherwise).
 *
 * opts: as for tile_rowsum_ex.  Strips may be split over several CTAs, with
 * the caller's workspace (see tile_colsum_workspace_bytes: tickets and
 * partial sums per strip, zero-filled, 256-byte aligned, left zero-filled)
 * or, when opts->workspace is NULL, the library's own for (device, stream),
 * exactly as tile_rowsum describes; opts->no_split = 1 reduces each strip
 * on a single CTA.  M = 0 writes N zeros; N = 0 writes nothing.
 */
int tile_colsum(const void *src, float *out, int64_t M, int64_t N, int tile_m,
                int tile_n, int stages, int dtype, void *stream);
int tile_colsum_ex(const void *src, float *out, int64_t M, int64_t N, int tile_m,
                   int tile_n, int stages, int dtype, void *stream,
                   const mbt_opts *opts);
int tile_colsum_workspace_bytes(int64_t M, int64_t N, int tile_m, int tile_n,
                                int stages, int dtype, const mbt_opts *opts,
                                size_t *bytes);

/* Workspace bytes tile_rowsum_ex needs on the current device for this shape
 * and these options (opts->workspace is ignored).  0 when no split helps or
 * opts->no_split is set. */
int tile_rowsum_workspace_bytes(int64_t M, int64_t N, int tile_m, int tile_n,
                                int stages, int dtype, const mbt_opts *opts,
                                size_t *bytes);
/* The same for tile_copy_rowsum_ex (its grid differs from tile_rowsum's). */
int tile_copy_rowsum_workspace_bytes(int64_t M, int64_t N, int tile_m, int tile_n,
                                     int stages, int dtype, const mbt_opts *opts,
                                     size_t *bytes);

/*
 * tile_rowsum_noalloc -- tile_rowsum_ex for callers that cannot allocate
 * device memory.
 *
 * Some callers may not call cudaMalloc: code whose device memory is all owned
 * by another allocator (a framework's pool, an embedding host), where a new
 * allocation would fail or fragment it, and latency-critical paths that must
 * not allocate or free because cudaMalloc / cudaFree can synchronise the
 * device.  This entry point computes exactly what tile_rowsum_ex computes but
 * allocates nothing: the band-split workspace is a static device array inside
 * the library, MBT_NOALLOC_SCRATCH_BYTES (1 MiB) per device that loads the
 * library, held until the process exits.  The caller still passes src and
 * out.  opts->workspace and opts->workspace_bytes must be 0 (MBT_ERR_ARG
 * otherwise).
 *
 * Errors: a shape whose plan needs more workspace than the array holds is
 * rejected with MBT_ERR_WORKSPACE before anything is launched (shapes that
 * need no workspace are always accepted).  Otherwise as tile_rowsum_ex.
 *
 * Set-up: the first call on a device looks up the array's device address
 * (with that device current) and keeps it for the device's context (after
 * cudaDeviceReset the next call looks it up again, and a call that fails
 * with MBT_ERR_CUDA drops it); make that first call before any stream
 * capture begins.  Every call clears the part of the array it uses (an
 * asynchronous memset on `stream`) before launching, so a call after one
 * that stopped on a timed-out wait starts clean.
 *
 * Sharing: every call on a device uses the same array, so calls whose work
 * overlaps on the GPU (different streams, or different host threads) race
 * with each other and may return wrong sums; serialise them, e.g. on one
 * stream.
 *
 * The pages have no counterpart of this entry point.
 */
#define MBT_NOALLOC_SCRATCH_BYTES (1u << 20)
int tile_rowsum_noalloc(const void *src, float *out, int64_t M, int64_t N,
                        int tile_m, int tile_n, int stages, int dtype,
                        void *stream, const mbt_opts *opts);

/*
 * tile_plan -- the launch plan for op (MBT_OP_COPY, MBT_OP_ROWSUM or
 * MBT_OP_COPY_ROWSUM), from
 * the device figures given as arguments; makes no CUDA call.
 *   num_sms        SMs of the device (> 0).
 *   smem_optin     opt-in dynamic shared memory limit per CTA, bytes.
 *   fit_per_sm     CTAs of this plan that fit on one SM (> 0).
 *   with_workspace row sum: plan for a split band (1) or whole bands (0).
 * Returns the same argument errors as the entry points.
 */
int tile_plan(int op, int64_t M, int64_t N, int tile_m, int tile_n, int stages,
              int dtype, const mbt_opts *opts, int num_sms, int smem_optin,
              int fit_per_sm, int with_workspace, mbt_plan *plan);

/*
 * tile_plan_device -- the plan a call of op (MBT_OP_*) with these arguments
 * runs on the current device: tile_plan with the device's SM count, shared
 * memory and the occupancy of the kernel the plan picks; row and column sums
 * planned as the call plans them (bands or strips split unless
 * opts->no_split).  Returns the argument errors of the calls, or
 * MBT_ERR_CUDA.
 */
int tile_plan_device(int op, int64_t M, int64_t N, int tile_m, int tile_n, int stages,
                     int dtype, const mbt_opts *opts, mbt_plan *plan);

/*
 * tile_stage_image -- debug: the raw shared-memory image of one staged tile.
 *
 * Loads tile (tile_row, tile_col) of src (M x N, row pitch ld elements, which
 * must be a multiple of 16 bytes) exactly as the pipelines do -- one 2-D bulk
 * tensor copy per 128-byte box with the 128-byte swizzle, completion counted
 * on an mbarrier -- and writes the stage's bytes to the device buffer `image`
 * (boxes x tile_m x 128 bytes, box after box, unswizzling nothing).  Used to
 * check the swizzle against "cute(11) Hopper TMA copy" §2.2.  One CTA, 1 KB
 * of slack plus the tile in shared memory.
 */
int tile_stage_image(const void *src, int64_t M, int64_t N, int64_t ld, int tile_m,
                     int tile_n, int dtype, int64_t tile_row, int64_t tile_col,
                     void *image, void *stream);

/*
 * Host-buffer forms: src, dst and out are HOST pointers (pinned memory from
 * cudaHostAlloc / cudaHostRegister lets the copies overlap; pageable memory
 * works but the driver then stages it).  The result is that of tile_copy_ex /
 * tile_rowsum_ex / tile_colsum_ex on the same matrix (sums: within the same
 * error bound, not necessarily bit-identical, since the work is split
 * differently).
 * The call is synchronous: on return every copy and kernel has finished.
 *
 * The matrix moves through the current device in slabs of whole row bands of
 * about MBT_HOST_SLAB_BYTES each, repacked there with a 16-byte row pitch (so
 * ld_src / ld_dst, in elements, may be any value >= N and host pointers need
 * no alignment).  Three slab slots and three streams pipeline the host-to-
 * device copy of slab k + 1, the kernel of slab k and the device-to-host copy
 * of slab k - 1.  The staging memory (3 x 2 slabs, plus a row-sum workspace)
 * comes from a per-device pool that the library owns; concurrent calls use
 * separate staging sets; tile_host_release frees the idle ones.
 *
 * opts: as for the device calls, except that log, workspace and
 * workspace_bytes must be NULL / 0 (the slab schedule owns them).  Returns
 * MBT_OK, an argument error before anything is copied, MBT_ERR_CUDA, or
 * MBT_ERR_TIMEOUT when a pipeline wait of this call ran out of its budget
 * (each staging set has its own device status buffer, so concurrent calls and
 * the per-device word do not see one another's timeouts).  opts->status must
 * be NULL.
 */
#define MBT_HOST_SLAB_BYTES (64ll << 20)
int tile_copy_host(const void *src, void *dst, int64_t M, int64_t N, int tile_m, int tile_n,
                   int stages, int dtype, const mbt_opts *opts);
int tile_rowsum_host(const void *src, float *out, int64_t M, int64_t N, int tile_m,
                     int tile_n, int stages, int dtype, const mbt_opts *opts);
/* Column sums of a host matrix (out: host fp32[N]).  Each slab's column sums
 * are added on the device in slab order, then copied out once; any host row
 * pitch (the slabs are repacked to a 16-byte pitch on the device). */
int tile_colsum_host(const void *src, float *out, int64_t M, int64_t N, int tile_m,
                     int tile_n, int stages, int dtype, const mbt_opts *opts);
/* Frees the current device's idle staging sets of the host-buffer forms. */
int tile_host_release(void);

/* Frees, in stream order (cudaFreeAsync on `stream`), the sum workspace the
 * library keeps for (current device, stream); the next row or column sum
 * without a caller's workspace on that stream allocates a new one.  MBT_OK
 * when there is none. */
int tile_workspace_release(void *stream);

/*
 * tile_read_checksum -- the read-bandwidth reference of the reductions:
 * *out = the XOR of all 32-bit words of the `bytes` bytes at src (a device
 * buffer, read once with 16-byte loads by a grid of whole CTAs per SM).
 *
 * Not an operation of the pages: row and column sums read their matrix and
 * write only its sums, so the copy's read + write bandwidth is not their
 * ceiling; the benchmark times this call on a buffer far larger than L2 and
 * states the sums' fraction of it beside their fraction of the copy peak.
 *   src    device pointer, 16-byte aligned; bytes a multiple of 16
 *          (MBT_ERR_ALIGN otherwise).  bytes == 0 gives 0.
 *   out    device pointer to one uint32, 4-byte aligned, overwritten (set to 0
 *          on `stream`, then XORed into by the kernel).
 * Asynchronous on `stream`.  Returns MBT_OK, MBT_ERR_ARG (out NULL or
 * misaligned, src NULL with bytes > 0), MBT_ERR_ALIGN or MBT_ERR_CUDA.
 */
int tile_read_checksum(const void *src, size_t bytes, uint32_t *out, void *stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * word.  info (may be NULL) receives {code, block, stage, role * 2 + parity}
 * of the first wait that timed out (role 0 = producer, 1 = consumer).
 * Returns MBT_OK, MBT_ERR_TIMEOUT, or MBT_ERR_CUDA. */
int tile_status(void *stream, int32_t info[4]);

/* Static description of a status code; never NULL. */
const char *tile_strerror(int code);

/* Figures of device `device`: SM count, opt-in shared memory per CTA and the
 * theoretical memory bandwidth 2 x memory clock x bus width (GB/s = 1e9 B/s).
 * Any output pointer may be NULL. */
int tile_device_info(int device, int *num_sms, int *smem_optin,
                     double *hbm_gbs_theoretical);

/*
 * Log records (opts->log).  Only CTA 0 records.  The buffer holds
 * 2 x log_capacity records of 4 int32 each: records [0, cap) belong to the
 * producer, [cap, 2 cap) to consumer warp 0.  Record k of a role is
 * {k, stage index, phase parity waited on, tile number}; tiles past the
 * capacity are not recorded.  The caller zero-fills the buffer beforehand.
 */

#ifdef __cplusplus
}
#endif

#endif /* MBTILE_H */
