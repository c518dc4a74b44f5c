// Internal interface between the host side of libmbtile (mbtile_host.cpp) and
// its kernels (mbtile_kernels.cu).  Not installed; the public ABI is mbtile.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mbtile.h"

namespace mbt {

constexpr int kMaxStages = 8;
constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxThreads = 32 * (1 + kMaxConsumerWarps);
// Row and column sums with one CTA per SM (stages too large for two) run a
// wide CTA instead: up to 16 consumer warps, in kernels built for one block
// per SM (so the two-per-SM kernels keep their register budget).
constexpr int kMaxWideConsumerWarps = 16;
constexpr int kMaxWideThreads = 32 * (2 + kMaxWideConsumerWarps);
constexpr int kBoxRowBytes = 128;      // one 128-byte swizzle span per box row
constexpr int kSwizzleAtomBytes = 1024;
constexpr uint64_t kDefaultWaitBudgetNs = 1000000000ull;  // 1 s
// Flat row sum: rows of at most this many bytes are summed one thread per row,
// element by element (fewer instructions per row than masked 16-byte chunks).
constexpr int kFlatElemRowBytes = 64;

// Fields every pipeline kernel needs.  Sizes in elements unless named *_bytes.
struct PipeArgs {
    int64_t M, N;              // logical shape
    int64_t tiles_n;           // tiles across the columns
    int64_t tiles_m;           // tiles down the rows
    int64_t num_tiles;         // tiles_m * tiles_n
    int32_t col_group;         // tile order of the producer.  0: row-major (tile t
                               // is (t / tiles_n, t % tiles_n)).  g >= 1: column
                               // strips in groups of g adjacent strips (the last
                               // group may be narrower); a group's tiles are taken
                               // band by band, left to right within a band
    int32_t pad_pipe_;
    int32_t tile_m;            // rows per tile (= rows per box)
    int32_t boxes;             // 128-byte boxes per tile row: 1, 2, 4 or 8
    int32_t box_inner;         // elements per box row (128 / esize)
    int32_t esize;             // bytes per element
    int32_t stages;
    int32_t consumer_warps;
    uint32_t box_stride;       // shared-memory bytes between box buffers
    uint32_t stage_stride;     // shared-memory bytes between stages
    uint32_t tx_bytes;         // bytes one tile delivers to its full barrier
    int32_t fault;             // test hook, see mbt_opts.fault
    int32_t empty_extra;       // arrivals on an empty barrier beyond one per
                               // consumer warp (1 when a bulk store also reads
                               // the stage)
    uint64_t wait_budget_ns;
    int32_t *log;
    int64_t log_cap;
    int32_t *status;           // the call's status buffer, or nullptr (g_status)
};

struct CopyArgs {
    PipeArgs p;
    char *dst;
    int64_t ld_dst_bytes;
    int32_t store_mode;        // 0: consumer warps store with st.global.v4;
                               // 1: one consumer thread issues bulk tensor stores
    int32_t pad_;
};

struct RowsumArgs {
    PipeArgs p;
    float *out;
    float *partial;            // [bands][kmax][tile_m], used when kmax > 1
    int32_t *ticket;           // [bands], zero between calls
    int32_t *clear_ticket;     // the library's own workspace: the other ticket
    int64_t clear_n;           // set, zeroed by this call for the next (n words)
    int64_t units;             // scheduling units = num_tiles / gran
    int64_t gran;              // tiles per scheduling unit (1 or tiles_n)
    int32_t kmax;
    int32_t fused;             // 1: also copy every tile to dst (bulk stores)
    int32_t boxed;             // 1: a full/empty barrier pair per (stage, box); the
                               // consumer warps of box b use only box b's pair
    int32_t pad2_;
    char *dst;                 // fused copy destination
    int64_t ld_dst_bytes;
};

// Column sums (mbtile_colsum.cuh): tiles in strip-major order, each column
// strip (tile_n columns) reduced down the rows.
constexpr int kMaxColGroup = 2;

// Records the consumers of a row sum may post ahead of the flush warp.
constexpr int kFlushSlots = 2;

// The column sum's flush ring has one slot: its consumers post once per strip
// group they leave (a few times per launch), and a second slot would cost the
// bf16 8192 x 65536 column sum with 64 x 256 tiles, 3 stages and 8 consumer
// warps its second CTA per SM (measured 6733 -> 5088 GB/s).
constexpr int kColsumRingSlots = 1;

// Dynamic shared memory of the column sum's flush ring, after the stages:
// kColsumRingSlots slots of one float per consumer thread, element of a
// 16-byte chunk (16 / es) and strip of a group.
constexpr int64_t colsum_ring_bytes(int consumer_warps, int es, int col_group) {
    return static_cast<int64_t>(kColsumRingSlots) * 32 * consumer_warps * (16 / es) * col_group *
           4;
}

// Position of tile t in the strip-group order (PipeArgs.col_group = g >= 1).
struct ColPos {
    int64_t gstart;            // order position of the group's first tile
    int32_t gi;                // group index
    int32_t band;              // tile row (row band)
    int32_t kloc, wg;          // strip within its group, strips in the group
    // (M, N < 2^31, so bands and strips fit 32 bits; order positions need 64)
};

__host__ __device__ inline ColPos col_pos(int64_t t, int64_t tiles_m, int64_t tiles_n, int g) {
    ColPos c;
    const int64_t per = tiles_m * g;
    const int64_t gi = t / per;
    c.gi = static_cast<int32_t>(gi);
    c.gstart = gi * per;
    const int64_t left = tiles_n - gi * g;
    c.wg = static_cast<int32_t>(left < g ? left : g);
    const int64_t local = t - c.gstart;
    c.band = static_cast<int32_t>(local / c.wg);
    c.kloc = static_cast<int32_t>(local - static_cast<int64_t>(c.band) * c.wg);
    return c;
}

__host__ __device__ inline int64_t col_strip(const ColPos &c, int g) {
    return static_cast<int64_t>(c.gi) * g + c.kloc;
}

// The position of the next tile in the same order (no divisions).
__host__ __device__ inline void col_next(ColPos &c, int64_t tiles_m, int64_t tiles_n, int g) {
    if (++c.kloc == c.wg) {
        c.kloc = 0;
        if (++c.band == tiles_m) {
            c.band = 0;
            ++c.gi;
            c.gstart += tiles_m * g;
            const int64_t left = tiles_n - static_cast<int64_t>(c.gi) * g;
            c.wg = static_cast<int32_t>(left < g ? left : g);
        }
    }
}

struct ColsumArgs {
    PipeArgs p;                // col_group >= 1
    float *out;                // [N]
    float *partial;            // [strips][kmax][tile_n], used when kmax > 1
    int32_t *ticket;           // [strips], zero between calls
    int32_t *clear_ticket;     // as in RowsumArgs
    int64_t clear_n;
    int64_t units;             // scheduling units = num_tiles / gran
    int64_t gran;              // tiles per scheduling unit (1 or tiles_m)
    int32_t kmax;
    int32_t tile_n;            // columns per tile
};

// Matrices whose row pitch is not a multiple of 16 bytes (mbtile_flat.cuh).
struct FlatArgs {
    PipeArgs p;                // M, N, esize, stages, consumer_warps, stage_stride, ...
    const char *src;
    char *dst;                 // copy
    float *out;                // row sum
    int64_t ld;                // row pitch (elements)
    int64_t total_bytes;       // ((M - 1) ld + N) * esize
    int64_t t_floor;           // total_bytes rounded down to 16
    int64_t cap_bytes;         // bytes one stage can take (multiple of 16)
    int64_t rows_per_window;   // row sum: whole rows per window, 0 => long rows
    int64_t piece_elems;       // row sum, long rows: elements per piece
    int64_t pieces_per_row;
    int32_t phase_shift;       // row sum, short rows: the row groups of one 8-lane
                               // shared-memory phase take rows 2^phase_shift apart
    int32_t elem_rows;         // row sum, rows of at most kFlatElemRowBytes: each
                               // thread sums whole rows element by element
    int32_t elem_period;       // ... lanes this many apart read rows whose starts
                               // share a shared-memory bank (0: no such lanes);
                               // lane l starts its row (l / elem_period) words in
    int32_t pad0;
};

// Launchers (mbtile_kernels.cu).  They only enqueue work on `stream`.
cudaError_t launch_copy(const CUtensorMap &map, const CUtensorMap &dst_map,
                        const CopyArgs &a, int grid, int threads, int smem,
                        cudaStream_t stream);
cudaError_t launch_rowsum(int dtype, const CUtensorMap &map, const CUtensorMap &dst_map,
                          const RowsumArgs &a, int grid, int threads, int smem,
                          cudaStream_t stream);
cudaError_t launch_colsum(int dtype, const CUtensorMap &map, const ColsumArgs &a, int grid,
                          int threads, int smem, cudaStream_t stream);
cudaError_t launch_copy_unified(const CUtensorMap &map, const CopyArgs &a, int grid,
                                int threads, int smem, cudaStream_t stream);
cudaError_t launch_copy_flat(const FlatArgs &a, int grid, int threads, int smem,
                             cudaStream_t stream);
cudaError_t launch_rowsum_flat(int dtype, const FlatArgs &a, int grid, int threads, int smem,
                               cudaStream_t stream);
cudaError_t launch_stage_image(const CUtensorMap &map, int32_t row0, int32_t col0, int32_t boxes,
                               int32_t box_inner, uint32_t box_bytes, uint32_t box_stride,
                               unsigned char *image, cudaStream_t stream);
cudaError_t launch_fill_zero(float *out, int64_t n, cudaStream_t stream);
// acc[i] = part[i] (first) or acc[i] + part[i], 0 <= i < n.
cudaError_t launch_accumulate(float *acc, const float *part, int64_t n, bool first,
                              cudaStream_t stream);
// Raise every kernel's dynamic shared-memory limit as far as the device's
// opt-in limit allows; `usable` receives the limit common to all kernels.
cudaError_t set_kernel_smem_limit(int optin, int *usable);
// CTAs of a kernel with this block/smem shape that fit on one SM; kernel
// MBT_OP_COPY, MBT_OP_ROWSUM, MBT_OP_COPY_ROWSUM, 3 = unified copy,
// 4 = flat copy, 5 = flat row sum, 6 = column sum, 7 = copy with bulk stores,
// 8 = row sum with a barrier pair per box, 9 = wide row sum, 10 = wide column
// sum.
cudaError_t kernel_fit_per_sm(int op, int dtype, int threads, int smem, int *fit);
// Read the device status word and clear it (synchronous).
cudaError_t read_and_clear_status(int32_t info[4]);

}  // namespace mbt
