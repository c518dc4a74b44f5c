// Host side of libmbtile: argument checks, launch planning, tensor-map
// encoding and the extern "C" entry points declared in mbtile.h.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <thread>
#include <tuple>

#include "internal.h"

namespace {

using mbt::CopyArgs;
using mbt::PipeArgs;
using mbt::RowsumArgs;

constexpr int kDefaultConsumerWarps = 4;         // copy
// Default CTAs per SM: enough that the stages of all CTAs on an SM hold about
// this many bytes, and never fewer than two.  Measured on GB300: one CTA per SM
// is consumer-bound; the copy (reads and writes share the DRAM) peaks with
// ~64 KB of stages per SM, the row sum (reads only) with ~128 KB; more data in
// flight lowers DRAM efficiency.  With bulk stores one stage per CTA is held by
// the store in progress, so it does not count.
constexpr int64_t kCopyBytesPerSm = 64 * 1024;
constexpr int64_t kRowsumBytesPerSm = 128 * 1024;
// Flat row sum (whatever the tile): windows of whole rows, at most
// kFlatShortWindowBytes while kFlatMinRowsPerWindow rows fit in that, else at
// most kFlatRowsumWindowBytes; rows too long for kFlatMinRowsPerWindow of them
// there are loaded in equal pieces of at most kFlatRowsumWindowBytes.  Both
// bounds shrink so that the stages fit in shared memory.  Its consumers hold a
// stage longer than the tiled row sum's, so the default grid keeps
// kFlatRowsumBytesPerSm of stages per SM.  Measured on GB300 (2 stages):
// 32 KB rows 4.6 -> 6.2 TB/s (fp16) and 5.0 -> 6.7 TB/s (fp32) against
// tile-sized windows of 16 KB and 128 KB per SM.
constexpr int64_t kFlatShortWindowBytes = 32 * 1024;
constexpr int64_t kFlatRowsumWindowBytes = 64 * 1024;
constexpr int64_t kFlatRowsumBytesPerSm = 192 * 1024;
// Long rows in pieces (flat_setup): the most flat row-sum CTAs an SM holds
// (with 4 consumer warps their registers allow no more), an SM's shared
// memory, and what a CTA takes besides its stages (static memory, the
// per-block reserve).
constexpr int64_t kFlatPiecesCtas = 4;
constexpr int64_t kSmemPerSmBytes = 228 * 1024;
constexpr int64_t kFlatCtaOverheadBytes = 2 * 1024;
constexpr int64_t kFlatMinRowsPerWindow = 8;
constexpr int kMaxDevices = 64;
// Smallest partial-sum area of the library's own workspace (most plans need
// far less; growing it costs an allocation on the stream).
constexpr int64_t kOwnedMinPartialBytes = 1 << 20;
constexpr int64_t kMaxCoord = 0x7fffffff;  // bulk-copy coordinates are int32

struct DeviceFigures {
    bool ready = false;
    int num_sms = 0;
    int smem_optin = 0;   // dynamic shared memory every kernel may use
};

std::mutex g_mutex;
DeviceFigures g_devices[kMaxDevices];
// CTAs per SM from the occupancy calculator, keyed by
// (device, op, dtype, threads, dynamic smem); the query is slow next to a launch.
std::map<std::tuple<int, int, int, int, int>, int> g_fit_cache;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int esize_of(int dtype) {
    switch (dtype) {
        case MBT_F16:
        case MBT_BF16: return 2;
        case MBT_F32: return 4;
        default: return 0;
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t m) { return ceil_div(a, m) * m; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks that need no device.  Fills the effective row pitches.
// *flat is set when the row pitch is not a multiple of 16 bytes and the
// operation can still run (through the 1-D bulk-copy kernels).
int check_args(int op, const void *src, const void *dst, int64_t M, int64_t N, int tile_m,
               int tile_n, int stages, int dtype, const mbt_opts &o, int64_t *ld_src,
               int64_t *ld_dst, bool *flat = nullptr, bool narrow_rows_flat = true) {
    if (flat) *flat = false;
    const int es = esize_of(dtype);
    if (es == 0) return MBT_ERR_ARG;
    if (op != MBT_OP_COPY && op != MBT_OP_ROWSUM && op != MBT_OP_COPY_ROWSUM &&
        op != MBT_OP_COLSUM)
        return MBT_ERR_ARG;
    const bool writes_dst = op == MBT_OP_COPY || op == MBT_OP_COPY_ROWSUM;
    const bool sums_only = op == MBT_OP_ROWSUM || op == MBT_OP_COLSUM;   // dst = fp32 sums
    if (M < 0 || N < 0) return MBT_ERR_ARG;
    if (tile_m < 1 || tile_m > 256 || tile_n < 1 || stages < 1 || stages > mbt::kMaxStages)
        return MBT_ERR_ARG;
    const int64_t row_bytes = static_cast<int64_t>(tile_n) * es;
    if (row_bytes != 128 && row_bytes != 256 && row_bytes != 512 && row_bytes != 1024)
        return MBT_ERR_UNSUPPORTED;
    if (o.consumer_warps < 0 || o.consumer_warps > mbt::kMaxWideConsumerWarps) return MBT_ERR_ARG;
    // more than 8 consumer warps: the wide row- and column-sum kernels only
    if (o.consumer_warps > mbt::kMaxConsumerWarps && op != MBT_OP_ROWSUM && op != MBT_OP_COLSUM)
        return MBT_ERR_ARG;
    if (o.ctas_per_sm < 0 || o.max_ctas < 0 || o.log_capacity < 0) return MBT_ERR_ARG;
    if (o.fault < 0 || o.fault > 2) return MBT_ERR_ARG;
    if (o.store_mode < 0 || o.store_mode > 2) return MBT_ERR_UNSUPPORTED;
    if (o.pipeline < 0 || o.pipeline > 3) return MBT_ERR_UNSUPPORTED;
    if (o.pipeline == 1 && op != MBT_OP_COPY) return MBT_ERR_ARG;
    if (o.pipeline >= 2 && op != MBT_OP_ROWSUM) return MBT_ERR_ARG;
    if (o.pipeline == 1 && o.store_mode == 1) return MBT_ERR_UNSUPPORTED;
    if (o.store_mode != 0 && op != MBT_OP_COPY) return MBT_ERR_ARG;
    if (o.reserved0 != 0 || o.reserved1 != 0) return MBT_ERR_ARG;
    if (o.no_split < 0 || o.no_split > 1) return MBT_ERR_ARG;
    if (o.no_split && (op == MBT_OP_COPY || o.workspace != nullptr)) return MBT_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(o.status) % 4 != 0) return MBT_ERR_ALIGN;
    if (o.host_slab_rows != 0) return MBT_ERR_ARG;   // host-buffer forms only
    if (o.log != nullptr && o.log_capacity == 0) return MBT_ERR_ARG;
    if (o.workspace == nullptr && o.workspace_bytes != 0) return MBT_ERR_ARG;
    if (M > kMaxCoord || N > kMaxCoord) return MBT_ERR_UNSUPPORTED;
    *ld_src = o.ld_src ? o.ld_src : N;
    *ld_dst = o.ld_dst ? o.ld_dst : N;
    if (*ld_src < N || *ld_dst < N || *ld_src < 0 || *ld_dst < 0) return MBT_ERR_ARG;
    if (sums_only && o.ld_dst != 0) return MBT_ERR_ARG;
    const bool empty = (M == 0 || N == 0);
    if (empty) {
        // Nothing is read; a row sum of empty rows still writes M zeros, a
        // column sum of empty columns N zeros.
        if (op == MBT_OP_ROWSUM && M > 0 && dst == nullptr) return MBT_ERR_ARG;
        if (op == MBT_OP_COLSUM && N > 0 && dst == nullptr) return MBT_ERR_ARG;
        return MBT_OK;
    }
    if (src == nullptr || dst == nullptr) return MBT_ERR_ARG;
    if (!aligned16(src)) return MBT_ERR_ALIGN;
    if (writes_dst && !aligned16(dst)) return MBT_ERR_ALIGN;
    if (sums_only && (reinterpret_cast<uintptr_t>(dst) & 3u) != 0) return MBT_ERR_ALIGN;
    const bool pitch_ok = (*ld_src * es) % 16 == 0 && (!writes_dst || (*ld_dst * es) % 16 == 0);
    if (!pitch_ok) {
        // Unaligned pitch: a row sum of any pitch, or a copy of a dense matrix
        // into a dense matrix (one contiguous byte array), through 1-D bulk copies.
        const bool flat_ok =
            op == MBT_OP_ROWSUM ||
            (op == MBT_OP_COPY && *ld_src == N && *ld_dst == N && o.store_mode != 1 &&
             o.pipeline == 0);
        if (!flat_ok) return MBT_ERR_ALIGN;
        if (o.consumer_warps > mbt::kMaxConsumerWarps) return MBT_ERR_ARG;   // 1-D kernels: <= 8
        if (flat) *flat = true;
        return MBT_OK;
    }
    if (static_cast<uint64_t>(*ld_src) * es >= (1ull << 40)) return MBT_ERR_UNSUPPORTED;
    // Row sums of rows of at most kFlatElemRowBytes take the 1-D kernels whatever
    // the pitch: a tile at least 128 bytes wide would carry mostly zero fill
    // (measured: bf16 rows of 8 elements, 64 x 256 tiles, 279 GB/s), while the
    // 1-D kernels sum such rows one thread a row.
    if (narrow_rows_flat && op == MBT_OP_ROWSUM && N * es <= mbt::kFlatElemRowBytes &&
        o.consumer_warps <= mbt::kMaxConsumerWarps) {
        if (flat) *flat = true;
    }
    return MBT_OK;
}

// CTA that owns tile x in a split of `units` units of `gran` tiles over G CTAs.
int64_t unit_owner(int64_t x, int64_t gran, int64_t units, int64_t G) {
    return ((x / gran + 1) * G - 1) / units;
}

// Most CTAs that share one band when `num_tiles` tiles are split tile by tile.
int32_t most_contributors(int64_t tiles_n, int64_t num_tiles, int64_t G) {
    int64_t kmax = 1;
    for (int64_t b = 1; b < G; ++b) {
        const int64_t start = b * num_tiles / G;
        if (start % tiles_n == 0) continue;   // boundary between bands
        const int64_t band = start / tiles_n;
        const int64_t x0 = band * tiles_n;
        const int64_t k = unit_owner(x0 + tiles_n - 1, 1, num_tiles, G) -
                          unit_owner(x0, 1, num_tiles, G) + 1;
        kmax = std::max(kmax, k);
    }
    return static_cast<int32_t>(kmax);
}

// Column sums: adjacent strips walked together so that a row's bytes in flight
// span at least this much (narrow tiles otherwise read scattered 128-byte
// pieces of each row: measured 4.1 against 5.7-6.2 TB/s for 256 bytes and up).
constexpr int64_t kColGroupBytes = 256;
// ... and at least this much where one CTA per SM streams alone: bf16
// 8192 x 65536 with 64 x 256 tiles at 4 stages ran at 4983 GB/s with one
// 512-byte strip at a time, 6219 with strip pairs (with two CTAs per SM, pairs
// lost 1.3 % at 2 stages).
constexpr int64_t kColGroupBytesOnePerSm = 1024;

int col_group_for(int tile_n, int es, bool one_per_sm = false) {
    const int64_t row = static_cast<int64_t>(tile_n) * es;
    const int64_t want = one_per_sm ? kColGroupBytesOnePerSm : kColGroupBytes;
    return static_cast<int>(
        std::min<int64_t>(mbt::kMaxColGroup, std::max<int64_t>(1, want / row)));
}

// Strips per group of a split column sum with W consumer warps: one for the
// wide CTA; a pair only where its tpc = 32 W / (8 boxes) threads per chunk
// column are a multiple of 8, so that each thread's rows share one swizzle
// term (the launch refuses other pairs).
int colsum_group(int W, int tile_n, int es, int boxes, bool one_per_sm) {
    if (W > mbt::kMaxConsumerWarps) return 1;
    const int cg = col_group_for(tile_n, es, one_per_sm);
    return cg > 1 && (32 * W / (8 * boxes)) % 8 != 0 ? 1 : cg;
}

// Most CTAs that share one column strip when num_tiles tiles in strip-group
// order (groups of g strips) are split tile by tile over G CTAs.
// A strip's tiles lie inside its group's range, so only groups that hold the
// start of some CTA's range can have more than one contributor.
int32_t colsum_contributors(int64_t tiles_m, int64_t tiles_n, int g, int64_t num_tiles,
                            int64_t G) {
    int64_t kmax = 1;
    const int64_t per = tiles_m * g;
    for (int64_t b = 1; b < G; ++b) {
        const int64_t gi = (b * num_tiles / G) / per;
        const int64_t gstart = gi * per;
        const int64_t wg = std::min<int64_t>(g, tiles_n - gi * g);
        for (int64_t k = 0; k < wg; ++k) {
            const int64_t first = gstart + k, last = gstart + (tiles_m - 1) * wg + k;
            kmax = std::max(kmax, unit_owner(last, 1, num_tiles, G) -
                                      unit_owner(first, 1, num_tiles, G) + 1);
        }
    }
    return static_cast<int32_t>(kmax);
}

// Copy: bulk tensor stores (one store-issuing warp) or 16-byte LSU stores by
// the consumer warps.  store_mode 0 picks bulk stores when rows end inside a
// 16-byte chunk (LSU stores then leave a partly written last sector per row:
// measured 6.17 against 6.62 TB/s for fp16 24577 x 16383), LSU stores
// otherwise; the unified pipeline always stores with LSU.  `n_mod` = N modulo
// the elements of a 16-byte chunk.
bool bulk_stores(int op, const mbt_opts &o, int64_t n_mod) {
    if (op != MBT_OP_COPY || o.pipeline == 1 || o.store_mode == 2) return false;
    return o.store_mode == 1 || n_mod != 0;
}

int wanted_ctas_per_sm(int op, const mbt_opts &o, int stages, int64_t stage_bytes, int64_t n_mod,
                       bool flat) {
    if (o.ctas_per_sm) return o.ctas_per_sm;
    const bool bulk = bulk_stores(op, o, n_mod) || op == MBT_OP_COPY_ROWSUM;
    const int64_t held = bulk ? 1 : 0;
    const int64_t live = std::max<int64_t>(1, stages - held);
    // reads only: row and column sums; the fused operation writes too
    const int64_t target = flat && op == MBT_OP_ROWSUM ? kFlatRowsumBytesPerSm
                           : op == MBT_OP_ROWSUM || op == MBT_OP_COLSUM ? kRowsumBytesPerSm
                                                                        : kCopyBytesPerSm;
    return static_cast<int>(std::max<int64_t>(2, ceil_div(target, live * stage_bytes)));
}

// Row sums: 8 consumer warps (256 threads: an even split of any power-of-two
// tile_m <= 256) when at most two CTAs share an SM; 4 warps when three or more
// do (then registers would not fit 8), unless the tile has more rows than 128
// threads can own.  The tiled row sum also takes 4 at 3 or more stages when
// two CTAs share an SM: measured on 32 KB tiles (bf16 64x256 and 32x512, fp16
// 128x128) at 3 stages, 4 warps beat 8 by 1.5-2.9 %, and on 16 KB tiles (fp32
// 128x32, fp16 128x64) at 4 stages by 3.0-5.0 %, while at 2 stages 8 beat 4
// by up to 4 %, and where only one 4-stage CTA fits an SM 4 warps lose a
// third.  Column sums that want four or more CTAs per SM take 2 warps, so that
// four fit the registers (with 4 warps only three do): fp32 12289 x 8191
// 128 x 32 and fp16 24577 x 16383 128 x 64 at 2 stages, +3.3-3.7 %.  Where
// only one CTA of the tiled row sum runs on an SM (`one_per_sm`: its stages
// leave no room for a second, or the caller asked for one): 8 warps where
// each thread then reads at most one round of 8 chunks of a tile row (boxes x
// tile_m <= 256; the 8-warp kernel then takes one base address per thread),
// else the wide kernel's 16.  Measured with one CTA per SM, 8 against 16
// warps: bf16 64 x 256 at 4 / 5 / 6 stages 6511 / 6641 / 6473 against 6102 /
// 6108 / 6102 GB/s, and 1-7 % ahead on 9 of 10 other one-round tiles (32 x
// 512, 256 x 64, 128 x 128, fp32 64 x 128 and 128 x 64); two-round tiles (fp32
// 128 x 128, bf16 128 x 256) 2-4.5 % behind.  The column sum keeps 8 unless
// asked (16 measured 2 % slower).
int consumer_warps_for(int op, int tile_m, int boxes, int stages, const mbt_opts &o,
                       int wanted_ctas, int64_t n_mod, bool flat, bool one_per_sm, bool wide_ok) {
    if (bulk_stores(op, o, n_mod)) return 1;   // one thread issues the stores
    if (o.consumer_warps) return o.consumer_warps;
    if (flat && op == MBT_OP_ROWSUM) return wanted_ctas <= 2 ? 8 : 4;   // no tile rows
    if (op == MBT_OP_ROWSUM && one_per_sm)
        return boxes * tile_m <= 256 || !wide_ok ? 8 : mbt::kMaxWideConsumerWarps;
    if (op == MBT_OP_ROWSUM && wanted_ctas == 2 && stages >= 3 && tile_m <= 128) return 4;
    if (op == MBT_OP_COLSUM && wanted_ctas >= 4) return 2;
    // The fused copy + row sum on tiles of one 128-byte box and at most 128
    // rows: 4 row-sum warps, whose reads of the stage compete less with the
    // store warp's (fp32 12289 x 8191 128 x 32, fp16 24577 x 16383 and 16384^2
    // 128 x 64, 2 CTAs per SM: +0.5-0.8 % at 3 stages, +0.8-1.8 % at 4).
    if (op == MBT_OP_COPY_ROWSUM && boxes == 1 && tile_m <= 128) return 4;
    if (op != MBT_OP_COPY) return (wanted_ctas <= 2 || tile_m > 128) ? 8 : 4;
    return kDefaultConsumerWarps;
}

// Window schedule of the 1-D bulk-copy kernels (pure; shared by planning and launch).
void flat_setup(int op, int64_t M, int64_t N, int64_t ld, int es, int tile_m, int tile_n,
                int stages, int smem_optin, mbt::FlatArgs *f) {
    f->ld = ld;
    f->total_bytes = M > 0 ? ((M - 1) * ld + N) * es : 0;
    f->t_floor = f->total_bytes & ~int64_t(15);
    f->cap_bytes = static_cast<int64_t>(tile_m) * tile_n * es;
    f->rows_per_window = 0;
    f->elem_rows = 0;
    f->elem_period = 0;
    f->piece_elems = 0;
    f->pieces_per_row = 0;
    if (op == MBT_OP_ROWSUM) {
        // Window bounds of the row sum: stages of at most `fit` bytes each
        // (whole 1 KB units) fill the shared memory at most.
        const int64_t fit =
            (static_cast<int64_t>(smem_optin) - mbt::kSwizzleAtomBytes) / std::max(stages, 1) /
            mbt::kSwizzleAtomBytes * mbt::kSwizzleAtomBytes;
        const int64_t longest = std::max<int64_t>(std::min(kFlatRowsumWindowBytes, fit), 64);
        const int64_t pitch_b = ld * es;
        f->cap_bytes = pitch_b * kFlatMinRowsPerWindow + 32 <= kFlatShortWindowBytes
                           ? std::min(kFlatShortWindowBytes, longest)
                           : longest;
    }
    if (op == MBT_OP_ROWSUM) {
        const int64_t row_bytes = N * es, pitch = ld * es, room = f->cap_bytes - 32;
        // Whole rows per window only when every consumer warp gets rows to
        // sum (a row's lanes stay inside one warp); else pieces of each row,
        // which all threads share.
        int64_t rows = room >= row_bytes ? (room - row_bytes) / pitch + 1 : 0;
        // A multiple of 32 rows spreads evenly over the consumer threads (129
        // rows on 128 threads would take two passes, the second for one row).
        if (rows >= 32) rows -= rows % 32;
        if (rows >= kFlatMinRowsPerWindow) {
            f->rows_per_window = rows;
            f->elem_rows = row_bytes <= mbt::kFlatElemRowBytes ? 1 : 0;
            // Rows a whole number w of 4-byte words apart start in the same bank
            // every 32 / gcd(w, 32) rows: the lanes that far apart read their
            // rows from different starting columns (measured on bf16 rows of 16
            // and 32 elements, dense: 8- and 16-way conflicts otherwise).
            if (f->elem_rows && pitch % 4 == 0) {
                int64_t g = pitch / 4, m = 32;
                while (m != 0) {
                    const int64_t t = g % m;
                    g = m;
                    m = t;
                }
                f->elem_period = g > 1 ? static_cast<int32_t>(32 / g) : 0;
            }
        } else {
            // Pieces of a long row: the count that puts the most bytes of stages
            // in flight on an SM (CTAs that fit its shared memory, at most
            // kFlatPiecesCtas, x stages x stage bytes), where that is at least
            // 5 % more than with the fewest pieces that fit the window.
            // Measured, dense rows, 2 stages, GB/s: bf16 131 KB rows 3 pieces
            // (2 CTAs per SM) 5434 -> 5 pieces (4) 6451; fp16 80 KB rows 2 -> 3
            // pieces 5438 -> 6529; bf16 60 KB rows 1 piece (1 CTA) 4605, 3
            // pieces (4 CTAs) 6273, 2 pieces (3 CTAs) 6453; bf16 200 KB rows
            // keep 4 pieces (2 CTAs, 6324; 7 pieces on 3 CTAs 5833).
            const int64_t most = room / es;
            const int64_t p_min = ceil_div(N, most);
            auto in_flight = [&](int64_t P, int64_t *ctas) {
                const int64_t stage_b =
                    round_up(ceil_div(N, P) * es + 32, mbt::kSwizzleAtomBytes);
                const int64_t per_cta =
                    std::max(stages, 1) * stage_b + mbt::kSwizzleAtomBytes + kFlatCtaOverheadBytes;
                *ctas = std::min<int64_t>(kFlatPiecesCtas, kSmemPerSmBytes / per_cta);
                return *ctas * std::max(stages, 1) * stage_b;
            };
            int64_t ctas = 0;
            const int64_t f_min = in_flight(p_min, &ctas);
            int64_t pieces = p_min, best = f_min;
            // Once kFlatPiecesCtas CTAs fit, more pieces only shrink the stages.
            for (int64_t P = p_min + 1; ctas < kFlatPiecesCtas && P <= N; ++P) {
                const int64_t fl = in_flight(P, &ctas);
                if (fl > best) {
                    best = fl;
                    if (fl * 100 >= f_min * 105) pieces = P;
                }
            }
            f->pieces_per_row = pieces;
            f->piece_elems = ceil_div(N, f->pieces_per_row);
        }
    }
}

// Flat row sum, short rows: lanes per row L for a window of `rows` rows on
// `nthr` consumer threads -- the kernel's rule (a power of two, as many lanes
// per row as the threads allow, up to a warp).
int flat_lanes_per_row(int64_t rows, int nthr) {
    int L = 1;
    while (L < 32 && 2 * L * rows <= nthr) L <<= 1;
    return L;
}

// Flat row sum, short rows: a 16-byte shared-memory load is served in phases
// of 8 lanes, one wavefront per 16-byte bank group (address / 16 mod 8) and
// distinct address in it.  A phase holds 8 / L rows' groups of L lanes; rows
// one pitch apart start in nearly the same bank group when the pitch is close
// to a multiple of 128 bytes (126-byte rows: ~23 wavefronts per load instead
// of 4).  The kernel therefore lets the groups of one phase take rows 2^shift
// apart; this picks the shift whose first loads spread best, by counting the
// wavefronts of sample phases (window start offsets 0, 4, 8, 12 mod 16, 8
// phases each).  The kernel pads a window's rows to a whole block of
// (8 / L) << shift rows, so a shift qualifies only if the padding adds no round
// of rows per lane group.  A shift is taken only if it cuts the wavefronts at
// least 3-fold: the row map costs a few instructions per row, and measured on
// rows whose lanes met 2-way conflicts (34- and 606-byte rows) removing them
// did not pay (-1.5 to -2.5 %), while 126-byte rows (~6 wavefronts per phase)
// gained 21 %.  0 when L >= 8 (a phase reads one row's consecutive chunks) or
// the rows are read 4 bytes at a time.
int flat_phase_shift(const mbt::FlatArgs &f, int64_t N, int es, int W) {
    if (f.rows_per_window <= 0 || f.elem_rows || N * es <= 16) return 0;
    const int L = flat_lanes_per_row(f.rows_per_window, 32 * W);
    if (L >= 8) return 0;
    const int64_t pitch = f.ld * es, rows = f.rows_per_window;
    // The answer depends on (pitch, rows per window, W) alone; callers repeat
    // shapes, so each host thread keeps its last one (the search below costs
    // a few microseconds).
    thread_local int64_t last_pitch = -1, last_rows = -1;
    thread_local int last_w = 0, last_shift = 0;
    if (pitch == last_pitch && rows == last_rows && W == last_w) return last_shift;
    const int per_phase = 8 / L;
    // Wavefronts of the first 16-byte loads of sample phases: per phase, the
    // most distinct chunks that share one bank group.
    auto wavefronts = [&](int shift) {
        int64_t total = 0;
        for (int off0 = 0; off0 < 16; off0 += 4) {
            for (int h = 0; h < 8; ++h) {
                int64_t chunk[8];
                int per_group[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                int n = 0, worst = 0;
                for (int q = 0; q < per_phase; ++q) {
                    const int64_t first =
                        (off0 + (h + (static_cast<int64_t>(q) << shift)) * pitch) / 16;
                    for (int gl = 0; gl < L; ++gl) {
                        const int64_t c = first + gl;
                        bool seen = false;
                        for (int k = 0; k < n; ++k) seen = seen || chunk[k] == c;
                        chunk[n++] = c;
                        if (!seen) worst = std::max(worst, ++per_group[c & 7]);
                    }
                }
                total += worst;
            }
        }
        return total;
    };
    const int64_t groups = 32 * W / L;
    const int64_t rounds = ceil_div(rows, groups);
    const int64_t base_cost = wavefronts(0);
    int best = 0;
    int64_t best_cost = base_cost;
    for (int shift = 1; shift <= 6; ++shift) {
        const int64_t blk = static_cast<int64_t>(per_phase) << shift;
        if (ceil_div(round_up(rows, blk), groups) != rounds) continue;
        const int64_t c = wavefronts(shift);
        if (c < best_cost) {
            best = shift;
            best_cost = c;
        }
    }
    last_pitch = pitch;
    last_rows = rows;
    last_w = W;
    last_shift = 3 * best_cost <= base_cost ? best : 0;
    return last_shift;
}

int64_t flat_windows(int op, const mbt::FlatArgs &f, int64_t M, int64_t G) {
    if (op == MBT_OP_COPY) return ceil_div(f.t_floor, f.cap_bytes);
    int64_t n = 0;
    for (int64_t b = 0; b < G; ++b) {
        const int64_t rows = (b + 1) * M / G - b * M / G;
        n += f.rows_per_window > 0 ? ceil_div(rows, f.rows_per_window)
                                   : rows * f.pieces_per_row;
    }
    return n;
}

// Row sum with a full/empty barrier pair per (stage, box): each consumer warp
// must read a single box.  The threads of a row split its boxes * 8 chunks
// into tpr = 32 W / tile_m contiguous blocks; that holds when every thread
// is active (tile_m divides 32 W), tpr is a multiple of the box count, and
// the threads serving one box, tile_m tpr / boxes of them, are whole warps.
// By default only with at most kBoxBarrierMaxStages stages: measured on the
// bf16 64 x 256 row sum, per-box pairs gain ~0.4% at 2 stages and lose ~1.6%
// at 3 (the boxes of one tile are then issued at different times, so the
// 512-byte row segments of a tile no longer reach DRAM together).
constexpr int kBoxBarrierMaxStages = 2;

bool box_barriers_apply(int op, int tile_m, int boxes, int W, int stages, const mbt_opts &o,
                        bool flat) {
    if (op != MBT_OP_ROWSUM || flat || boxes < 2 || boxes > 8) return false;
    if (W > mbt::kMaxConsumerWarps) return false;   // the wide kernel has stage-wide pairs
    if (o.pipeline == 2 || (o.pipeline == 0 && stages > kBoxBarrierMaxStages)) return false;
    const int nthr = 32 * W;
    if (nthr % tile_m != 0) return false;
    const int tpr = nthr / tile_m;
    if (tpr % boxes != 0) return false;
    return (tile_m * (tpr / boxes)) % 32 == 0;
}

// fit_per_sm: CTAs of this plan's kernel that fit on one SM; 0 = not known yet
// (a first pass, before the occupancy query: planned as if two fit).
int plan_impl(int op, int64_t M, int64_t N, int tile_m, int tile_n, int stages, int dtype,
              const mbt_opts &o, int num_sms, int smem_optin, int fit_per_sm,
              int with_workspace, mbt_plan *plan, bool flat = false) {
    if (plan == nullptr || num_sms < 1 || fit_per_sm < 0) return MBT_ERR_ARG;
    const int es = esize_of(dtype);
    std::memset(plan, 0, sizeof *plan);
    plan->box_inner = mbt::kBoxRowBytes / es;
    plan->boxes = tile_n * es / mbt::kBoxRowBytes;
    plan->box_rows = tile_m;
    const int64_t box_stride = round_up(static_cast<int64_t>(tile_m) * mbt::kBoxRowBytes,
                                        mbt::kSwizzleAtomBytes);
    plan->stage_bytes = static_cast<int32_t>(plan->boxes * box_stride);
    if (flat && op == MBT_OP_ROWSUM) {
        // The flat row sum's windows do not follow the tile (flat_setup):
        // whole rows, or equal pieces of a long row.  Stages are sized to the
        // largest window it really loads (+ 16-byte rounding at both ends),
        // and the grid by those bytes in flight.
        mbt::FlatArgs f{};
        flat_setup(op, M, N, o.ld_src ? o.ld_src : N, es, tile_m, tile_n, stages, smem_optin, &f);
        const int64_t pitch = (o.ld_src ? o.ld_src : N) * es;
        const int64_t window = f.rows_per_window > 0
                                   ? (std::min(f.rows_per_window, std::max<int64_t>(M, 1)) - 1) *
                                             pitch + N * es
                                   : f.piece_elems * es;
        plan->stage_bytes = static_cast<int32_t>(
            round_up(std::min<int64_t>(window + 32, f.cap_bytes), mbt::kSwizzleAtomBytes));
    }
    const int64_t n_mod = N % (16 / es);
    const int wanted = wanted_ctas_per_sm(op, o, stages, plan->stage_bytes, n_mod, flat);
    const bool one_per_sm = wanted == 1 || fit_per_sm == 1;
    // wide column sums walk one strip at a time (a split plan of 128-byte tiles
    // walks two)
    const bool wide_ok = op == MBT_OP_ROWSUM || !with_workspace || col_group_for(tile_n, es) == 1;
    const int W = consumer_warps_for(op, tile_m, plan->boxes, stages, o, wanted, n_mod, flat,
                                     one_per_sm, wide_ok);
    plan->bulk_stores = bulk_stores(op, o, n_mod) || op == MBT_OP_COPY_ROWSUM ? 1 : 0;
    // Row sums: at least one thread per tile row; column sums: at least one
    // thread per 16-byte chunk column of a tile row.
    if (op == MBT_OP_COLSUM) {
        if (W * 32 < plan->boxes * 8) return MBT_ERR_UNSUPPORTED;
    } else if (op != MBT_OP_COPY && !flat && W * 32 < tile_m) {
        return MBT_ERR_UNSUPPORTED;
    }
    plan->consumer_warps = W;
    // producer warp + consumer warps (+ the fused operation's store warp, or
    // the flush warp of the tiled row sum and the column sum); the unified
    // pipeline has no producer warp
    const bool second_warp = op == MBT_OP_COPY_ROWSUM || op == MBT_OP_COLSUM ||
                             (op == MBT_OP_ROWSUM && !flat);
    plan->threads = 32 * ((o.pipeline == 1 ? 0 : 1) + W + (second_warp ? 1 : 0) +
                          (op == MBT_OP_COPY_ROWSUM ? 1 : 0));   // the fused flush warp
    plan->tx_bytes = plan->boxes * tile_m * mbt::kBoxRowBytes;
    int64_t smem = static_cast<int64_t>(stages) * plan->stage_bytes + mbt::kSwizzleAtomBytes;
    if (op == MBT_OP_COLSUM) {
        // the flush ring, sized for the widest strip group the plan may take
        // (the same rule as the split plan's below)
        const int cg_max = colsum_group(W, tile_n, es, plan->boxes, one_per_sm);
        smem += mbt::colsum_ring_bytes(W, es, cg_max);
    }
    if (smem > smem_optin) return MBT_ERR_SMEM;
    plan->smem_bytes = static_cast<int32_t>(smem);
    plan->tiles_m = ceil_div(M, tile_m);
    plan->tiles_n = ceil_div(N, tile_n);
    plan->num_tiles = plan->tiles_m * plan->tiles_n;
    int64_t per_sm = fit_per_sm > 0 ? std::min(wanted, fit_per_sm) : wanted;
    int64_t cap = per_sm * num_sms;
    if (o.max_ctas) cap = std::min<int64_t>(cap, o.max_ctas);
    plan->flat = flat ? 1 : 0;
    plan->box_barriers = box_barriers_apply(op, tile_m, plan->boxes, W, stages, o, flat) ? 1 : 0;
    if (plan->num_tiles == 0) return MBT_OK;
    if (flat) {
        mbt::FlatArgs f{};
        const int64_t ld = o.ld_src ? o.ld_src : N;
        flat_setup(op, M, N, ld, es, tile_m, tile_n, stages, smem_optin, &f);
        int64_t G = 1;
        if (op == MBT_OP_COPY) {
            G = std::max<int64_t>(1, std::min<int64_t>(ceil_div(f.t_floor, f.cap_bytes), cap));
        } else {
            G = std::min<int64_t>(M, cap);
        }
        plan->grid = static_cast<int32_t>(G);
        plan->num_tiles = flat_windows(op, f, M, G);
        plan->kmax = 1;
        plan->phase_shift = op == MBT_OP_ROWSUM ? flat_phase_shift(f, N, es, W) : 0;
        return MBT_OK;
    }
    if (op == MBT_OP_COPY) {
        plan->grid = static_cast<int32_t>(std::min<int64_t>(plan->num_tiles, cap));
        plan->kmax = 1;
        return MBT_OK;
    }
    // Reduction groups: row bands (tiles_n tiles of tile_m sums each) for row
    // sums, column strips (tiles_m tiles of tile_n sums each) for column sums.
    const bool cols = op == MBT_OP_COLSUM;
    const int64_t groups = cols ? plan->tiles_n : plan->tiles_m;
    const int64_t group_tiles = cols ? plan->tiles_m : plan->tiles_n;
    const int64_t sums_per_group = cols ? tile_n : tile_m;
    if (with_workspace) {
        const int64_t G = std::min<int64_t>(plan->num_tiles, cap);
        const int cg = cols ? colsum_group(W, tile_n, es, plan->boxes, one_per_sm) : 0;
        const int32_t kmax =
            cols ? colsum_contributors(plan->tiles_m, plan->tiles_n, cg, plan->num_tiles, G)
                 : most_contributors(group_tiles, plan->num_tiles, G);
        if (kmax > 1) {
            plan->grid = static_cast<int32_t>(G);
            plan->split = 1;
            plan->kmax = kmax;
            plan->workspace_bytes = static_cast<size_t>(round_up(groups * 4, 256) +
                                                        groups * kmax * sums_per_group * 4);
            plan->col_group = cg;
            return MBT_OK;
        }
    }
    plan->col_group = cols ? 1 : 0;   // whole strips, one CTA each
    plan->grid = static_cast<int32_t>(std::min<int64_t>(groups, cap));
    plan->split = 0;
    plan->kmax = 1;
    return MBT_OK;
}

int device_figures(DeviceFigures *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MBT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceFigures &d = g_devices[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return MBT_ERR_CUDA;
        int usable = 0;
        if (mbt::set_kernel_smem_limit(d.smem_optin, &usable) != cudaSuccess) return MBT_ERR_CUDA;
        d.smem_optin = usable;
        d.ready = true;
    }
    *out = d;
    return MBT_OK;
}

int encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
            return MBT_ERR_DRIVER;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    *fn = g_encode;
    return MBT_OK;
}

// 2-D tiled map over the logical M x N matrix: box = 128 bytes x tile_m rows,
// 128-byte swizzle, zero fill outside the matrix.
int encode_map(CUtensorMap *map, const void *src, int64_t M, int64_t N, int64_t ld, int dtype,
               int tile_m) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    int rc = encoder(&fn);
    if (rc != MBT_OK) return rc;
    const int es = esize_of(dtype);
    const CUtensorMapDataType type = dtype == MBT_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                     : dtype == MBT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(mbt::kBoxRowBytes / es),
                               static_cast<cuuint32_t>(tile_m)};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = fn(map, type, 2, const_cast<void *>(src), dims, strides, box, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MBT_OK : MBT_ERR_DRIVER;
}

// Map for bulk tensor stores: it ends at the last whole 16-byte chunk of a row
// (the copy engine clips stores only at 16-byte granularity; the partial chunk
// is stored by the kernel's lanes).  No map when a row has no whole chunk.
int encode_store_map(CUtensorMap *map, void *dst, int64_t M, int64_t N, int64_t ld, int dtype,
                     int tile_m) {
    const int64_t vec = 16 / esize_of(dtype);
    const int64_t n_whole = N - N % vec;
    if (n_whole == 0) return MBT_OK;   // every tile is stored by lanes
    return encode_map(map, dst, M, n_whole, ld, dtype, tile_m);
}

// Occupancy kernel id of a plan (see mbt::kernel_fit_per_sm).
int kernel_id_of(int op, const mbt_opts &o, const mbt_plan &plan, bool flat) {
    const bool wide = plan.consumer_warps > mbt::kMaxConsumerWarps;
    return flat                                          ? (op == MBT_OP_COPY ? 4 : 5)
           : op == MBT_OP_COLSUM                         ? (wide ? 10 : 6)
           : op == MBT_OP_COPY && o.pipeline == 1        ? 3
           : op == MBT_OP_COPY && plan.bulk_stores       ? 7
           : op == MBT_OP_ROWSUM && wide                 ? 9
           : op == MBT_OP_ROWSUM && plan.box_barriers    ? 8
                                                         : op;
}

// Plan for the current device (occupancy included): a first pass without the
// CTAs that fit an SM, the occupancy of its kernel, and the plan again with
// it; when that picks another kernel (the wide sums where only one CTA fits),
// its occupancy and a last pass.
int plan_on_device(int op, int64_t M, int64_t N, int tile_m, int tile_n, int stages, int dtype,
                   const mbt_opts &o, int with_workspace, mbt_plan *plan, bool flat = false) {
    DeviceFigures d;
    int rc = device_figures(&d);
    if (rc != MBT_OK) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MBT_ERR_CUDA;
    auto fit_of = [&](const mbt_plan &pl, int *fit) {
        const int kernel_id = kernel_id_of(op, o, pl, flat);
        const auto key = std::make_tuple(dev, kernel_id, op != MBT_OP_COPY ? dtype : 0,
                                         pl.threads, pl.smem_bytes);
        *fit = 0;
        {
            std::lock_guard<std::mutex> lock(g_mutex);
            auto it = g_fit_cache.find(key);
            if (it != g_fit_cache.end()) *fit = it->second;
        }
        if (*fit == 0) {
            if (mbt::kernel_fit_per_sm(kernel_id, dtype, pl.threads, pl.smem_bytes, fit) !=
                cudaSuccess)
                return MBT_ERR_CUDA;
            if (*fit < 1) return MBT_ERR_SMEM;
            std::lock_guard<std::mutex> lock(g_mutex);
            g_fit_cache[key] = *fit;
        }
        return MBT_OK;
    };
    rc = plan_impl(op, M, N, tile_m, tile_n, stages, dtype, o, d.num_sms, d.smem_optin, 0,
                   with_workspace, plan, flat);
    if (rc != MBT_OK) return rc;
    int fit = 0;
    rc = fit_of(*plan, &fit);
    if (rc != MBT_OK) return rc;
    const int threads = plan->threads, smem = plan->smem_bytes;
    rc = plan_impl(op, M, N, tile_m, tile_n, stages, dtype, o, d.num_sms, d.smem_optin, fit,
                   with_workspace, plan, flat);
    // (the second pass may change the warps, or the column sum's flush ring
    // with its strip group: then the occupancy is asked again)
    if (rc != MBT_OK || (plan->threads == threads && plan->smem_bytes == smem)) return rc;
    rc = fit_of(*plan, &fit);
    if (rc != MBT_OK) return rc;
    return plan_impl(op, M, N, tile_m, tile_n, stages, dtype, o, d.num_sms, d.smem_optin, fit,
                     with_workspace, plan, flat);
}

PipeArgs pipe_args(const mbt_plan &plan, int64_t M, int64_t N, int tile_m, int stages, int dtype,
                   const mbt_opts &o) {
    PipeArgs p{};
    p.M = M;
    p.N = N;
    p.tiles_n = plan.tiles_n;
    p.tiles_m = plan.tiles_m;
    p.num_tiles = plan.num_tiles;
    p.tile_m = tile_m;
    p.boxes = plan.boxes;
    p.box_inner = plan.box_inner;
    p.esize = esize_of(dtype);
    p.stages = stages;
    p.consumer_warps = plan.consumer_warps;
    p.box_stride = static_cast<uint32_t>(plan.stage_bytes / plan.boxes);
    p.stage_stride = static_cast<uint32_t>(plan.stage_bytes);
    p.tx_bytes = static_cast<uint32_t>(plan.tx_bytes);
    p.fault = o.fault;
    p.wait_budget_ns = o.wait_budget_ns ? o.wait_budget_ns : mbt::kDefaultWaitBudgetNs;
    p.log = o.log;
    p.log_cap = o.log_capacity;
    p.status = o.status;
    return p;
}

mbt_opts opts_or_default(const mbt_opts *opts) {
    mbt_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts) o = *opts;
    return o;
}

// Launch of the 1-D bulk-copy kernels (pitch not a multiple of 16 bytes).
int flat_launch(int op, const void *src, void *dst, float *out, int64_t M, int64_t N, int64_t ld,
                int tile_m, int tile_n, int stages, int dtype, void *stream, const mbt_opts &o) {
    mbt_plan plan;
    int rc = plan_on_device(op, M, N, tile_m, tile_n, stages, dtype, o, 0, &plan, true);
    if (rc != MBT_OK) return rc;
    mbt::FlatArgs f{};
    f.p = pipe_args(plan, M, N, tile_m, stages, dtype, o);
    f.src = static_cast<const char *>(src);
    f.dst = static_cast<char *>(dst);
    f.out = out;
    DeviceFigures d;
    rc = device_figures(&d);
    if (rc != MBT_OK) return rc;
    flat_setup(op, M, N, ld, esize_of(dtype), tile_m, tile_n, stages, d.smem_optin, &f);
    f.phase_shift = plan.phase_shift;
    const cudaError_t e =
        op == MBT_OP_COPY
            ? mbt::launch_copy_flat(f, plan.grid, plan.threads, plan.smem_bytes,
                                    static_cast<cudaStream_t>(stream))
            : mbt::launch_rowsum_flat(dtype, f, plan.grid, plan.threads, plan.smem_bytes,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

// The library's own sum workspace, for row and column sums called without one
// (and without no_split): one buffer per (device, stream), allocated in stream
// order on first use and grown when a plan needs more.  Layout: two ticket
// sets of ticket_cap words each, then the partial sums.  Successive calls
// alternate between the two sets; each call's kernel zeroes the set it does
// not use (clear_next_tickets), so the next call on the stream starts from
// zeroed tickets even if a call before it stopped on a timed-out wait.  The
// partial slots need no clearing: a band's last contributor reads only slots
// its co-contributors wrote in the same call.  The per-thread default stream
// is a different stream in every host thread, so its key includes the thread.
struct OwnedWorkspace {
    char *base = nullptr;
    int64_t ticket_cap = 0;     // words per ticket set (a multiple of 64)
    size_t partial_bytes = 0;
    uint64_t uses = 0;
};

std::mutex g_owned_mutex;
std::map<std::tuple<int, uintptr_t, size_t>, OwnedWorkspace> g_owned;

std::tuple<int, uintptr_t, size_t> owned_key(int dev, void *stream) {
    const size_t thread =
        stream == static_cast<void *>(cudaStreamPerThread)
            ? std::hash<std::thread::id>()(std::this_thread::get_id())
            : 0;
    return std::make_tuple(dev, reinterpret_cast<uintptr_t>(stream), thread);
}

// Tickets for `groups` reduction groups and `partial_bytes` of partial sums
// from the library's workspace for (current device, stream).
int owned_workspace(void *stream, int64_t groups, size_t partial_bytes, int32_t **ticket,
                    int32_t **clear, int64_t *clear_n, float **partial) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MBT_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_owned_mutex);
    OwnedWorkspace &w = g_owned[owned_key(dev, stream)];
    if (w.base == nullptr || w.ticket_cap < groups || w.partial_bytes < partial_bytes) {
        // Allocating inside a stream capture would end the capture with an error.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return MBT_ERR_CUDA;
        if (cap != cudaStreamCaptureStatusNone) return MBT_ERR_WORKSPACE;
        OwnedWorkspace nw;
        nw.ticket_cap = round_up(std::max<int64_t>({groups, w.ticket_cap, 64}), 64);
        nw.partial_bytes = static_cast<size_t>(round_up(
            static_cast<int64_t>(std::max({partial_bytes, w.partial_bytes,
                                           static_cast<size_t>(kOwnedMinPartialBytes)})),
            256));
        const size_t total = static_cast<size_t>(2 * nw.ticket_cap * 4) + nw.partial_bytes;
        void *p = nullptr;
        if (cudaMallocAsync(&p, total, s) != cudaSuccess) return MBT_ERR_CUDA;
        if (cudaMemsetAsync(p, 0, total, s) != cudaSuccess) {
            cudaFreeAsync(p, s);
            return MBT_ERR_CUDA;
        }
        // The old buffer served this stream only: freed after its last use.
        if (w.base != nullptr && cudaFreeAsync(w.base, s) != cudaSuccess) {
            cudaFreeAsync(p, s);
            return MBT_ERR_CUDA;
        }
        nw.base = static_cast<char *>(p);
        w = nw;
    }
    const int64_t parity = static_cast<int64_t>(w.uses++ & 1u);
    int32_t *sets = reinterpret_cast<int32_t *>(w.base);
    *ticket = sets + parity * w.ticket_cap;
    *clear = sets + (1 - parity) * w.ticket_cap;
    *clear_n = w.ticket_cap;
    *partial = reinterpret_cast<float *>(w.base + 2 * w.ticket_cap * 4);
    return MBT_OK;
}

// Row sums (and, with dst != nullptr, the fused copy) after argument checks.
int rowsum_launch(const void *src, void *dst, float *out, int64_t M, int64_t N, int64_t ld_src,
                  int64_t ld_dst, int tile_m, int tile_n, int stages, int dtype, void *stream,
                  const mbt_opts &o) {
    const int op = dst != nullptr ? MBT_OP_COPY_ROWSUM : MBT_OP_ROWSUM;
    if (M == 0) return MBT_OK;
    if (N == 0) {
        return mbt::launch_fill_zero(out, M, static_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? MBT_OK
                   : MBT_ERR_CUDA;
    }
    mbt_plan plan;
    int rc = plan_on_device(op, M, N, tile_m, tile_n, stages, dtype, o, !o.no_split, &plan);
    if (rc != MBT_OK) return rc;
    const bool own = plan.split && o.workspace == nullptr;
    if (plan.split && !own) {
        if (o.workspace_bytes < plan.workspace_bytes) return MBT_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(o.workspace) & 255u) != 0) return MBT_ERR_ALIGN;
    }
    alignas(64) CUtensorMap map;
    rc = encode_map(&map, src, M, N, ld_src, dtype, tile_m);
    if (rc != MBT_OK) return rc;
    alignas(64) CUtensorMap dst_map;
    std::memset(&dst_map, 0, sizeof dst_map);
    if (dst != nullptr) {
        rc = encode_store_map(&dst_map, dst, M, N, ld_dst, dtype, tile_m);
        if (rc != MBT_OK) return rc;
    }
    RowsumArgs a{};
    a.p = pipe_args(plan, M, N, tile_m, stages, dtype, o);
    a.out = out;
    if (own) {
        rc = owned_workspace(stream, plan.tiles_m,
                             plan.workspace_bytes - round_up(plan.tiles_m * 4, 256), &a.ticket,
                             &a.clear_ticket, &a.clear_n, &a.partial);
        if (rc != MBT_OK) return rc;
    } else if (plan.split) {
        char *ws = static_cast<char *>(o.workspace);
        a.ticket = reinterpret_cast<int32_t *>(ws);
        a.partial = reinterpret_cast<float *>(ws + round_up(plan.tiles_m * 4, 256));
    }
    if (plan.split) {
        a.gran = 1;
        a.units = plan.num_tiles;
    } else {
        a.gran = plan.tiles_n;
        a.units = plan.tiles_m;
    }
    a.kmax = plan.kmax;
    a.boxed = plan.box_barriers;
    if (dst != nullptr) {
        a.fused = 1;
        a.dst = static_cast<char *>(dst);
        a.ld_dst_bytes = ld_dst * esize_of(dtype);
        a.p.empty_extra = 1;   // the bulk store's reads of each stage
    }
    const cudaError_t e = mbt::launch_rowsum(dtype, map, dst_map, a, plan.grid, plan.threads,
                                             plan.smem_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

// Column sums after argument checks.
int colsum_launch(const void *src, float *out, int64_t M, int64_t N, int64_t ld_src, int tile_m,
                  int tile_n, int stages, int dtype, void *stream, const mbt_opts &o) {
    if (N == 0) return MBT_OK;
    if (M == 0) {
        return mbt::launch_fill_zero(out, N, static_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? MBT_OK
                   : MBT_ERR_CUDA;
    }
    mbt_plan plan;
    int rc = plan_on_device(MBT_OP_COLSUM, M, N, tile_m, tile_n, stages, dtype, o, !o.no_split,
                            &plan);
    if (rc != MBT_OK) return rc;
    const bool own = plan.split && o.workspace == nullptr;
    if (plan.split && !own) {
        if (o.workspace_bytes < plan.workspace_bytes) return MBT_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(o.workspace) & 255u) != 0) return MBT_ERR_ALIGN;
    }
    alignas(64) CUtensorMap map;
    rc = encode_map(&map, src, M, N, ld_src, dtype, tile_m);
    if (rc != MBT_OK) return rc;
    mbt::ColsumArgs a{};
    a.p = pipe_args(plan, M, N, tile_m, stages, dtype, o);
    a.p.col_group = plan.col_group;
    a.out = out;
    if (own) {
        rc = owned_workspace(stream, plan.tiles_n,
                             plan.workspace_bytes - round_up(plan.tiles_n * 4, 256), &a.ticket,
                             &a.clear_ticket, &a.clear_n, &a.partial);
        if (rc != MBT_OK) return rc;
    } else if (plan.split) {
        char *ws = static_cast<char *>(o.workspace);
        a.ticket = reinterpret_cast<int32_t *>(ws);
        a.partial = reinterpret_cast<float *>(ws + round_up(plan.tiles_n * 4, 256));
    }
    if (plan.split) {
        a.gran = 1;
        a.units = plan.num_tiles;
    } else {
        a.gran = plan.tiles_m;
        a.units = plan.tiles_n;
    }
    a.kmax = plan.kmax;
    a.tile_n = tile_n;
    // strip pairs: the consumers' row stride must keep the swizzle term
    if (plan.col_group == 2 && (plan.consumer_warps * 32 / (plan.boxes * 8)) % 8 != 0)
        return MBT_ERR_UNSUPPORTED;
    const cudaError_t e = mbt::launch_colsum(dtype, map, a, plan.grid, plan.threads,
                                             plan.smem_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

int workspace_bytes(int op, int64_t M, int64_t N, int tile_m, int tile_n, int stages, int dtype,
                    const mbt_opts *opts, size_t *bytes) {
    if (bytes == nullptr) return MBT_ERR_ARG;
    mbt_opts o = opts_or_default(opts);
    o.workspace = nullptr;
    o.workspace_bytes = 0;
    int64_t ld_src = 0, ld_dst = 0;
    static const char dummy[16] __attribute__((aligned(16))) = {0};
    bool flat = false;
    int rc = check_args(op, dummy, dummy, M, N, tile_m, tile_n, stages, dtype, o, &ld_src,
                        &ld_dst, &flat);
    if (rc != MBT_OK) return rc;
    *bytes = 0;
    // flat row sums need no workspace, nor sums that are never split
    if (M == 0 || N == 0 || flat || o.no_split) return MBT_OK;
    mbt_plan plan;
    rc = plan_on_device(op, M, N, tile_m, tile_n, stages, dtype, o, 1, &plan);
    if (rc != MBT_OK) return rc;
    *bytes = plan.workspace_bytes;
    return MBT_OK;
}

}  // namespace

extern "C" {

int tile_plan(int op, int64_t M, int64_t N, int tile_m, int tile_n, int stages, int dtype,
              const mbt_opts *opts, int num_sms, int smem_optin, int fit_per_sm,
              int with_workspace, mbt_plan *plan) {
    const mbt_opts o = opts_or_default(opts);
    int64_t ld_src = 0, ld_dst = 0;
    // Shape checks only: pointers are not part of a plan.
    static const char dummy[16] __attribute__((aligned(16))) = {0};
    bool flat = false;
    int rc = check_args(op, dummy, dummy, M, N, tile_m, tile_n, stages, dtype, o, &ld_src, &ld_dst,
                        &flat);
    if (rc != MBT_OK) return rc;
    return plan_impl(op, M, N, tile_m, tile_n, stages, dtype, o, num_sms, smem_optin, fit_per_sm,
                     with_workspace, plan, flat);
}

int tile_plan_device(int op, int64_t M, int64_t N, int tile_m, int tile_n, int stages,
                     int dtype, const mbt_opts *opts, mbt_plan *plan) {
    if (plan == nullptr) return MBT_ERR_ARG;
    const mbt_opts o = opts_or_default(opts);
    int64_t ld_src = 0, ld_dst = 0;
    static const char dummy[16] __attribute__((aligned(16))) = {0};
    bool flat = false;
    int rc = check_args(op, dummy, dummy, M, N, tile_m, tile_n, stages, dtype, o, &ld_src,
                        &ld_dst, &flat);
    if (rc != MBT_OK) return rc;
    const bool sums = op != MBT_OP_COPY;
    return plan_on_device(op, M, N, tile_m, tile_n, stages, dtype, o,
                          sums && !o.no_split ? 1 : 0, plan, flat);
}

int tile_copy_ex(const void *src, void *dst, int64_t M, int64_t N, int tile_m, int tile_n,
                 int stages, int dtype, void *stream, const mbt_opts *opts) {
    const mbt_opts o = opts_or_default(opts);
    int64_t ld_src = 0, ld_dst = 0;
    bool flat = false;
    int rc = check_args(MBT_OP_COPY, src, dst, M, N, tile_m, tile_n, stages, dtype, o, &ld_src,
                        &ld_dst, &flat);
    if (rc != MBT_OK) return rc;
    if (M == 0 || N == 0) return MBT_OK;
    if (flat)
        return flat_launch(MBT_OP_COPY, src, dst, nullptr, M, N, ld_src, tile_m, tile_n, stages,
                           dtype, stream, o);
    mbt_plan plan;
    rc = plan_on_device(MBT_OP_COPY, M, N, tile_m, tile_n, stages, dtype, o, 0, &plan);
    if (rc != MBT_OK) return rc;
    alignas(64) CUtensorMap map;
    rc = encode_map(&map, src, M, N, ld_src, dtype, tile_m);
    if (rc != MBT_OK) return rc;
    alignas(64) CUtensorMap dst_map;
    std::memset(&dst_map, 0, sizeof dst_map);
    if (plan.bulk_stores) {
        rc = encode_store_map(&dst_map, dst, M, N, ld_dst, dtype, tile_m);
        if (rc != MBT_OK) return rc;
    }
    CopyArgs a{};
    a.p = pipe_args(plan, M, N, tile_m, stages, dtype, o);
    a.dst = static_cast<char *>(dst);
    a.ld_dst_bytes = ld_dst * esize_of(dtype);
    a.store_mode = plan.bulk_stores;
    const cudaError_t e =
        o.pipeline == 1
            ? mbt::launch_copy_unified(map, a, plan.grid, plan.threads, plan.smem_bytes,
                                       static_cast<cudaStream_t>(stream))
            : mbt::launch_copy(map, dst_map, a, plan.grid, plan.threads, plan.smem_bytes,
                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

int tile_copy(const void *src, void *dst, int64_t M, int64_t N, int tile_m, int tile_n,
              int stages, int dtype, void *stream) {
    return tile_copy_ex(src, dst, M, N, tile_m, tile_n, stages, dtype, stream, nullptr);
}

int tile_rowsum_ex(const void *src, float *out, int64_t M, int64_t N, int tile_m, int tile_n,
                   int stages, int dtype, void *stream, const mbt_opts *opts) {
    const mbt_opts o = opts_or_default(opts);
    int64_t ld_src = 0, ld_dst = 0;
    bool flat = false;
    int rc = check_args(MBT_OP_ROWSUM, src, out, M, N, tile_m, tile_n, stages, dtype, o, &ld_src,
                        &ld_dst, &flat);
    if (rc != MBT_OK) return rc;
    if (flat && M > 0 && N > 0)
        return flat_launch(MBT_OP_ROWSUM, src, nullptr, out, M, N, ld_src, tile_m, tile_n, stages,
                           dtype, stream, o);
    return rowsum_launch(src, nullptr, out, M, N, ld_src, 0, tile_m, tile_n, stages, dtype,
                         stream, o);
}

int tile_copy_rowsum_ex(const void *src, void *dst, float *out, int64_t M, int64_t N, int tile_m,
                        int tile_n, int stages, int dtype, void *stream, const mbt_opts *opts) {
    const mbt_opts o = opts_or_default(opts);
    if (o.store_mode != 0) return MBT_ERR_ARG;
    int64_t ld_src = 0, ld_dst = 0;
    int rc = check_args(MBT_OP_COPY_ROWSUM, src, dst, M, N, tile_m, tile_n, stages, dtype, o,
                        &ld_src, &ld_dst);
    if (rc != MBT_OK) return rc;
    if (M > 0 && out == nullptr) return MBT_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0) return MBT_ERR_ALIGN;
    return rowsum_launch(src, dst, out, M, N, ld_src, ld_dst, tile_m, tile_n, stages, dtype,
                         stream, o);
}

int tile_copy_rowsum(const void *src, void *dst, float *out, int64_t M, int64_t N, int tile_m,
                     int tile_n, int stages, int dtype, void *stream) {
    return tile_copy_rowsum_ex(src, dst, out, M, N, tile_m, tile_n, stages, dtype, stream,
                               nullptr);
}

int tile_rowsum(const void *src, float *out, int64_t M, int64_t N, int tile_m, int tile_n,
                int stages, int dtype, void *stream) {
    return tile_rowsum_ex(src, out, M, N, tile_m, tile_n, stages, dtype, stream, nullptr);
}

int tile_colsum_ex(const void *src, float *out, int64_t M, int64_t N, int tile_m, int tile_n,
                   int stages, int dtype, void *stream, const mbt_opts *opts) {
    const mbt_opts o = opts_or_default(opts);
    int64_t ld_src = 0, ld_dst = 0;
    bool flat = false;
    int rc = check_args(MBT_OP_COLSUM, src, out, M, N, tile_m, tile_n, stages, dtype, o, &ld_src,
                        &ld_dst, &flat);
    if (rc != MBT_OK) return rc;
    if (flat) return MBT_ERR_ALIGN;   // column sums need a 16-byte row pitch
    return colsum_launch(src, out, M, N, ld_src, tile_m, tile_n, stages, dtype, stream, o);
}

int tile_colsum(const void *src, float *out, int64_t M, int64_t N, int tile_m, int tile_n,
                int stages, int dtype, void *stream) {
    return tile_colsum_ex(src, out, M, N, tile_m, tile_n, stages, dtype, stream, nullptr);
}

int tile_colsum_workspace_bytes(int64_t M, int64_t N, int tile_m, int tile_n, int stages,
                                int dtype, const mbt_opts *opts, size_t *bytes) {
    return workspace_bytes(MBT_OP_COLSUM, M, N, tile_m, tile_n, stages, dtype, opts, bytes);
}

int tile_rowsum_workspace_bytes(int64_t M, int64_t N, int tile_m, int tile_n, int stages,
                                int dtype, const mbt_opts *opts, size_t *bytes) {
    return workspace_bytes(MBT_OP_ROWSUM, M, N, tile_m, tile_n, stages, dtype, opts, bytes);
}

int tile_copy_rowsum_workspace_bytes(int64_t M, int64_t N, int tile_m, int tile_n, int stages,
                                     int dtype, const mbt_opts *opts, size_t *bytes) {
    return workspace_bytes(MBT_OP_COPY_ROWSUM, M, N, tile_m, tile_n, stages, dtype, opts, bytes);
}

int tile_stage_image(const void *src, int64_t M, int64_t N, int64_t ld, int tile_m, int tile_n,
                     int dtype, int64_t tile_row, int64_t tile_col, void *image, void *stream) {
    mbt_opts o;
    std::memset(&o, 0, sizeof o);
    o.ld_src = ld;
    int64_t ld_src = 0, ld_dst = 0;
    bool flat = false;
    int rc = check_args(MBT_OP_ROWSUM, src, image, M, N, tile_m, tile_n, 1, dtype, o, &ld_src,
                        &ld_dst, &flat, false);
    if (rc != MBT_OK) return rc;
    if (flat || M == 0 || N == 0 || image == nullptr) return MBT_ERR_ARG;
    if (tile_row < 0 || tile_col < 0 || tile_row * tile_m >= M || tile_col * tile_n >= N)
        return MBT_ERR_ARG;
    const int es = esize_of(dtype);
    const int boxes = tile_n * es / mbt::kBoxRowBytes;
    const uint32_t box_bytes = static_cast<uint32_t>(tile_m) * mbt::kBoxRowBytes;
    const uint32_t box_stride = static_cast<uint32_t>(round_up(box_bytes, mbt::kSwizzleAtomBytes));
    DeviceFigures d;
    rc = device_figures(&d);
    if (rc != MBT_OK) return rc;
    if (static_cast<int64_t>(boxes) * box_stride + 1024 > d.smem_optin) return MBT_ERR_SMEM;
    alignas(64) CUtensorMap map;
    rc = encode_map(&map, src, M, N, ld_src, dtype, tile_m);
    if (rc != MBT_OK) return rc;
    const cudaError_t e = mbt::launch_stage_image(
        map, static_cast<int32_t>(tile_row * tile_m), static_cast<int32_t>(tile_col * tile_n),
        boxes, mbt::kBoxRowBytes / es, box_bytes, box_stride, static_cast<unsigned char *>(image),
        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

int tile_workspace_release(void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MBT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_owned_mutex);
    auto it = g_owned.find(owned_key(dev, stream));
    if (it == g_owned.end()) return MBT_OK;
    const cudaError_t e =
        it->second.base ? cudaFreeAsync(it->second.base, static_cast<cudaStream_t>(stream))
                        : cudaSuccess;
    g_owned.erase(it);
    return e == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}

int tile_status(void *stream, int32_t info[4]) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MBT_ERR_CUDA;
    int32_t local[4];
    if (mbt::read_and_clear_status(local) != cudaSuccess) return MBT_ERR_CUDA;
    if (info)
        for (int i = 0; i < 4; ++i) info[i] = local[i];
    return local[0] == 0 ? MBT_OK : local[0];
}

const char *tile_strerror(int code) {
    switch (code) {
        case MBT_OK: return "success";
        case MBT_ERR_ARG: return "invalid argument (pointer, size, shape, enum or option)";
        case MBT_ERR_ALIGN: return "base pointer or row pitch not 16-byte aligned";
        case MBT_ERR_UNSUPPORTED: return "tile shape, size or warp count not supported";
        case MBT_ERR_SMEM: return "stages x tile exceed the shared memory of one CTA";
        case MBT_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
        case MBT_ERR_TIMEOUT: return "an mbarrier wait exceeded its time budget";
        case MBT_ERR_DRIVER: return "tensor-map encoder unavailable or rejected the map";
        case MBT_ERR_WORKSPACE: return "workspace smaller than required";
        default: return "unknown status code";
    }
}

int tile_device_info(int device, int *num_sms, int *smem_optin, double *hbm_gbs_theoretical) {
    int sms = 0, optin = 0, mem_khz = 0, bus_bits = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess)
        return MBT_ERR_CUDA;
    // Memory clock and bus width may be unreported; then the figure is 0.
    if (cudaDeviceGetAttribute(&mem_khz, cudaDevAttrMemoryClockRate, device) != cudaSuccess)
        mem_khz = 0;
    if (cudaDeviceGetAttribute(&bus_bits, cudaDevAttrGlobalMemoryBusWidth, device) != cudaSuccess)
        bus_bits = 0;
    cudaGetLastError();
    if (num_sms) *num_sms = sms;
    if (smem_optin) *smem_optin = optin;
    if (hbm_gbs_theoretical)
        *hbm_gbs_theoretical = 2.0 * mem_khz * 1e3 * (bus_bits / 8.0) / 1e9;
    return MBT_OK;
}

}  // extern "C"
