// Kernels of libmbtile: a warp-specialised, mbarrier-synchronised bulk-tensor
// tile pipeline for sm_103a, with a copy consumer and a row-sum consumer.
//
// CTA layout: warp 0 is the producer (one elected lane issues every bulk
// tensor copy); warps 1..W are consumers.  Shared memory holds S stages; a
// stage is `boxes` box buffers of tile_m rows x 128 bytes, each aligned to
// 1024 bytes so that the hardware's 128-byte swizzle (16-byte chunk c of row r
// stored at chunk c ^ (r mod 8)) is relative to the buffer start.
//
// Per stage s there is a full barrier (expects 1 arrival + the tile's bytes)
// and an empty barrier (expects one arrival per consumer warp).  The producer
// waits on empty[s] with its cursor parity (starting at 1, because every
// buffer is free at the start), registers the bytes with arrive.expect_tx and
// issues the copies; consumers wait on full[s] with their parity (starting at
// 0), read the stage, and one lane per warp arrives on empty[s] once the whole
// warp has finished its shared-memory reads.  Sources: "cute(12)
// async_pipeline" §1-§3, §6 and §7; "cute(11) Hopper TMA copy" §3 and §6;
// "异步协作：mbarrier"; "CUDA features 10: Pipelines" §4.10.4-4.10.5.
//
// Every wait is bounded (time budget from the host).  A wait that runs out
// records MBT_ERR_TIMEOUT in the call's status buffer (or, without one, in
// g_status), raises a CTA-local abort flag that makes the CTA's other waits
// give up early, and the producer then waits (again
// bounded) for the bulk copies it still has in flight before the CTA exits.
//
// Kernels: mbt_copy_kernel<bulk> (LSU stores, or bulk tensor stores from one
// consumer warp), mbt_copy_unified_kernel (no warp specialisation; a CTA
// barrier releases each stage), mbt_rowsum_kernel<dtype, fused, boxed> (row sums;
// fused adds a store warp that also writes the tile out; without it, where
// each consumer warp reads one 128-byte box, every box of a stage may have
// its own full/empty pair); in mbtile_flat.cuh, the 1-D bulk-copy kernels for
// row pitches that are not a multiple of 16 bytes; in mbtile_colsum.cuh,
// mbt_colsum_kernel (column sums, tiles taken down the column strips).
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"

namespace mbt {

__device__ int32_t g_status[4];

namespace {

constexpr int kVec = 8;  // 16-byte chunks a consumer thread holds per round
static_assert(kVec == 8, "the row-sum consumer's box-aligned addressing assumes 8 chunks a round");

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the copy engine before first use.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One probe of the barrier: true once the phase with parity `parity` is over.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 1-D bulk copy of `bytes` bytes (16-byte aligned address and size) from
// global memory into shared memory; completion is counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void *src, uint32_t bytes,
                                             uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Bulk tensor copy of one 2-D box at element coordinates (x = column, y = row)
// into shared memory; completion is counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map,
                                            int32_t x, int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Bulk tensor copy of one 2-D box from shared memory to global memory at
// element coordinates (x, y); elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most one committed bulk store group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_allow1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void stg128(void *ptr, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Byte offset of 16-byte chunk q (counted across all boxes of a tile row) of
// tile row `row`, relative to the stage base.
__device__ __forceinline__ uint32_t chunk_offset(int row, int q, uint32_t box_stride) {
    return static_cast<uint32_t>(q >> 3) * box_stride +
           static_cast<uint32_t>(row) * kBoxRowBytes +
           (static_cast<uint32_t>((q & 7) ^ (row & 7)) << 4);
}

// ---------------------------------------------------------------------------
// Bounded waits and the failure record
// ---------------------------------------------------------------------------
struct WaitCtl {
    uint64_t budget_ns;
    volatile int *abort;
    int32_t *status;    // where a timed-out wait is recorded: the call's own
                        // status buffer (mbt_opts.status) or g_status
};

__device__ __forceinline__ int32_t *status_of(const PipeArgs &p) {
    return p.status != nullptr ? p.status : g_status;
}

__device__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl &w,
                             bool heed_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    // Each probe costs well over 8 ns, so this iteration cap is reached only
    // if the timer itself stalls; it keeps the loop finite regardless.
    const uint64_t max_iter = w.budget_ns / 8 + 4096;
    for (uint64_t it = 0; it < max_iter; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7) == 7) {
            if (heed_abort && *w.abort) return false;
            if (global_ns() - t0 > w.budget_ns) return false;
        }
    }
    return false;
}

__device__ void report_timeout(const WaitCtl &w, int role, uint32_t stage, uint32_t parity) {
    int32_t *st = w.status;
    if (atomicCAS(&st[0], 0, static_cast<int32_t>(MBT_ERR_TIMEOUT)) == 0) {
        st[1] = static_cast<int32_t>(blockIdx.x);
        st[2] = static_cast<int32_t>(stage);
        st[3] = role * 2 + static_cast<int32_t>(parity);
    }
}

__device__ __forceinline__ void log_record(const PipeArgs &p, int role, int64_t k,
                                           uint32_t stage, uint32_t parity,
                                           int64_t tile) {
    if (p.log != nullptr && blockIdx.x == 0 && k < p.log_cap) {
        int32_t *r = p.log + 4 * (role * p.log_cap + k);
        r[0] = static_cast<int32_t>(k);
        r[1] = static_cast<int32_t>(stage);
        r[2] = static_cast<int32_t>(parity);
        r[3] = static_cast<int32_t>(tile);
    }
}

// ---------------------------------------------------------------------------
// Shared pipeline skeleton
// ---------------------------------------------------------------------------
struct Smem {
    uint32_t base;    // 1024-aligned start of stage 0
    uint32_t full0;   // full barrier of stage 0 (stage s at + 8 s)
    uint32_t empty0;  // empty barrier of stage 0
    // Per-box barriers (row sum, boxed mode): box b of stage s at + 8 (8 s + b).
    uint32_t fullb0 = 0;
    uint32_t emptyb0 = 0;
};

__device__ __forceinline__ uint32_t box_bar(uint32_t base, uint32_t stage, int box) {
    return base + 8u * (stage * 8u + static_cast<uint32_t>(box));
}

// Producer of the copy and column-sum kernels: one elected lane.  Loads
// `count` tiles, tile j being first + j * step in row-major tile order (or,
// with p.col_group, in strip-group order), then drains (producer tail).
__device__ void produce(const CUtensorMap *map, const PipeArgs &p, const Smem &sm,
                        const WaitCtl &w, int64_t first, int64_t step, int64_t count) {
    uint32_t stage = 0;
    uint32_t phase = (p.fault == 1) ? 0u : 1u;  // free buffers: start at phase 1
    int64_t issued = 0;
    bool ok = true;
    for (int64_t j = 0; j < count; ++j) {
        // Wait for the stage first, then work out the tile (measured: this
        // order kept the 3-stage row sum 1.3% faster than computing the
        // coordinates ahead of the wait, and the 3-stage column sum 3% faster
        // than stepping its strip-group position incrementally after the wait
        // -- a short gap between a stage's release and its next copy helps,
        // though the incremental step does less work).
        if (!wait_bounded(sm.empty0 + 8u * stage, phase, w, true)) {
            report_timeout(w, 0, stage, phase);
            *w.abort = 1;
            ok = false;
            break;
        }
        const int64_t tile = first + j * step;
        int64_t tm, tn;
        if (p.col_group) {
            const ColPos c = col_pos(tile, p.tiles_m, p.tiles_n, p.col_group);
            tm = c.band;
            tn = col_strip(c, p.col_group);
        } else {
            tm = tile / p.tiles_n;
            tn = tile - tm * p.tiles_n;
        }
        const int32_t y = static_cast<int32_t>(tm * p.tile_m);
        const int32_t x0 = static_cast<int32_t>(tn * p.boxes * p.box_inner);
        const uint32_t dst = sm.base + stage * p.stage_stride;
        const uint32_t full_bar = sm.full0 + 8u * stage;
        mbar_arrive_expect_tx(full_bar, p.tx_bytes);
        for (int b = 0; b < p.boxes; ++b)
            tma_load_2d(dst + b * p.box_stride, map, x0 + b * p.box_inner, y, full_bar);
        log_record(p, 0, j, stage, phase, tile);
        ++issued;
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (ok) {
        // Tail: wait until the consumers have released every stage once more,
        // so the CTA never exits with a stage still being read or filled.
        for (int s = 0; s < p.stages; ++s) {
            if (!wait_bounded(sm.empty0 + 8u * stage, phase, w, true)) {
                report_timeout(w, 0, stage, phase);
                *w.abort = 1;
                ok = false;
                break;
            }
            if (++stage == static_cast<uint32_t>(p.stages)) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        // Abort: wait (bounded) for the copies this CTA may still have in
        // flight -- the last min(issued, S) tiles -- before leaving.
        const int64_t from = issued > p.stages ? issued - p.stages : 0;
        for (int64_t t = from; t < issued; ++t) {
            const uint32_t s = static_cast<uint32_t>(t % p.stages);
            const uint32_t par = static_cast<uint32_t>((t / p.stages) & 1);
            wait_bounded(sm.full0 + 8u * s, par, w, false);
        }
    }
}

// What the row-sum producer publishes for each stage (each box with per-box
// barriers): the band the tile belongs to (-1 marks the end) and the tile's
// coordinates, so that the consumers do no division between a full barrier
// and their first read.
struct StageInfo {
    int64_t key;
    int32_t tm, tn;
};

// Producer of the row-sum kernels: loads the tiles [first, last) in order.
// Besides loading, it publishes each stage's band and tile coordinates (each
// box's, with `boxed`) in `info` before the stage's full barrier is armed --
// the arrive releases them to the consumers, which then need no division of
// their own between the barrier and their first read (measured without a
// workspace: +5.6 % on the bf16 8192 x 65536 row sum, +21.6 / +16.9 % on the
// fp32 12289 x 8191 / fp16 24577 x 16383 ones) -- and closes the ring with an
// end mark (key -1) on a stage whose full barrier completes by a plain arrive.
template <bool boxed>
__device__ void produce_rows(const CUtensorMap *map, const RowsumArgs &a, const Smem &sm,
                             const WaitCtl &w, int64_t first, int64_t last,
                             volatile StageInfo *info) {
    const PipeArgs &p = a.p;
    uint32_t stage = 0;
    uint32_t phase = (p.fault == 1) ? 0u : 1u;  // free buffers: start at phase 1
    int64_t issued = 0;
    int last_boxes = p.boxes;   // boxes issued of tile issued - 1
    bool ok = true;
    const uint32_t box_tx = p.tx_bytes / static_cast<uint32_t>(p.boxes);
    // The run of tiles being issued: columns [tn, tn_end) of band tm (the
    // band is the consumers' segment key), one run per band.
    int64_t tm = 0, tn = 0, tn_end = 0, t_next = first;
    auto open_run = [&]() {
        if (t_next >= last) return false;
        tm = t_next / p.tiles_n;
        tn = t_next - tm * p.tiles_n;
        tn_end = last - tm * p.tiles_n < p.tiles_n ? last - tm * p.tiles_n : p.tiles_n;
        t_next = tm * p.tiles_n + tn_end;
        return true;
    };
    bool more = open_run();
    for (int64_t j = 0;; ++j) {
        // Work out the next tile (or the end mark) before waiting for a stage.
        const bool end = !more;
        const int64_t ctm = tm, ctn = tn, ckey = end ? -1 : tm;
        if (!end && ++tn == tn_end) more = open_run();
        if (!boxed && !wait_bounded(sm.empty0 + 8u * stage, phase, w, true)) {
            report_timeout(w, 0, stage, phase);
            *w.abort = 1;
            ok = false;
            break;
        }
        const int64_t tile = end ? -1 : ctm * p.tiles_n + ctn;
        const int32_t y = static_cast<int32_t>(ctm * p.tile_m);
        const int32_t x0 = static_cast<int32_t>(ctn * p.boxes * p.box_inner);
        const uint32_t dst = sm.base + stage * p.stage_stride;
        if (boxed) {
            for (int b = 0; b < p.boxes; ++b) {
                if (!wait_bounded(box_bar(sm.emptyb0, stage, b), phase, w, true)) {
                    report_timeout(w, 0, stage, phase);
                    *w.abort = 1;
                    ok = false;
                    if (b > 0 && tile >= 0) {   // boxes 0 .. b-1 of this tile are in flight
                        ++issued;
                        last_boxes = b;
                    }
                    break;
                }
                info[stage * 8 + b].key = ckey;
                info[stage * 8 + b].tm = static_cast<int32_t>(ctm);
                info[stage * 8 + b].tn = static_cast<int32_t>(ctn);
                const uint32_t full_bar = box_bar(sm.fullb0, stage, b);
                if (tile < 0) {
                    mbar_arrive(full_bar);
                } else {
                    mbar_arrive_expect_tx(full_bar, box_tx);
                    tma_load_2d(dst + b * p.box_stride, map, x0 + b * p.box_inner, y, full_bar);
                }
            }
            if (!ok) break;
        } else {
            info[stage * 8].key = ckey;
            info[stage * 8].tm = static_cast<int32_t>(ctm);
            info[stage * 8].tn = static_cast<int32_t>(ctn);
            const uint32_t full_bar = sm.full0 + 8u * stage;
            if (tile < 0) {
                mbar_arrive(full_bar);
            } else {
                mbar_arrive_expect_tx(full_bar, p.tx_bytes);
                for (int b = 0; b < p.boxes; ++b)
                    tma_load_2d(dst + b * p.box_stride, map, x0 + b * p.box_inner, y, full_bar);
            }
        }
        if (tile >= 0) {
            log_record(p, 0, j, stage, phase, tile);
            ++issued;
        }
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
        if (tile < 0) break;
    }
    if (ok) {
        // Tail: wait until the consumers have released every stage once more,
        // so the CTA never exits with a stage still being read or filled.
        for (int s = 0; s < p.stages && ok; ++s) {
            const int nb = boxed ? p.boxes : 1;
            for (int b = 0; b < nb; ++b) {
                const uint32_t bar = boxed ? box_bar(sm.emptyb0, stage, b) : sm.empty0 + 8u * stage;
                if (!wait_bounded(bar, phase, w, true)) {
                    report_timeout(w, 0, stage, phase);
                    *w.abort = 1;
                    ok = false;
                    break;
                }
            }
            if (++stage == static_cast<uint32_t>(p.stages)) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        // Abort: wait (bounded) for the copies this CTA may still have in
        // flight -- the last min(issued, S) tiles -- before leaving.  (Stages
        // are used in order, the end mark after the last tile, so tile k went
        // to stage k mod S.)
        const int64_t from = issued > p.stages ? issued - p.stages : 0;
        for (int64_t k = from; k < issued; ++k) {
            const uint32_t s = static_cast<uint32_t>(k % p.stages);
            const uint32_t par = static_cast<uint32_t>((k / p.stages) & 1);
            if (boxed) {
                const int nb = k == issued - 1 ? last_boxes : p.boxes;
                for (int b = 0; b < nb; ++b) wait_bounded(box_bar(sm.fullb0, s, b), par, w, false);
            } else {
                wait_bounded(sm.full0 + 8u * s, par, w, false);
            }
        }
    }
}

// `bars` holds 2 kMaxStages barriers, or 16 kMaxStages when `boxed`: then
// each (stage, box) gets a full barrier (one arrival + the box's bytes) and an
// empty barrier that the box's consumer warps -- consumer_warps / boxes of
// them -- release.
__device__ __forceinline__ void init_pipeline(const PipeArgs &p, Smem &sm,
                                              uint64_t *bars, volatile int *abort_flag,
                                              unsigned char *dyn, bool boxed = false) {
    sm.base = (smem_u32(dyn) + (kSwizzleAtomBytes - 1)) & ~uint32_t(kSwizzleAtomBytes - 1);
    sm.full0 = smem_u32(&bars[0]);
    sm.empty0 = smem_u32(&bars[kMaxStages]);
    if (boxed) {
        sm.fullb0 = smem_u32(&bars[0]);
        sm.emptyb0 = smem_u32(&bars[8 * kMaxStages]);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            if (boxed) {
                for (int b = 0; b < p.boxes; ++b) {
                    mbar_init(box_bar(sm.fullb0, s, b), 1);
                    mbar_init(box_bar(sm.emptyb0, s, b),
                              static_cast<uint32_t>(p.consumer_warps / p.boxes + p.empty_extra));
                }
                continue;
            }
            mbar_init(sm.full0 + 8u * s, 1);
            mbar_init(sm.empty0 + 8u * s,
                      static_cast<uint32_t>(p.consumer_warps + p.empty_extra));
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Programmatic dependent launch (the launchers allow it): this CTA may have
    // been launched while the previous kernel of the stream was completing.
    // Nothing above touches global memory; every global access below comes
    // after that kernel has completed and its writes are visible.  A no-op for
    // a launch without the attribute.  The kernel does not signal its own
    // dependents early (they start as its CTAs exit): with an early signal the
    // next kernel's CTAs were placed beside this one's on whichever SMs had
    // room, which unbalanced a following kernel of another kind (copy and row
    // sum alternating on one stream: 0.337 -> 0.377 ms per pair).
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The library's own sum workspace holds two ticket sets and successive calls
// alternate between them: each call zeroes the set it does not use, spread
// over every thread of its grid, right after init_pipeline (so before any wait
// that could run out of time).  The next call, ordered after this one on the
// stream, then starts from zeroed tickets even if a call before this one
// stopped half way.  n == 0 (a caller's workspace, or none): nothing to do.
__device__ __forceinline__ void clear_next_tickets(int32_t *t, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride)
        t[i] = 0;
}

// ---------------------------------------------------------------------------
// Copy
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_tail(char *d, const uint4 &v, int nbytes, int esize) {
    // A 16-byte chunk that straddles column N: store only its in-bounds elements.
    auto word = [&v](int k) { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; };
    if (esize == 4) {
        for (int k = 0; k < nbytes / 4; ++k) reinterpret_cast<uint32_t *>(d)[k] = word(k);
    } else {
        for (int k = 0; k < nbytes / 2; ++k)
            reinterpret_cast<uint16_t *>(d)[k] =
                static_cast<uint16_t>(word(k >> 1) >> ((k & 1) * 16));
    }
}

// Copy one landed stage to the destination with 16-byte LSU stores, using
// `nthr` threads (ctid = 0 .. nthr-1, whole warps).  Every warp releases the
// stage (one arrive on `release_bar` per warp, unless release_bar == 0) right
// after its last shared-memory loads, before its global stores.
__device__ __forceinline__ void copy_tile_lsu(const PipeArgs &p, char *dst, int64_t ld_dst_bytes,
                                              uint32_t sbase, int64_t row0, int64_t col0,
                                              int ctid, int nthr, uint32_t release_bar) {
    const int lane = threadIdx.x & 31;
    const int cpr = p.boxes * 8;                    // 16-byte chunks per tile row
    const int cpr_log2 = __ffs(cpr) - 1;
    const int items = p.tile_m * cpr;
    const int rounds = (items + nthr * kVec - 1) / (nthr * kVec);
    const int vec_elems = 16 / p.esize;
    for (int r = 0; r < rounds; ++r) {
        uint4 v[kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const int i = ctid + (r * kVec + u) * nthr;
            if (i < items) v[u] = lds128(sbase + chunk_offset(i >> cpr_log2, i & (cpr - 1), p.box_stride));
        }
        if (r == rounds - 1) {
            // Every lane's reads of this stage are done: release it.
            __syncwarp();
            if (lane == 0 && release_bar != 0) mbar_arrive(release_bar);
        }
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const int i = ctid + (r * kVec + u) * nthr;
            if (i >= items) continue;
            const int64_t grow = row0 + (i >> cpr_log2);
            const int64_t gcol = col0 + static_cast<int64_t>(i & (cpr - 1)) * vec_elems;
            if (grow >= p.M || gcol >= p.N) continue;
            char *d = dst + grow * ld_dst_bytes + gcol * p.esize;
            if (gcol + vec_elems <= p.N)
                stg128(d, v[u]);
            else
                store_tail(d, v[u], static_cast<int>(p.N - gcol) * p.esize, p.esize);
        }
    }
}

__device__ void consume_copy(const CopyArgs &a, const Smem &sm, const WaitCtl &w,
                             int64_t first, int64_t step, int64_t count) {
    const PipeArgs &p = a.p;
    const int ctid = static_cast<int>(threadIdx.x) - 32;
    const int lane = threadIdx.x & 31;
    const int nthr = p.consumer_warps * 32;
    uint32_t stage = 0, phase = 0;
    for (int64_t j = 0; j < count; ++j) {
        const uint32_t full_bar = sm.full0 + 8u * stage;
        bool ok = wait_bounded(full_bar, phase, w, true);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) {
                report_timeout(w, 1, stage, phase);
                *w.abort = 1;
            }
            break;
        }
        const int64_t tile = first + j * step;
        if (threadIdx.x == 32) log_record(p, 1, j, stage, phase, tile);
        const int64_t tm = tile / p.tiles_n;
        const int64_t row0 = tm * p.tile_m;
        const int64_t col0 = (tile - tm * p.tiles_n) * p.boxes * p.box_inner;
        copy_tile_lsu(p, a.dst, a.ld_dst_bytes, sm.base + stage * p.stage_stride, row0, col0,
                      ctid, nthr, p.fault != 2 ? sm.empty0 + 8u * stage : 0u);
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// Bulk tensor stores of landed stages, issued by one thread.  A stage is
// released (one arrival on its empty barrier) once its store has finished
// reading shared memory: with two or more stages one store is left in flight
// and its stage released after the next store is issued; a single stage is
// released right away.  Loads and stores both run in the async proxy; the
// proxy fence orders the thread's view of the completed phase before the
// store's reads.
struct BulkStores {
    bool pending = false;      // a committed store whose stage is not released yet
    uint32_t prev_stage = 0;

    // Store the tile's boxes that start before column n_map (the extent of
    // dst_map: the columns held in whole 16-byte chunks); the copy engine
    // clips each box there.
    __device__ void store_tile(const CUtensorMap *dst_map, const PipeArgs &p, const Smem &sm,
                               uint32_t stage, int64_t row0, int64_t col0, int64_t n_map) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t sbase = sm.base + stage * p.stage_stride;
        for (int b = 0; b < p.boxes; ++b)
            if (col0 + static_cast<int64_t>(b) * p.box_inner < n_map)
                tma_store_2d(dst_map, sbase + b * p.box_stride,
                             static_cast<int32_t>(col0) + b * p.box_inner,
                             static_cast<int32_t>(row0));
        bulk_commit_group();
        if (p.stages == 1) {
            bulk_wait_read_all();
            if (p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
            return;
        }
        if (pending) {
            bulk_wait_read_allow1();
            if (p.fault != 2) mbar_arrive(sm.empty0 + 8u * prev_stage);
        }
        pending = true;
        prev_stage = stage;
    }

    // Release the stage of the store in flight now (before a tile that no
    // store will follow soon: the producer may need that stage next).
    __device__ void release_pending(const PipeArgs &p, const Smem &sm) {
        if (!pending) return;
        bulk_wait_read_all();
        if (p.fault != 2) mbar_arrive(sm.empty0 + 8u * prev_stage);
        pending = false;
    }

    __device__ void finish(const PipeArgs &p, const Smem &sm, bool aborted) {
        bulk_wait_read_all();
        if (pending && !aborted && p.fault != 2) mbar_arrive(sm.empty0 + 8u * prev_stage);
        pending = false;
        bulk_wait_all();
    }
};

// The partial 16-byte chunk that ends each row of the tile at column N
// (columns [n_whole, N), fewer than 16 bytes), stored element by element by
// the 32 lanes of one warp.
__device__ __forceinline__ void store_partial_chunks(const PipeArgs &p, char *dst,
                                                     int64_t ld_dst_bytes, uint32_t sbase,
                                                     int64_t row0, int64_t col0,
                                                     int64_t n_whole, int lane) {
    const int64_t c_lo = n_whole > col0 ? n_whole : col0;
    const int q = static_cast<int>((c_lo - col0) * p.esize / 16);   // chunk in the tile row
    const int nbytes = static_cast<int>((p.N - c_lo) * p.esize);
    const int64_t left = p.M - row0;
    const int rows = left < p.tile_m ? static_cast<int>(left) : p.tile_m;
    for (int r = lane; r < rows; r += 32) {
        const uint4 v = lds128(sbase + chunk_offset(r, q, p.box_stride));
        store_tail(dst + (row0 + r) * ld_dst_bytes + c_lo * p.esize, v, nbytes, p.esize);
    }
}

// Copy consumer with bulk tensor stores (one consumer warp): lane 0 stores
// each landed stage straight from shared memory (same swizzled box layout) to
// the destination.  The copy engine clips a store's innermost dimension only
// at 16-byte granularity, so dst_map ends at the last whole 16-byte chunk of a
// row (n_whole columns): a tile holding the partial chunk at column N has its
// whole chunks stored in bulk and that chunk stored by the warp's lanes.
// With `info` (the row-sum kernels' store warp) the tiles are those the
// producer published per stage, up to its end mark; else first + j step, j < count.
__device__ void consume_copy_bulk(const CUtensorMap *dst_map, const CopyArgs &a, const Smem &sm,
                                  const WaitCtl &w, int64_t first, int64_t step, int64_t count,
                                  bool do_log = true, const volatile StageInfo *info = nullptr) {
    const PipeArgs &p = a.p;
    const int lane = threadIdx.x & 31;
    const int vec_elems = 16 / p.esize;
    const int64_t n_whole = p.N - p.N % vec_elems;   // columns in whole 16-byte chunks
    const int64_t tile_n = static_cast<int64_t>(p.boxes) * p.box_inner;
    BulkStores bs;
    uint32_t stage = 0, phase = 0;
    for (int64_t j = 0; info != nullptr || j < count; ++j) {
        bool ok = wait_bounded(sm.full0 + 8u * stage, phase, w, true);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) {
                report_timeout(w, 1, stage, phase);
                *w.abort = 1;
            }
            break;
        }
        int64_t tm, tn;
        if (info != nullptr) {
            if (info[stage * 8].key < 0) {   // end mark: release it after the stores in flight
                if (lane == 0) {
                    bs.release_pending(p, sm);
                    if (p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
                }
                break;
            }
            tm = info[stage * 8].tm;
            tn = info[stage * 8].tn;
        } else {
            const int64_t tile = first + j * step;
            tm = tile / p.tiles_n;
            tn = tile - tm * p.tiles_n;
        }
        if (do_log && lane == 0) log_record(p, 1, j, stage, phase, tm * p.tiles_n + tn);
        const int64_t row0 = tm * p.tile_m;
        const int64_t col0 = tn * tile_n;
        if (col0 + tile_n > n_whole && n_whole != p.N) {
            store_partial_chunks(p, a.dst, a.ld_dst_bytes, sm.base + stage * p.stage_stride,
                                 row0, col0, n_whole, lane);
            __syncwarp();   // every lane's reads of the stage are done
            if (lane == 0) {
                if (col0 < n_whole) {
                    bs.store_tile(dst_map, p, sm, stage, row0, col0, n_whole);
                } else {    // nothing in whole chunks: release the stage now
                    bs.release_pending(p, sm);
                    if (p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
                }
            }
        } else if (lane == 0) {
            bs.store_tile(dst_map, p, sm, stage, row0, col0, n_whole);
        }
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (lane == 0) bs.finish(p, sm, *w.abort != 0);
}

// BULK: bulk tensor stores from one consumer warp; else the consumer warps'
// 16-byte LSU stores.  Two instantiations, so that neither carries the other's
// code (one kernel with both paths ran the LSU copy 1.5% slower).
template <bool BULK>
__global__ void __launch_bounds__(kMaxThreads, 2)
    mbt_copy_kernel(const __grid_constant__ CUtensorMap map,
                    const __grid_constant__ CUtensorMap dst_map, const CopyArgs a) {
    extern __shared__ __align__(1024) unsigned char dyn_smem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
    __shared__ int abort_flag;
    Smem sm;
    init_pipeline(a.p, sm, bars, &abort_flag, dyn_smem);
    WaitCtl w{a.p.wait_budget_ns, &abort_flag, status_of(a.p)};
    // Tiles b, b + G, b + 2G, ... in row-major tile order.
    const int64_t G = gridDim.x;
    const int64_t first = blockIdx.x;
    const int64_t count = first < a.p.num_tiles ? (a.p.num_tiles - first + G - 1) / G : 0;
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) produce(&map, a.p, sm, w, first, G, count);
        return;
    }
    if constexpr (BULK)
        consume_copy_bulk(&dst_map, a, sm, w, first, G, count);   // one consumer warp
    else
        consume_copy(a, sm, w, first, G, count);
}

// ---------------------------------------------------------------------------
// Unified (not warp-specialised) copy pipeline
// ---------------------------------------------------------------------------
// Every warp consumes.  Thread 0 issues tile j + S - 1 at the top of
// iteration j (prologue: tiles 0 .. S-2 before the loop); all threads wait on
// full[j mod S], copy the stage out, and a CTA-wide barrier -- which also
// votes on whether any wait gave up -- marks the stage free for the issue at
// the top of the next iteration.  No empty barriers.  Source: "CUDA features
// 10: Pipelines" §4.10.7 (prologue fills S-1 stages; steady state issues the
// next tile, waits for and uses the current one, releases it; epilogue).
__global__ void __launch_bounds__(kMaxThreads, 2)
    mbt_copy_unified_kernel(const __grid_constant__ CUtensorMap map, const CopyArgs a) {
    extern __shared__ __align__(1024) unsigned char dyn_smem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
    __shared__ int abort_flag;
    Smem sm;
    init_pipeline(a.p, sm, bars, &abort_flag, dyn_smem);
    const PipeArgs &p = a.p;
    WaitCtl w{p.wait_budget_ns, &abort_flag, status_of(p)};
    const int64_t G = gridDim.x;
    const int64_t first = blockIdx.x;
    const int64_t count = first < p.num_tiles ? (p.num_tiles - first + G - 1) / G : 0;
    const int nthr = static_cast<int>(blockDim.x);
    const int64_t ahead = p.stages - 1;
    auto issue = [&](int64_t j) {
        const uint32_t s = static_cast<uint32_t>(j % p.stages);
        const int64_t tile = first + j * G;
        const int64_t tm = tile / p.tiles_n;
        const int32_t y = static_cast<int32_t>(tm * p.tile_m);
        const int32_t x0 = static_cast<int32_t>((tile - tm * p.tiles_n) * p.boxes * p.box_inner);
        const uint32_t full_bar = sm.full0 + 8u * s;
        mbar_arrive_expect_tx(full_bar, p.tx_bytes);
        for (int b = 0; b < p.boxes; ++b)
            tma_load_2d(sm.base + s * p.stage_stride + b * p.box_stride, &map,
                        x0 + b * p.box_inner, y, full_bar);
        log_record(p, 0, j, s, 0, tile);
    };
    int64_t issued = 0;
    if (threadIdx.x == 0)
        for (; issued < ahead && issued < count; ++issued) issue(issued);
    for (int64_t j = 0; j < count; ++j) {
        const uint32_t s = static_cast<uint32_t>(j % p.stages);
        const uint32_t par = static_cast<uint32_t>((j / p.stages) & 1);
        // The stage of tile j + S - 1 held tile j - 1, released by the
        // barrier that ended the previous iteration.
        if (threadIdx.x == 0 && issued == j + ahead && issued < count) issue(issued++);
        const bool ok = wait_bounded(sm.full0 + 8u * s, par, w, true);
        if (ok) {
            if (threadIdx.x == 0) log_record(p, 1, j, s, par, first + j * G);
            const int64_t tile = first + j * G;
            const int64_t tm = tile / p.tiles_n;
            copy_tile_lsu(p, a.dst, a.ld_dst_bytes, sm.base + s * p.stage_stride, tm * p.tile_m,
                          (tile - tm * p.tiles_n) * p.boxes * p.box_inner,
                          static_cast<int>(threadIdx.x), nthr, 0u);
        } else if ((threadIdx.x & 31) == 0) {
            report_timeout(w, 1, s, par);
            *w.abort = 1;
        }
        if (__syncthreads_or(!ok)) break;
    }
    if (threadIdx.x == 0 && *w.abort) {
        // Wait (bounded) for loads still in flight before the CTA exits.
        const int64_t from = issued > p.stages ? issued - p.stages : 0;
        for (int64_t t = from; t < issued; ++t)
            wait_bounded(sm.full0 + 8u * static_cast<uint32_t>(t % p.stages),
                         static_cast<uint32_t>((t / p.stages) & 1), w, false);
    }
}

// ---------------------------------------------------------------------------
// Row sum
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ float chunk_sum(const uint4 &v) {
    if constexpr (DT == MBT_F32) {
        return (__uint_as_float(v.x) + __uint_as_float(v.y)) +
               (__uint_as_float(v.z) + __uint_as_float(v.w));
    } else if constexpr (DT == MBT_BF16) {
        // bf16 -> fp32 is exact: the 16 bits are the top half of the fp32.
        auto pair = [](uint32_t u) {
            return __uint_as_float(u << 16) + __uint_as_float(u & 0xffff0000u);
        };
        return (pair(v.x) + pair(v.y)) + (pair(v.z) + pair(v.w));
    } else {
        auto pair = [](uint32_t u) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u));
            return f.x + f.y;
        };
        return (pair(v.x) + pair(v.y)) + (pair(v.z) + pair(v.w));
    }
}

// CTA that owns tile x when `units` units of `gran` tiles are split evenly
// over G CTAs (CTA b owns units [b U / G, (b + 1) U / G)).
__device__ __forceinline__ int64_t unit_owner(int64_t x, int64_t gran, int64_t units, int64_t G) {
    return ((x / gran + 1) * G - 1) / units;
}

// Where a finished segment (a CTA's part of band `key`) goes: the band's K
// contributors are the CTAs owning its units, this CTA's slot its rank among
// them.
struct FlushTarget {
    int64_t band, K, slot;
};

__device__ __forceinline__ FlushTarget flush_target(const RowsumArgs &a, int64_t key) {
    FlushTarget t;
    const int64_t G = gridDim.x;
    const int64_t x0 = key * a.p.tiles_n;
    const int64_t b_first = unit_owner(x0, a.gran, a.units, G);
    t.band = key;
    t.K = unit_owner(x0 + a.p.tiles_n - 1, a.gran, a.units, G) - b_first + 1;
    t.slot = blockIdx.x - b_first;
    return t;
}

// One warp adds K partial slots (`stride` floats apart) for the entries
// lane, lane + 32, ... < n: per entry in slot order (so the same bits for
// every grid); writes dst[c] for c < valid and leaves the slots zero.
// Each lane's entries (at most PL) and B slots are loaded together, so the
// addition takes about K / B load round trips instead of one per entry.
template <int PL, int B>
__device__ __forceinline__ void warp_add_slots(float *base, int64_t K, int64_t stride, int n,
                                               float *dst, int64_t valid) {
    const int lane = threadIdx.x & 31;
    float acc[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) acc[i] = 0.f;
    for (int64_t k0 = 0; k0 < K; k0 += B) {
        float v[B][PL];
#pragma unroll
        for (int u = 0; u < B; ++u)
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                const int c = lane + 32 * i;
                v[u][i] = k0 + u < K && c < n ? __ldcg(base + (k0 + u) * stride + c) : 0.f;
            }
#pragma unroll
        for (int u = 0; u < B; ++u)
#pragma unroll
            for (int i = 0; i < PL; ++i)
                if (k0 + u < K && lane + 32 * i < n) acc[i] += v[u][i];
    }
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int c = lane + 32 * i;
        if (c < n && c < valid) dst[c] = acc[i];
    }
    for (int64_t k = 0; k < K; ++k)
#pragma unroll
        for (int i = 0; i < PL; ++i)
            if (lane + 32 * i < n) base[k * stride + lane + 32 * i] = 0.f;
}

// Orders this thread's earlier memory accesses (and those it has synchronised
// with) before its later ones at GPU scope: release before a ticket, acquire
// after it.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Flush ring of the row sum: the consumers hand each finished segment (the
// CTA's part of a band) -- one fp32 per consumer thread and the segment's key
// -- to a flush warp through a ring of shared-memory slots (full: all
// consumer warps arrived; empty: the flush warp has read the slot), and go on
// with the next segment at once.  The flush warp combines each row's threads
// in `sub` order and does the global part (the row sums, or the segment's
// partials, the band's ticket and the last contributor's ordered addition),
// so the global round trips of a segment change never stall the pipeline.
// (Measured when the consumers still did that part themselves, between
// rendezvous of all consumer warps: the CTAs crossing a band change stalled
// ~3 us; in the fused kernel, moving it to a flush warp gained 0.2-0.5 %.)
constexpr int kMaxConsumerThreads = 32 * kMaxConsumerWarps;
constexpr int kMaxWideConsumerThreads = 32 * kMaxWideConsumerWarps;

struct FlushRing {
    uint32_t full0;    // full[slot] at + 8 slot, counts consumer warps
    uint32_t empty0;   // empty[slot] at + 8 slot, counts the flush warp
    uint32_t k;        // records posted (consumers) or taken (flush warp)
    volatile int64_t *key;   // key[slot]: the segment's key, -1 = no more segments
};

// Slot and phase parity of record k in a ring of NS slots.
template <int NS = kFlushSlots>
__device__ __forceinline__ uint32_t ring_slot(uint32_t k) {
    return k % NS;
}
template <int NS = kFlushSlots>
__device__ __forceinline__ uint32_t ring_parity(uint32_t k) {
    return (k / NS) & 1u;
}

// Post a segment (key >= 0, red: this thread's share) or the end (key < 0).
// CT: consumer threads a ring slot holds.
template <int CT>
__device__ bool flush_post(FlushRing &fr, float *red, float acc, int64_t key, int ctid,
                           const WaitCtl &w) {
    const uint32_t slot = ring_slot(fr.k);
    bool ok = wait_bounded(fr.empty0 + 8u * slot, ring_parity(fr.k) ^ 1u, w, true);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        if ((threadIdx.x & 31) == 0) {
            report_timeout(w, 1, kMaxStages + 1, slot);
            *w.abort = 1;
        }
        return false;
    }
    red[slot * CT + ctid] = acc;
    if (ctid == 0) fr.key[slot] = key;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(fr.full0 + 8u * slot);
    ++fr.k;
    return true;
}

// The flush warp: takes the consumers' records in order until the end mark.
// A band this CTA reduced alone gets its row sums written; otherwise the
// CTA's partials go to its slot and the band's last contributor to arrive
// adds the K slots in slot order.
template <int CT>
__device__ void flush_warp(const RowsumArgs &a, const float *red, FlushRing fr,
                           const WaitCtl &w) {
    const PipeArgs &p = a.p;
    const int lane = threadIdx.x & 31;
    const int tpr = p.consumer_warps * 32 / p.tile_m;
    for (;;) {
        const uint32_t slot = ring_slot(fr.k);
        bool ok = wait_bounded(fr.full0 + 8u * slot, ring_parity(fr.k), w, true);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) {
                report_timeout(w, 1, kMaxStages + 2, slot);
                *w.abort = 1;
            }
            return;
        }
        const int64_t key = fr.key[slot];
        if (key < 0) return;   // the consumers are done
        const float *r = red + slot * CT;
        const FlushTarget ft = flush_target(a, key);
        float *part = ft.K > 1 ? a.partial + (ft.band * a.kmax + ft.slot) * p.tile_m : nullptr;
        for (int row = lane; row < p.tile_m; row += 32) {
            float v = r[row];
            for (int s = 1; s < tpr; ++s) v += r[row + s * p.tile_m];
            const int64_t grow = ft.band * p.tile_m + row;
            if (ft.K == 1) {
                if (grow < p.M) a.out[grow] = v;
            } else {
                part[row] = v;
            }
        }
        if (ft.K > 1) fence_acq_rel_gpu();   // partials visible before the ticket
        __syncwarp();
        if (lane == 0) mbar_arrive(fr.empty0 + 8u * slot);   // r[] is no longer read
        ++fr.k;
        if (ft.K == 1) continue;
        int is_last = 0;
        if (lane == 0) is_last = atomicAdd(&a.ticket[ft.band], 1) == ft.K - 1;
        is_last = __shfl_sync(0xffffffffu, is_last, 0);
        if (is_last) {
            fence_acq_rel_gpu();   // the other contributors' partials, before reading them
            // Bands of at most 128 rows: 8 slots per load round trip (a band
            // of the fp32 12289 x 8191 row sum has 5-6 contributors).  Not in
            // the wide kernel, whose consumers lost speed when its register
            // count went up.
            if (CT <= kMaxConsumerThreads && p.tile_m <= 128)
                warp_add_slots<4, 8>(a.partial + ft.band * a.kmax * p.tile_m, ft.K, p.tile_m,
                                     p.tile_m, a.out + ft.band * p.tile_m,
                                     p.M - ft.band * p.tile_m);
            else
                warp_add_slots<8, 4>(a.partial + ft.band * a.kmax * p.tile_m, ft.K, p.tile_m,
                                     p.tile_m, a.out + ft.band * p.tile_m,
                                     p.M - ft.band * p.tile_m);
            __syncwarp();
            if (lane == 0) a.ticket[ft.band] = 0;
        }
    }
}

// Row-sum consumer warps; the first of them is warp `cwarp0` of the CTA.
// Thread (row, sub) of the tpr threads per row sums the contiguous block of
// 16-byte chunks [sub cpr / tpr, (sub + 1) cpr / tpr) of its row (cpr chunks
// per tile row), in chunk order; the per-thread sums are combined in `sub`
// order.  This order does not depend on the barrier layout, so the fused and
// the per-box kernels give bit-identical sums.  With `boxed` (host-checked:
// tpr a multiple of boxes, and the threads of one box whole warps) every warp
// reads one box only, and waits for and releases that box alone.
template <int DT, bool boxed, int CT>
__device__ void consume_rowsum(const RowsumArgs &a, const Smem &sm, const WaitCtl &w,
                               const volatile StageInfo *info, float *red, FlushRing &fr,
                               int cwarp0) {
    const PipeArgs &p = a.p;
    const int ctid = static_cast<int>(threadIdx.x) - 32 * cwarp0;
    const int lane = threadIdx.x & 31;
    const int nthr = p.consumer_warps * 32;
    const int tpr = nthr / p.tile_m;                 // threads per row (>= 1)
    const bool active = ctid < p.tile_m * tpr;
    const int row = active ? ctid % p.tile_m : 0;
    const int sub = active ? ctid / p.tile_m : 0;
    const int cpr = p.boxes * 8;
    const int lo = sub * cpr / tpr;
    const int mine = active ? (sub + 1) * cpr / tpr - lo : 0;
    const int most = (cpr + tpr - 1) / tpr;
    const int rounds = (most + kVec - 1) / kVec;
    const int box = boxed ? (ctid / p.tile_m) / (tpr / p.boxes) : 0;
    // Where this thread's chunk block starts on a box boundary and takes one
    // round (the default plans at 2 stages and of 128-byte tiles), chunk lo + u
    // of its row lies at box_base + ((u ^ (row mod 8)) << 4): one base per
    // thread instead of a chunk_offset per load.  Measured: +1.5-1.9 % on the
    // ragged 128-byte tiles; with two rounds (4 warps at 3 stages) the general
    // form was 1.7 % faster, and the wide CTA's 4-chunk blocks (S=4) lost 4 %
    // with both forms compiled in, so its kernel keeps the general form only.
    constexpr bool kWide = CT > kMaxConsumerThreads;
    const bool box_aligned = !kWide && (lo & 7) == 0 && rounds == 1;
    const uint32_t box_base =
        static_cast<uint32_t>(lo >> 3) * p.box_stride + static_cast<uint32_t>(row) * kBoxRowBytes;
    const int rx = row & 7;
    float acc = 0.f;
    int64_t key = -1;   // band being summed
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int64_t j = 0;; ++j) {
        const uint32_t full_bar = boxed ? box_bar(sm.fullb0, stage, box) : sm.full0 + 8u * stage;
        const uint32_t empty_bar = boxed ? box_bar(sm.emptyb0, stage, box) : sm.empty0 + 8u * stage;
        bool got = wait_bounded(full_bar, phase, w, true);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
            if (lane == 0) {
                report_timeout(w, 1, stage, phase);
                *w.abort = 1;
            }
            ok = false;
            break;
        }
        const int64_t k = info[stage * 8 + box].key;
        if (k < 0) {   // end mark: release its stage, no more tiles
            __syncwarp();
            if (lane == 0 && p.fault != 2) mbar_arrive(empty_bar);
            break;
        }
        if (k != key) {
            if (key >= 0 && !flush_post<CT>(fr, red, acc, key, ctid, w)) {
                ok = false;
                break;
            }
            key = k;
            acc = 0.f;
        }
        if (ctid == 0 && p.log != nullptr)
            log_record(p, 1, j, stage, phase,
                       static_cast<int64_t>(info[stage * 8 + box].tm) * p.tiles_n +
                           info[stage * 8 + box].tn);
        const uint32_t rbase = sm.base + stage * p.stage_stride;
        float tsum = 0.f;
        for (int r = 0; r < rounds; ++r) {
            uint4 v[kVec];
            if (box_aligned) {
#pragma unroll
                for (int u = 0; u < kVec; ++u)
                    if (r * kVec + u < mine)
                        v[u] = lds128(rbase + box_base + r * p.box_stride +
                                      (static_cast<uint32_t>(u ^ rx) << 4));
            } else {
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    const int c = r * kVec + u;
                    if (c < mine) v[u] = lds128(rbase + chunk_offset(row, lo + c, p.box_stride));
                }
            }
            if (r == rounds - 1) {
                __syncwarp();
                if (lane == 0 && p.fault != 2) mbar_arrive(empty_bar);
            }
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int c = r * kVec + u;
                if (c < mine) tsum += chunk_sum<DT>(v[u]);
            }
        }
        acc += tsum;
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (!ok) return;
    if (key >= 0) ok = flush_post<CT>(fr, red, acc, key, ctid, w);
    if (ok) flush_post<CT>(fr, red, 0.f, -1, ctid, w);   // end mark for the flush warp
}

// FUSED: warp 1 writes every landed stage to dst (bulk tensor stores; LSU
// stores for tiles with a partial 16-byte chunk at column N) and is the one
// extra arrival on each empty barrier, warp 2 is the flush warp (see
// flush_warp) and the row-sum warps follow.  Without it, warp 1 is the flush
// warp.
// BOXED: a full/empty pair per (stage, box) (never with FUSED).  Each barrier
// layout is its own instantiation, so neither carries the other's code.
// WIDE: up to 16 consumer warps, one CTA per SM (stage-wide pairs, no store
// warp).
template <int DT, bool FUSED, bool BOXED, bool WIDE = false>
__global__ void __launch_bounds__(WIDE ? kMaxWideThreads : kMaxThreads + (FUSED ? 64 : 32),
                                  WIDE ? 1 : 2)
    mbt_rowsum_kernel(const __grid_constant__ CUtensorMap map,
                      const __grid_constant__ CUtensorMap dst_map, const RowsumArgs a) {
    extern __shared__ __align__(1024) unsigned char dyn_smem[];
    // Per-box barrier pairs only without the store warp (which reads whole stages).
    static_assert(!(FUSED && BOXED), "the store warp reads whole stages");
    static_assert(!(WIDE && (FUSED || BOXED)), "wide CTAs: stage-wide pairs, no store warp");
    constexpr int CT = WIDE ? kMaxWideConsumerThreads : kMaxConsumerThreads;
    __shared__ __align__(8) uint64_t bars[BOXED ? 16 * kMaxStages : 2 * kMaxStages];
    __shared__ __align__(8) uint64_t ring_bars[2 * kFlushSlots];   // flush ring: full, empty
    // By row-sum consumer thread, one block per flush-ring slot.
    __shared__ float red[kFlushSlots * CT];
    __shared__ int abort_flag;
    __shared__ StageInfo info[8 * kMaxStages];   // per (stage, box), from the producer
    __shared__ int64_t ring_key[kFlushSlots];
    Smem sm;
    constexpr bool boxed = BOXED;
    FlushRing fr{smem_u32(&ring_bars[0]), smem_u32(&ring_bars[kFlushSlots]), 0u, ring_key};
    if (threadIdx.x == 0) {
        for (int k = 0; k < kFlushSlots; ++k) {
            mbar_init(fr.full0 + 8u * k, static_cast<uint32_t>(a.p.consumer_warps));
            mbar_init(fr.empty0 + 8u * k, 1);
        }
    }
    init_pipeline(a.p, sm, bars, &abort_flag, dyn_smem, boxed);   // fences the inits
    clear_next_tickets(a.clear_ticket, a.clear_n);
    WaitCtl w{a.p.wait_budget_ns, &abort_flag, status_of(a.p)};
    // Contiguous, evenly split range of scheduling units, in band-major order.
    const int64_t G = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t first = (b * a.units / G) * a.gran;
    const int64_t last = ((b + 1) * a.units / G) * a.gran;
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) produce_rows<boxed>(&map, a, sm, w, first, last, info);
        return;
    }
    if (threadIdx.x < 64) {
        if constexpr (FUSED) {
            CopyArgs c{};
            c.p = a.p;
            c.dst = a.dst;
            c.ld_dst_bytes = a.ld_dst_bytes;
            c.store_mode = 1;
            consume_copy_bulk(&dst_map, c, sm, w, 0, 0, 0, false, info);
        } else {
            flush_warp<CT>(a, red, fr, w);
        }
        return;
    }
    if (FUSED && threadIdx.x < 96) {   // the fused kernel's flush warp
        flush_warp<CT>(a, red, fr, w);
        return;
    }
    consume_rowsum<DT, boxed, CT>(a, sm, w, info, red, fr, FUSED ? 3 : 2);
}

__global__ void mbt_accumulate_kernel(float *acc, const float *part, int64_t n, int first) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        acc[i] = first ? part[i] : acc[i] + part[i];
}

__global__ void mbt_fill_zero_kernel(float *out, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = 0.f;
}

#include "mbtile_flat.cuh"
#include "mbtile_colsum.cuh"

// Debug: one CTA loads tile (row0, col0) exactly as the pipelines do (one
// bulk tensor copy per 128-byte box, completion on an mbarrier with the
// tile's bytes registered) and writes the stage's raw shared-memory bytes,
// box after box, to `image` -- the swizzled layout the copy engine produced.
__global__ void mbt_stage_image_kernel(const __grid_constant__ CUtensorMap map, int32_t row0,
                                       int32_t col0, int32_t boxes, int32_t box_inner,
                                       uint32_t box_bytes, uint32_t box_stride,
                                       uint64_t budget_ns, unsigned char *image) {
    extern __shared__ __align__(1024) unsigned char dyn_smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t base = (smem_u32(dyn_smem) + 1023u) & ~1023u;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(b, box_bytes * boxes);
        for (int k = 0; k < boxes; ++k)
            tma_load_2d(base + k * box_stride, &map, col0 + k * box_inner, row0, b);
    }
    WaitCtl w{budget_ns, &abort_flag, g_status};
    const bool ok = wait_bounded(b, 0, w, false);
    if (!ok && threadIdx.x == 0) report_timeout(w, 1, 0, 0);
    const unsigned char *stage = dyn_smem + (base - smem_u32(dyn_smem));
    if (ok)
        for (uint32_t i = threadIdx.x; i < box_bytes * boxes; i += blockDim.x) {
            const uint32_t k = i / box_bytes, off = i - k * box_bytes;
            image[i] = stage[k * box_stride + off];
        }
}

}  // namespace

// ---------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------

// Launch of a pipeline kernel with programmatic stream serialization: it may be
// launched, and its CTAs set up their shared memory, while the previous kernel
// of the stream completes (a host launch otherwise starts ~3 us after it
// ends); init_pipeline holds every global access until that kernel has
// completed.
template <class... P, class... A>
cudaError_t launch_pipeline(void (*kernel)(P...), int grid, int threads, int smem,
                            cudaStream_t stream, const A &...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_copy(const CUtensorMap &map, const CUtensorMap &dst_map, const CopyArgs &a,
                        int grid, int threads, int smem, cudaStream_t stream) {
    if (a.store_mode == 1)
        return launch_pipeline(mbt_copy_kernel<true>, grid, threads, smem, stream, map, dst_map,
                               a);
    return launch_pipeline(mbt_copy_kernel<false>, grid, threads, smem, stream, map, dst_map, a);
}

template <bool FUSED, bool BOXED, bool WIDE = false>
cudaError_t launch_rowsum_t(int dtype, const CUtensorMap &map, const CUtensorMap &dst_map,
                            const RowsumArgs &a, int grid, int threads, int smem,
                            cudaStream_t stream) {
    switch (dtype) {
        case MBT_F16:
            return launch_pipeline(mbt_rowsum_kernel<MBT_F16, FUSED, BOXED, WIDE>, grid, threads,
                                   smem, stream, map, dst_map, a);
        case MBT_BF16:
            return launch_pipeline(mbt_rowsum_kernel<MBT_BF16, FUSED, BOXED, WIDE>, grid, threads,
                                   smem, stream, map, dst_map, a);
        default:
            return launch_pipeline(mbt_rowsum_kernel<MBT_F32, FUSED, BOXED, WIDE>, grid, threads,
                                   smem, stream, map, dst_map, a);
    }
}

cudaError_t launch_rowsum(int dtype, const CUtensorMap &map, const CUtensorMap &dst_map,
                          const RowsumArgs &a, int grid, int threads, int smem,
                          cudaStream_t stream) {
    const bool wide = a.p.consumer_warps > kMaxConsumerWarps;
    if (wide && (a.fused || a.boxed)) return cudaErrorInvalidValue;
    if (a.fused)
        return launch_rowsum_t<true, false>(dtype, map, dst_map, a, grid, threads, smem, stream);
    if (a.boxed)
        return launch_rowsum_t<false, true>(dtype, map, dst_map, a, grid, threads, smem, stream);
    if (wide)
        return launch_rowsum_t<false, false, true>(dtype, map, dst_map, a, grid, threads, smem,
                                                   stream);
    return launch_rowsum_t<false, false>(dtype, map, dst_map, a, grid, threads, smem, stream);
}

template <int GMAX, bool WIDE = false>
cudaError_t launch_colsum_t(int dtype, const CUtensorMap &map, const ColsumArgs &a, int grid,
                            int threads, int smem, cudaStream_t stream) {
    switch (dtype) {
        case MBT_F16:
            return launch_pipeline(mbt_colsum_kernel<MBT_F16, GMAX, WIDE>, grid, threads, smem,
                                   stream, map, a);
        case MBT_BF16:
            return launch_pipeline(mbt_colsum_kernel<MBT_BF16, GMAX, WIDE>, grid, threads, smem,
                                   stream, map, a);
        default:
            return launch_pipeline(mbt_colsum_kernel<MBT_F32, GMAX, WIDE>, grid, threads, smem,
                                   stream, map, a);
    }
}

cudaError_t launch_colsum(int dtype, const CUtensorMap &map, const ColsumArgs &a, int grid,
                          int threads, int smem, cudaStream_t stream) {
    if (a.p.col_group < 1 || a.p.col_group > kMaxColGroup) return cudaErrorInvalidValue;
    const bool wide = a.p.consumer_warps > kMaxConsumerWarps;
    if (wide) {   // planned for strips walked one at a time only
        if (a.p.col_group != 1) return cudaErrorInvalidValue;
        return launch_colsum_t<1, true>(dtype, map, a, grid, threads, smem, stream);
    }
    if (a.p.col_group == 1) return launch_colsum_t<1>(dtype, map, a, grid, threads, smem, stream);
    return launch_colsum_t<2>(dtype, map, a, grid, threads, smem, stream);
}

cudaError_t launch_copy_unified(const CUtensorMap &map, const CopyArgs &a, int grid, int threads,
                                int smem, cudaStream_t stream) {
    return launch_pipeline(mbt_copy_unified_kernel, grid, threads, smem, stream, map, a);
}

cudaError_t launch_copy_flat(const FlatArgs &a, int grid, int threads, int smem,
                             cudaStream_t stream) {
    return launch_pipeline(mbt_copy_flat_kernel, grid, threads, smem, stream, a);
}

template <bool ELEM>
cudaError_t launch_rowsum_flat_t(int dtype, const FlatArgs &a, int grid, int threads, int smem,
                                 cudaStream_t stream) {
    switch (dtype) {
        case MBT_F16:
            return launch_pipeline(mbt_rowsum_flat_kernel<MBT_F16, ELEM>, grid, threads, smem,
                                   stream, a);
        case MBT_BF16:
            return launch_pipeline(mbt_rowsum_flat_kernel<MBT_BF16, ELEM>, grid, threads, smem,
                                   stream, a);
        default:
            return launch_pipeline(mbt_rowsum_flat_kernel<MBT_F32, ELEM>, grid, threads, smem,
                                   stream, a);
    }
}

// Rows of at most kFlatElemRowBytes, whole rows per window: the element
// instantiation (same launch bound as the other, so the occupancy the planner
// asked of the other holds for it).
cudaError_t launch_rowsum_flat(int dtype, const FlatArgs &a, int grid, int threads, int smem,
                               cudaStream_t stream) {
    if (a.rows_per_window > 0 && a.elem_rows)
        return launch_rowsum_flat_t<true>(dtype, a, grid, threads, smem, stream);
    return launch_rowsum_flat_t<false>(dtype, a, grid, threads, smem, stream);
}

cudaError_t launch_stage_image(const CUtensorMap &map, int32_t row0, int32_t col0, int32_t boxes,
                               int32_t box_inner, uint32_t box_bytes, uint32_t box_stride,
                               unsigned char *image, cudaStream_t stream) {
    const int smem = static_cast<int>(boxes * box_stride + 1024);
    cudaError_t e = cudaFuncSetAttribute(mbt_stage_image_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    mbt_stage_image_kernel<<<1, 128, smem, stream>>>(map, row0, col0, boxes, box_inner, box_bytes,
                                                     box_stride, kDefaultWaitBudgetNs, image);
    return cudaGetLastError();
}

cudaError_t launch_fill_zero(float *out, int64_t n, cudaStream_t stream) {
    const int threads = 256;
    const int64_t blocks64 = (n + threads - 1) / threads;
    const int blocks = static_cast<int>(blocks64 < 1024 ? (blocks64 < 1 ? 1 : blocks64) : 1024);
    mbt_fill_zero_kernel<<<blocks, threads, 0, stream>>>(out, n);
    return cudaGetLastError();
}

cudaError_t launch_accumulate(float *acc, const float *part, int64_t n, bool first,
                              cudaStream_t stream) {
    const int threads = 256;
    const int64_t blocks64 = (n + threads - 1) / threads;
    const int blocks = static_cast<int>(blocks64 < 1024 ? (blocks64 < 1 ? 1 : blocks64) : 1024);
    mbt_accumulate_kernel<<<blocks, threads, 0, stream>>>(acc, part, n, first ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t set_kernel_smem_limit(int optin, int *usable) {
    // Each kernel may use the opt-in limit minus its own static shared memory;
    // the plan uses the smallest of these so that any kernel can launch it.
    const void *fns[] = {reinterpret_cast<const void *>(mbt_copy_kernel<false>),
                         reinterpret_cast<const void *>(mbt_copy_kernel<true>),
                         reinterpret_cast<const void *>(mbt_copy_unified_kernel),
                         reinterpret_cast<const void *>(mbt_copy_flat_kernel),
                         reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_F16>),
                         reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_BF16>),
                         reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_F32>),
                         reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_F16, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_BF16, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_F32, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, false, false>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, false, false>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, false, false>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, false, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, false, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, false, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, true, false>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, true, false>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, true, false>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F16, 1>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_BF16, 1>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F32, 1>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F16, 2>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_BF16, 2>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F32, 2>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, false, false, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, false, false, true>),
                         reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, false, false, true>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F16, 1, true>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_BF16, 1, true>),
                         reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F32, 1, true>)};
    int least = optin;
    for (const void *fn : fns) {
        cudaFuncAttributes attr{};
        cudaError_t e = cudaFuncGetAttributes(&attr, fn);
        if (e != cudaSuccess) return e;
        const int dyn = optin - static_cast<int>(attr.sharedSizeBytes);
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        if (e != cudaSuccess) return e;
        if (dyn < least) least = dyn;
    }
    *usable = least;
    return cudaSuccess;
}

cudaError_t kernel_fit_per_sm(int op, int dtype, int threads, int smem, int *fit) {
    const void *fn = reinterpret_cast<const void *>(mbt_copy_kernel<false>);
    if (op == 7) fn = reinterpret_cast<const void *>(mbt_copy_kernel<true>);
    if (op == 3) fn = reinterpret_cast<const void *>(mbt_copy_unified_kernel);
    if (op == 4) fn = reinterpret_cast<const void *>(mbt_copy_flat_kernel);
    if (op == 5)
        fn = dtype == MBT_F16    ? reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_F16>)
             : dtype == MBT_BF16 ? reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_BF16>)
                                 : reinterpret_cast<const void *>(mbt_rowsum_flat_kernel<MBT_F32>);
    if (op == MBT_OP_ROWSUM)
        fn = dtype == MBT_F16    ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, false, false>)
             : dtype == MBT_BF16 ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, false, false>)
                                 : reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, false, false>);
    if (op == 8)
        fn = dtype == MBT_F16    ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, false, true>)
             : dtype == MBT_BF16 ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, false, true>)
                                 : reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, false, true>);
    if (op == MBT_OP_COPY_ROWSUM)
        fn = dtype == MBT_F16    ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, true, false>)
             : dtype == MBT_BF16 ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, true, false>)
                                 : reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, true, false>);
    if (op == 6)   // both group widths have the same block shape and limits
        fn = dtype == MBT_F16    ? reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F16, 2>)
             : dtype == MBT_BF16 ? reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_BF16, 2>)
                                 : reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F32, 2>);
    if (op == 9)   // wide row sum
        fn = dtype == MBT_F16    ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F16, false, false, true>)
             : dtype == MBT_BF16 ? reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_BF16, false, false, true>)
                                 : reinterpret_cast<const void *>(mbt_rowsum_kernel<MBT_F32, false, false, true>);
    if (op == 10)  // wide column sum
        fn = dtype == MBT_F16    ? reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F16, 1, true>)
             : dtype == MBT_BF16 ? reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_BF16, 1, true>)
                                 : reinterpret_cast<const void *>(mbt_colsum_kernel<MBT_F32, 1, true>);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(fit, fn, threads, smem);
}

cudaError_t read_and_clear_status(int32_t info[4]) {
    int32_t host[4] = {0, 0, 0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(host, g_status, sizeof host);
    if (e != cudaSuccess) return e;
    const int32_t zero[4] = {0, 0, 0, 0};
    e = cudaMemcpyToSymbol(g_status, zero, sizeof zero);
    for (int i = 0; i < 4; ++i) info[i] = host[i];
    return e;
}

}  // namespace mbt
