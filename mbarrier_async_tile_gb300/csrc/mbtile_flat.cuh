// Pipelines over matrices whose row pitch is not a multiple of 16 bytes.
//
// A bulk tensor copy needs 16-byte global strides, so such a matrix cannot be
// described by a 2-D tensor map.  Here the stages are filled with 1-D bulk
// copies (cp.async.bulk, 16-byte-aligned address and size) of windows of the
// matrix's bytes: the same producer / consumer ring, full and empty barriers,
// expect_tx byte counts and parity cursors as the tiled kernels, but linear
// (unswizzled) stages.  A window starts at the 16-byte boundary at or below its
// first byte and ends at the one at or above its last byte, clipped to the
// last 16-byte boundary of the array; bytes past that clip (at most 15, at the
// very end of the array) are read from global memory directly.
//
// Included by mbtile_kernels.cu inside its anonymous namespace: it uses that
// file's PTX wrappers, bounded waits and status word.

struct Window {
    int64_t ws;     // first byte (16-byte aligned) loaded into the stage
    int64_t size;   // bytes loaded (multiple of 16, may be 0)
};

__device__ __forceinline__ Window make_window(int64_t b0, int64_t b1, int64_t t_floor) {
    Window w;
    w.ws = b0 & ~int64_t(15);
    int64_t we = (b1 + 15) & ~int64_t(15);
    if (we > t_floor) we = t_floor;
    w.size = we > w.ws ? we - w.ws : 0;
    return w;
}

// Element range [e0, e1) of window j of this CTA (row-sum schedule).
struct RowWindow {
    int64_t r0, r1;     // rows [r0, r1) -- whole rows (short rows) or one row
    int64_t e0, e1;     // element indices covered (global, counted along the pitch)
    int64_t piece;      // long rows: which piece of row r0
};

__device__ __forceinline__ RowWindow rowsum_window(const FlatArgs &a, int64_t ra, int64_t rb,
                                                   int64_t j) {
    RowWindow w;
    if (a.rows_per_window > 0) {
        w.r0 = ra + j * a.rows_per_window;
        w.r1 = w.r0 + a.rows_per_window < rb ? w.r0 + a.rows_per_window : rb;
        w.piece = 0;
        w.e0 = w.r0 * a.ld;
        w.e1 = (w.r1 - 1) * a.ld + a.p.N;
    } else {
        w.r0 = ra + j / a.pieces_per_row;
        w.r1 = w.r0 + 1;
        w.piece = j % a.pieces_per_row;
        const int64_t c0 = w.piece * a.piece_elems;
        const int64_t c1 = c0 + a.piece_elems < a.p.N ? c0 + a.piece_elems : a.p.N;
        w.e0 = w.r0 * a.ld + c0;
        w.e1 = w.r0 * a.ld + c1;
    }
    return w;
}

__device__ __forceinline__ int64_t flat_rowsum_windows(const FlatArgs &a, int64_t ra, int64_t rb) {
    if (rb <= ra) return 0;
    if (a.rows_per_window > 0) return (rb - ra + a.rows_per_window - 1) / a.rows_per_window;
    return (rb - ra) * a.pieces_per_row;
}

// Window of the copy schedule: bytes [w C, (w + 1) C) of the 16-byte-aligned
// part of the array.
__device__ __forceinline__ Window copy_window(const FlatArgs &a, int64_t w) {
    Window win;
    win.ws = w * a.cap_bytes;
    const int64_t end = win.ws + a.cap_bytes < a.t_floor ? win.ws + a.cap_bytes : a.t_floor;
    win.size = end - win.ws;
    return win;
}

// Producer of the flat pipelines: loads `count` windows (window j given by
// `win(j)`) into the ring, then drains it.  A window of size 0 (all of it in
// the unaligned tail) completes its phase with a plain arrive.
template <class WinFn>
__device__ void produce_flat(const FlatArgs &a, const Smem &sm, const WaitCtl &w, int64_t count,
                             WinFn win) {
    const PipeArgs &p = a.p;
    uint32_t stage = 0;
    uint32_t phase = (p.fault == 1) ? 0u : 1u;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t j = 0; j < count; ++j) {
        if (!wait_bounded(sm.empty0 + 8u * stage, phase, w, true)) {
            report_timeout(w, 0, stage, phase);
            *w.abort = 1;
            ok = false;
            break;
        }
        const Window wj = win(j);
        const uint32_t full_bar = sm.full0 + 8u * stage;
        if (wj.size > 0) {
            mbar_arrive_expect_tx(full_bar, static_cast<uint32_t>(wj.size));
            bulk_load_1d(sm.base + stage * p.stage_stride, a.src + wj.ws,
                         static_cast<uint32_t>(wj.size), full_bar);
        } else {
            mbar_arrive(full_bar);
        }
        log_record(p, 0, j, stage, phase, j);
        ++issued;
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (ok) {
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
        const int64_t from = issued > p.stages ? issued - p.stages : 0;
        for (int64_t t = from; t < issued; ++t)
            wait_bounded(sm.full0 + 8u * static_cast<uint32_t>(t % p.stages),
                         static_cast<uint32_t>((t / p.stages) & 1), w, false);
    }
}

__device__ __forceinline__ void copy_element(char *d, const char *s, int esize) {
    if (esize == 4)
        *reinterpret_cast<uint32_t *>(d) = *reinterpret_cast<const uint32_t *>(s);
    else
        *reinterpret_cast<uint16_t *>(d) = *reinterpret_cast<const uint16_t *>(s);
}

// ---------------------------------------------------------------------------
// Flat copy (dense source and destination, ld = N, row bytes not a multiple
// of 16): the matrix is one contiguous byte array; CTA b copies windows
// b, b + G, ... with 16-byte LSU stores at the same offsets.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMaxThreads, 2)
    mbt_copy_flat_kernel(const FlatArgs a) {
    extern __shared__ __align__(1024) unsigned char dyn_smem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
    __shared__ int abort_flag;
    Smem sm;
    init_pipeline(a.p, sm, bars, &abort_flag, dyn_smem);
    const PipeArgs &p = a.p;
    WaitCtl w{p.wait_budget_ns, &abort_flag, status_of(p)};
    const int64_t G = gridDim.x;
    const int64_t nwin = (a.t_floor + a.cap_bytes - 1) / a.cap_bytes;
    const int64_t first = blockIdx.x;
    const int64_t count = first < nwin ? (nwin - first + G - 1) / G : 0;
    auto win = [&](int64_t j) { return copy_window(a, first + j * G); };
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) produce_flat(a, sm, w, count, win);
        return;
    }
    const int ctid = static_cast<int>(threadIdx.x) - 32;
    const int lane = threadIdx.x & 31;
    const int nthr = p.consumer_warps * 32;
    if (blockIdx.x == 0) {
        // The unaligned tail of the array (fewer than 16 bytes).
        for (int64_t b = a.t_floor + ctid * p.esize; b < a.total_bytes; b += nthr * p.esize)
            copy_element(a.dst + b, a.src + b, p.esize);
    }
    uint32_t stage = 0, phase = 0;
    for (int64_t j = 0; j < count; ++j) {
        bool ok = wait_bounded(sm.full0 + 8u * stage, phase, w, true);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) {
                report_timeout(w, 1, stage, phase);
                *w.abort = 1;
            }
            break;
        }
        if (ctid == 0) log_record(p, 1, j, stage, phase, first + j * G);
        const Window wj = win(j);
        const uint32_t sbase = sm.base + stage * p.stage_stride;
        const int chunks = static_cast<int>(wj.size >> 4);
        const int rounds = (chunks + nthr * kVec - 1) / (nthr * kVec);
        for (int r = 0; r < rounds; ++r) {
            uint4 v[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int c = ctid + (r * kVec + u) * nthr;
                if (c < chunks) v[u] = lds128(sbase + 16u * c);
            }
            if (r == rounds - 1) {
                __syncwarp();
                if (lane == 0 && p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
            }
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int c = ctid + (r * kVec + u) * nthr;
                if (c < chunks) stg128(a.dst + wj.ws + 16 * static_cast<int64_t>(c), v[u]);
            }
        }
        if (rounds == 0) {
            __syncwarp();
            if (lane == 0 && p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
        }
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// ---------------------------------------------------------------------------
// Flat row sum (any row pitch): CTA b owns rows [b M / G, (b + 1) M / G).
// Rows of at most kFlatElemRowBytes: a window holds many whole rows and each
// thread sums whole rows, element by element.  Other short rows: a window
// holds several whole rows; each row goes to a group of L lanes of one warp
// (as many lanes per row as the CTA's threads allow, a power of two up to 32),
// which add the row's 16-byte chunks masked to the row and finish with a
// shuffle tree: no rendezvous per window.  Long rows: a window
// holds one piece of one row; every thread keeps its share of the row across
// the row's pieces; at the row's last piece each warp's shuffle tree deposits
// a partial, and warp 0 adds the partials in warp order (the other warps do
// not wait for it).  Each row is summed by one CTA, so no
// workspace is needed.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ float element_value(uint32_t bits) {
    if constexpr (DT == MBT_F32) {
        return __uint_as_float(bits);
    } else if constexpr (DT == MBT_BF16) {
        return __uint_as_float(bits << 16);
    } else {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
    }
}

template <int DT>
__device__ __forceinline__ uint32_t element_bits(const unsigned char *p) {
    if constexpr (DT == MBT_F32)
        return *reinterpret_cast<const uint32_t *>(p);
    else
        return *reinterpret_cast<const uint16_t *>(p);
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// One element of the stage at shared address addr, widened exactly.
template <int DT>
__device__ __forceinline__ float lds_element(uint32_t addr) {
    if constexpr (DT == MBT_F32)
        return __uint_as_float(lds32(addr));
    else
        return element_value<DT>(lds16(addr));
}

// Sum of the NN elements of a row starting at shared address addr, in column
// order.
template <int DT, int NN>
__device__ __forceinline__ float row_sum_fixed(uint32_t addr) {
    constexpr int es = DT == MBT_F32 ? 4 : 2;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < NN; ++c) s += lds_element<DT>(addr + es * c);
    return s;
}

// The same for a row of n elements (n at most kFlatElemRowBytes / element size).
template <int DT>
__device__ __forceinline__ float row_sum_elems(uint32_t addr, int n) {
    constexpr int es = DT == MBT_F32 ? 4 : 2;
    switch (n) {
        case 1: return row_sum_fixed<DT, 1>(addr);
        case 2: return row_sum_fixed<DT, 2>(addr);
        case 3: return row_sum_fixed<DT, 3>(addr);
        case 4: return row_sum_fixed<DT, 4>(addr);
        case 5: return row_sum_fixed<DT, 5>(addr);
        case 6: return row_sum_fixed<DT, 6>(addr);
        case 7: return row_sum_fixed<DT, 7>(addr);
        case 8: return row_sum_fixed<DT, 8>(addr);
        default: {
            float s = 0.f;
            int c = 0;
            for (; c + 4 <= n; c += 4) {
                const float x0 = lds_element<DT>(addr + es * c);
                const float x1 = lds_element<DT>(addr + es * (c + 1));
                const float x2 = lds_element<DT>(addr + es * (c + 2));
                const float x3 = lds_element<DT>(addr + es * (c + 3));
                s += x0;
                s += x1;
                s += x2;
                s += x3;
            }
            for (; c < n; ++c) s += lds_element<DT>(addr + es * c);
            return s;
        }
    }
}

// Rows whose pitch is a whole number of 4-byte words sharing a factor with 32:
// the sum from column r round to column r - 1 (r, r + 1, ..., NN - 1, 0, ...,
// r - 1; 0 <= r < NN), lanes starting at different columns so that their
// reads fall in different banks.
template <int DT, int NN>
__device__ __forceinline__ float row_sum_fixed_rot(uint32_t addr, int r) {
    constexpr int es = DT == MBT_F32 ? 4 : 2;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NN; ++k) {
        const int c = k + r < NN ? k + r : k + r - NN;
        s += lds_element<DT>(addr + es * c);
    }
    return s;
}

template <int DT>
__device__ __forceinline__ float row_sum_elems_rot(uint32_t addr, int n, int r) {
    constexpr int es = DT == MBT_F32 ? 4 : 2;
    switch (n) {
        case 1: return row_sum_fixed_rot<DT, 1>(addr, r);
        case 2: return row_sum_fixed_rot<DT, 2>(addr, r);
        case 3: return row_sum_fixed_rot<DT, 3>(addr, r);
        case 4: return row_sum_fixed_rot<DT, 4>(addr, r);
        case 5: return row_sum_fixed_rot<DT, 5>(addr, r);
        case 6: return row_sum_fixed_rot<DT, 6>(addr, r);
        case 7: return row_sum_fixed_rot<DT, 7>(addr, r);
        case 8: return row_sum_fixed_rot<DT, 8>(addr, r);
        default: {
            float s = 0.f;
            for (int k = 0; k < n; ++k) {
                const int c = k + r < n ? k + r : k + r - n;
                s += lds_element<DT>(addr + es * c);
            }
            return s;
        }
    }
}

// The two 16-bit elements of one 4-byte word of the stage, widened exactly
// as element_value does (the lower address first).
template <int DT>
__device__ __forceinline__ float2 pair_value(uint32_t w) {
    if constexpr (DT == MBT_BF16)
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    else
        return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(w))),
                           __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))));
}

// The sum of row_sum_fixed for 16-bit rows of NN elements on a 4-byte
// boundary: the same elements in the same order, two per 32-bit load (an odd
// row's last element alone).
template <int DT, int NN>
__device__ __forceinline__ float row_sum_pairs_fixed(uint32_t addr) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k + 1 < NN; k += 2) {
        const float2 f = pair_value<DT>(lds32(addr + 2 * k));
        s += f.x;
        s += f.y;
    }
    if constexpr (NN % 2 == 1) s += lds_element<DT>(addr + 2 * (NN - 1));
    return s;
}

template <int DT>
__device__ __forceinline__ float row_sum_pairs(uint32_t addr, int n) {
    float s = 0.f;
    int c = 0;
    for (; c + 4 <= n; c += 4) {
        const uint32_t w0 = lds32(addr + 2 * c), w1 = lds32(addr + 2 * c + 4);
        const float2 f0 = pair_value<DT>(w0), f1 = pair_value<DT>(w1);
        s += f0.x;
        s += f0.y;
        s += f1.x;
        s += f1.y;
    }
    for (; c + 2 <= n; c += 2) {
        const float2 f = pair_value<DT>(lds32(addr + 2 * c));
        s += f.x;
        s += f.y;
    }
    if (c < n) s += lds_element<DT>(addr + 2 * c);
    return s;
}

// The rotated sum of row_sum_fixed_rot for 16-bit rows of 2 NP elements on a
// 4-byte boundary whose starting column is even (2 rp): the same elements in
// the same order, two per 32-bit load, and one wrap test per pair.
template <int DT, int NP>
__device__ __forceinline__ float row_sum_pairs_rot_fixed(uint32_t addr, int rp) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        const int c = k + rp < NP ? k + rp : k + rp - NP;
        const float2 f = pair_value<DT>(lds32(addr + 4 * c));
        s += f.x;
        s += f.y;
    }
    return s;
}

template <int DT>
__device__ __forceinline__ float row_sum_pairs_rot(uint32_t addr, int np, int rp) {
    float s = 0.f;
    int c = rp;
    int k = 0;
    for (; k + 2 <= np; k += 2) {
        const int c1 = c + 1 == np ? 0 : c + 1;
        const uint32_t w0 = lds32(addr + 4 * c), w1 = lds32(addr + 4 * c1);
        const float2 f0 = pair_value<DT>(w0), f1 = pair_value<DT>(w1);
        s += f0.x;
        s += f0.y;
        s += f1.x;
        s += f1.y;
        c = c1 + 1 == np ? 0 : c1 + 1;
    }
    if (k < np) {
        const float2 f = pair_value<DT>(lds32(addr + 4 * c));
        s += f.x;
        s += f.y;
    }
    return s;
}

// Sum of the elements of the 16-byte chunk `v` at window byte offset cb whose
// bytes lie in [b0, b1) (window-relative offsets, so 32 bits do), in element order.
template <int DT>
__device__ __forceinline__ float masked_chunk_sum_rel(const uint4 &v, int cb, int b0, int b1) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    float s = 0.f;
    if constexpr (DT == MBT_F32) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (cb + 4 * k >= b0 && cb + 4 * k < b1) s += __uint_as_float(w4[k]);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t bits = (w4[k >> 1] >> ((k & 1) * 16)) & 0xffffu;
            if (cb + 2 * k >= b0 && cb + 2 * k < b1) s += element_value<DT>(bits);
        }
    }
    return s;
}

// Window j + 1 of the row-sum schedule from window j (no divisions).
__device__ __forceinline__ void next_row_window(const FlatArgs &a, int64_t rb, RowWindow &w) {
    if (a.rows_per_window > 0) {
        w.r0 += a.rows_per_window;
        w.r1 = w.r0 + a.rows_per_window < rb ? w.r0 + a.rows_per_window : rb;
        w.e0 = w.r0 * a.ld;
        w.e1 = (w.r1 - 1) * a.ld + a.p.N;
    } else {
        if (++w.piece == a.pieces_per_row) {
            w.piece = 0;
            ++w.r0;
            w.r1 = w.r0 + 1;
        }
        const int64_t c0 = w.piece * a.piece_elems;
        const int64_t c1 = c0 + a.piece_elems < a.p.N ? c0 + a.piece_elems : a.p.N;
        w.e0 = w.r0 * a.ld + c0;
        w.e1 = w.r0 * a.ld + c1;
    }
}

// Long rows: slots for the warp partials of rows still being combined.  A
// window is reloaded only after every warp released it, so another warp can
// finish row lr + K before warp 0 has read row lr's partials only if
// K P <= stages (P pieces per row, P >= 1): 16 slots hold for up to 15 stages.
constexpr int kFlatRowSlots = 16;
constexpr int kFlatVec = 4;   // chunks a thread holds per round (register budget)

// ELEM: the instantiation launched for rows of at most kFlatElemRowBytes
// summed whole by one thread each (modes 2-5: a.elem_rows and whole rows per
// window); the other holds only the window modes (0, 1), which alone take 88
// registers instead of 94-96 (bf16 rows of 100 / 2047 elements: +3.4 / +3.6 %).
template <int DT, bool ELEM = false>
__global__ void __launch_bounds__(kMaxThreads, 2)
    mbt_rowsum_flat_kernel(const FlatArgs a) {
    extern __shared__ __align__(1024) unsigned char dyn_smem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
    // Long rows: warp partials of row lr in red[lr % kFlatRowSlots]; its
    // row_bar completes when every consumer warp has deposited its partial.
    __shared__ __align__(8) uint64_t row_bar[kFlatRowSlots];
    __shared__ float red[kFlatRowSlots][kMaxConsumerWarps];
    __shared__ int abort_flag;
    Smem sm;
    if (threadIdx.x == 0)
        for (int k = 0; k < kFlatRowSlots; ++k)
            mbar_init(smem_u32(&row_bar[k]), static_cast<uint32_t>(a.p.consumer_warps));
    init_pipeline(a.p, sm, bars, &abort_flag, dyn_smem);   // fences the inits
    const PipeArgs &p = a.p;
    WaitCtl w{p.wait_budget_ns, &abort_flag, status_of(p)};
    const int64_t G = gridDim.x;
    const int64_t ra = static_cast<int64_t>(blockIdx.x) * p.M / G;
    const int64_t rb = (static_cast<int64_t>(blockIdx.x) + 1) * p.M / G;
    const int64_t count = flat_rowsum_windows(a, ra, rb);
    auto win = [&](int64_t j) {
        const RowWindow rw = rowsum_window(a, ra, rb, j);
        return make_window(rw.e0 * p.esize, rw.e1 * p.esize, a.t_floor);
    };
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) produce_flat(a, sm, w, count, win);
        return;
    }
    const int ctid = static_cast<int>(threadIdx.x) - 32;
    const int lane = threadIdx.x & 31;
    const int warp = ctid >> 5;
    const int nthr = p.consumer_warps * 32;
    const unsigned char *gsrc = reinterpret_cast<const unsigned char *>(a.src);
    // One instantiation of the window loop per row shape -- pieces of long rows
    // (0), whole rows summed by lane groups (1), whole rows of at most
    // kFlatElemRowBytes summed element by element (2; 3 with the lanes'
    // starting columns rotated): none carries another's state.
    auto run = [&](auto mode) {
        constexpr int kMode = decltype(mode)::value;
        constexpr bool kShort = kMode != 0;
        float row_acc = 0.f;            // long rows: this thread's share of the current row
        // Short rows: every row of a window goes to a group of L lanes of one warp
        // (a power of two, 1..32: as many lanes per row as the threads allow for
        // this CTA's fullest window; a shorter last window leaves groups idle).
        // The pp = 8 / L groups of one 8-lane shared-memory phase take rows
        // 2^phase_shift apart (group g of a block of pp << phase_shift groups sums
        // row h + q 2^phase_shift, q = g mod pp, h = g / pp), so that their 16-byte
        // reads fall in different bank groups.
        const int64_t full_rows = a.rows_per_window < rb - ra ? a.rows_per_window : rb - ra;
        int L = 1;
        while (L < 32 && 2 * L * full_rows <= nthr) L <<= 1;
        const int groups = nthr / L;
        const int gidx = ctid / L, gl = ctid % L;
        const int pp_log = L < 8 ? 3 - (__ffs(L) - 1) : 0;
        const int sh = pp_log > 0 ? a.phase_shift : 0;
        const int blk = 1 << (pp_log + sh);
        uint32_t stage = 0, phase = 0;
        RowWindow rw = rowsum_window(a, ra, rb, 0);
        for (int64_t j = 0; j < count; ++j, next_row_window(a, rb, rw)) {
            bool ok = wait_bounded(sm.full0 + 8u * stage, phase, w, true);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) {
                    report_timeout(w, 1, stage, phase);
                    *w.abort = 1;
                }
                break;
            }
            if (ctid == 0) log_record(p, 1, j, stage, phase, j);
            const Window wj = make_window(rw.e0 * p.esize, rw.e1 * p.esize, a.t_floor);
            const int64_t we = wj.ws + wj.size;
            const int chunks = static_cast<int>(wj.size >> 4);
            const uint32_t sbase = sm.base + stage * p.stage_stride;
            if constexpr (kMode >= 2) {
                // Rows of at most kFlatElemRowBytes: thread t sums rows t, t + nthr,
                // ... of the window element by element, from its starting column
                // round to the one before it.  Consecutive lanes take consecutive
                // rows (nearby shared-memory addresses, and coalesced stores of the
                // sums).
                const int nrows = static_cast<int>(rw.r1 - rw.r0);
                const int pitch_b = static_cast<int>(a.ld * p.esize);
                const int off0 = static_cast<int>(rw.e0 * p.esize - wj.ws);
                const int row_b = static_cast<int>(p.N) * p.esize;
                const int n = static_cast<int>(p.N);
                // Starting column of this lane's rows: lanes elem_period apart would
                // otherwise read the same bank at every step.
                const int rot = kMode >= 3 ? (lane / a.elem_period) * (4 / p.esize) % n : 0;
                // One row loop per row length up to 12 (the row's sum unrolled inside,
                // no branch on the length per row), one for longer rows.  Measured,
                // same box, bf16 dense: 1 / 3 / 8 columns 2377 -> 4437 / 3483 -> 5753
                // / 5144 -> 6650 GB/s; 16-32 columns 2-3 % slower than with the
                // length switch inside the row loop (and 20-25 % slower with the
                // longer rows' loop in a separate, non-inlined function).
                auto rows = [&](auto len) {
                    constexpr int NN = decltype(len)::value;   // 0: the length n at run time
                    for (int lr = ctid; lr < nrows; lr += nthr) {
                        const int b0 = off0 + lr * pitch_b;
                        float s;
                        if (b0 + row_b <= wj.size) {
                            const uint32_t ra = sbase + static_cast<uint32_t>(b0);
                            if constexpr (kMode == 5 && NN > 0)
                                s = row_sum_pairs_fixed<DT, NN>(ra);
                            else if constexpr (kMode == 5)
                                s = row_sum_pairs<DT>(ra, n);
                            else if constexpr (kMode == 4 && NN > 0 && NN % 2 == 0)
                                s = row_sum_pairs_rot_fixed<DT, NN / 2>(ra, rot / 2);
                            else if constexpr (kMode == 4)
                                s = row_sum_pairs_rot<DT>(ra, n / 2, rot / 2);
                            else if constexpr (kMode == 3 && NN > 0)
                                s = row_sum_fixed_rot<DT, NN>(ra, rot);
                            else if constexpr (kMode == 3)
                                s = row_sum_elems_rot<DT>(ra, n, rot);
                            else if constexpr (NN > 0)
                                s = row_sum_fixed<DT, NN>(ra);
                            else
                                s = row_sum_elems<DT>(ra, n);
                        } else {
                            // The array's last row: bytes past its last 16-byte
                            // boundary were not loaded.
                            s = 0.f;
                            for (int c = 0; c < n; ++c) {
                                const int64_t bb = b0 + static_cast<int64_t>(c) * p.esize;
                                s += bb < wj.size
                                         ? lds_element<DT>(sbase + static_cast<uint32_t>(bb))
                                         : element_value<DT>(element_bits<DT>(gsrc + wj.ws + bb));
                            }
                        }
                        a.out[rw.r0 + lr] = s;
                    }
                };
                switch (n) {
                    case 1: rows(std::integral_constant<int, 1>{}); break;
                    case 2: rows(std::integral_constant<int, 2>{}); break;
                    case 3: rows(std::integral_constant<int, 3>{}); break;
                    case 4: rows(std::integral_constant<int, 4>{}); break;
                    case 5: rows(std::integral_constant<int, 5>{}); break;
                    case 6: rows(std::integral_constant<int, 6>{}); break;
                    case 7: rows(std::integral_constant<int, 7>{}); break;
                    case 8: rows(std::integral_constant<int, 8>{}); break;
                    default:
                        // Rows of 9-12 elements unrolled too (dense bf16 9 / 11
                        // columns 4032 / 4194 -> 6832 / 6771 GB/s, fp32 10 / 12
                        // columns 5045 / 5662 -> 6737 / 6748; longer unrolled rows
                        // made the kernel spill).
                        if constexpr (kMode >= 2) {
                            switch (n) {
                                case 9: rows(std::integral_constant<int, 9>{}); break;
                                case 10: rows(std::integral_constant<int, 10>{}); break;
                                case 11: rows(std::integral_constant<int, 11>{}); break;
                                case 12: rows(std::integral_constant<int, 12>{}); break;
                                default: rows(std::integral_constant<int, 0>{}); break;
                            }
                        } else {
                            rows(std::integral_constant<int, 0>{});
                        }
                        break;
                }
                __syncwarp();
                if (lane == 0 && p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
            } else if constexpr (kShort) {
                // Short rows: the group's lanes add the row's chunks, masked to
                // the row, and a shuffle tree inside the group gives the row's sum.
                // No thread needs another warp's results, so the window needs no
                // rendezvous.  The rows are padded to whole blocks of the row map.
                const int nrows = static_cast<int>(rw.r1 - rw.r0);
                const int padded = (nrows + blk - 1) & ~(blk - 1);
                const int iters = (padded + groups - 1) / groups;
                for (int it = 0; it < iters; ++it) {
                    int lr = gidx + it * groups;
                    if (sh != 0) {
                        const int gi = lr & (blk - 1);
                        lr += (gi >> pp_log) + ((gi & ((1 << pp_log) - 1)) << sh) - gi;
                    }
                    float s = 0.f;
                    if (lr < nrows) {
                        const int64_t e0 = (rw.r0 + lr) * a.ld, e1 = e0 + p.N;
                        const int64_t b0 = e0 * p.esize - wj.ws, b1 = e1 * p.esize - wj.ws;
                        const int64_t loaded = b1 < wj.size ? b1 : wj.size;
                        if (loaded > b0) {
                            const int rb0 = static_cast<int>(b0), rb1 = static_cast<int>(b1);
                            const int cs = rb0 >> 4;
                            const int ce = static_cast<int>((loaded - 1) >> 4);
                            for (int c = cs + gl; c <= ce; c += L) {
                                const uint4 v = lds128(sbase + 16u * c);
                                const int cb = 16 * c;
                                s += (cb >= rb0 && cb + 16 <= rb1)
                                         ? chunk_sum<DT>(v)
                                         : masked_chunk_sum_rel<DT>(v, cb, rb0, rb1);
                            }
                        }
                        // Bytes past the array's last 16-byte boundary (never loaded).
                        if (gl == 0)
                            for (int64_t bb = loaded > b0 ? loaded : b0; bb < b1; bb += p.esize)
                                s += element_value<DT>(element_bits<DT>(gsrc + wj.ws + bb));
                    }
                    for (int off = L >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                    if (lr < nrows && gl == 0) a.out[rw.r0 + lr] = s;
                }
                __syncwarp();
                if (lane == 0 && p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
            } else {
                // Long rows: the window is one piece of row r0; threads keep their
                // share of the row across its pieces and reduce once per row.
                const int pb0 = static_cast<int>(rw.e0 * p.esize - wj.ws);   // piece bytes in
                const int pb1 = static_cast<int>(rw.e1 * p.esize - wj.ws);   // the window
                for (int c0 = 0; c0 < chunks; c0 += nthr * kFlatVec) {
                    uint4 v[kFlatVec];
    #pragma unroll
                    for (int u = 0; u < kFlatVec; ++u) {
                        const int c = c0 + ctid + u * nthr;
                        if (c < chunks) v[u] = lds128(sbase + 16u * c);
                    }
                    if (c0 + nthr * kFlatVec >= chunks) {
                        __syncwarp();
                        if (lane == 0 && p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
                    }
    #pragma unroll
                    for (int u = 0; u < kFlatVec; ++u) {
                        const int c = c0 + ctid + u * nthr;
                        if (c >= chunks) continue;
                        const int cb = 16 * c;
                        row_acc += (cb >= pb0 && cb + 16 <= pb1)
                                       ? chunk_sum<DT>(v[u])
                                       : masked_chunk_sum_rel<DT>(v[u], cb, pb0, pb1);
                    }
                }
                if (chunks == 0) {
                    __syncwarp();
                    if (lane == 0 && p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
                }
                if (ctid == 0) {
                    // Elements past the array's last 16-byte boundary.
                    for (int64_t g = (we > rw.e0 * p.esize ? we / p.esize : rw.e0); g < rw.e1; ++g)
                        row_acc += element_value<DT>(element_bits<DT>(gsrc + g * p.esize));
                }
                if (rw.piece == a.pieces_per_row - 1) {
                    float s = row_acc;
                    row_acc = 0.f;
    #pragma unroll
                    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                    // Deposit the warp's partial; warp 0 alone waits for the row's
                    // other partials and adds them in warp order, so the other
                    // warps go on to the next row at once.
                    const int64_t lr = rw.r0 - ra;
                    const int slot = static_cast<int>(lr % kFlatRowSlots);
                    const uint32_t bar = smem_u32(&row_bar[slot]);
                    if (lane == 0) {
                        red[slot][warp] = s;
                        mbar_arrive(bar);
                    }
                    if (warp == 0) {
                        bool got = wait_bounded(bar, static_cast<uint32_t>((lr / kFlatRowSlots) & 1),
                                                w, true);
                        got = __all_sync(0xffffffffu, got);
                        if (!got) {
                            if (lane == 0) {
                                report_timeout(w, 1, kMaxStages, static_cast<uint32_t>(slot));
                                *w.abort = 1;
                            }
                            break;
                        }
                        if (lane == 0) {
                            float total = 0.f;
                            for (int k = 0; k < p.consumer_warps; ++k) total += red[slot][k];
                            a.out[rw.r0] = total;
                        }
                    }
                }
            }
            if (++stage == static_cast<uint32_t>(p.stages)) {
                stage = 0;
                phase ^= 1u;
            }
        }
    };
    // Mode 4: the rotated rows of mode 3 for 16-bit elements and an even row
    // length, so that the starting column (a whole 4-byte word) is even and a
    // pair never straddles the row's end: two elements per load.
    // Mode 5: the rows of mode 2 for 16-bit elements where the pitch is a
    // whole number of 4-byte words (so every row starts on one): two elements
    // per load.
    if constexpr (ELEM) {
        // (every mode: the element rows' code measured 6-10 % slower on rows of
        // 13-31 elements when compiled without the window modes beside it)
        if constexpr (DT != MBT_F32) {
            if (a.rows_per_window > 0 && a.elem_rows && a.elem_period > 0 &&
                (a.p.N & 1) == 0) {
                run(std::integral_constant<int, 4>{});
                return;
            }
            if (a.rows_per_window > 0 && a.elem_rows && a.elem_period == 0 &&
                (a.ld * a.p.esize) % 4 == 0) {
                run(std::integral_constant<int, 5>{});
                return;
            }
        }
        if (a.rows_per_window > 0 && a.elem_rows && a.elem_period > 0)
            run(std::integral_constant<int, 3>{});
        else if (a.rows_per_window > 0 && a.elem_rows)
            run(std::integral_constant<int, 2>{});
        else if (a.rows_per_window > 0)
            run(std::integral_constant<int, 1>{});
        else
            run(std::integral_constant<int, 0>{});
    } else {
        if (a.rows_per_window > 0)
            run(std::integral_constant<int, 1>{});
        else
            run(std::integral_constant<int, 0>{});
    }
}
