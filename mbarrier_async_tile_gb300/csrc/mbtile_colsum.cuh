// Column sums through the tile pipeline: out[j] = sum over rows i < M of
// x[i][j], fp32.
//
// The same producer / consumer ring as the row sum (one elected producer
// thread issues each tile's bulk tensor copies against the stage's full
// barrier, consumer warps wait on it, read the swizzled stage and release it
// with one arrive per warp), but the tiles are taken down the column strips
// (tile_n columns each), so each consumer thread keeps its columns' sums in
// registers across a strip's tiles.
//
// Order.  The column strips are taken in groups of col_group adjacent strips
// (2 strips where a tile row is 128 bytes, so that the copies in flight read
// 256 contiguous bytes of each row, not scattered 128-byte pieces; and where one
// CTA per SM streams alone, 2 strips of up to 512 bytes, 1 KB per row); within
// a group the tiles go band by band, left to right.  Each consumer thread keeps
// one set of accumulators per strip of the group.
//
// Consumer mapping.  A tile row holds cpr = boxes x 8 chunks of 16 bytes;
// tpc = 32 W / cpr threads share each chunk column: thread (q, g) with
// q = ctid / tpc, g = ctid % tpc sums rows g, g + tpc, ... of chunk column q
// into EPC fp32 accumulators (EPC = elements per chunk: 8, or 4 for fp32).
// Eight consecutive threads read eight consecutive rows of the same chunk,
// which the 128-byte swizzle spreads over all banks.  When a CTA leaves a
// group, the tpc partial sums of each column are added in g order (by the
// flush warp); a strip that several CTAs share is combined by the last of them
// in CTA order (tickets and partials in the workspace, left zeroed).
//
// Included by mbtile_kernels.cu inside its anonymous namespace: it uses that
// file's PTX wrappers, bounded waits, producer, status word and log.

template <int DT>
__device__ __forceinline__ void chunk_accumulate(float *acc, const uint4 &v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (DT == MBT_F32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] += __uint_as_float(w[k]);
    } else if constexpr (DT == MBT_BF16) {
        // bf16 -> fp32 is exact: the 16 bits are the top half of the fp32.
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc[2 * k] += __uint_as_float(w[k] << 16);
            acc[2 * k + 1] += __uint_as_float(w[k] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            acc[2 * k] += f.x;
            acc[2 * k + 1] += f.y;
        }
    }
}

// Flush ring of the column sum: when a CTA leaves a group, each consumer
// thread drops its accumulators into the next ring slot (in dynamic shared
// memory after the stages: kColsumRingSlots slots of 32 W x EPC x GMAX floats,
// thread (q, g)'s sums of strip k at g (GMAX tn) + k tn + q EPC) and its warp
// arrives; no consumer waits for another.  The flush warp adds the tpc
// partials of each column in g order and does the global part: the column
// sums (sole contributor), or the CTA's partials, fence, ticket, and for the
// last contributor the addition of all contributors' partials in CTA order.
// Measured on the fp32 12289 x 8191 column sum with 128 x 32 tiles: adding
// the partials in the consumers, between two rendezvous of all consumer
// warps per strip, stalled the consumers of a CTA that changes strip pair
// half way through its range by ~4 us.
template <int EPC, int GMAX>
__device__ bool post_group(int tn, int64_t gstart, float (*acc)[EPC], bool active, int q,
                           int g, float *ring, int slot_floats, FlushRing &fr, const WaitCtl &w,
                           int ctid) {
    const uint32_t slot = ring_slot<kColsumRingSlots>(fr.k);
    bool ok = wait_bounded(fr.empty0 + 8u * slot, ring_parity<kColsumRingSlots>(fr.k) ^ 1u, w,
                           true);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        if ((threadIdx.x & 31) == 0) {
            report_timeout(w, 1, kMaxStages + 1, slot);
            *w.abort = 1;
        }
        return false;
    }
    if (gstart >= 0 && active) {
        float *dst = ring + slot * slot_floats + g * (GMAX * tn) + q * EPC;
#pragma unroll
        for (int k = 0; k < GMAX; ++k)
#pragma unroll
            for (int e = 0; e < EPC; e += 4)
                *reinterpret_cast<float4 *>(dst + k * tn + e) =
                    make_float4(acc[k][e], acc[k][e + 1], acc[k][e + 2], acc[k][e + 3]);
    }
    if (ctid == 0) fr.key[slot] = gstart;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(fr.full0 + 8u * slot);
    ++fr.k;
    return true;
}

// The last contributor's addition for the strips of a pair that this CTA
// completes (bit k of `lasts`: strip k of the pair).  Entry e = k tn + c
// (strip k, column c) of a 128-entry chunk of the pair belongs to lane
// e % 32; for each entry the K_k partial slots are added in slot order (as
// warp_add_slots does, so the same bits), the column sum is written and the
// slots are left zero.  A lane's 4 entries and 8 slots are loaded together,
// both strips at once: a pair of 128-byte strips (at most 2 x 64 columns, one
// chunk) with 5 contributors each costs one load round trip, not three per
// strip one strip after the other.  Wider strips (pairs where one CTA per SM
// runs) take one chunk after another.
__device__ __forceinline__ void combine_pair(const ColsumArgs &a, const int64_t *strip_k,
                                             const int64_t *K_k, unsigned lasts, int tn) {
    constexpr int PL = 4, B = 8;
    const int lane = threadIdx.x & 31;
    for (int e0 = 0; e0 < 2 * tn; e0 += 32 * PL) {
        float *slot0[PL];
        int kn[PL];
        int kmax_all = 0;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = e0 + lane + 32 * i;
            const int k = e >= tn ? 1 : 0;
            const bool on = e < 2 * tn && ((lasts >> k) & 1u);
            slot0[i] = a.partial + (k ? strip_k[1] : strip_k[0]) * a.kmax * tn + (e - k * tn);
            kn[i] = on ? static_cast<int>(k ? K_k[1] : K_k[0]) : 0;
            kmax_all = kn[i] > kmax_all ? kn[i] : kmax_all;
        }
        float acc[PL];
#pragma unroll
        for (int i = 0; i < PL; ++i) acc[i] = 0.f;
        for (int k0 = 0; k0 < kmax_all; k0 += B) {
            float v[B][PL];
#pragma unroll
            for (int u = 0; u < B; ++u)
#pragma unroll
                for (int i = 0; i < PL; ++i)
                    v[u][i] = k0 + u < kn[i]
                                  ? __ldcg(slot0[i] + static_cast<int64_t>(k0 + u) * tn)
                                  : 0.f;
#pragma unroll
            for (int u = 0; u < B; ++u)
#pragma unroll
                for (int i = 0; i < PL; ++i)
                    if (k0 + u < kn[i]) acc[i] += v[u][i];
        }
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            if (kn[i] == 0) continue;
            const int e = e0 + lane + 32 * i;
            const int k = e >= tn ? 1 : 0;
            const int64_t col = (k ? strip_k[1] : strip_k[0]) * tn + (e - k * tn);
            if (col < a.p.N) a.out[col] = acc[i];
            for (int j = 0; j < kn[i]; ++j) slot0[i][static_cast<int64_t>(j) * tn] = 0.f;
        }
    }
}

// The column sum's flush warp: takes the consumers' records in order until
// the end mark (key -1).
template <int GMAX>
__device__ void colsum_flush_warp(const ColsumArgs &a, const float *ring, int slot_floats,
                                  int tpc, FlushRing fr, const WaitCtl &w) {
    const PipeArgs &p = a.p;
    const int lane = threadIdx.x & 31;
    const int tn = a.tile_n;
    const int gw = GMAX * tn;   // floats per partial row of a slot
    const int64_t G = gridDim.x;
    for (;;) {
        const uint32_t slot = ring_slot<kColsumRingSlots>(fr.k);
        bool ok = wait_bounded(fr.full0 + 8u * slot, ring_parity<kColsumRingSlots>(fr.k), w, true);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) {
                report_timeout(w, 1, kMaxStages + 2, slot);
                *w.abort = 1;
            }
            return;
        }
        const int64_t gstart = fr.key[slot];
        if (gstart < 0) return;   // the consumers are done
        const float *data = ring + slot * slot_floats;
        const ColPos c0 = col_pos(gstart, p.tiles_m, p.tiles_n, GMAX);
        int64_t strip_k[GMAX], K_k[GMAX];
        bool any_split = false;
#pragma unroll
        for (int k = 0; k < GMAX; ++k) {
            strip_k[k] = 0;
            K_k[k] = 0;
            if (k >= c0.wg) continue;
            const int64_t pos_first = gstart + k;
            const int64_t pos_last = gstart + (p.tiles_m - 1) * c0.wg + k;
            const int64_t b_first = unit_owner(pos_first, a.gran, a.units, G);
            const int64_t b_last = unit_owner(pos_last, a.gran, a.units, G);
            if (static_cast<int64_t>(blockIdx.x) < b_first ||
                static_cast<int64_t>(blockIdx.x) > b_last)
                continue;   // not a contributor of this strip
            const int64_t strip = col_strip(c0, GMAX) + k;
            const int64_t K = b_last - b_first + 1;
            strip_k[k] = strip;
            K_k[k] = K;
            const int64_t col0 = strip * tn;
            float *part = a.partial + (strip * a.kmax + (blockIdx.x - b_first)) * tn;
            for (int c = lane; c < tn; c += 32) {
                // the tpc partials of the column, in g order (4 loads at a time)
                const float *col = data + k * tn + c;
                float v = col[0];
                int s = 1;
                for (; s + 4 <= tpc; s += 4) {
                    const float t0 = col[s * gw], t1 = col[(s + 1) * gw];
                    const float t2 = col[(s + 2) * gw], t3 = col[(s + 3) * gw];
                    v += t0;
                    v += t1;
                    v += t2;
                    v += t3;
                }
                for (; s < tpc; ++s) v += col[s * gw];
                if (K == 1) {
                    if (col0 + c < p.N) a.out[col0 + c] = v;
                } else {
                    part[c] = v;
                }
            }
            any_split |= K > 1;
        }
        if (any_split) fence_acq_rel_gpu();   // partials visible before the tickets
        __syncwarp();
        if (lane == 0) mbar_arrive(fr.empty0 + 8u * slot);   // data[] is no longer read
        ++fr.k;
        if (!any_split) continue;
        // The tickets of the group's split strips, taken together (lane k:
        // strip k of the group).
        int64_t my_strip = 0, my_K = 0;
#pragma unroll
        for (int k = 0; k < GMAX; ++k)
            if (lane == k) {
                my_strip = strip_k[k];
                my_K = K_k[k];
            }
        const bool my_last = my_K > 1 && atomicAdd(&a.ticket[my_strip], 1) == my_K - 1;
        const unsigned lasts = __ballot_sync(0xffffffffu, my_last);
        if (lasts == 0) continue;
        fence_acq_rel_gpu();   // the other contributors' partials, before reading them
        if constexpr (GMAX == 2) {
            combine_pair(a, strip_k, K_k, lasts, tn);
        } else {
            warp_add_slots<16, 2>(a.partial + strip_k[0] * a.kmax * tn, K_k[0], tn, tn,
                                  a.out + strip_k[0] * tn, p.N - strip_k[0] * tn);
        }
        __syncwarp();
        if (my_last) a.ticket[my_strip] = 0;
    }
}

// GMAX: strips per group (= p.col_group; the launch picks the instantiation).
template <int DT, int GMAX>
__device__ void consume_colsum(const ColsumArgs &a, const Smem &sm, const WaitCtl &w,
                               int64_t first, int64_t count, float *ring, int slot_floats,
                               FlushRing &fr) {
    constexpr int EPC = DT == MBT_F32 ? 4 : 8;
    const PipeArgs &p = a.p;
    const int ctid = static_cast<int>(threadIdx.x) - 64;   // warp 0 produces, warp 1 flushes
    const int lane = threadIdx.x & 31;
    const int nthr = p.consumer_warps * 32;
    const int cpr = p.boxes * 8;
    const int tpc = nthr / cpr;                      // threads per chunk column (>= 1)
    const bool active = ctid < cpr * tpc;
    const int q = active ? ctid / tpc : 0;
    const int g = active ? ctid % tpc : 0;
    float acc[GMAX][EPC];
#pragma unroll
    for (int k = 0; k < GMAX; ++k)
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc[k][e] = 0.f;
    // 16-byte loads in flight per thread and round (fewer when a thread keeps
    // two strips' accumulators, to stay within the registers of 2 CTAs/SM).
    constexpr int CV = GMAX == 1 ? kVec : kVec / 2;
    int64_t group = -1;   // order position of the current group's first tile
    const int most = (p.tile_m + tpc - 1) / tpc;
    const int rounds = (most + CV - 1) / CV;
    // Strip pairs are planned with tpc a multiple of 8, so
    // rows g, g + tpc, ... of chunk q share one swizzle term: their stage
    // offsets are one per-thread base plus k tpc 128 bytes, and a whole-height
    // tile gives every thread the same row count.  Measured on fp16 24577 x
    // 16383 with 128 x 64 tiles: 5.49 -> 6.19 TB/s; for one strip at a time
    // (at the register limit) the general form was 2 % faster.
    const int mine_full = active && g < p.tile_m ? (p.tile_m - g + tpc - 1) / tpc : 0;
    const uint32_t base_off = chunk_offset(g, q, p.box_stride);
    const uint32_t row_step = static_cast<uint32_t>(tpc) * kBoxRowBytes;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    // The launch picks GMAX = p.col_group, so the group width is a constant here.
    ColPos c = col_pos(first, p.tiles_m, p.tiles_n, GMAX);
    for (int64_t j = 0; j < count; ++j, col_next(c, p.tiles_m, p.tiles_n, GMAX)) {
        const int64_t tile = first + j;
        if (c.gstart != group) {
            if (group >= 0 && !post_group<EPC, GMAX>(a.tile_n, group, acc, active, q, g, ring,
                                                     slot_floats, fr, w, ctid)) {
                ok = false;
                break;
            }
            group = c.gstart;
#pragma unroll
            for (int k = 0; k < GMAX; ++k)
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[k][e] = 0.f;
        }
        const uint32_t full_bar = sm.full0 + 8u * stage;
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
        if (ctid == 0) log_record(p, 1, j, stage, phase, tile);
        // Rows of this tile inside the matrix (the copy engine zero-fills the
        // rest; skipping them saves the reads).
        const int64_t left = p.M - static_cast<int64_t>(c.band) * p.tile_m;
        const int rows = left < p.tile_m ? static_cast<int>(left) : p.tile_m;
        int mine;
        if constexpr (GMAX == 2)
            mine = rows == p.tile_m ? mine_full : (active && g < rows ? (rows - g + tpc - 1) / tpc : 0);
        else
            mine = active && g < rows ? (rows - g + tpc - 1) / tpc : 0;
        const uint32_t rbase = sm.base + stage * p.stage_stride;
        for (int r = 0; r < rounds; ++r) {
            uint4 v[CV];
#pragma unroll
            for (int u = 0; u < CV; ++u) {
                const int k = r * CV + u;
                if (k < mine) {
                    if constexpr (GMAX == 2)
                        v[u] = lds128(rbase + base_off + k * row_step);
                    else
                        v[u] = lds128(rbase + chunk_offset(g + k * tpc, q, p.box_stride));
                }
            }
            if (r == rounds - 1) {
                __syncwarp();
                if (lane == 0 && p.fault != 2) mbar_arrive(sm.empty0 + 8u * stage);
            }
            // The strip's accumulators, selected without indexing registers
            // by a run-time value.
#pragma unroll
            for (int s = 0; s < GMAX; ++s) {
                if (s != c.kloc) continue;
#pragma unroll
                for (int u = 0; u < CV; ++u) {
                    const int k = r * CV + u;
                    if (k < mine) chunk_accumulate<DT>(acc[s], v[u]);
                }
            }
        }
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (ok && group >= 0)
        ok = post_group<EPC, GMAX>(a.tile_n, group, acc, active, q, g, ring, slot_floats, fr,
                                   w, ctid);
    if (ok)   // the end mark for the flush warp
        post_group<EPC, GMAX>(a.tile_n, -1, acc, active, q, g, ring, slot_floats, fr, w, ctid);
}

// WIDE: up to 16 consumer warps, one CTA per SM.
template <int DT, int GMAX, bool WIDE = false>
__global__ void __launch_bounds__(WIDE ? kMaxWideThreads : kMaxThreads + 32, WIDE ? 1 : 2)
    mbt_colsum_kernel(const __grid_constant__ CUtensorMap map, const ColsumArgs a) {
    extern __shared__ __align__(1024) unsigned char dyn_smem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
    __shared__ __align__(8) uint64_t ring_bars[2 * kColsumRingSlots];   // flush ring: full, empty
    __shared__ int64_t ring_key[kColsumRingSlots];
    __shared__ int abort_flag;
    Smem sm;
    FlushRing fr{smem_u32(&ring_bars[0]), smem_u32(&ring_bars[kColsumRingSlots]), 0u, ring_key};
    if (threadIdx.x == 0) {
        for (int k = 0; k < kColsumRingSlots; ++k) {
            mbar_init(fr.full0 + 8u * k, static_cast<uint32_t>(a.p.consumer_warps));
            mbar_init(fr.empty0 + 8u * k, 1);
        }
    }
    init_pipeline(a.p, sm, bars, &abort_flag, dyn_smem);   // fences the inits
    clear_next_tickets(a.clear_ticket, a.clear_n);
    WaitCtl w{a.p.wait_budget_ns, &abort_flag, status_of(a.p)};
    // The flush ring's slots, after the stages (the host sized the dynamic
    // shared memory for them: colsum_ring_bytes).
    constexpr int EPC = DT == MBT_F32 ? 4 : 8;
    const int slot_floats = 32 * a.p.consumer_warps * EPC * GMAX;
    float *ring = reinterpret_cast<float *>(dyn_smem + (sm.base - smem_u32(dyn_smem)) +
                                            a.p.stages * a.p.stage_stride);
    // Contiguous, evenly split range of scheduling units, in strip-major order.
    const int64_t G = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t first = (b * a.units / G) * a.gran;
    const int64_t last = ((b + 1) * a.units / G) * a.gran;
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) produce(&map, a.p, sm, w, first, 1, last - first);
        return;
    }
    if (threadIdx.x < 64) {
        colsum_flush_warp<GMAX>(a, ring, slot_floats, a.p.consumer_warps * 32 / (a.p.boxes * 8),
                                fr, w);
        return;
    }
    consume_colsum<DT, GMAX>(a, sm, w, first, last - first, ring, slot_floats, fr);
}
