// Host-buffer forms of tile_copy, tile_rowsum and tile_colsum: the matrix
// lives in host memory, the library moves it through the device in row slabs.
//
// Each call takes a staging set from a per-device pool: kSlots slab-sized
// device buffers plus three streams (host-to-device copies, kernels,
// device-to-host copies) and per-slot events.  Slab k is copied in on the
// first stream, processed by the device entry point on the second once its
// copy has landed, and copied out on the third once the kernel is done; slot
// k mod kSlots is refilled only after slab k - kSlots has left the device.
// With pinned host memory the copy-in of slab k + 1 therefore overlaps the
// kernel and the copy-out of slab k, and the link carries both directions at
// once.  The slabs are repacked on the device with a 16-byte row pitch, so the
// 2-D bulk tensor copies of the pipeline apply whatever the host pitch is.
//
// The operations are those of tile_copy_ex / tile_rowsum_ex / tile_colsum_ex
// (see mbtile.h); this file schedules copies and calls those entry points, and
// for column sums adds the slabs' sums on the device in slab order.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <memory>
#include <mutex>
#include <vector>

#include "internal.h"

namespace {

constexpr int kSlots = 3;
constexpr int64_t kSlabBytes = MBT_HOST_SLAB_BYTES;
constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int esize_of(int dtype) {
    return dtype == MBT_F16 || dtype == MBT_BF16 ? 2 : dtype == MBT_F32 ? 4 : 0;
}

struct Staging {
    int device = -1;
    bool busy = false;
    char *base = nullptr;
    size_t bytes = 0;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t in[kSlots] = {}, kdone[kSlots] = {}, out[kSlots] = {};

    int create(int dev) {
        device = dev;
        const unsigned f = cudaStreamNonBlocking;
        if (cudaStreamCreateWithFlags(&h2d, f) != cudaSuccess ||
            cudaStreamCreateWithFlags(&comp, f) != cudaSuccess ||
            cudaStreamCreateWithFlags(&d2h, f) != cudaSuccess)
            return MBT_ERR_CUDA;
        for (int s = 0; s < kSlots; ++s)
            if (cudaEventCreateWithFlags(&in[s], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&kdone[s], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&out[s], cudaEventDisableTiming) != cudaSuccess)
                return MBT_ERR_CUDA;
        return MBT_OK;
    }

    // Device memory of at least `need` bytes (grown, never shrunk).
    int reserve(size_t need) {
        if (bytes >= need) return MBT_OK;
        if (base != nullptr) {
            cudaFree(base);
            base = nullptr;
            bytes = 0;
        }
        if (cudaMalloc(&base, need) != cudaSuccess) {
            cudaGetLastError();
            return MBT_ERR_CUDA;
        }
        bytes = need;
        return MBT_OK;
    }

    void destroy() {
        if (base) cudaFree(base);
        for (int s = 0; s < kSlots; ++s) {
            if (in[s]) cudaEventDestroy(in[s]);
            if (kdone[s]) cudaEventDestroy(kdone[s]);
            if (out[s]) cudaEventDestroy(out[s]);
        }
        if (h2d) cudaStreamDestroy(h2d);
        if (comp) cudaStreamDestroy(comp);
        if (d2h) cudaStreamDestroy(d2h);
        *this = Staging{};
    }
};

std::mutex g_pool_mutex;
std::vector<std::unique_ptr<Staging>> g_pool;

// A free staging set of the current device with at least `need` bytes.
int acquire(size_t need, Staging **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MBT_ERR_CUDA;
    Staging *st = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_pool_mutex);
        for (auto &s : g_pool)
            if (!s->busy && s->device == dev && (st == nullptr || s->bytes > st->bytes))
                st = s.get();
        if (st == nullptr) {
            g_pool.push_back(std::make_unique<Staging>());
            st = g_pool.back().get();
            st->device = dev;
        }
        st->busy = true;
    }
    int rc = st->h2d == nullptr ? st->create(dev) : MBT_OK;
    if (rc == MBT_OK) rc = st->reserve(need);
    if (rc != MBT_OK) {
        std::lock_guard<std::mutex> lock(g_pool_mutex);
        st->busy = false;
        return rc;
    }
    *out = st;
    return MBT_OK;
}

void release(Staging *st) {
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    st->busy = false;
}

mbt_opts opts_or_default(const mbt_opts *opts) {
    mbt_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts) o = *opts;
    return o;
}

// op: MBT_OP_COPY (src -> dst), MBT_OP_ROWSUM (out[M]) or MBT_OP_COLSUM
// (out[N]: each slab's column sums, added on the device in slab order).
int host_run(int op, const void *src, void *dst, float *out, int64_t M, int64_t N, int tile_m,
             int tile_n, int stages, int dtype, const mbt_opts *opts) {
    const mbt_opts o = opts_or_default(opts);
    const int es = esize_of(dtype);
    const bool is_copy = op == MBT_OP_COPY, cols = op == MBT_OP_COLSUM;
    if (es == 0 || M < 0 || N < 0) return MBT_ERR_ARG;
    // Device-side options that the slab schedule owns.
    if (o.log != nullptr || o.workspace != nullptr || o.workspace_bytes != 0 ||
        o.status != nullptr)
        return MBT_ERR_ARG;
    const int64_t ld_src = o.ld_src ? o.ld_src : N;
    const int64_t ld_dst = o.ld_dst ? o.ld_dst : N;
    if (ld_src < N || ld_dst < N || (!is_copy && o.ld_dst != 0)) return MBT_ERR_ARG;
    if (o.host_slab_rows < 0) return MBT_ERR_ARG;
    const int64_t nsums = cols ? N : M;
    if (!is_copy && nsums > 0 && out == nullptr) return MBT_ERR_ARG;
    if (M == 0 || N == 0) {   // nothing to read: no copy, zero sums
        if (!is_copy) std::fill(out, out + nsums, 0.f);
        return MBT_OK;
    }
    if (src == nullptr || (is_copy && dst == nullptr)) return MBT_ERR_ARG;
    const size_t row_bytes = static_cast<size_t>(N) * es;
    const size_t dpitch = round_up(row_bytes, 16);
    int64_t R = o.host_slab_rows;
    if (R == 0) {
        R = std::max<int64_t>(1, kSlabBytes / static_cast<int64_t>(dpitch));
        if (R >= tile_m && tile_m > 0) R -= R % tile_m;   // whole row bands per slab
    }
    R = std::min(R, M);

    // Shape and option checks of the device call on one slab, before any copy
    // (host-only planning; the shared-memory limit is checked by the device
    // call itself, which the first slab reaches before anything is copied out).
    mbt_opts dev_o = o;
    dev_o.host_slab_rows = 0;
    dev_o.ld_src = static_cast<int64_t>(dpitch / es);
    dev_o.ld_dst = is_copy ? dev_o.ld_src : 0;
    mbt_plan plan;
    int rc = tile_plan(op, R, N, tile_m, tile_n, stages, dtype, &dev_o, 1, 1 << 30, 1, 0, &plan);
    if (rc != MBT_OK) return rc;
    // Sum workspace: the larger of what a full slab and the last slab need.
    size_t ws_bytes = 0;
    if (!is_copy) {
        const int64_t tail = M % R;
        for (int64_t rows : {R, tail}) {
            if (rows == 0) continue;
            size_t b = 0;
            rc = cols ? tile_colsum_workspace_bytes(rows, N, tile_m, tile_n, stages, dtype, &dev_o,
                                                    &b)
                      : tile_rowsum_workspace_bytes(rows, N, tile_m, tile_n, stages, dtype, &dev_o,
                                                    &b);
            if (rc != MBT_OK) return rc;
            ws_bytes = std::max(ws_bytes, b);
        }
    }
    const size_t slab_in = round_up(static_cast<size_t>(R) * dpitch, kAlign);
    const size_t slab_out =
        is_copy ? slab_in
                : round_up(static_cast<size_t>(cols ? N : R) * sizeof(float), kAlign);
    const size_t acc_bytes = cols ? round_up(static_cast<size_t>(N) * sizeof(float), kAlign) : 0;
    const size_t ws_region = round_up(ws_bytes, kAlign);
    // Layout: the call's status buffer (int32[4]), the sum workspace, the
    // column-sum accumulator, then the slab slots.
    const size_t status_region = kAlign;
    const size_t need = status_region + ws_region + acc_bytes + kSlots * (slab_in + slab_out);

    Staging *st = nullptr;
    rc = acquire(need, &st);
    if (rc != MBT_OK) return rc;
    int32_t *status = reinterpret_cast<int32_t *>(st->base);
    char *ws = st->base + status_region;
    float *acc = reinterpret_cast<float *>(ws + ws_region);
    auto slot_in = [&](int s) {
        return ws + ws_region + acc_bytes + s * (slab_in + slab_out);
    };
    auto slot_out = [&](int s) { return slot_in(s) + slab_in; };
    if (cudaMemsetAsync(st->base, 0, status_region + ws_bytes, st->comp) != cudaSuccess)
        rc = MBT_ERR_CUDA;
    dev_o.workspace = ws_bytes > 0 ? ws : nullptr;
    dev_o.workspace_bytes = ws_bytes;
    if (ws_bytes == 0 && !is_copy) dev_o.no_split = 1;   // never the library's own workspace
    dev_o.status = status;   // this call's timeouts only

    const char *hsrc = static_cast<const char *>(src);
    const size_t spitch = static_cast<size_t>(ld_src) * es;
    const size_t hdpitch = static_cast<size_t>(ld_dst) * es;
    const int64_t slabs = (M + R - 1) / R;
    for (int64_t k = 0; k < slabs && rc == MBT_OK; ++k) {
        const int s = static_cast<int>(k % kSlots);
        const int64_t r0 = k * R;
        const int64_t rows = std::min<int64_t>(R, M - r0);
        // Slot s is free once slab k - kSlots has been copied out (column
        // sums: once its kernel and the addition of its sums have run).
        if (k >= kSlots &&
            cudaStreamWaitEvent(st->h2d, cols ? st->kdone[s] : st->out[s], 0) != cudaSuccess) {
            rc = MBT_ERR_CUDA;
            break;
        }
        if (cudaMemcpy2DAsync(slot_in(s), dpitch, hsrc + r0 * spitch, spitch, row_bytes,
                              static_cast<size_t>(rows), cudaMemcpyHostToDevice,
                              st->h2d) != cudaSuccess ||
            cudaEventRecord(st->in[s], st->h2d) != cudaSuccess ||
            cudaStreamWaitEvent(st->comp, st->in[s], 0) != cudaSuccess) {
            rc = MBT_ERR_CUDA;
            break;
        }
        float *sums = reinterpret_cast<float *>(slot_out(s));
        if (is_copy)
            rc = tile_copy_ex(slot_in(s), slot_out(s), rows, N, tile_m, tile_n, stages, dtype,
                              st->comp, &dev_o);
        else if (cols)
            rc = tile_colsum_ex(slot_in(s), sums, rows, N, tile_m, tile_n, stages, dtype,
                                st->comp, &dev_o);
        else
            rc = tile_rowsum_ex(slot_in(s), sums, rows, N, tile_m, tile_n, stages, dtype,
                                st->comp, &dev_o);
        if (rc != MBT_OK) break;
        if (cols && mbt::launch_accumulate(acc, sums, N, k == 0, st->comp) != cudaSuccess) {
            rc = MBT_ERR_CUDA;
            break;
        }
        if (cudaEventRecord(st->kdone[s], st->comp) != cudaSuccess) {
            rc = MBT_ERR_CUDA;
            break;
        }
        if (cols) continue;   // copied out once, after the last slab
        if (cudaStreamWaitEvent(st->d2h, st->kdone[s], 0) != cudaSuccess) {
            rc = MBT_ERR_CUDA;
            break;
        }
        const cudaError_t e =
            is_copy ? cudaMemcpy2DAsync(static_cast<char *>(dst) + r0 * hdpitch, hdpitch,
                                        slot_out(s), dpitch, row_bytes,
                                        static_cast<size_t>(rows), cudaMemcpyDeviceToHost,
                                        st->d2h)
                    : cudaMemcpyAsync(out + r0, sums, static_cast<size_t>(rows) * 4,
                                      cudaMemcpyDeviceToHost, st->d2h);
        if (e != cudaSuccess || cudaEventRecord(st->out[s], st->d2h) != cudaSuccess) {
            rc = MBT_ERR_CUDA;
            break;
        }
    }
    if (cols && rc == MBT_OK &&
        cudaMemcpyAsync(out, acc, static_cast<size_t>(N) * 4, cudaMemcpyDeviceToHost,
                        st->comp) != cudaSuccess)
        rc = MBT_ERR_CUDA;
    // Nothing may still read or write the caller's host memory after return.
    const bool synced = cudaStreamSynchronize(st->h2d) == cudaSuccess &&
                        cudaStreamSynchronize(st->comp) == cudaSuccess &&
                        cudaStreamSynchronize(st->d2h) == cudaSuccess;
    if (!synced && rc == MBT_OK) rc = MBT_ERR_CUDA;
    int32_t info[4] = {0, 0, 0, 0};
    if (cudaMemcpyAsync(info, status, sizeof info, cudaMemcpyDeviceToHost, st->comp) !=
            cudaSuccess ||
        cudaStreamSynchronize(st->comp) != cudaSuccess) {
        if (rc == MBT_OK) rc = MBT_ERR_CUDA;
    } else if (info[0] != 0 && rc == MBT_OK) {
        rc = info[0];   // MBT_ERR_TIMEOUT
    }
    release(st);
    return rc;
}

}  // namespace

extern "C" {

int tile_copy_host(const void *src, void *dst, int64_t M, int64_t N, int tile_m, int tile_n,
                   int stages, int dtype, const mbt_opts *opts) {
    return host_run(MBT_OP_COPY, src, dst, nullptr, M, N, tile_m, tile_n, stages, dtype, opts);
}

int tile_rowsum_host(const void *src, float *out, int64_t M, int64_t N, int tile_m, int tile_n,
                     int stages, int dtype, const mbt_opts *opts) {
    return host_run(MBT_OP_ROWSUM, src, nullptr, out, M, N, tile_m, tile_n, stages, dtype, opts);
}

int tile_colsum_host(const void *src, float *out, int64_t M, int64_t N, int tile_m, int tile_n,
                     int stages, int dtype, const mbt_opts *opts) {
    return host_run(MBT_OP_COLSUM, src, nullptr, out, M, N, tile_m, tile_n, stages, dtype, opts);
}

int tile_host_release(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MBT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    for (auto &s : g_pool)
        if (!s->busy && s->device == dev) s->destroy();
    g_pool.erase(std::remove_if(g_pool.begin(), g_pool.end(),
                                [](const std::unique_ptr<Staging> &s) { return s->device < 0; }),
                 g_pool.end());
    return MBT_OK;
}

}  // extern "C"
