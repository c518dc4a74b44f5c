// tile_rowsum_noalloc: the row sum for callers that cannot allocate device
// memory.  The band-split workspace that tile_rowsum_ex takes from its caller
// lives here instead, in a fixed-size array of the library's own.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// One copy per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MBT_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
struct ScratchAddress {
    void *ptr = nullptr;
    unsigned long long ctx_id = 0;   // context the address belongs to
};
ScratchAddress g_scratch_address[kMaxDevices];
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// Unique id of the current context (never reused within a process), 0 if
// the driver does not tell.  cudaDeviceReset destroys the device's context;
// the array then lives at a new address in the next one.
unsigned long long current_context_id() {
    if (g_ctx_current == nullptr || g_ctx_id == nullptr) {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa{}, qb{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault,
                                             &qa) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess ||
            qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || g_ctx_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the array on the current device.  In host code the
// array's name only stands for it, so the address comes from the runtime,
// once per device (and again if the device's context was rebuilt), with that
// device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MBT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddress &a = g_scratch_address[dev];
    if (a.ptr == nullptr || a.ctx_id == 0 || a.ctx_id != current_context_id()) {
        void *p = nullptr;
        // (creates the device's context if there is none yet)
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            a.ptr = nullptr;
            return MBT_ERR_CUDA;
        }
        a.ptr = p;
        a.ctx_id = current_context_id();
    }
    *out = a.ptr;
    return MBT_OK;
}

// A failed call drops the cached address: the next call looks it up again.
void forget_scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    g_scratch_address[dev].ptr = nullptr;
}

}  // namespace

extern "C" int tile_rowsum_noalloc(const void *src, float *out, int64_t M, int64_t N,
                                   int tile_m, int tile_n, int stages, int dtype, void *stream,
                                   const mbt_opts *opts) {
    mbt_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts) o = *opts;
    if (o.workspace != nullptr || o.workspace_bytes != 0) return MBT_ERR_ARG;
    size_t need = 0;
    int rc = tile_rowsum_workspace_bytes(M, N, tile_m, tile_n, stages, dtype, &o, &need);
    if (rc != MBT_OK) return rc;
    if (need > MBT_NOALLOC_SCRATCH_BYTES) return MBT_ERR_WORKSPACE;
    if (need > 0) {
        void *scratch = nullptr;
        rc = scratch_address(&scratch);
        if (rc != MBT_OK) return rc;
        // The array keeps whatever the previous call left; the band tickets
        // and partial sums must start at zero.
        if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
            forget_scratch_address();
            return MBT_ERR_CUDA;
        }
        o.workspace = scratch;
        o.workspace_bytes = MBT_NOALLOC_SCRATCH_BYTES;
    }
    rc = tile_rowsum_ex(src, out, M, N, tile_m, tile_n, stages, dtype, stream, &o);
    if (rc == MBT_ERR_CUDA) forget_scratch_address();
    return rc;
}
