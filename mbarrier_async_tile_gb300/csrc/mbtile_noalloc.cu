// tile_rowsum_noalloc: the row sum for callers that cannot allocate device
// memory.  The band-split workspace that tile_rowsum_ex takes from its caller
// lives here instead, in a fixed-size array of the library's own.
#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// One copy per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MBT_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void *g_scratch_address[kMaxDevices];

// Device address of the array on the current device.  In host code the
// array's name only stands for it, so the address comes from the runtime,
// once per device, with that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MBT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MBT_ERR_CUDA;
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return MBT_OK;
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
        if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return MBT_ERR_CUDA;
        o.workspace = scratch;
        o.workspace_bytes = MBT_NOALLOC_SCRATCH_BYTES;
    }
    return tile_rowsum_ex(src, out, M, N, tile_m, tile_n, stages, dtype, stream, &o);
}
