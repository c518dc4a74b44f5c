// tile_read_checksum: the read-bandwidth reference of the reductions.
//
// Row and column sums only read the matrix (plus a few bytes of sums), so the
// copy's read + write bandwidth is not their ceiling.  This kernel states the
// read-only one on the same device: it streams a buffer once with 16-byte
// loads and folds every 32-bit word into one XOR checksum (a result the tests
// check against the oracle; XOR is associative and commutative, so the
// grouping of the fold does not change it).  A grid of whole CTAs per SM
// strides through the buffer: consecutive threads read consecutive 16-byte
// vectors (each warp 512 contiguous bytes per load), every thread keeps
// kProbeUnroll loads in flight, and each warp's fold reaches `out` with one
// atomic XOR.
#include <mutex>

#include "internal.h"

namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 8;   // 16-byte loads in flight per thread
constexpr int kMaxDevices = 64;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kProbeThreads)
    mbt_read_checksum_kernel(const uint4 *src, int64_t n16, uint32_t *out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    uint32_t x = 0;
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) v[u] = ld_stream(src + i + u * stride);
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) x ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = ld_stream(src + i);
        x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0 && x != 0) atomicXor(out, x);
}

std::mutex g_probe_mutex;
int g_probe_grid[kMaxDevices];

// Whole CTAs per SM times the SM count, once per device.
int probe_grid(int *grid) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MBT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_probe_mutex);
    if (g_probe_grid[dev] == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mbt_read_checksum_kernel,
                                                          kProbeThreads, 0) != cudaSuccess ||
            sms < 1 || per_sm < 1)
            return MBT_ERR_CUDA;
        g_probe_grid[dev] = sms * per_sm;
    }
    *grid = g_probe_grid[dev];
    return MBT_OK;
}

}  // namespace

extern "C" int tile_read_checksum(const void *src, size_t bytes, uint32_t *out, void *stream) {
    if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 3u) != 0) return MBT_ERR_ARG;
    if (bytes > 0 && src == nullptr) return MBT_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0 || bytes % 16 != 0) return MBT_ERR_ALIGN;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(out, 0, sizeof(uint32_t), s) != cudaSuccess) return MBT_ERR_CUDA;
    if (bytes == 0) return MBT_OK;
    int grid = 0;
    const int rc = probe_grid(&grid);
    if (rc != MBT_OK) return rc;
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    const int64_t most = (n16 + kProbeThreads - 1) / kProbeThreads;
    if (most < grid) grid = static_cast<int>(most);
    mbt_read_checksum_kernel<<<grid, kProbeThreads, 0, s>>>(static_cast<const uint4 *>(src), n16,
                                                            out);
    return cudaGetLastError() == cudaSuccess ? MBT_OK : MBT_ERR_CUDA;
}
