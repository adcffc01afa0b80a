// colsum_noalloc.cu -- the bias-gradient column sum for callers that cannot
// allocate device memory.
//
// tpmlp_backward takes its column-sum scratch (per-split partial sums) from a
// workspace the caller allocates.  Some callers have no way to provide one:
// a library embedded in another runtime whose device memory belongs to that
// runtime's own pool (a cudaMalloc there bypasses its budget, and cudaFree
// synchronises the whole device), or a latency-critical loop that forbids any
// allocation once it has started.  This file gives them the same reduction
// with the scratch in a fixed, library-owned array instead.
//
// The array is a file-scope __device__ variable of kNoallocScratchFloats
// floats (4 MiB).  Every GPU that loads the library holds it until the
// process exits, and every call on that GPU shares it: calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// it.  Each call writes every partial sum it later reads, so nothing in the
// array needs to start at zero and the previous call's contents do no harm.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "tpmlp.h"
#include "colsum.cuh"

#define TPMLP_NOALLOC_API extern "C" __attribute__((visibility("default")))

namespace tpmlp {
namespace {

constexpr long long kNoallocScratchFloats = 1LL << 20;  // 4 MiB of partial sums
constexpr int kNoallocMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoallocMaxDevices] = {};
int g_noalloc_sms[kNoallocMaxDevices] = {};

// Once per device, with that device current: the device address of the
// scratch array (the host-side name is only a stand-in, not an address the
// GPU can use), plus the SM count used to size the grid.
tpmlp_status noalloc_setup(int dev, float** scratch, int* sms) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TPMLP_ERR_CUDA;
        if (major != 10 || minor != 3) return TPMLP_ERR_UNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return TPMLP_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<float*>(p);
        g_noalloc_sms[dev] = count;
    }
    *scratch = g_noalloc_ptr[dev];
    *sms = g_noalloc_sms[dev];
    return TPMLP_OK;
}

}  // namespace
}  // namespace tpmlp

TPMLP_NOALLOC_API tpmlp_status tpmlp_column_sums_noalloc(const void* src, int64_t rows,
                                                         int64_t cols, void* out, void* stream) {
    using namespace tpmlp;
    if (!src || !out || rows < 0 || cols <= 0) return TPMLP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
        return TPMLP_ERR_UNSUPPORTED;
    if (cols % 8 != 0 || cols > kNoallocScratchFloats || rows > (int64_t(1) << 31) - 1)
        return TPMLP_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TPMLP_ERR_CUDA;
    if (dev < 0 || dev >= kNoallocMaxDevices) return TPMLP_ERR_UNSUPPORTED;
    float* scratch = nullptr;
    int sms = 0;
    const tpmlp_status s = noalloc_setup(dev, &scratch, &sms);
    if (s != TPMLP_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (rows == 0) {
        return cudaMemsetAsync(out, 0, static_cast<size_t>(cols) * sizeof(float), st) == cudaSuccess
                   ? TPMLP_OK
                   : TPMLP_ERR_CUDA;
    }
    ColsumParams c;
    std::memset(&c, 0, sizeof(c));
    c.src[0] = src;
    c.nparts = 1;
    c.rows_per_part = rows;
    c.ncols = static_cast<int>(cols);
    c.mode = CS_ROWS_CONCAT;
    c.out = static_cast<float*>(out);
    c.partial = scratch;
    dim3 grid = colsum_plan(c, sms);
    // keep the partial sums [splits][cols] inside the static array
    const long long max_splits = kNoallocScratchFloats / cols;
    if (c.splits > max_splits) {
        c.splits = static_cast<int>(max_splits);
        c.rows_per_split = (rows + c.splits - 1) / c.splits;
        grid.y = static_cast<unsigned>(c.splits);
    }
    return launch_colsum(c, grid, st, nullptr) == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}
