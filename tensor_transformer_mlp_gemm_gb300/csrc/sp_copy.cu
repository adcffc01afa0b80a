// sp_copy.cu -- explicit sequence-parallel gather and scatter of token chunks
// (declared in include/tpmlp.h).
//
// "Megatron-LM：NVIDIA 的大规模并行训练方案", "并行训练范式 / 序列并行": with
// sequence parallelism each rank holds a chunk of the sequence; the tensor-
// parallel block gathers the chunks before its column-parallel GEMM and
// reduce-scatters its output to chunks after the row-parallel GEMM.  The
// block's own calls do both without copies (one TMA tensor map per chunk, an
// epilogue that writes each row into its chunk).  These calls make the copies
// explicit, for callers that want the gathered tensor itself and to measure
// what addressing the chunks saves: gather = concatenation of the t chunks
// along tokens, scatter = the split of a [T, cols] tensor into them.
#include <cuda_runtime.h>

#include <cstdint>

#include "abi_internal.h"
#include "tpmlp.h"

#define TPMLP_API extern "C" __attribute__((visibility("default")))

namespace tpmlp {
namespace {

constexpr int kCopyMaxChunks = 8;

struct ChunkCopy {
    const void* src[kCopyMaxChunks];  // gather: the chunks; scatter: [0] = the whole tensor
    void* dst[kCopyMaxChunks];        // gather: [0] = the whole tensor; scatter: the chunks
    long long rows_per_chunk;
    long long vec_per_row;            // 16-byte vectors per row (cols / 8)
    long long total;                  // vectors in the [T, cols] tensor
    int gather;
};

// One 16-byte vector per thread and grid-stride step: vector v of the whole
// tensor is row v / vec_per_row, which lies in chunk row / rows_per_chunk.
__global__ void __launch_bounds__(256) chunk_copy_kernel(const ChunkCopy c) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < c.total;
         v += stride) {
        const long long row = v / c.vec_per_row;
        const int j = static_cast<int>(row / c.rows_per_chunk);
        const long long local = v - static_cast<long long>(j) * c.rows_per_chunk * c.vec_per_row;
        if (c.gather) {
            const uint4 x = __ldg(static_cast<const uint4*>(c.src[j]) + local);
            static_cast<uint4*>(c.dst[0])[v] = x;
        } else {
            const uint4 x = __ldg(static_cast<const uint4*>(c.src[0]) + v);
            static_cast<uint4*>(c.dst[j])[local] = x;
        }
    }
}

tpmlp_status chunk_copy(const tpmlp_dims* dims, int64_t cols, const void* const* chunks_in,
                        void* const* chunks_out, const void* whole_in, void* whole_out,
                        bool gather, cudaStream_t st) {
    if (!dims || cols <= 0 || dims->tokens < 0 || dims->seq_chunks <= 0) return TPMLP_ERR_INVALID_ARG;
    if (dims->seq_chunks > kCopyMaxChunks) return TPMLP_ERR_UNSUPPORTED;
    if (dims->tokens % dims->seq_chunks != 0) return TPMLP_ERR_INVALID_ARG;
    if (cols % 8 != 0) return TPMLP_ERR_UNSUPPORTED;
    const int n = dims->seq_chunks;
    ChunkCopy c{};
    if (gather) {
        TPMLP_TRY(abi::check_ptrs(chunks_in, n));
        TPMLP_TRY(abi::check_ptr(whole_out));
        for (int j = 0; j < n; ++j) c.src[j] = chunks_in[j];
        c.dst[0] = whole_out;
    } else {
        TPMLP_TRY(abi::check_ptrs(reinterpret_cast<const void* const*>(chunks_out), n));
        TPMLP_TRY(abi::check_ptr(whole_in));
        for (int j = 0; j < n; ++j) c.dst[j] = chunks_out[j];
        c.src[0] = whole_in;
    }
    abi::DeviceInfo* dev = nullptr;
    TPMLP_TRY(abi::device_info(&dev));
    if (dims->tokens == 0) return TPMLP_OK;
    c.rows_per_chunk = dims->tokens / n;
    c.vec_per_row = cols / 8;
    c.total = static_cast<long long>(dims->tokens) * c.vec_per_row;
    c.gather = gather ? 1 : 0;
    // a few CTAs per SM, each looping over the tensor
    const long long want = (c.total + 255) / 256;
    const long long cap = static_cast<long long>(dev->sm_count) * 8;
    const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
    TPMLP_CUDA(abi::timed(TPMLP_KERNEL_SP_COPY, 1, st, [&] {
        chunk_copy_kernel<<<blocks, 256, 0, st>>>(c);
        return cudaGetLastError();
    }));
    return TPMLP_OK;
}

}  // namespace
}  // namespace tpmlp

TPMLP_API tpmlp_status tpmlp_sp_gather(const tpmlp_dims* dims, const void* const* chunks,
                                       int64_t cols, void* out, void* stream) {
    return tpmlp::chunk_copy(dims, cols, chunks, nullptr, nullptr, out, true,
                             static_cast<cudaStream_t>(stream));
}

TPMLP_API tpmlp_status tpmlp_sp_scatter(const tpmlp_dims* dims, const void* in, int64_t cols,
                                        void* const* chunks, void* stream) {
    return tpmlp::chunk_copy(dims, cols, nullptr, chunks, in, nullptr, false,
                             static_cast<cudaStream_t>(stream));
}
