// colsum.cu -- HBM-bound column sums for the bias gradients db1 and db2.
//
// CTA = 256 threads over a 64-column strip: thread (slot, vec) reads the
// 16-byte vector of 8 bf16 at columns vec*8.. of rows slot, slot+32, ...
// (each warp covers four full 128-byte rows per load, coalesced; eight loads
// in flight per thread), keeps 8 fp32 partial sums in registers, and the 32
// row slots are then combined in a fixed order through shared memory.  With
// row splits, a second kernel adds the per-split partial sums in split order.
// No atomics, so the result is bitwise reproducible.
#include <cuda_bf16.h>

#include "colsum.cuh"

namespace tpmlp {

__device__ __forceinline__ void add_bf16x8(const uint4& u, float (&acc)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Moves (part, local row) d rows on, parts of rpp rows each.
__device__ __forceinline__ void step_row(int& part, long long& lr, long long d, long long rpp) {
    lr += d;
    while (lr >= rpp) {
        lr -= rpp;
        ++part;
    }
}

// p.src[i] by selects (indexing the parameter array with a run-time index
// makes the compiler copy the whole parameter block to local memory per thread).
__device__ __forceinline__ const void* part_src(const ColsumParams& p, int i) {
    const void* s = p.src[0];
#pragma unroll
    for (int k = 1; k < CS_MAX_PARTS; ++k) s = i == k ? p.src[k] : s;
    return s;
}

// The 16-byte vector at columns col.. of the row d rows after (part, lr).
__device__ __forceinline__ uint4 load_row(const ColsumParams& p, int part, long long lr,
                                          long long d, long long rpp, int col) {
    step_row(part, lr, d, rpp);
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(part_src(p, part));
    return __ldg(reinterpret_cast<const uint4*>(src + lr * p.ncols + col));
}

__global__ void __launch_bounds__(CS_THREADS) colsum_kernel(const ColsumParams p) {
    __shared__ float red[32][CS_COLS + 1];
    const int vec = threadIdx.x & 7;
    const int slot = threadIdx.x >> 3;
    const int grp = blockIdx.z;
    const int col = blockIdx.x * CS_COLS + vec * 8;
    const long long total_rows =
        p.mode == CS_ROWS_CONCAT ? p.rows_per_part * p.nparts : p.rows_per_part;
    const long long r0 = static_cast<long long>(blockIdx.y) * p.rows_per_split;
    const long long r1 = min(total_rows, r0 + p.rows_per_split);

    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;

    if (col < p.ncols && r0 + slot < r1) {
        // part and local row of this thread's row, stepped without a division
        const long long rpp = p.mode == CS_ROWS_CONCAT ? p.rows_per_part : total_rows + 1;
        long long r = r0 + slot;
        int part = p.mode == CS_ROWS_CONCAT ? static_cast<int>(r / rpp) : grp;
        long long lr = p.mode == CS_ROWS_CONCAT ? r - part * rpp : r;
        // eight, then four independent loads in flight per thread, added in row order
        for (; r + 224 < r1; r += 256) {
            uint4 u[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) u[q] = load_row(p, part, lr, 32 * q, rpp, col);
#pragma unroll
            for (int q = 0; q < 8; ++q) add_bf16x8(u[q], acc);
            step_row(part, lr, 256, rpp);
        }
        for (; r + 96 < r1; r += 128) {
            uint4 u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) u[q] = load_row(p, part, lr, 32 * q, rpp, col);
#pragma unroll
            for (int q = 0; q < 4; ++q) add_bf16x8(u[q], acc);
            step_row(part, lr, 128, rpp);
        }
        for (; r < r1; r += 32) {
            add_bf16x8(load_row(p, part, lr, 0, rpp, col), acc);
            step_row(part, lr, 32, rpp);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) red[slot][vec * 8 + j] = acc[j];
    __syncthreads();
    if (threadIdx.x < CS_COLS) {
        const int c = blockIdx.x * CS_COLS + threadIdx.x;
        if (c < p.ncols) {
            float s = 0.f;
            for (int k = 0; k < 32; ++k) s += red[k][threadIdx.x];
            const long long n_out =
                p.mode == CS_ROWS_CONCAT ? p.ncols : static_cast<long long>(p.ncols) * p.nparts;
            const long long o = (p.mode == CS_COLS_CONCAT ? static_cast<long long>(grp) * p.ncols : 0) + c;
            if (p.splits == 1)
                p.out[o] = s;
            else
                p.partial[static_cast<long long>(blockIdx.y) * n_out + o] = s;
        }
    }
}

__global__ void colsum_finish_kernel(const float* __restrict__ partial, int splits,
                                     long long n_out, float* __restrict__ out) {
    const long long o = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (o >= n_out) return;
    float s = 0.f;
    for (int k = 0; k < splits; ++k) s += partial[k * n_out + o];
    out[o] = s;
}

// CTA = 16 column quads (64 columns) x 16 row lanes; lane r sums rows r,
// r + 16, ... of its four columns with 16-byte loads (eight in flight, added
// in row order), then the 16 lanes are combined in a fixed order.  Column
// c < split goes to out0[c], the others to out1[c - split].
__global__ void __launch_bounds__(256) colsum_f32_kernel(const float* __restrict__ part,
                                                         long long rows, long long ld,
                                                         long long ncols, long long split,
                                                         float* __restrict__ out0,
                                                         float* __restrict__ out1) {
    __shared__ float4 red[16][16];
    const int quad = threadIdx.x & 15;
    const int lane_r = threadIdx.x >> 4;
    const long long c = (static_cast<long long>(blockIdx.x) * 16 + quad) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < ncols) {
        auto add = [&](const float4& v) {
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        };
        long long r = lane_r;
        for (; r + 7 * 16 < rows; r += 8 * 16) {
            float4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = __ldg(reinterpret_cast<const float4*>(part + (r + 16 * k) * ld + c));
#pragma unroll
            for (int k = 0; k < 8; ++k) add(v[k]);
        }
        for (; r < rows; r += 16) add(__ldg(reinterpret_cast<const float4*>(part + r * ld + c)));
    }
    red[lane_r][quad] = acc;
    __syncthreads();
    if (lane_r == 0 && c < ncols) {
        float4 s = red[0][quad];
        for (int k = 1; k < 16; ++k) {
            const float4 v = red[k][quad];
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        *reinterpret_cast<float4*>(c < split ? out0 + c : out1 + (c - split)) = s;
    }
}

cudaError_t launch_colsum_f32(const float* part, long long rows, long long ld, long long ncols,
                              float* out, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((ncols + 63) / 64);
    if (blocks == 0) return cudaSuccess;
    colsum_f32_kernel<<<blocks, 256, 0, stream>>>(part, rows, ld, ncols, ncols, out, out);
    return cudaGetLastError();
}

cudaError_t launch_colsum_f32_pair(const float* part, long long rows, long long ld,
                                   long long ncols, float* out0, float* out1,
                                   cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((2 * ncols + 63) / 64);
    if (blocks == 0) return cudaSuccess;
    colsum_f32_kernel<<<blocks, 256, 0, stream>>>(part, rows, ld, 2 * ncols, ncols, out0, out1);
    return cudaGetLastError();
}

dim3 colsum_plan(ColsumParams& p, int sm_count) {
    const int strips = (p.ncols + CS_COLS - 1) / CS_COLS;
    const int groups = p.mode == CS_COLS_CONCAT ? p.nparts : 1;
    const long long total_rows =
        p.mode == CS_ROWS_CONCAT ? p.rows_per_part * p.nparts : p.rows_per_part;
    const long long base = static_cast<long long>(strips) * groups;
    // about four CTAs per SM (one wave), at least 256 rows (eight per thread)
    // each, so every thread keeps eight loads in flight
    long long splits = (4LL * sm_count + base - 1) / base;
    const long long max_by_rows = total_rows / 256 > 0 ? total_rows / 256 : 1;
    if (splits > max_by_rows) splits = max_by_rows;
    if (splits > CS_MAX_SPLITS) splits = CS_MAX_SPLITS;
    if (splits < 1) splits = 1;
    p.splits = static_cast<int>(splits);
    p.rows_per_split = (total_rows + splits - 1) / splits;
    if (p.rows_per_split < 1) p.rows_per_split = 1;
    return dim3(strips, p.splits, groups);
}

cudaError_t launch_colsum(const ColsumParams& p, dim3 grid, cudaStream_t stream, int* launches) {
    colsum_kernel<<<grid, CS_THREADS, 0, stream>>>(p);
    int n = 1;
    if (p.splits > 1) {
        const long long n_out =
            p.mode == CS_ROWS_CONCAT ? p.ncols : static_cast<long long>(p.ncols) * p.nparts;
        const int threads = 256;
        const unsigned blocks = static_cast<unsigned>((n_out + threads - 1) / threads);
        colsum_finish_kernel<<<blocks, threads, 0, stream>>>(p.partial, p.splits, n_out, p.out);
        ++n;
    }
    if (launches) *launches = n;
    return cudaGetLastError();
}

}  // namespace tpmlp
