// layernorm.cu -- LayerNorm forward/backward and dropout backward of the
// sequence-parallel sublayer (see layernorm.cuh).  One CTA of 256 threads per
// token row in the forward pass and in the dX pass of the backward; each
// thread holds up to eight 8-element vectors of its row in registers, so every
// input is read once and every output written once.  dgamma and dbeta come
// from a separate column-reduction pass over dXn and X.
// Reductions run warp-shuffle then one warp over the partial sums, always in
// the same order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "layernorm.cuh"

namespace tpmlp {
namespace {

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the CTA's LN_THREADS threads; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
    constexpr int W = LN_THREADS / 32;
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();  // the previous call's result has been read
    if (l == 0) red[w] = v;
    __syncthreads();
    if (w == 0) {
        float t = l < W ? red[l] : 0.0f;
        t = warp_sum(t);
        if (l == 0) red[W] = t;
    }
    __syncthreads();
    return red[W];
}

// Token row r lives in chunk r / rows at local row r % rows.
__device__ __forceinline__ long long chunk_row(long long r, long long rows, int& j) {
    j = static_cast<int>(r / rows);
    return r - static_cast<long long>(j) * rows;
}

// VEC = 8-element vectors per thread (h <= VEC * 8 * LN_THREADS): the row's
// registers are sized to the row, so narrow rows keep more CTAs per SM.
template <int VEC>
__global__ void __launch_bounds__(LN_THREADS) ln_forward_kernel(const LnForwardParams p) {
    __shared__ float red[LN_THREADS / 32 + 1];
    const long long r = blockIdx.x;
    int j;
    const long long rr = chunk_row(r, p.x.rows, j);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x.in[j]) + rr * p.h;
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y[j]) + rr * p.h;
    uint4 v[VEC];
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        if (c < p.h) {
            v[i] = *reinterpret_cast<const uint4*>(x + c);
            float f[8];
            unpack8(v[i], f);
#pragma unroll
            for (int k = 0; k < 8; ++k) s += f[k];
        }
    }
    const float mean = block_sum(s, red) / static_cast<float>(p.h);
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        if (c < p.h) {
            float f[8];
            unpack8(v[i], f);
#pragma unroll
            for (int k = 0; k < 8; ++k) q += (f[k] - mean) * (f[k] - mean);
        }
    }
    const float var = block_sum(q, red) / static_cast<float>(p.h);
    const float rs = 1.0f / sqrtf(var + p.eps);
    const __nv_bfloat16* gm = static_cast<const __nv_bfloat16*>(p.gamma);
    const __nv_bfloat16* bt = static_cast<const __nv_bfloat16*>(p.beta);
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        if (c < p.h) {
            float f[8], g[8], b[8], o[8];
            unpack8(v[i], f);
            unpack8(__ldg(reinterpret_cast<const uint4*>(gm + c)), g);
            unpack8(__ldg(reinterpret_cast<const uint4*>(bt + c)), b);
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = (f[k] - mean) * rs * g[k] + b[k];
            *reinterpret_cast<uint4*>(y + c) = pack8(o);
        }
    }
    if (threadIdx.x == 0) {
        p.mean[r] = mean;
        p.rstd[r] = rs;
    }
}

// grid (T, ceil(h / 8 / LN_THREADS)): one 8-element vector per thread
__global__ void __launch_bounds__(LN_THREADS) dropout_backward_kernel(const DropoutBackwardParams p) {
    const long long r = blockIdx.x;
    const int c = (blockIdx.y * LN_THREADS + threadIdx.x) * 8;
    if (c >= p.h) return;
    int j;
    const long long rr = chunk_row(r, p.dout.rows, j);
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.dout.in[j]) + rr * p.h + c;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.dz[j]) + rr * p.h + c;
    const uint64_t e0 = static_cast<uint64_t>(r) * static_cast<uint64_t>(p.h) +
                        static_cast<uint64_t>(c);  // a multiple of 8
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(src), f);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const PhiloxOut o = philox4x32_10(p.drop.offset + e0 / 4 + q, p.drop.seed);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const bool keep = static_cast<uint64_t>(o.w[k]) < p.drop.thresh;
            f[4 * q + k] = keep ? f[4 * q + k] * p.drop.scale : 0.0f;
        }
    }
    *reinterpret_cast<uint4*>(dst) = pack8(f);
}

// Sum of two values over the CTA in one pass (both orders fixed).
__device__ __forceinline__ float2 block_sum2(float a, float b, float* red) {
    constexpr int W = LN_THREADS / 32;
    a = warp_sum(a);
    b = warp_sum(b);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) {
        red[w] = a;
        red[W + w] = b;
    }
    __syncthreads();
    if (w == 0) {
        float ta = l < W ? red[l] : 0.0f, tb = l < W ? red[W + l] : 0.0f;
        ta = warp_sum(ta);
        tb = warp_sum(tb);
        if (l == 0) {
            red[2 * W] = ta;
            red[2 * W + 1] = tb;
        }
    }
    __syncthreads();
    return make_float2(red[2 * W], red[2 * W + 1]);
}

// dX of one token row per CTA:
//   dX = rstd * (g - mean(g) - xhat * mean(g * xhat)) + dres,  g = dXn * gamma
template <int VEC>
__global__ void __launch_bounds__(LN_THREADS) ln_dx_kernel(const LnBackwardParams p) {
    __shared__ float red[2 * (LN_THREADS / 32) + 2];
    const int h = p.h;
    const long long r = blockIdx.x;
    int j;
    const long long off = chunk_row(r, p.x.rows, j) * h;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x.in[j]) + off;
    const __nv_bfloat16* dy = static_cast<const __nv_bfloat16*>(p.dxn[j]) + off;
    const __nv_bfloat16* dres = static_cast<const __nv_bfloat16*>(p.dres[j]) + off;
    __nv_bfloat16* dx = static_cast<__nv_bfloat16*>(p.dx[j]) + off;
    const __nv_bfloat16* gm = static_cast<const __nv_bfloat16*>(p.gamma);
    const float mean = p.mean[r], rs = p.rstd[r];
    uint4 xv[VEC], dv[VEC];
    float sg = 0.0f, sgx = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        if (c < h) {
            xv[i] = *reinterpret_cast<const uint4*>(x + c);
            dv[i] = *reinterpret_cast<const uint4*>(dy + c);
        }
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        if (c < h) {
            float xf[8], df[8], gf[8];
            unpack8(xv[i], xf);
            unpack8(dv[i], df);
            unpack8(__ldg(reinterpret_cast<const uint4*>(gm + c)), gf);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float g = df[k] * gf[k];
                sg += g;
                sgx += g * (xf[k] - mean) * rs;
            }
        }
    }
    const float2 sums = block_sum2(sg, sgx, red);
    const float mg = sums.x / static_cast<float>(h), mgx = sums.y / static_cast<float>(h);
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        if (c < h) {
            float xf[8], df[8], gf[8], rf[8], o[8];
            unpack8(xv[i], xf);
            unpack8(dv[i], df);
            unpack8(*reinterpret_cast<const uint4*>(dres + c), rf);
            unpack8(__ldg(reinterpret_cast<const uint4*>(gm + c)), gf);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                o[k] = rs * (df[k] * gf[k] - mg - (xf[k] - mean) * rs * mgx) + rf[k];
            *reinterpret_cast<uint4*>(dx + c) = pack8(o);
        }
    }
}

// dgamma / dbeta partial column sums: CTA = a 64-column strip x 32 row slots
// over the rows of split blockIdx.y; thread (slot, vec) accumulates columns
// vec*8 .. vec*8+7 of rows slot, slot + 32, ...; the slots are then added in
// order through shared memory.  part[split][0][c] = sum dXn * xhat,
// part[split][1][c] = sum dXn.
__global__ void __launch_bounds__(LN_THREADS) ln_param_grad_kernel(const LnBackwardParams p,
                                                                   long long T) {
    constexpr int COLS = 64;
    __shared__ float red[2][32][COLS + 1];
    const int h = p.h;
    const int vec = threadIdx.x & 7, slot = threadIdx.x >> 3;
    const int col = blockIdx.x * COLS + vec * 8;
    const long long r0 = static_cast<long long>(blockIdx.y) * p.rows_per_block;
    const long long r1 = r0 + p.rows_per_block < T ? r0 + p.rows_per_block : T;
    float ag[8], ab[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) ag[k] = ab[k] = 0.0f;
    if (col < h) {
        for (long long r = r0 + slot; r < r1; r += 32) {
            int j;
            const long long off = chunk_row(r, p.x.rows, j) * h + col;
            float xf[8], df[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(
                        static_cast<const __nv_bfloat16*>(p.x.in[j]) + off)), xf);
            unpack8(__ldg(reinterpret_cast<const uint4*>(
                        static_cast<const __nv_bfloat16*>(p.dxn[j]) + off)), df);
            const float mean = __ldg(p.mean + r), rs = __ldg(p.rstd + r);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                ag[k] += df[k] * ((xf[k] - mean) * rs);
                ab[k] += df[k];
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        red[0][slot][vec * 8 + k] = ag[k];
        red[1][slot][vec * 8 + k] = ab[k];
    }
    __syncthreads();
    if (threadIdx.x < 2 * COLS) {
        const int which = threadIdx.x / COLS, cc = threadIdx.x % COLS;
        const int c = blockIdx.x * COLS + cc;
        if (c < h) {
            float s = 0.0f;
            for (int k = 0; k < 32; ++k) s += red[which][k][cc];
            p.part[(static_cast<size_t>(blockIdx.y) * 2 + which) * h + c] = s;
        }
    }
}

// dgamma[c] = sum_b part[b][0][c], dbeta[c] = sum_b part[b][1][c], b in order
__global__ void ln_finish_kernel(const float* part, int splits, int h, float* dgamma,
                                 float* dbeta) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= h) return;
    float g = 0.0f, b = 0.0f;
    for (int k = 0; k < splits; ++k) {
        g += part[static_cast<size_t>(k) * 2 * h + c];
        b += part[static_cast<size_t>(k) * 2 * h + h + c];
    }
    dgamma[c] = g;
    dbeta[c] = b;
}

// Vectors per thread for rows of h elements: the smallest of 1, 2, 4, 8 that covers h.
int ln_vec(int h) {
    const int v = (h + 8 * LN_THREADS - 1) / (8 * LN_THREADS);
    return v <= 1 ? 1 : v <= 2 ? 2 : v <= 4 ? 4 : 8;
}

}  // namespace

cudaError_t launch_ln_forward(const LnForwardParams& p, long long T, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>(T);
    switch (ln_vec(p.h)) {
        case 1: ln_forward_kernel<1><<<grid, LN_THREADS, 0, st>>>(p); break;
        case 2: ln_forward_kernel<2><<<grid, LN_THREADS, 0, st>>>(p); break;
        case 4: ln_forward_kernel<4><<<grid, LN_THREADS, 0, st>>>(p); break;
        default: ln_forward_kernel<8><<<grid, LN_THREADS, 0, st>>>(p); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_dropout_backward(const DropoutBackwardParams& p, long long T, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const int vecs = (p.h + 7) / 8;
    const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>((vecs + LN_THREADS - 1) / LN_THREADS));
    dropout_backward_kernel<<<grid, LN_THREADS, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_ln_backward(const LnBackwardParams& p, long long T, int splits, float* dgamma,
                               float* dbeta, cudaStream_t st) {
    if (T > 0) {
        const unsigned grid = static_cast<unsigned>(T);
        switch (ln_vec(p.h)) {
            case 1: ln_dx_kernel<1><<<grid, LN_THREADS, 0, st>>>(p); break;
            case 2: ln_dx_kernel<2><<<grid, LN_THREADS, 0, st>>>(p); break;
            case 4: ln_dx_kernel<4><<<grid, LN_THREADS, 0, st>>>(p); break;
            default: ln_dx_kernel<8><<<grid, LN_THREADS, 0, st>>>(p); break;
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>((p.h + 63) / 64), static_cast<unsigned>(splits));
    ln_param_grad_kernel<<<grid, LN_THREADS, 0, st>>>(p, T);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ln_finish_kernel<<<(p.h + 255) / 256, 256, 0, st>>>(p.part, splits, p.h, dgamma, dbeta);
    return cudaGetLastError();
}

}  // namespace tpmlp
