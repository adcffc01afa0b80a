// layernorm.cu -- LayerNorm forward/backward and dropout backward of the
// sequence-parallel sublayer (see layernorm.cuh).  The forward pass runs one
// warp per token row for rows of up to 4096 elements and one CTA of 256
// threads per row beyond that; each thread holds its vectors of the row in
// registers, so every input is read once and every output written once.  The
// backward pass, for rows of up to 4096 elements, walks blocks of token rows
// with one CTA each: dX row by row and the dgamma / dbeta partial sums of its
// columns in registers, in one pass over X, dXn and dOut.  Wider rows take a
// dX pass (one CTA per row) and a separate column-reduction pass over dXn
// and X.  The dropout backward reads the keep bits the forward pass stored
// and sums dZ's columns (db2) as it goes.  Reductions run warp-shuffle then
// over the warps' partial sums, always in the same order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "colsum.cuh"
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

// Chunk and local row of a token row, moved along without a division (the
// strip kernels step each thread's row by a fixed stride).
struct ChunkPos {
    int j;
    long long lr;
};

__device__ __forceinline__ ChunkPos chunk_pos(long long r, long long rows) {
    ChunkPos c;
    c.lr = chunk_row(r, rows, c.j);
    return c;
}

__device__ __forceinline__ ChunkPos chunk_advance(ChunkPos c, long long d, long long rows) {
    c.lr += d;
    while (c.lr >= rows) {
        c.lr -= rows;
        ++c.j;
    }
    return c;
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

// One warp per token row, for rows of at most 32 * 8 * V elements (h a
// multiple of 8): lane l holds the row's vectors l, l + 32, ...; the mean and
// variance are warp-shuffle sums (no block barrier), so a warp starts its
// row's loads as soon as it is scheduled and an SM keeps sixteen rows' loads
// in flight.
template <int V>
__global__ void __launch_bounds__(LN_THREADS, 2) ln_forward_warp_kernel(const LnForwardParams p,
                                                                        long long T) {
    const int lane = threadIdx.x & 31;
    const long long r = static_cast<long long>(blockIdx.x) * (LN_THREADS / 32) + (threadIdx.x >> 5);
    if (r >= T) return;
    int j;
    const long long rr = chunk_row(r, p.x.rows, j);
    const int h = p.h;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x.in[j]) + rr * h;
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y[j]) + rr * h;
    uint4 v[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int c = (lane + 32 * i) * 8;
        if (c < h) v[i] = *reinterpret_cast<const uint4*>(x + c);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        if ((lane + 32 * i) * 8 < h) {
            float f[8];
            unpack8(v[i], f);
#pragma unroll
            for (int k = 0; k < 8; ++k) s += f[k];
        }
    }
    const float mean = warp_sum(s) / static_cast<float>(h);
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        if ((lane + 32 * i) * 8 < h) {
            float f[8];
            unpack8(v[i], f);
#pragma unroll
            for (int k = 0; k < 8; ++k) q += (f[k] - mean) * (f[k] - mean);
        }
    }
    const float var = warp_sum(q) / static_cast<float>(h);
    const float rs = 1.0f / sqrtf(var + p.eps);
    const __nv_bfloat16* gm = static_cast<const __nv_bfloat16*>(p.gamma);
    const __nv_bfloat16* bt = static_cast<const __nv_bfloat16*>(p.beta);
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int c = (lane + 32 * i) * 8;
        if (c < h) {
            float f[8], g[8], b[8], o[8];
            unpack8(v[i], f);
            unpack8(__ldg(reinterpret_cast<const uint4*>(gm + c)), g);
            unpack8(__ldg(reinterpret_cast<const uint4*>(bt + c)), b);
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = (f[k] - mean) * rs * g[k] + b[k];
            *reinterpret_cast<uint4*>(y + c) = pack8(o);
        }
    }
    if (lane == 0) {
        p.mean[r] = mean;
        p.rstd[r] = rs;
    }
}

// One 8-element vector of the dropout backward pass: dOut at token row r
// (chunk position c), columns col.., and the keep bits of its 32-column word.
__device__ __forceinline__ void dropout_load(const DropoutBackwardParams& p, ChunkPos c,
                                             long long r, int col, uint4& u, uint32_t& word) {
    const long long off = c.lr * p.h + col;
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.dout.in[c.j]);
    u = __ldg(reinterpret_cast<const uint4*>(src + off));
    word = __ldg(p.drop.mask + r * p.drop.mask_words + col / 32);
}

// dZ for that vector, stored; its bf16 values added to acc.
__device__ __forceinline__ void dropout_apply(const DropoutBackwardParams& p, ChunkPos c, int col,
                                              const uint4& u, uint32_t word, float (&acc)[8]) {
    const long long off = c.lr * p.h + col;
    const uint32_t bits = word >> (col & 31);
    float f[8];
    unpack8(u, f);
#pragma unroll
    for (int k = 0; k < 8; ++k) f[k] = ((bits >> k) & 1u) ? f[k] * p.drop.scale : 0.0f;
    const uint4 o = pack8(f);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dz[c.j]) + off) = o;
    float g[8];
    unpack8(o, g);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] += g[k];
}

// dZ = keep ? dOut * scale : 0 from the keep bits the forward pass stored,
// and the column sums of dZ (as rounded to bf16) per row split: CTA = a
// 64-column strip x 32 row slots over the rows of split blockIdx.y; thread
// (slot, vec) handles columns vec*8 .. vec*8+7 of rows slot, slot + 32, ...
// (four rows' loads in flight, added in row order), and the slots are added
// in order through shared memory into part[split][col].
__global__ void __launch_bounds__(LN_THREADS, 3) dropout_backward_kernel(const DropoutBackwardParams p,
                                                                      long long T) {
    constexpr int COLS = 64;
    __shared__ float red[32][COLS + 1];
    const int h = p.h;
    const int vec = threadIdx.x & 7, slot = threadIdx.x >> 3;
    const int col = blockIdx.x * COLS + vec * 8;
    const long long r0 = static_cast<long long>(blockIdx.y) * p.rows_per_split;
    const long long r1 = r0 + p.rows_per_split < T ? r0 + p.rows_per_split : T;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    if (col < h && r0 + slot < r1) {
        const long long rows = p.dout.rows;
        long long r = r0 + slot;
        ChunkPos c = chunk_pos(r, rows);
        for (; r + 96 < r1; r += 128) {
            uint4 u[4];
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dropout_load(p, chunk_advance(c, 32 * q, rows), r + 32 * q, col, u[q], w[q]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dropout_apply(p, chunk_advance(c, 32 * q, rows), col, u[q], w[q], acc);
            c = chunk_advance(c, 128, rows);
        }
        for (; r < r1; r += 32) {
            uint4 u;
            uint32_t w;
            dropout_load(p, c, r, col, u, w);
            dropout_apply(p, c, col, u, w, acc);
            c = chunk_advance(c, 32, rows);
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) red[slot][vec * 8 + k] = acc[k];
    __syncthreads();
    if (threadIdx.x < COLS) {
        const int c = blockIdx.x * COLS + threadIdx.x;
        if (c < h) {
            float sum = 0.0f;
            for (int k = 0; k < 32; ++k) sum += red[k][threadIdx.x];
            p.part[static_cast<long long>(blockIdx.y) * h + c] = sum;
        }
    }
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

// Sum of two values over the CTA with one barrier: red holds two buffers of
// 2 x (LN_THREADS / 32) floats, used by alternate calls (buf = 0, 1, 0, ...),
// so a call's writes cannot meet the previous call's reads; every thread adds
// the warps' partial sums in the same order.
__device__ __forceinline__ float2 block_sum2_1bar(float a, float b, float* red, int buf) {
    constexpr int W = LN_THREADS / 32;
    a = warp_sum(a);
    b = warp_sum(b);
    float* rb = red + buf * 2 * W;
    if ((threadIdx.x & 31) == 0) {
        rb[threadIdx.x >> 5] = a;
        rb[W + (threadIdx.x >> 5)] = b;
    }
    __syncthreads();
    float ta = rb[0], tb = rb[W];
#pragma unroll
    for (int w = 1; w < W; ++w) {
        ta += rb[w];
        tb += rb[W + w];
    }
    return make_float2(ta, tb);
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

// Rows of at most LN_WARP_MAX_H elements: dX and the dgamma / dbeta partial
// sums in one pass.  CTA b walks token rows [b * rows_per_block, ...) in
// order with the next row's X, dXn and residual gradient loads in flight;
// each thread keeps gamma and the partial sums of its columns in registers,
// so X and dXn are read once:
// part[b][0][c] = sum dXn * xhat, part[b][1][c] = sum dXn, added over the
// blocks in a fixed order by the finishing kernels.
template <int VEC>
__global__ void __launch_bounds__(LN_THREADS, 2) ln_backward_fused_kernel(const LnBackwardParams p,
                                                                          long long T) {
    __shared__ float red[4 * (LN_THREADS / 32)];
    const int h = p.h;
    const long long rows = p.x.rows;
    const long long r0 = static_cast<long long>(blockIdx.x) * p.rows_per_block;
    const long long r1 = r0 + p.rows_per_block < T ? r0 + p.rows_per_block : T;
    const __nv_bfloat16* gm = static_cast<const __nv_bfloat16*>(p.gamma);
    float ag[VEC][8], ab[VEC][8];
    uint4 gv[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        gv[i] = c < h ? __ldg(reinterpret_cast<const uint4*>(gm + c)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < 8; ++k) ag[i][k] = ab[i][k] = 0.0f;
    }
    // row r's X, dXn and residual gradient vectors, at chunk position cp
    auto load = [&](ChunkPos cp, uint4 (&xv)[VEC], uint4 (&dv)[VEC], uint4 (&rv)[VEC]) {
        const long long off = cp.lr * h;
        const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x.in[cp.j]) + off;
        const __nv_bfloat16* dy = static_cast<const __nv_bfloat16*>(p.dxn[cp.j]) + off;
        const __nv_bfloat16* dr = static_cast<const __nv_bfloat16*>(p.dres[cp.j]) + off;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const int c = (threadIdx.x + i * LN_THREADS) * 8;
            if (c < h) {
                xv[i] = __ldg(reinterpret_cast<const uint4*>(x + c));
                dv[i] = __ldg(reinterpret_cast<const uint4*>(dy + c));
                rv[i] = __ldg(reinterpret_cast<const uint4*>(dr + c));
            }
        }
    };
    uint4 xv[VEC], dv[VEC], rv[VEC], nx[VEC], nd[VEC], nr[VEC];
    ChunkPos cp{0, 0};
    if (r0 < r1) {
        cp = chunk_pos(r0, rows);
        load(cp, xv, dv, rv);
    }
    for (long long r = r0; r < r1; ++r) {
        const ChunkPos cn = chunk_advance(cp, 1, rows);
        if (r + 1 < r1) load(cn, nx, nd, nr);
        const float mean = __ldg(p.mean + r), rs = __ldg(p.rstd + r);
        const float nmr = -mean * rs;  // xhat = x * rstd - mean * rstd
        float sg = 0.0f, sgx = 0.0f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            if ((threadIdx.x + i * LN_THREADS) * 8 < h) {
                float xf[8], df[8], gf[8];
                unpack8(xv[i], xf);
                unpack8(dv[i], df);
                unpack8(gv[i], gf);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float xh = fmaf(xf[k], rs, nmr);
                    const float g = df[k] * gf[k];
                    sg += g;
                    sgx = fmaf(g, xh, sgx);
                    ag[i][k] = fmaf(df[k], xh, ag[i][k]);
                    ab[i][k] += df[k];
                }
            }
        }
        const float2 sums = block_sum2_1bar(sg, sgx, red, static_cast<int>((r - r0) & 1));
        // dX = rstd * g - rstd * mean(g) - xhat * rstd * mean(g * xhat) + dres
        //    = rstd * g + c3 * x + (c4 + dres)
        const float c2 = -rs * (sums.y / static_cast<float>(h));
        const float c3 = c2 * rs;
        const float c4 = fmaf(c2, nmr, -rs * (sums.x / static_cast<float>(h)));
        __nv_bfloat16* dx = static_cast<__nv_bfloat16*>(p.dx[cp.j]) + cp.lr * h;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const int c = (threadIdx.x + i * LN_THREADS) * 8;
            if (c < h) {
                float xf[8], df[8], gf[8], rf[8], o[8];
                unpack8(xv[i], xf);
                unpack8(dv[i], df);
                unpack8(gv[i], gf);
                unpack8(rv[i], rf);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    o[k] = fmaf(rs, df[k] * gf[k], fmaf(c3, xf[k], rf[k] + c4));
                *reinterpret_cast<uint4*>(dx + c) = pack8(o);
            }
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            xv[i] = nx[i];
            dv[i] = nd[i];
            rv[i] = nr[i];
        }
        cp = cn;
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int c = (threadIdx.x + i * LN_THREADS) * 8;
        if (c < h) {
            float* pg = p.part + (static_cast<size_t>(blockIdx.x) * 2) * h + c;
            float* pb = pg + h;
            *reinterpret_cast<float4*>(pg) = make_float4(ag[i][0], ag[i][1], ag[i][2], ag[i][3]);
            *reinterpret_cast<float4*>(pg + 4) = make_float4(ag[i][4], ag[i][5], ag[i][6], ag[i][7]);
            *reinterpret_cast<float4*>(pb) = make_float4(ab[i][0], ab[i][1], ab[i][2], ab[i][3]);
            *reinterpret_cast<float4*>(pb + 4) = make_float4(ab[i][4], ab[i][5], ab[i][6], ab[i][7]);
        }
    }
}

// dgamma / dbeta partial column sums: CTA = a 64-column strip x 32 row slots
// over the rows of split blockIdx.y; thread (slot, vec) accumulates columns
// vec*8 .. vec*8+7 of rows slot, slot + 32, ... (four rows' loads in flight,
// added in row order); the slots are then added in order through shared
// memory.  part[split][0][c] = sum dXn * xhat, part[split][1][c] = sum dXn.
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
    // row r's inputs, then its terms added to the sums
    auto load = [&](ChunkPos c, long long r, uint4& xu, uint4& du, float& mean, float& rs) {
        const long long off = c.lr * h + col;
        const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(p.x.in[c.j]);
        const __nv_bfloat16* ds = static_cast<const __nv_bfloat16*>(p.dxn[c.j]);
        xu = __ldg(reinterpret_cast<const uint4*>(xs + off));
        du = __ldg(reinterpret_cast<const uint4*>(ds + off));
        mean = __ldg(p.mean + r);
        rs = __ldg(p.rstd + r);
    };
    auto add = [&](const uint4& xu, const uint4& du, float mean, float rs) {
        float xf[8], df[8];
        unpack8(xu, xf);
        unpack8(du, df);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            ag[k] += df[k] * ((xf[k] - mean) * rs);
            ab[k] += df[k];
        }
    };
    if (col < h && r0 + slot < r1) {
        const long long rows = p.x.rows;
        long long r = r0 + slot;
        ChunkPos c = chunk_pos(r, rows);
        for (; r + 96 < r1; r += 128) {
            uint4 xu[4], du[4];
            float mn[4], rs[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                load(chunk_advance(c, 32 * q, rows), r + 32 * q, xu[q], du[q], mn[q], rs[q]);
#pragma unroll
            for (int q = 0; q < 4; ++q) add(xu[q], du[q], mn[q], rs[q]);
            c = chunk_advance(c, 128, rows);
        }
        for (; r < r1; r += 32) {
            uint4 xu, du;
            float mn, rs;
            load(c, r, xu, du, mn, rs);
            add(xu, du, mn, rs);
            c = chunk_advance(c, 32, rows);
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

// Vectors per thread for rows of h elements: the smallest of 1, 2, 4, 8 that covers h.
int ln_vec(int h) {
    const int v = (h + 8 * LN_THREADS - 1) / (8 * LN_THREADS);
    return v <= 1 ? 1 : v <= 2 ? 2 : v <= 4 ? 4 : 8;
}

}  // namespace

cudaError_t launch_ln_forward(const LnForwardParams& p, long long T, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    if (p.h % 8 == 0 && p.h <= LN_WARP_MAX_H) {
        // rows of up to 4096 elements: one warp per row
        constexpr int RPB = LN_THREADS / 32;
        const unsigned blocks = static_cast<unsigned>((T + RPB - 1) / RPB);
        if (p.h <= 1024)
            ln_forward_warp_kernel<4><<<blocks, LN_THREADS, 0, st>>>(p, T);
        else if (p.h <= 2048)
            ln_forward_warp_kernel<8><<<blocks, LN_THREADS, 0, st>>>(p, T);
        else
            ln_forward_warp_kernel<16><<<blocks, LN_THREADS, 0, st>>>(p, T);
        return cudaGetLastError();
    }
    const unsigned grid = static_cast<unsigned>(T);
    switch (ln_vec(p.h)) {
        case 1: ln_forward_kernel<1><<<grid, LN_THREADS, 0, st>>>(p); break;
        case 2: ln_forward_kernel<2><<<grid, LN_THREADS, 0, st>>>(p); break;
        case 4: ln_forward_kernel<4><<<grid, LN_THREADS, 0, st>>>(p); break;
        default: ln_forward_kernel<8><<<grid, LN_THREADS, 0, st>>>(p); break;
    }
    return cudaGetLastError();
}

int dropout_splits(long long T, long long h, int sm_count) {
    const long long strips = (h + 63) / 64;
    long long sp = (16LL * sm_count + strips - 1) / strips;
    const long long by_rows = T / 128 > 0 ? T / 128 : 1;
    if (sp > by_rows) sp = by_rows;
    if (sp > LN_MAX_SPLITS) sp = LN_MAX_SPLITS;
    return static_cast<int>(sp < 1 ? 1 : sp);
}

cudaError_t launch_dropout_backward(const DropoutBackwardParams& p, long long T, float* db2,
                                    cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((p.h + 63) / 64), static_cast<unsigned>(p.splits));
    dropout_backward_kernel<<<grid, LN_THREADS, 0, st>>>(p, T);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_colsum_f32(p.part, p.splits, p.h, p.h, db2, st);
}

cudaError_t launch_ln_backward(const LnBackwardParams& p, long long T, int splits, float* dgamma,
                               float* dbeta, cudaStream_t st) {
    if (ln_backward_fused(p.h)) {
        // dX and the partial sums in one pass over row blocks, then the finish
        const unsigned grid = static_cast<unsigned>(splits);
        if (p.h <= LN_THREADS * 8)
            ln_backward_fused_kernel<1><<<grid, LN_THREADS, 0, st>>>(p, T);
        else
            ln_backward_fused_kernel<2><<<grid, LN_THREADS, 0, st>>>(p, T);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_colsum_f32_pair(p.part, splits, 2LL * p.h, p.h, dgamma, dbeta, st);
    }
    if (T > 0) {
        const unsigned grid = static_cast<unsigned>(T);
        // rows wider than LN_WARP_MAX_H: four or eight vectors per thread
        if (ln_vec(p.h) <= 4)
            ln_dx_kernel<4><<<grid, LN_THREADS, 0, st>>>(p);
        else
            ln_dx_kernel<8><<<grid, LN_THREADS, 0, st>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>((p.h + 63) / 64), static_cast<unsigned>(splits));
    ln_param_grad_kernel<<<grid, LN_THREADS, 0, st>>>(p, T);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // dgamma = sum of part[s][0][:], dbeta = sum of part[s][1][:] over the splits
    return launch_colsum_f32_pair(p.part, splits, 2LL * p.h, p.h, dgamma, dbeta, st);
}

}  // namespace tpmlp
