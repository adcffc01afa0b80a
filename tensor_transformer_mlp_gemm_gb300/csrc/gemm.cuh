// gemm.cuh -- the tcgen05 GEMM behind every contraction of the tensor-parallel
// MLP block, with the block's elementwise work fused into its epilogue.
//
// Sources (page title, section):
//   [FGO]   "Megatron-LM：NVIDIA 的大规模并行训练方案", "Megatron-LM 核心架构 /
//           张量并行原理" (column- and row-parallel linear layers, MLP = column
//           then row).
//   [FGO-F] same page, "融合优化技术" (Bias + GeLU fused into one kernel).
//   [CH2]   "2、分布式训练基础：数据并行、模型并行、流水线并行的基本概念与区别",
//           "2.2 模型并行 —— 张量并行 / 核心原理".
//
// One kernel computes, for every group g and output tile,
//     C_g[m, n] = sum_{s < ksegs} sum_{k < K} Aop_{g,s}[m, k] * Bop_{g,s}[n, k]
// where the operands are bf16 matrices reached through TMA tensor maps and the
// sum runs in fp32 in tensor memory.  "Groups" are independent GEMMs that
// share a launch (the t column-parallel shards); "k-segments" are summed into
// the same accumulator (the t row-parallel shards: the AllReduce of the pages
// becomes split-K accumulation in TMEM, with no separate reduction pass).
//
// Each operand is either K-major (row-major [rows, K]) or MN-major (row-major
// [K, rows]); the weight-gradient GEMMs contract over tokens and read both
// operands MN-major straight from the token-major activations.
//
// Work unit: a CTA pair (cluster of 2, one CTA per SM) owns a 256 x 256
// output tile and computes it with tcgen05.mma.cta_group::2 (256 x 256 x 16
// per instruction, issued by the even CTA).  Each CTA stages its own 128 rows
// of A and its own 128 rows of B per K step (32 KB), so a 6-deep ring fits in
// shared memory and each SM keeps 192 KB of operands in flight while needing
// only 64 B per clock at full MMA rate (a single-CTA 128 x 256 tile needs 96).
// The pair's accumulator rows live in each CTA's own tensor memory.  A
// wider variant (256 x 512 tiles, one accumulator in two halves, see Tile)
// moves a quarter fewer operand bytes per FLOP; the host picks the width.
//
// CTA layout (192 threads, persistent over tiles; both CTAs of the pair):
//   warp 0      TMA producer (one elected thread): this CTA's A and B halves
//               into the shared-memory ring; their bytes are counted on the
//               even CTA's "full" barrier
//   warp 1      owns the tensor memory (pair allocation); in the even CTA one
//               elected thread issues the pair MMAs and commits them to both
//               CTAs' "empty" / "accumulator full" barriers
//   warps 2..5  epilogue: tcgen05.ld of this CTA's accumulator rows, fused
//               elementwise work, TMA stores; then they release the
//               accumulator on the even CTA's "accumulator empty" barrier
// Two 256-column fp32 accumulators in TMEM let the epilogue of one tile run
// under the main loop of the next (256-wide tiles).
//
// Every mbarrier wait is bounded (GemmParams::timeout_ns).  A wait that
// expires sets a CTA-wide abort flag and a bit of the device error word;
// every role of that CTA then leaves its loop (the peer's waits expire in
// turn), the even CTA's producer waits (bounded) for copies in flight, the
// MMA issuer waits (bounded) for its MMAs, and after a final cluster barrier
// both CTAs free their tensor memory and return.  Before leaving, each
// producer also waits until every stage it filled has been released, and the
// MMA issuer until the last accumulators have been released, so no
// asynchronous arrive can land in a CTA that has exited.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gemm_params.h"
#include "ptx.cuh"

namespace tpmlp {

// ---- tanh-form GeLU ----------------------------------------------------------
// GeLU(y)  = 0.5 y (1 + tanh(u)),  u = sqrt(2/pi) (y + 0.044715 y^3)
// GeLU'(y) = 0.5 (1 + tanh u) + 0.5 y (1 - tanh^2 u) du, du = sqrt(2/pi) (1 + 3*0.044715 y^2)
constexpr float kGeluK0 = 0.7978845608028654f;  // sqrt(2/pi)
constexpr float kGeluK1 = 0.044715f;

__device__ __forceinline__ float gelu_f(float y) {
    const float u = kGeluK0 * fmaf(kGeluK1 * y, y * y, y);
    return 0.5f * y * (1.0f + ptx::tanh_approx(u));
}

// The same derivative regrouped for the epilogue's instruction count: with
// a = 0.5 y du = y (0.5 sqrt(2/pi) + 1.5 sqrt(2/pi) 0.044715 y^2),
// GeLU'(y) = (0.5 + a) + th (0.5 - a th).
__device__ __forceinline__ float gelu_grad_f(float y) {
    const float y2 = y * y;
    const float th = ptx::tanh_approx(kGeluK0 * fmaf(kGeluK1 * y, y2, y));
    const float a = y * fmaf(1.5f * kGeluK0 * kGeluK1, y2, 0.5f * kGeluK0);
    return fmaf(th, fmaf(-a, th, 0.5f), 0.5f + a);
}

// ---- bounded waits -------------------------------------------------------------

// Sleeps in short naps until this SM's clock reaches `deadline` (returns at once
// if it already has).  The deadline is at most a few thousand clocks ahead; the
// nap count is capped all the same.
__device__ __forceinline__ void pace_until(long long deadline) {
    for (int i = 0; i < 4096 && clock64() < deadline; ++i) __nanosleep(32);
}

// Waits for phase `parity` of `bar`.  Gives up (returns false) when another
// role has aborted, or when timeout_ns has elapsed (then this role aborts the
// CTA and records `code` in the device error word).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, const GemmParams& p,
                                             unsigned code) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            atomicOr(p.err, code);
            return false;
        }
    }
}

// Same, with cluster-scope acquire (for barriers the peer CTA arrives on).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                     volatile int* abort_flag,
                                                     const GemmParams& p, unsigned code) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            atomicOr(p.err, code);
            return false;
        }
    }
}

// Teardown wait: ignores the abort flag, still bounded.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const GemmParams& p) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.err, ERR_DRAIN);
            return false;
        }
    }
    return true;
}

// ---- tile schedule ---------------------------------------------------------------
// Tiles are walked in bands of `band` M-tiles; inside a band the M-tile index
// runs fastest, so the CTAs that run at the same time share their B tiles
// (and, across the band, their A panels) through L2.  (group, n-tile) pairs
// form one combined N axis.
template <int TN>
__device__ __forceinline__ void decode_tile(const GemmParams& p, int tile, int& g, int& m0,
                                            int& n0) {
    const int nt_total = p.ntiles * p.groups;
    const int band_tiles = p.band * nt_total;
    const int b = tile / band_tiles;
    const int r = tile - b * band_tiles;
    const int mt_first = b * p.band;
    const int rows_here = min(p.band, p.mtiles - mt_first);
    const int mt = mt_first + r % rows_here;
    const int ntg = r / rows_here;
    g = ntg / p.ntiles;
    n0 = (ntg - g * p.ntiles) * TN;
    m0 = mt * CLUSTER_M;
}

// ---- work items -------------------------------------------------------------------
// Pair c takes whole tiles c, c + P, ... below dp_tiles, then split unit c (if
// c < units): K steps [kbeg, kend) of leftover tile dp_tiles + c / splits.
// Every role of both CTAs walks the same sequence.  With the units last, all
// pairs start their whole tiles together, so the pairs that share an operand
// panel stay closer in step and re-read less of it from DRAM (measured:
// +0.6 % per step at the 175B-class layer against units first).
struct WorkItem {
    int tile;
    int kbeg, kend;
    int unit;  // split unit index, or -1 for a whole tile
};

__device__ __forceinline__ bool work_item(const GemmParams& p, int c, int P, int j, int nk,
                                          WorkItem& it) {
    const int tile = c + j * P;
    if (tile < p.dp_tiles) {
        it.tile = tile;
        it.kbeg = 0;
        it.kend = nk;
        it.unit = -1;
        return true;
    }
    // the unit is the item right after the pair's last whole tile
    if (c >= p.units || (j > 0 && tile - P >= p.dp_tiles)) return false;
    const int sidx = c % p.splits;
    it.unit = c;
    it.tile = p.dp_tiles + c / p.splits;
    it.kbeg = sidx * nk / p.splits;
    it.kend = (sidx + 1) * nk / p.splits;
    return true;
}

// Named barrier among the four epilogue warps of a CTA.
__device__ __forceinline__ void epilogue_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(EPI_WARPS * 32) : "memory");
}

// ---- operand loads -----------------------------------------------------------------
// K-major operand: tensor [rows, K] (inner K), box {BK, ROWS}; one copy.
// MN-major operand: tensor [K, rows] (inner rows), box {64, BK}; ROWS/64
// copies, box j landing at dst + j * MN_CHUNK_BYTES.  The bytes complete on
// `bar`, a shared::cluster address (the even CTA's barrier).
// PART_ROW: a tile whose rows start past the last token chunk (the second
// CTA of a pair tile when T is not a multiple of 256) reads the last chunk's
// map at out-of-range rows, which TMA fills with zeros; the map index never
// leaves the encoded maps.
struct OperandCursor {
    const CUtensorMap* map;
    int r;      // row (M or N) coordinate of this CTA's box
    int kbase;  // K coordinate of the segment's first element
    int mn3d;   // MN-major operand encoded as a 3-D map {64, K, rows / 64}
};

__device__ __forceinline__ OperandCursor operand_cursor(const CUtensorMap* maps, int part,
                                                        int rows_per_map, int nmaps, int g,
                                                        int s, int row0, int K, int mn3d) {
    OperandCursor c{maps, row0, s * K, mn3d};
    if (part == PART_GROUP) {
        c.map = maps + g;
    } else if (part == PART_KSEG) {
        c.map = maps + s;
        c.kbase = 0;
    } else if (part == PART_ROW) {
        const int idx = min(row0 / rows_per_map, nmaps - 1);
        c.map = maps + idx;
        c.r = row0 - idx * rows_per_map;
    }
    return c;
}

template <bool MN, int ROWS>
__device__ __forceinline__ void load_operand(const OperandCursor& c, int kc, uint32_t dst,
                                             uint32_t bar) {
    const int k = c.kbase + kc;
    if constexpr (!MN) {
        ptx::tma_load_2d_pair(dst, c.map, k, c.r, bar);
    } else {
        if (c.mn3d) {
            // box {64, BK, ROWS / 64}: chunk j lands at dst + j * MN_CHUNK_BYTES
            ptx::tma_load_3d_pair(dst, c.map, 0, k, c.r / MN_CHUNK, bar);
        } else {
#pragma unroll
            for (int j = 0; j < ROWS / MN_CHUNK; ++j)
                ptx::tma_load_2d_pair(dst + j * MN_CHUNK_BYTES, c.map, c.r + j * MN_CHUNK, k, bar);
        }
    }
}

// The same boxes as load_operand, prefetched into L2 only.
template <bool MN, int ROWS>
__device__ __forceinline__ void prefetch_operand(const OperandCursor& c, int kc) {
    const int k = c.kbase + kc;
    if constexpr (!MN) {
        ptx::tma_prefetch_2d(c.map, k, c.r);
    } else {
        if (c.mn3d) {
            ptx::tma_prefetch_3d(c.map, 0, k, c.r / MN_CHUNK);
        } else {
#pragma unroll
            for (int j = 0; j < ROWS / MN_CHUNK; ++j)
                ptx::tma_prefetch_2d(c.map, c.r + j * MN_CHUNK, k);
        }
    }
}

// Descriptor of the 16-wide K slice `kk` (0..3) of a stage's operand tile.
//   K-major:  rows of 128 B, 8-row swizzle atoms stacked every 1024 B (SBO);
//             the K slice starts 32 B further along the row.
//   MN-major: [rows/64 boxes][BK K-rows][64 elements]; 8-K-row atoms every
//             1024 B (SBO), 64-element boxes every MN_CHUNK_BYTES (LBO); the
//             K slice starts 16 rows (2048 B) further down.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile, int kk) {
    if constexpr (!MN)
        return ptx::smem_desc_sw128(tile + kk * 32, 16, 1024);
    else
        return ptx::smem_desc_sw128(tile + kk * 2048, MN_CHUNK_BYTES, 1024);
}

// ---- epilogue ----------------------------------------------------------------------
// Each epilogue warp owns 32 accumulator rows (its TMEM lane quarter) and walks
// the tile's columns 32 at a time: tcgen05.ld -> fused elementwise work in
// fp32 -> one row per lane written into a swizzled 32 x 32 staging buffer ->
// one lane issues a TMA bulk tensor store.  The store clips rows and columns
// outside the tensor, so ragged edges need no masks.  Two staging buffers
// per warp let the stores of chunk c-1 drain while chunk c is being staged.

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Row `r` (32 fp32 values) into a 32 x 32 fp32 box staged with the 128-byte
// swizzle: 16-byte chunk c of row r lives at chunk c ^ (r % 8).
__device__ __forceinline__ void stage_row_f32(uint8_t* buf, int r, const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float4 v = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
        *reinterpret_cast<float4*>(buf + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
}

// Row `r` (32 bf16 values) into a 32 x 32 bf16 box staged with the 64-byte
// swizzle: 16-byte chunk c of row r lives at chunk c ^ ((r / 2) % 4).
__device__ __forceinline__ void stage_row_bf16(uint8_t* buf, int r, const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float* a = x + 8 * c;
        uint4 v = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                             pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
        *reinterpret_cast<uint4*>(buf + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) = v;
    }
}

// Epilogues that read a second input per output element (the saved Y of the
// dGeLU epilogues, the residual of the dropout epilogue).
template <int EPI>
struct EpiReadsIn0 {
    static constexpr bool value =
        EPI == EPI_DGELU || EPI == EPI_DGELU_H || EPI == EPI_BIAS_DROP_RES;
};

// That input for one thread's 32 values (row `row` of part `part`, columns
// [n, n + 32)), as four 16-byte vectors.  Issued ahead of the accumulator
// chunk it belongs to, so its latency overlaps the previous chunk's work.
template <int EPI>
__device__ __forceinline__ void load_in0(const GemmParams& p, int part, long long row, int m,
                                         int n, uint4 (&u)[4]) {
    if constexpr (EpiReadsIn0<EPI>::value) {
        if (m < p.M && n < p.N) {
            const __nv_bfloat16* src =
                static_cast<const __nv_bfloat16*>(p.in0[part]) + row * p.ld_in + n;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (n + 8 * q < p.N) u[q] = *reinterpret_cast<const uint4*>(src + 8 * q);
        }
    }
}

// Epilogues that add a bias per output column.
template <int EPI>
struct EpiReadsBias {
    static constexpr bool value = EPI == EPI_BIAS_GELU || EPI == EPI_BIAS || EPI == EPI_BIAS_DROP_RES;
};

// The bias of columns [n, n + 32) of group g as four 16-byte vectors (every
// lane reads the same ones); issued a chunk ahead like load_in0.
template <int EPI>
__device__ __forceinline__ void load_bias(const GemmParams& p, int g, int n, uint4 (&b)[4]) {
    if constexpr (EpiReadsBias<EPI>::value) {
        const __nv_bfloat16* src =
            static_cast<const __nv_bfloat16*>(p.bias) + n + g * p.bias_group_stride;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (n + 8 * q < p.N) b[q] = __ldg(reinterpret_cast<const uint4*>(src + 8 * q));
    }
}

// Elementwise work on one thread's 32 values: row m, columns [n, n + 32);
// `in` holds the second input (load_in0) for the epilogues that read one,
// `bias` the columns' bias (load_bias) for those that add one.
template <int EPI>
__device__ __forceinline__ void epilogue_math(const GemmParams& p, int g, int part, long long row,
                                              int m, int n, float (&x)[32], float (&x2)[32],
                                              const uint4 (&in)[4], const uint4 (&bias)[4]) {
    if constexpr (EpiReadsBias<EPI>::value) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (n + 8 * q < p.N) {
                float bf[8];
                unpack_bf16x8(bias[q], bf);
#pragma unroll
                for (int j = 0; j < 8; ++j) x[8 * q + j] += bf[j];
            }
        }
        if constexpr (EPI == EPI_BIAS_GELU) {
#pragma unroll
            for (int j = 0; j < 32; ++j) x2[j] = gelu_f(x[j]);
        }
    }
    if constexpr (EPI == EPI_BIAS_DROP_RES) {
        // Out = in0 + Dropout(acc + bias): the 32 columns of this row are the
        // elements e0 .. e0 + 31 of the [M, N] output, e0 = m * N + n (a multiple
        // of 4), i.e. eight Philox counters offset + e0 / 4 + q
        if (m < p.M) {
            const uint64_t e0 = static_cast<uint64_t>(m) * static_cast<uint64_t>(p.N) +
                                static_cast<uint64_t>(n);
            uint32_t bits = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const PhiloxOut o = philox4x32_10(p.drop.offset + e0 / 4 + q, p.drop.seed);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool keep = static_cast<uint64_t>(o.w[j]) < p.drop.thresh;
                    x[4 * q + j] = keep ? x[4 * q + j] * p.drop.scale : 0.0f;
                    bits |= (keep ? 1u : 0u) << (4 * q + j);
                }
            }
            // the mask's bits for the backward pass (n is a multiple of 32)
            if (p.drop.mask)
                p.drop.mask[static_cast<long long>(m) * p.drop.mask_words + n / 32] = bits;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (n + 8 * q < p.N) {
                    float rf[8];
                    unpack_bf16x8(in[q], rf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[8 * q + j] += rf[j];
                }
            }
        }
    }
    if constexpr (EPI == EPI_DGELU || EPI == EPI_DGELU_H) {
        if (m < p.M) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (n + 8 * q < p.N) {
                    float yf[8];
                    unpack_bf16x8(in[q], yf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        x[8 * q + j] *= gelu_grad_f(yf[j]);
                        if constexpr (EPI == EPI_DGELU_H) x2[8 * q + j] = gelu_f(yf[j]);
                    }
                }
            }
        }
    }
}

// Column sums of one warp's 32 x 32 block of the fp32 output (lane = row,
// x[j] = column n + j), rows at or past M counted as zero: a butterfly of 31
// shuffles leaves lane j with the sum of column n + j over the 32 rows, which
// it stores into the partial row of this 32-row group (one 128-byte store per
// warp).  The order of the additions is fixed, so the sums are reproducible.
// Works in place: x is consumed (called after the values have been staged).
__device__ __forceinline__ void warp_column_sums(const GemmParams& p, int g, int first_row, int m,
                                                 int n, int lane, float (&x)[32]) {
    if (m >= p.M) {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.f;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = upper ? x[i] : x[i + o];
            const float keep = upper ? x[i + o] : x[i];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    if (first_row < p.M && n + lane < p.N)
        p.colsum_part[static_cast<long long>(first_row / 32) * p.colsum_ld +
                      static_cast<long long>(g) * p.N + n + lane] = x[0];
}

// ---- the kernel ---------------------------------------------------------------------

// Tile shapes.  A pair computes a CLUSTER_M x TN output tile, TN = 256 (two
// 256-column accumulators in TMEM, so a tile's epilogue runs under the next
// tile's MMAs) or TN = 512 (one 512-column accumulator of two 256-column
// halves; a K step that feeds both halves moves 48 KB per CTA for twice the
// FLOPs of a 32 KB narrow step, a quarter fewer operand bytes per FLOP).
//
// A wide tile overlaps its epilogue with MMAs by splitting its K steps
// [kbeg, kend) into three phases, L = wide_lookahead(kend - kbeg):
//   A  steps kbeg .. kbeg+L-1   half 0 only   (stage: A + B half 0)
//   B  steps kbeg+L .. kend-1   both halves   (stage: A + both B halves)
//   C  steps kbeg .. kbeg+L-1   half 1 only   (stage: A again + B half 1)
// Half 0 is complete after phase B and is drained under phase C; half 1 is
// complete after phase C and is drained under the next tile's phase A.  Half
// 1 sums its K steps starting at kbeg+L (a rotation of the narrow order).
template <int TN>
struct Tile {
    static_assert(TN == 256 || TN == 512, "tile width 256 or 512");
    static constexpr int kStages = TN == 512 ? 4 : STAGES;
    static constexpr int kStageBytes = A_STAGE_BYTES + (TN / 256) * B_STAGE_BYTES;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + EPI_STAGE_BYTES + BAR_BYTES;
    static constexpr int kChunks = TN / EPI_CHUNK;  // epilogue chunks per tile
    static constexpr int kHalves = TN / 256;        // 256-column MMA halves
};
static_assert(Tile<512>::kSmemBytes <= 232448, "the wide tile's shared memory fits a CTA");

// K steps of a wide tile's phases A and C (none for a one-step tile).
constexpr int WIDE_LOOKAHEAD = 32;
__device__ __forceinline__ int wide_lookahead(int nks) {
    return min(WIDE_LOOKAHEAD, nks / 2);
}

template <bool A_MN, bool B_MN, int EPI, int TN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    tpmlp_gemm_kernel(const __grid_constant__ GemmParams p) {
    using TL = Tile<TN>;
    constexpr int NST = TL::kStages;
    constexpr int SB = TL::kStageBytes;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* epi_area = smem_raw + (base - raw) + NST * SB;
    uint8_t* bar_area = epi_area + EPI_STAGE_BYTES;
    const uint32_t epi0 = base + NST * SB;
    const uint32_t bar0 = epi0 + EPI_STAGE_BYTES;
    const uint32_t bar_full = bar0;                      // [NST] used in the even CTA
    const uint32_t bar_empty = bar0 + 8 * NST;           // [NST] both CTAs
    const uint32_t bar_tfull = bar0 + 16 * NST;          // [2] both CTAs
    const uint32_t bar_tempty = bar_tfull + 16;          // [2] used in the even CTA
    const uint32_t bar_drain = bar_tempty + 16;          // [1] even CTA
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 16 * NST + 40);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 16 * NST + 44);
    volatile int* last_flag = reinterpret_cast<volatile int*>(bar_area + 16 * NST + 48);
    volatile int* epi_fail = reinterpret_cast<volatile int*>(bar_area + 16 * NST + 52);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(ptx::cluster_ctarank());  // CTA within its pair
    const int cluster = blockIdx.x / 2;
    const int nclusters = gridDim.x / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, 1);
        }
        // TN = 256: accumulator a full / empty.  TN = 512: tfull[0] = the
        // accumulator full, tempty[h] = its half h drained.
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bar_tfull + 8 * a, 1);
            ptx::mbar_init(bar_tempty + 8 * a, 2 * EPI_WARPS * 32);  // both CTAs' epilogues
        }
        ptx::mbar_init(bar_drain, 1);
        *abort_flag = 0;
        *last_flag = 0;
        *epi_fail = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < p.a_nmaps; ++i) ptx::prefetch_tensormap(&p.a_map[i]);
        for (int i = 0; i < p.b_nmaps; ++i) ptx::prefetch_tensormap(&p.b_map[i]);
    }
    // both CTAs' barriers and tensor memory exist before anything crosses
    ptx::tc_fence_before();
    __syncwarp();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the previous kernel in the
    // stream: the set-up above overlaps that kernel's last wave; nothing
    // below touches global memory before it has completed.  The producer
    // lets the next kernel be scheduled when it starts this CTA's last tile.
    ptx::griddep_wait();

    const int kblocks = (p.K + BK - 1) / BK;
    const int nk = kblocks * p.ksegs;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            const uint32_t even_full = ptx::mapa_shared(bar_full, 0);
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            WorkItem it;
            for (int j = 0; ok && work_item(p, cluster, nclusters, j, nk, it); ++j) {
                // Last tile of this CTA: the next kernel in the stream may be
                // scheduled (its CTAs take the SMs this grid leaves and wait
                // for it to complete before touching memory).  Triggered at
                // the start instead, it slowed the weight-gradient GEMMs by
                // ~15 % (measured) for no gain.
                {
                    WorkItem nx;
                    if (!work_item(p, cluster, nclusters, j + 1, nk, nx))
                        ptx::griddep_launch_dependents();
                }
                int g, m0, n0;
                decode_tile<TN>(p, it.tile, g, m0, n0);
                const int a_row = m0 + rank * BM;
                // B rows of half h staged by this CTA: n0 + 256 h + 128 rank
                const int b_row = n0 + rank * B_ROWS;
                // segment and K step advance by increments; the map and row of each
                // operand change only with the segment
                int seg = it.kbeg / kblocks;
                int kb = it.kbeg - seg * kblocks;
                OperandCursor ca = operand_cursor(p.a_map, p.a_part, p.a_rows_per_map, p.a_nmaps,
                                                  g, seg, a_row, p.K, p.a_mn3d);
                OperandCursor cb = operand_cursor(p.b_map, p.b_part, p.b_rows_per_map, p.b_nmaps,
                                                  g, seg, b_row, p.K, p.b_mn3d);
                OperandCursor cb1 = cb;
                if (TN == 512)
                    cb1 = operand_cursor(p.b_map, p.b_part, p.b_rows_per_map, p.b_nmaps, g, seg,
                                         b_row + 256, p.K, p.b_mn3d);
                // head prefetch: the first K steps of this pair's next tile go to L2
                // now, a whole tile ahead of their loads (short-K GEMMs, where
                // every tile start would otherwise wait for first-touch data)
                if (p.head_prefetch > 0 && !p.stall_producer) {
                    WorkItem nx;
                    if (work_item(p, cluster, nclusters, j + 1, nk, nx)) {
                        int ng, nm0, nn0;
                        decode_tile<TN>(p, nx.tile, ng, nm0, nn0);
                        const int nseg = nx.kbeg / kblocks;
                        const int nkb = nx.kbeg - nseg * kblocks;
                        const OperandCursor pa =
                            operand_cursor(p.a_map, p.a_part, p.a_rows_per_map, p.a_nmaps, ng,
                                           nseg, nm0 + rank * BM, p.K, p.a_mn3d);
                        const OperandCursor pb =
                            operand_cursor(p.b_map, p.b_part, p.b_rows_per_map, p.b_nmaps, ng,
                                           nseg, nn0 + rank * B_ROWS, p.K, p.b_mn3d);
                        const int stop = min(nkb + p.head_prefetch, kblocks);
                        for (int q = nkb; q < stop && nseg * kblocks + q < nx.kend; ++q) {
                            prefetch_operand<A_MN, BM>(pa, q * BK);
                            prefetch_operand<B_MN, B_ROWS>(pb, q * BK);
                        }
                    }
                }
                const int nks = it.kend - it.kbeg;
                const int la = TN == 512 ? wide_lookahead(nks) : 0;
                for (int st = 0; st < nks + la; ++st) {
                    if (TN == 512 && st == nks) {
                        // phase C: back to the first K step of the item
                        seg = it.kbeg / kblocks;
                        kb = it.kbeg - seg * kblocks;
                        ca = operand_cursor(p.a_map, p.a_part, p.a_rows_per_map, p.a_nmaps, g,
                                            seg, a_row, p.K, p.a_mn3d);
                        cb1 = operand_cursor(p.b_map, p.b_part, p.b_rows_per_map, p.b_nmaps, g,
                                             seg, b_row + 256, p.K, p.b_mn3d);
                    } else if (kb == kblocks) {
                        kb = 0;
                        ++seg;
                        ca = operand_cursor(p.a_map, p.a_part, p.a_rows_per_map, p.a_nmaps, g,
                                            seg, a_row, p.K, p.a_mn3d);
                        cb = operand_cursor(p.b_map, p.b_part, p.b_rows_per_map, p.b_nmaps, g,
                                            seg, b_row, p.K, p.b_mn3d);
                        if (TN == 512)
                            cb1 = operand_cursor(p.b_map, p.b_part, p.b_rows_per_map, p.b_nmaps, g,
                                                 seg, b_row + 256, p.K, p.b_mn3d);
                    }
                    // halves this step feeds: bit 0 = half 0, bit 1 = half 1
                    const int hmask = TN == 256 ? 1 : (st < la ? 1 : (st < nks ? 3 : 2));
                    {
                        if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p,
                                          ERR_PRODUCER)) {
                            ok = false;
                            break;
                        }
                        if (!p.stall_producer) {
                            const uint32_t full = even_full + 8 * stage;
                            const uint32_t sa = base + stage * SB;
                            const uint32_t bytes =
                                A_STAGE_BYTES + (hmask == 3 ? 2 : 1) * B_STAGE_BYTES;
                            if (rank == 0)  // counts both CTAs' bytes
                                ptx::mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * bytes);
                            load_operand<A_MN, BM>(ca, kb * BK, sa, full);
                            if (hmask & 1)
                                load_operand<B_MN, B_ROWS>(cb, kb * BK, sa + A_STAGE_BYTES, full);
                            if (hmask & 2)
                                load_operand<B_MN, B_ROWS>(
                                    cb1, kb * BK, sa + A_STAGE_BYTES + B_STAGE_BYTES, full);
                            ++fills;
                        }
                        if (++stage == NST) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    ++kb;
                }
            }
            if (ok) {
                // Producer tail: the even CTA's MMA releases each stage with an
                // asynchronous arrive on both CTAs' "empty" barriers.  Wait until
                // every stage filled here has been released, so no such arrive
                // can land after this CTA has exited.
                for (int i = 0; i < NST; ++i) {
                    if (!wait_drain(bar_empty + 8 * stage, phase ^ 1u, p)) break;
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            } else if (rank == 0) {
                // Wait for the pair's copies still in flight (the last NST
                // fills, counted on this CTA's barriers) before leaving.
                for (long long f = (fills > NST ? fills - NST : 0); f < fills; ++f) {
                    const int st = static_cast<int>(f % NST);
                    const uint32_t par = static_cast<uint32_t>((f / NST) & 1);
                    if (!wait_drain(bar_full + 8 * st, par, p)) break;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (even CTA) ----------------
            constexpr uint32_t IDESC = ptx::idesc_bf16_f32(CLUSTER_M, 256, A_MN, B_MN);
            constexpr uint32_t B_HALF_BYTES = 128 * BK * 2;  // half h of a CTA's B tile
            int stage = 0;
            uint32_t phase = 0;
            int lt = 0;
            bool ok = true;
            // the MMAs of N-half h of one stage (h = 0 for TN = 256)
            auto issue = [&](int h, uint32_t d_tmem, bool first) {
                const uint32_t sa = base + stage * SB;
                const uint32_t sb = sa + A_STAGE_BYTES + h * B_HALF_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    ptx::mma_bf16_pair(d_tmem + h * 256, operand_desc<A_MN>(sa, k),
                                       operand_desc<B_MN>(sb, k), IDESC,
                                       (!first || k > 0) ? 1u : 0u);
                }
            };
            auto advance = [&]() {
                if (++stage == NST) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            WorkItem it;
            for (int j = 0; ok && work_item(p, cluster, nclusters, j, nk, it); ++j, ++lt) {
                if constexpr (TN == 256) {
                    const int acc = lt & 1;
                    const uint32_t acc_phase = static_cast<uint32_t>((lt >> 1) & 1);
                    if (!wait_bounded_cluster(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag,
                                              p, ERR_MMA)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * 256);
                    for (int kk = it.kbeg; kk < it.kend; ++kk) {
                        if (!wait_bounded(bar_full + 8 * stage, phase, abort_flag, p, ERR_MMA)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        issue(0, d_tmem, kk == it.kbeg);
                        // the stage is free again in both CTAs of the pair
                        ptx::mma_commit_pair_multicast(bar_empty + 8 * stage, 0x3);
                        advance();
                    }
                    if (ok) ptx::mma_commit_pair_multicast(bar_tfull + 8 * acc, 0x3);
                } else {
                    // One accumulator in two halves, K steps in phases A, B, C
                    const uint32_t ph = static_cast<uint32_t>(lt & 1);
                    const int nks = it.kend - it.kbeg;
                    const int la = wide_lookahead(nks);
                    for (int st = 0; st < nks + la; ++st) {
                        // half 0 (phase A) needs the previous tile's half 0
                        // drained, half 1 (phase B on) its half 1
                        if (st == 0 &&
                            !wait_bounded_cluster(bar_tempty, ph ^ 1u, abort_flag, p, ERR_MMA)) {
                            ok = false;
                            break;
                        }
                        if (st == la && !wait_bounded_cluster(bar_tempty + 8, ph ^ 1u, abort_flag,
                                                              p, ERR_MMA)) {
                            ok = false;
                            break;
                        }
                        if (!wait_bounded(bar_full + 8 * stage, phase, abort_flag, p, ERR_MMA)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        if (st < nks) issue(0, tmem, st == 0);
                        if (st >= la) issue(1, tmem, st == la);
                        ptx::mma_commit_pair_multicast(bar_empty + 8 * stage, 0x3);
                        // half 0 complete after phase B, half 1 after phase C
                        if (st == nks - 1) ptx::mma_commit_pair_multicast(bar_tfull, 0x3);
                        if (st == nks + la - 1) ptx::mma_commit_pair_multicast(bar_tfull + 8, 0x3);
                        advance();
                    }
                }
            }
            // Every MMA this thread issued must finish before TMEM is freed.
            ptx::mma_commit_pair(bar_drain);
            wait_drain(bar_drain, 0, p);
            // MMA tail: both CTAs' epilogues release the last accumulators with
            // arrives on this CTA's barriers; wait for them before leaving.
            if (ok) {
                if constexpr (TN == 256) {
                    for (int j = (lt > 2 ? lt - 2 : 0); j < lt; ++j) {
                        if (!wait_drain(bar_tempty + 8 * (j & 1),
                                        static_cast<uint32_t>((j >> 1) & 1), p))
                            break;
                    }
                } else if (lt > 0) {
                    const uint32_t par = static_cast<uint32_t>((lt - 1) & 1);
                    if (wait_drain(bar_tempty, par, p)) wait_drain(bar_tempty + 8, par, p);
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;
        uint8_t* stage_buf = epi_area + (warp - 2) * (2 * EPI_BUF_BYTES);
        const uint32_t stage_u32 = epi0 + (warp - 2) * (2 * EPI_BUF_BYTES);
        const uint32_t even_tempty = ptx::mapa_shared(bar_tempty, 0);
        int chunk_seq = 0;

        // Stage 32 values per lane as this warp's 32 x 32 box and store it
        // through `map` at (x, y) (and the second output for EPI_BIAS_GELU).
        auto store_box = [&](const CUtensorMap* map, const CUtensorMap* map2, int x, int y,
                             const float (&v)[32], const float (&v2)[32], bool f32) {
            const int b = chunk_seq & 1;
            ++chunk_seq;
            if (lane == 0) ptx::bulk_wait_group_read<1>();
            __syncwarp();
            uint8_t* buf = stage_buf + b * EPI_BUF_BYTES;
            if (f32) {
                stage_row_f32(buf, lane, v);
            } else {
                stage_row_bf16(buf, lane, v);
                if (map2) stage_row_bf16(buf + 2048, lane, v2);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const uint32_t sb = stage_u32 + b * EPI_BUF_BYTES;
                ptx::tma_store_2d(map, sb, x, y);
                if (!f32 && map2) ptx::tma_store_2d(map2, sb + 2048, x, y);
                ptx::bulk_commit_group();
            }
        };
        // Releases accumulator part `a` (TN = 256: accumulator a; TN = 512:
        // half a) once this warp's loads from it have completed.
        auto release = [&](int a) {
            ptx::tc_fence_before();
            ptx::mbar_arrive_cluster(even_tempty + 8 * a);
        };

        // fp32 outputs (the weight gradients: short K, 128 KB per CTA per tile)
        // are stored paced over most of the time the next tile's MMAs take:
        // stored in one burst, all pairs' stores would meet the next tiles' first
        // loads.  The schedule is a deadline per chunk in SM clocks, derived from
        // the tile's K steps, not from the measured time between tiles: a paced
        // epilogue that falls behind (slow stores) does not wait, so the pacing
        // cannot feed back into a longer tile period.
        int lt = 0;
        WorkItem it;
        for (int j = 0; work_item(p, cluster, nclusters, j, nk, it); ++j, ++lt) {
            int g, mp, n0;
            decode_tile<TN>(p, it.tile, g, mp, n0);
            const int m0 = mp + rank * BM;  // this CTA's first row
            const int acc = TN == 256 ? (lt & 1) : 0;
            const uint32_t acc_phase =
                static_cast<uint32_t>(TN == 256 ? ((lt >> 1) & 1) : (lt & 1));
            // output map and row coordinate of this warp's 32 rows
            int part = g;
            int y0 = m0 + quarter * 32;
            if (p.out_part == PART_ROW && m0 < p.M) {
                part = m0 / p.out_rows_per_part;
                y0 -= part * p.out_rows_per_part;
            }
            const int m = m0 + row;
            const long long in_row = static_cast<long long>(y0) + lane;
            // the second input of the first chunk is read before the accumulator is ready
            uint4 pre[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                            make_uint4(0, 0, 0, 0)};
            uint4 bpre[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                             make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            if (it.unit < 0) {
                load_in0<EPI>(p, part, in_row, m, n0, pre);
                if constexpr (EPI != EPI_BIAS_DROP_RES) load_bias<EPI>(p, g, n0, bpre);
            }
            // Waits for accumulator part b (TN = 256: accumulator b; TN = 512:
            // half b); all four epilogue warps give up together (they share
            // named barriers).
            auto acc_ready = [&](int b) -> bool {
                const bool ok = wait_bounded(bar_tfull + 8 * b, acc_phase, abort_flag, p,
                                             ERR_EPILOGUE);
                if (!ok) *epi_fail = 1;
                epilogue_bar();
                if (*epi_fail) return false;
                __syncwarp();
                ptx::tc_fence_after();
                return true;
            };
            if (!acc_ready(acc)) break;
            long long pace_t0 = 0, pace_clk = 0;
            if constexpr (EPI == EPI_F32 && TN == 256) {
                // only while this pair has a next tile whose main loop the stores can
                // hide under; the last tile's stores go out at once
                WorkItem nx;
                if (it.unit < 0 && work_item(p, cluster, nclusters, j + 1, nk, nx)) {
                    pace_clk = static_cast<long long>(it.kend - it.kbeg) * PACE_CLK_PER_KBLOCK;
                    pace_t0 = clock64();
                }
            }
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * 256);
            const CUtensorMap* out1 = &p.out_map[part];
            const CUtensorMap* out2 = (EPI == EPI_BIAS_GELU || EPI == EPI_DGELU_H)
                                          ? &p.out_map[MAX_MAPS + part]
                                          : nullptr;
            constexpr bool OUT_F32 = EPI == EPI_F32;
            constexpr int NCH = TL::kChunks;

            if (it.unit < 0) {
                // whole tile: fused epilogue straight from the accumulator
                bool failed = false;
#pragma unroll 1
                for (int c = 0; c < NCH; ++c) {
                    if (TN == 512 && c == NCH / 2) {
                        release(0);  // half 0 drained
                        if (!acc_ready(1)) {
                            failed = true;
                            break;
                        }
                    }
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(taddr + c * EPI_CHUNK, v);
                    uint4 cur[4] = {pre[0], pre[1], pre[2], pre[3]};
                    uint4 curb[4] = {bpre[0], bpre[1], bpre[2], bpre[3]};
                    // the next chunk's second input and bias, in flight meanwhile (the
                    // dropout epilogue, short of registers, reads its bias when used)
                    if (c + 1 < NCH) {
                        load_in0<EPI>(p, part, in_row, m, n0 + (c + 1) * EPI_CHUNK, pre);
                        if constexpr (EPI != EPI_BIAS_DROP_RES)
                            load_bias<EPI>(p, g, n0 + (c + 1) * EPI_CHUNK, bpre);
                    }
                    if constexpr (EPI == EPI_BIAS_DROP_RES)
                        load_bias<EPI>(p, g, n0 + c * EPI_CHUNK, curb);
                    ptx::tmem_ld_wait();
                    const int n = n0 + c * EPI_CHUNK;
                    if (n >= p.N || m0 >= p.M) continue;  // outside the tensor (warp-uniform)
                    float x[32], x2[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) x[q] = __uint_as_float(v[q]);
                    epilogue_math<EPI>(p, g, part, in_row, m, n, x, x2, cur, curb);
                    if (pace_clk && c > 0) pace_until(pace_t0 + c * pace_clk);
                    store_box(out1, out2, n, y0, x, x2, OUT_F32);
                    if constexpr (EPI == EPI_DGELU || EPI == EPI_DGELU_H) {
                        if (p.colsum_part) warp_column_sums(p, g, m0 + quarter * 32, m, n, lane, x);
                    }
                }
                if (failed) break;
                release(TN == 256 ? acc : 1);
                continue;
            }

            // split unit: store this unit's raw partial rows, then count it.
            // Partial row block v = unit * halves + h holds N-half h of the unit.
            bool failed = false;
#pragma unroll 1
            for (int c = 0; c < NCH; ++c) {
                if (TN == 512 && c == NCH / 2) {
                    release(0);
                    if (!acc_ready(1)) {
                        failed = true;
                        break;
                    }
                }
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(taddr + c * EPI_CHUNK, v);
                ptx::tmem_ld_wait();
                const int n = n0 + c * EPI_CHUNK;
                if (n >= p.N || m0 >= p.M) continue;
                float x[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) x[q] = __uint_as_float(v[q]);
                const int vblk = it.unit * TL::kHalves + (c >> 3);
                const int prow = (vblk * 2 + rank) * BM + quarter * 32;
                store_box(&p.part_map, nullptr, (c & 7) * EPI_CHUNK, prow, x, x, true);
            }
            if (failed) break;
            release(TN == 256 ? acc : 1);
            // the partial is complete and visible before it is counted
            if (lane == 0) {
                ptx::bulk_wait_group<0>();
                ptx::fence_proxy_async_global();
            }
            __syncwarp();
            epilogue_bar();
            const int slot = (it.tile - p.dp_tiles) * 2 + rank;
            if (warp == 2 && lane == 0) {
                __threadfence();
                const int before = atomicAdd(&p.counters[slot], 1);
                *last_flag = (before == p.splits - 1) ? 1 : 0;
            }
            epilogue_bar();
            if (*last_flag) {
                // last unit of this tile: sum all partials in unit order, then
                // the fused epilogue
                __threadfence();
                const int u0 = (it.tile - p.dp_tiles) * p.splits;
#pragma unroll 1
                for (int c = 0; c < NCH; ++c) {
                    const int n = n0 + c * EPI_CHUNK;
                    if (n >= p.N || m0 >= p.M) continue;
                    float x[32], x2[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) x[q] = 0.f;
                    // SU units' rows in flight per round (the loads are
                    // independent), added in unit order; two for the epilogue
                    // that also produces H, whose registers are fuller
                    constexpr int SU = EPI == EPI_DGELU_H ? 2 : 4;
                    for (int sp0 = 0; sp0 < p.splits; sp0 += SU) {
                        float4 f[SU][8];
#pragma unroll
                        for (int u = 0; u < SU; ++u) {
                            if (sp0 + u < p.splits) {
                                const int vblk = (u0 + sp0 + u) * TL::kHalves + (c >> 3);
                                const long long r =
                                    static_cast<long long>(vblk * 2 + rank) * BM + row;
                                const float4* src = reinterpret_cast<const float4*>(
                                    p.partial + r * BN + (c & 7) * EPI_CHUNK);
#pragma unroll
                                for (int q = 0; q < 8; ++q) f[u][q] = __ldcg(src + q);
                            }
                        }
#pragma unroll
                        for (int u = 0; u < SU; ++u) {
                            if (sp0 + u < p.splits) {
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    x[4 * q] += f[u][q].x;
                                    x[4 * q + 1] += f[u][q].y;
                                    x[4 * q + 2] += f[u][q].z;
                                    x[4 * q + 3] += f[u][q].w;
                                }
                            }
                        }
                    }
                    uint4 in[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                   make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
                    uint4 bv[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                   make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
                    load_in0<EPI>(p, part, in_row, m, n, in);
                    load_bias<EPI>(p, g, n, bv);
                    epilogue_math<EPI>(p, g, part, in_row, m, n, x, x2, in, bv);
                    store_box(out1, out2, n, y0, x, x2, OUT_F32);
                    if constexpr (EPI == EPI_DGELU || EPI == EPI_DGELU_H) {
                        if (p.colsum_part) warp_column_sums(p, g, m0 + quarter * 32, m, n, lane, x);
                    }
                }
                if (warp == 2 && lane == 0) p.counters[slot] = 0;  // ready for the next launch
            }
        }
        // every store must have finished before the CTA leaves
        if (lane == 0) ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    // neither CTA frees its tensor memory or leaves before the pair's MMAs
    // (which write both CTAs' tensor memory) have drained
    ptx::tc_fence_before();
    __syncwarp();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// CTA pairs of this kernel variant that fit on the GPU at once (queried once
// per variant).
template <bool A_MN, bool B_MN, int EPI, int TN>
cudaError_t max_active_clusters(int& out) {
    static int max_clusters = 0;
    if (max_clusters == 0) {
        auto kern = tpmlp_gemm_kernel<A_MN, B_MN, EPI, TN>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Tile<TN>::kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = Tile<TN>::kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_clusters = n;
    }
    out = max_clusters;
    return cudaSuccess;
}

// Launched as a programmatic dependent of the previous kernel in the stream.
template <bool A_MN, bool B_MN, int EPI, int TN>
cudaError_t launch_variant(const GemmParams& p, int clusters, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Tile<TN>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tpmlp_gemm_kernel<A_MN, B_MN, EPI, TN>, p);
}

// Persistent launch, capped at the pairs that fit on the GPU at once; the
// tiles of an incomplete last wave get their K range split across the pairs
// that would otherwise idle.  A wide tile's split unit takes two partial-tile
// slots of the workspace (one per N-half).
template <bool A_MN, bool B_MN, int EPI, int TN>
cudaError_t launch_tiles(const GemmParams& p_in, cudaStream_t stream) {
    GemmParams p = p_in;
    int P = 0;
    cudaError_t e = max_active_clusters<A_MN, B_MN, EPI, TN>(P);
    if (e != cudaSuccess) return e;
    const int nk = ((p.K + BK - 1) / BK) * p.ksegs;
    const int full = p.total_tiles / P;
    const int left = p.total_tiles % P;
    constexpr int max_units = MAX_SPLIT_UNITS / Tile<TN>::kHalves;
    p.dp_tiles = p.total_tiles;
    p.units = 0;
    p.splits = 1;
    if (p.counters && p.split_min_kblocks > 0 && nk >= p.split_min_kblocks && left > 0) {
        int splits = P / left;
        if (splits > MAX_SPLITS) splits = MAX_SPLITS;
        if (splits > nk) splits = nk;
        if (splits >= 2 && left * splits <= max_units) {
            p.splits = splits;
            p.units = left * splits;
            p.dp_tiles = p.total_tiles - left;
        }
    }
    int clusters = p.total_tiles < P ? p.total_tiles : P;
    if (p.units > 0) {
        clusters = full > 0 ? P : p.units;
        e = cudaMemsetAsync(p.counters, 0, sizeof(int) * 2 * left, stream);
        if (e != cudaSuccess) return e;
    }
    return launch_variant<A_MN, B_MN, EPI, TN>(p, clusters, stream);
}

// The tile width the host chose (GemmParams::tn); fp32-output GEMMs (the
// weight gradients, short K and a large epilogue) always run narrow tiles.
template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_clusters(const GemmParams& p, cudaStream_t stream) {
    if constexpr (EPI != EPI_F32) {
        if (p.tn == 512) return launch_tiles<A_MN, B_MN, EPI, 512>(p, stream);
    }
    if (p.tn != 256) return cudaErrorInvalidValue;
    return launch_tiles<A_MN, B_MN, EPI, 256>(p, stream);
}

#define TPMLP_GEMM_LAUNCHER(NAME, A_MN, B_MN, EPI)               \
    cudaError_t NAME(const GemmParams& p, cudaStream_t stream) {  \
        return launch_clusters<A_MN, B_MN, EPI>(p, stream);       \
    }

}  // namespace tpmlp
