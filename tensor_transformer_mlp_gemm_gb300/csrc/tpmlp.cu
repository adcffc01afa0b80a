// tpmlp.cu -- the C ABI of libtpmlp (declared in include/tpmlp.h).
//
// Validates arguments, encodes the TMA tensor maps of every operand, lays out
// the workspace, and enqueues the kernels of the forward and backward passes
// of the tensor-parallel MLP block on the caller's stream:
//
//   forward   column_fwd  Y_i = X.A_i + b1_i, H_i = GeLU(Y_i)     (t groups)
//             row_fwd     Z = sum_i H_i.B_i + b2                  (t k-segments)
//   backward  dgrad_h     dY_i = (dZ.B_i^T) * GeLU'(Y_i)          (t groups)
//             dgrad_x     dX = sum_i dY_i.A_i^T                   (t k-segments)
//             wgrad       dB_i = H_i^T.dZ                         (t groups)
//             wgrad       dA_i = X^T.dY_i                         (t groups)
//             colsum      db1 = sum_T dY, db2 = sum_T dZ
//
// Sources (page title, section): "Megatron-LM：NVIDIA 的大规模并行训练方案",
// "Megatron-LM 核心架构 / 张量并行原理" (column then row parallel MLP),
// "融合优化技术" (Bias + GeLU fusion), "并行训练范式 / 序列并行" (sequence
// parallelism); "2、分布式训练基础：数据并行、模型并行、流水线并行的基本概念与区别",
// "2.2 模型并行 —— 张量并行 / 核心原理".
//
// Sequence parallelism: X and dZ come as seq_chunks token chunks, addressed
// through one tensor map per chunk (the gather happens inside the TMA loads),
// and the epilogues of the split-K GEMMs write each output row into its chunk
// (the reduce-scatter); no staging copies.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "abi_internal.h"
#include "block_internal.h"
#include "colsum.cuh"
#include "gemm_params.h"
#include "map_cache.h"
#include "tpmlp.h"

#define TPMLP_API extern "C" __attribute__((visibility("default")))

namespace tpmlp {

// Device error word: kernels OR a bit in when a bounded wait expires.
__device__ unsigned int g_error_word;

namespace abi {

namespace {
constexpr int kMaxDevices = 64;
}  // namespace

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
unsigned long long g_timeout_ns = 2000000000ULL;
int g_split_min_kblocks = DEFAULT_SPLIT_MIN_KBLOCKS;
int g_head_prefetch = 0;
int g_wide_tiles = WIDE_TILES_DEEP_K;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// ---- profiling ------------------------------------------------------------------
std::mutex g_prof_mu;
bool g_prof_on = false;
uint32_t g_prof_kinds = ~0u;  // kinds that get event pairs while profiling
std::vector<ProfRec> g_prof_pool;
size_t g_prof_used = 0;

ProfRec* prof_next(int kind, int kernels) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on || g_prof_used >= g_prof_pool.size()) return nullptr;
    if (kind < 0 || kind >= 32 || !((g_prof_kinds >> kind) & 1u)) return nullptr;
    ProfRec* r = &g_prof_pool[g_prof_used++];
    r->kind = kind;
    r->kernels = kernels;
    return r;
}

// ---- device / driver ----------------------------------------------------------------
tpmlp_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TPMLP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TPMLP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return TPMLP_ERR_CUDA;
        d.supported = (prop.major == 10 && prop.minor == 3);
        d.sm_count = prop.multiProcessorCount;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return TPMLP_ERR_CUDA;
            d.err = static_cast<unsigned int*>(p);
            if (cudaMemset(d.err, 0, sizeof(unsigned int)) != cudaSuccess) return TPMLP_ERR_CUDA;
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return TPMLP_ERR_CUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    if (!d.supported) return TPMLP_ERR_UNSUPPORTED;
    *out = &d;
    return TPMLP_OK;
}

// ---- tensor maps -------------------------------------------------------------------------
// Every map goes through the cache: encoded once per (address, shape, box,
// swizzle), then copied.
constexpr size_t kMapCacheCapacity = 4096;
MapCache g_maps(kMapCacheCapacity);

static bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dtype, uint32_t rank, const void* ptr,
                         const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                         CUtensorMapSwizzle swizzle, CUtensorMapL2promotion l2promo) {
    const MapKey key = make_map_key(dtype, rank, ptr, dims, strides, box, swizzle, l2promo);
    return g_maps.get(key, m, [&](CUtensorMap* out) {
        const cuuint32_t estr[3] = {1, 1, 1};
        return g_encode(out, dtype, rank, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, l2promo,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

// bf16 row-major matrix [outer, inner] with leading dimension ld (elements).
//   K-major operand tile: box {BK, box_rows} (BK along the contiguous K axis)
//   MN-major operand tile: box {64, BK}      (64 along the contiguous M/N axis)
static bool encode_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                 uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

bool encode_kmajor(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, int box_rows) {
    return encode_bf16(m, ptr, K, rows, K, BK, static_cast<uint32_t>(box_rows));
}

bool encode_mnmajor(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t K, int* mn3d,
                    int box_rows) {
    if (rows % MN_CHUNK != 0 || rows < static_cast<uint64_t>(box_rows)) {
        // 2-D map {rows, K}: a box is fetched as box_rows / 64 copies of {64, BK}
        *mn3d = 0;
        return encode_bf16(m, ptr, rows, K, rows, MN_CHUNK, BK);
    }
    // {64 elements, K rows, rows / 64 chunks}: chunk j starts 128 bytes after
    // chunk j - 1, so a box {64, BK, 2} is two neighbouring 64-element columns
    *mn3d = 1;
    cuuint64_t dims[3] = {MN_CHUNK, K, rows / MN_CHUNK};
    cuuint64_t strides[2] = {rows * 2, MN_CHUNK * 2};
    cuuint32_t box[3] = {MN_CHUNK, BK, static_cast<cuuint32_t>(box_rows / MN_CHUNK)};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// Epilogue store map: row-major [rows, cols] output, box 32 x 32; fp32 boxes
// are staged with the 128-byte swizzle, bf16 boxes with the 64-byte swizzle.
bool encode_out(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, bool f32) {
    const uint64_t esize = f32 ? 4 : 2;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * esize};
    cuuint32_t box[2] = {EPI_CHUNK, 32};
    return encode_tiled(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, ptr, dims, strides, box,
                        f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

tpmlp_status check_ptrs(const void* const* arr, int n) {
    if (!arr) return TPMLP_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        if (!arr[i]) return TPMLP_ERR_INVALID_ARG;
        if (!aligned16(arr[i])) return TPMLP_ERR_UNSUPPORTED;
    }
    return TPMLP_OK;
}

tpmlp_status check_ptr(const void* p) {
    if (!p) return TPMLP_ERR_INVALID_ARG;
    return aligned16(p) ? TPMLP_OK : TPMLP_ERR_UNSUPPORTED;
}

// ---- GEMM set-up ------------------------------------------------------------------------
void base_params(GemmParams& p, const DeviceInfo& dev, int M, int N, int K, int groups,
                 int ksegs) {
    std::memset(&p, 0, sizeof(p));
    p.a_nmaps = 1;
    p.b_nmaps = 1;
    p.M = M;
    p.N = N;
    p.K = K;
    p.groups = groups;
    p.ksegs = ksegs;
    p.tn = BN;
    p.mtiles = (M + CLUSTER_M - 1) / CLUSTER_M;
    p.ntiles = (N + BN - 1) / BN;
    p.total_tiles = p.mtiles * p.ntiles * groups;
    p.band = p.mtiles < kBand ? p.mtiles : kBand;
    p.err = dev.err;
    p.timeout_ns = g_timeout_ns;
    p.stall_producer = 0;
    p.bias = nullptr;
    p.bias_group_stride = 0;
    p.ld_in = 0;
    for (int i = 0; i < MAX_MAPS; ++i) p.in0[i] = nullptr;
}

// Waves of pair tiles a GEMM takes at tile width tn on `pairs` pairs, with the
// tail split's division of an incomplete last wave (as the launcher applies it).
static double tile_waves(const GemmParams& p, int tn, int pairs) {
    const long long ntiles = (p.N + tn - 1) / tn;
    const long long tiles = static_cast<long long>(p.mtiles) * ntiles * p.groups;
    const long long full = tiles / pairs, left = tiles % pairs;
    if (left == 0) return static_cast<double>(full);
    const int nk = ((p.K + BK - 1) / BK) * p.ksegs;
    long long splits = pairs / left;
    if (splits > MAX_SPLITS) splits = MAX_SPLITS;
    if (splits > nk) splits = nk;
    const bool split = g_split_min_kblocks > 0 && nk >= g_split_min_kblocks && splits >= 2 &&
                       left * splits <= MAX_SPLIT_UNITS / (tn / BN);
    return static_cast<double>(full) + (split ? 1.0 / static_cast<double>(splits) : 1.0);
}

void choose_tile_width(GemmParams& p, const DeviceInfo& dev) {
    int tn = BN;
    const int nk = ((p.K + BK - 1) / BK) * p.ksegs;
    if (g_wide_tiles == 2) {
        tn = BN_WIDE;
    } else if (g_wide_tiles == WIDE_TILES_DEEP_K) {
        // deep K: the one-half phases are a small share of a tile's K steps,
        // and the quarter fewer operand bytes per FLOP lower the power the
        // GEMM draws, which under the power cap raises the clock of every
        // kernel of the step (measured: the 175B-class layer's row and dX
        // GEMMs, 768 K steps, +1.2 % per step; 16384 x 4096, 256 K steps,
        // +1.9 %; 128 K steps, -0.3 to -0.9 %)
        if (nk >= WIDE_MIN_KSTEPS) tn = BN_WIDE;
    } else if (g_wide_tiles == 1) {
        // the same work in no more time: waves x tile width (a wide tile is
        // twice a narrow one's work); ties go to the wide tile, which moves a
        // quarter fewer operand bytes per FLOP
        const int pairs = dev.sm_count / 2 > 0 ? dev.sm_count / 2 : 1;
        if (tile_waves(p, BN_WIDE, pairs) * BN_WIDE <= tile_waves(p, BN, pairs) * BN) tn = BN_WIDE;
    }
    p.tn = tn;
    p.ntiles = (p.N + tn - 1) / tn;
    p.total_tiles = p.mtiles * p.ntiles * p.groups;
}

bool attach_split(GemmParams& p, void* split_part, void* split_cnt) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(BN),
                          static_cast<cuuint64_t>(MAX_SPLIT_UNITS) * CLUSTER_M};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(BN) * 4};
    cuuint32_t box[2] = {EPI_CHUNK, 32};
    if (!encode_tiled(&p.part_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, split_part, dims, strides,
                      box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE))
        return false;
    p.partial = reinterpret_cast<const float*>(split_part);
    p.counters = reinterpret_cast<int*>(split_cnt);
    p.split_min_kblocks = g_split_min_kblocks;
    p.head_prefetch = g_head_prefetch;
    return true;
}

}  // namespace abi

namespace block {

using namespace abi;

// ---- workspace ---------------------------------------------------------------------------
Layout layout_of(const tpmlp_dims& d) {
    Layout L;
    const size_t act = align256(static_cast<size_t>(d.tokens) * static_cast<size_t>(d.ffn) * 2);
    L.y = 0;
    L.h = act;
    L.dy = 2 * act;
    L.part1 = 3 * act;
    // db1: the dH GEMM's epilogue writes one row of column sums per 32 token rows
    const size_t groups = static_cast<size_t>((d.tokens + 31) / 32);
    const size_t db1_part = groups * static_cast<size_t>(d.ffn) * sizeof(float);
    L.part2 = L.part1 + align256(db1_part > 0 ? db1_part : 256);
    L.split_part = L.part2 + align256(colsum_scratch_bytes(d.hidden));
    L.split_cnt = L.split_part + split_part_bytes();
    L.total = L.split_cnt + split_cnt_bytes();
    return L;
}

tpmlp_status check_dims(const tpmlp_dims* d) {
    if (!d) return TPMLP_ERR_INVALID_ARG;
    if (d->tokens < 0 || d->hidden <= 0 || d->ffn <= 0 || d->t <= 0 || d->seq_chunks <= 0)
        return TPMLP_ERR_INVALID_ARG;
    if (d->ffn % d->t != 0) return TPMLP_ERR_INVALID_ARG;
    if (d->tokens % d->seq_chunks != 0) return TPMLP_ERR_INVALID_ARG;
    if (d->t > kMaxShards || d->seq_chunks > kMaxShards) return TPMLP_ERR_UNSUPPORTED;
    const int64_t fi = d->ffn / d->t;
    if (d->hidden % 8 != 0 || fi % 8 != 0) return TPMLP_ERR_UNSUPPORTED;
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (d->tokens > lim || d->hidden > lim || d->ffn > lim) return TPMLP_ERR_UNSUPPORTED;
    if (d->seq_chunks > 1 && (d->tokens / d->seq_chunks) % BM != 0) return TPMLP_ERR_UNSUPPORTED;
    return TPMLP_OK;
}

Regions regions_of(uint8_t* ws, const Layout& L) {
    return Regions{ws + L.y, ws + L.h, ws + L.dy, ws + L.part1, ws + L.part2, ws + L.split_part,
                   ws + L.split_cnt};
}

// The recompute calls: saved = Y only; scratch = everything after Y in the
// standard layout (H first), at the same relative offsets.
Regions recompute_regions(uint8_t* saved, uint8_t* scratch, const Layout& L) {
    return Regions{saved,
                   scratch,
                   scratch + (L.dy - L.h),
                   scratch + (L.part1 - L.h),
                   scratch + (L.part2 - L.h),
                   scratch + (L.split_part - L.h),
                   scratch + (L.split_cnt - L.h)};
}

bool attach_split(GemmParams& p, const Regions& R) {
    return abi::attach_split(p, R.split_part, R.split_cnt);
}

Shapes shapes_of(const tpmlp_dims& d) {
    Shapes s;
    s.T = static_cast<int>(d.tokens);
    s.h = static_cast<int>(d.hidden);
    s.f = static_cast<int>(d.ffn);
    s.t = d.t;
    s.fi = s.f / s.t;
    s.chunks = d.seq_chunks;
    s.Tc = s.T / s.chunks;
    return s;
}

namespace {
inline const void* shard_ptr(const void* base, int i, const Shapes& s) {
    return static_cast<const uint8_t*>(base) + static_cast<size_t>(i) * s.T * s.fi * 2;
}
}  // namespace

// With no tokens the weight and bias gradients are zero.
tpmlp_status zero_weight_grads(const Shapes& s, void* const* dA_shards, void* db1,
                               void* const* dB_shards, void* db2, cudaStream_t st) {
    const size_t wbytes = static_cast<size_t>(s.h) * s.fi * sizeof(float);
    for (int i = 0; i < s.t; ++i) {
        TPMLP_CUDA(cudaMemsetAsync(dA_shards[i], 0, wbytes, st));
        TPMLP_CUDA(cudaMemsetAsync(dB_shards[i], 0, wbytes, st));
    }
    TPMLP_CUDA(cudaMemsetAsync(db1, 0, static_cast<size_t>(s.f) * sizeof(float), st));
    TPMLP_CUDA(cudaMemsetAsync(db2, 0, static_cast<size_t>(s.h) * sizeof(float), st));
    return TPMLP_OK;
}

// ---- the passes, on explicit device buffers (arguments already validated) ----------------

tpmlp_status run_forward(const Shapes& s, const DeviceInfo* dev, const void* const* X,
                         const void* const* A_shards, const void* b1,
                         const void* const* B_shards, const void* b2, void* const* Z,
                         const Regions& R, cudaStream_t st, const RowEpilogue* ep) {
    const void* Y = R.y;
    const void* H = R.h;

    // column-parallel GEMM + bias + GeLU: t groups, M = T, N = fi, K = h
    {
        GemmParams p;
        base_params(p, *dev, s.T, s.fi, s.h, s.t, 1);
        choose_tile_width(p, *dev);
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_kmajor(&p.a_map[j], X[j], s.h, s.Tc, BM)) return TPMLP_ERR_UNSUPPORTED;
        p.a_part = PART_ROW;
        p.a_nmaps = s.chunks;
        p.b_nmaps = s.t;
        p.a_rows_per_map = s.Tc;
        for (int i = 0; i < s.t; ++i)
            if (!encode_mnmajor(&p.b_map[i], A_shards[i], s.fi, s.h, &p.b_mn3d))
                return TPMLP_ERR_UNSUPPORTED;
        p.b_part = PART_GROUP;
        p.b_rows_per_map = 0;
        for (int i = 0; i < s.t; ++i) {
            if (!encode_out(&p.out_map[i], shard_ptr(Y, i, s), s.fi, s.T, false) ||
                !encode_out(&p.out_map[MAX_MAPS + i], shard_ptr(H, i, s), s.fi, s.T, false))
                return TPMLP_ERR_UNSUPPORTED;
        }
        p.out_part = PART_GROUP;
        p.out_rows_per_part = 0;
        p.bias = b1;
        p.bias_group_stride = s.fi;
        if (!attach_split(p, R)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_COLUMN_FWD, 1, st,
                         [&] { return launch_column_fwd(p, st); }));
    }
    // row-parallel GEMM, shard split-K + b2: M = T, N = h, K = fi per segment
    {
        GemmParams p;
        base_params(p, *dev, s.T, s.h, s.fi, 1, s.t);
        choose_tile_width(p, *dev);
        for (int i = 0; i < s.t; ++i) {
            if (!encode_kmajor(&p.a_map[i], shard_ptr(H, i, s), s.fi, s.T, BM))
                return TPMLP_ERR_UNSUPPORTED;
            if (!encode_mnmajor(&p.b_map[i], B_shards[i], s.h, s.fi, &p.b_mn3d))
                return TPMLP_ERR_UNSUPPORTED;
        }
        p.a_part = PART_KSEG;
        p.a_nmaps = s.t;
        p.b_nmaps = s.t;
        p.b_part = PART_KSEG;
        p.a_rows_per_map = p.b_rows_per_map = 0;
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_out(&p.out_map[j], Z[j], s.h, s.Tc, false)) return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_ROW;
        p.out_rows_per_part = s.Tc;
        p.bias = b2;
        if (ep) {
            // Out = residual + Dropout(Z): the residual is read per token chunk
            for (int j = 0; j < s.chunks; ++j) p.in0[j] = ep->residual[j];
            p.ld_in = s.h;
            p.drop = ep->drop;
        }
        if (!attach_split(p, R)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_ROW_FWD, 1, st, [&] {
            return ep ? launch_row_fwd_dropout(p, st) : launch_row_fwd(p, st);
        }));
    }
    return TPMLP_OK;
}

// recompute = true: H is not read from a saved copy but rebuilt from the saved
// Y by the dH GEMM's epilogue before the dB GEMM uses it.
tpmlp_status run_backward(const Shapes& s, const DeviceInfo* dev, const void* const* dZ,
                          const void* const* X, const void* const* A_shards,
                          const void* const* B_shards, void* const* dX, void* const* dA_shards,
                          void* db1, void* const* dB_shards, void* db2, const Regions& R,
                          bool recompute, cudaStream_t st, bool db2_given) {
    const void* Y = R.y;
    const void* H = R.h;
    const void* dY = R.dy;

    // dY_i = (dZ.B_i^T) * GeLU'(Y_i): t groups, M = T, N = fi, K = h
    {
        GemmParams p;
        base_params(p, *dev, s.T, s.fi, s.h, s.t, 1);
        choose_tile_width(p, *dev);
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_kmajor(&p.a_map[j], dZ[j], s.h, s.Tc, BM)) return TPMLP_ERR_UNSUPPORTED;
        p.a_part = PART_ROW;
        p.a_nmaps = s.chunks;
        p.b_nmaps = s.t;
        p.a_rows_per_map = s.Tc;
        for (int i = 0; i < s.t; ++i)
            if (!encode_kmajor(&p.b_map[i], B_shards[i], s.h, s.fi, B_ROWS))
                return TPMLP_ERR_UNSUPPORTED;
        p.b_part = PART_GROUP;
        p.b_rows_per_map = 0;
        for (int i = 0; i < s.t; ++i) {
            if (!encode_out(&p.out_map[i], shard_ptr(dY, i, s), s.fi, s.T, false))
                return TPMLP_ERR_UNSUPPORTED;
            // selective recompute: the same epilogue rebuilds H_i = GeLU(Y_i)
            if (recompute &&
                !encode_out(&p.out_map[MAX_MAPS + i], shard_ptr(H, i, s), s.fi, s.T, false))
                return TPMLP_ERR_UNSUPPORTED;
            p.in0[i] = shard_ptr(Y, i, s);
        }
        p.ld_in = s.fi;
        p.out_part = PART_GROUP;
        p.out_rows_per_part = 0;
        // db1 partial sums: one row per 32 token rows, the t shards side by side
        p.colsum_part = reinterpret_cast<float*>(R.part1);
        p.colsum_ld = s.f;
        if (!attach_split(p, R)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_DGRAD_H, 1, st,
                         [&] {
                             return recompute ? launch_dgrad_h_recompute(p, st)
                                              : launch_dgrad_h(p, st);
                         }));
    }
    // dX = sum_i dY_i.A_i^T: M = T, N = h, K = fi per segment
    {
        GemmParams p;
        base_params(p, *dev, s.T, s.h, s.fi, 1, s.t);
        choose_tile_width(p, *dev);
        for (int i = 0; i < s.t; ++i) {
            if (!encode_kmajor(&p.a_map[i], shard_ptr(dY, i, s), s.fi, s.T, BM))
                return TPMLP_ERR_UNSUPPORTED;
            if (!encode_kmajor(&p.b_map[i], A_shards[i], s.fi, s.h, B_ROWS))
                return TPMLP_ERR_UNSUPPORTED;
        }
        p.a_part = PART_KSEG;
        p.a_nmaps = s.t;
        p.b_nmaps = s.t;
        p.b_part = PART_KSEG;
        p.a_rows_per_map = p.b_rows_per_map = 0;
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_out(&p.out_map[j], dX[j], s.h, s.Tc, false)) return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_ROW;
        p.out_rows_per_part = s.Tc;
        if (!attach_split(p, R)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_DGRAD_X, 1, st,
                         [&] { return launch_dgrad_x(p, st); }));
    }
    // dB_i = H_i^T.dZ: t groups, M = fi, N = h, K = Tc per chunk segment
    {
        GemmParams p;
        base_params(p, *dev, s.fi, s.h, s.Tc, s.t, s.chunks);
        for (int i = 0; i < s.t; ++i)
            if (!encode_mnmajor(&p.a_map[i], shard_ptr(H, i, s), s.fi, s.T, &p.a_mn3d))
                return TPMLP_ERR_UNSUPPORTED;
        p.a_part = PART_GROUP;
        p.a_nmaps = s.t;
        p.b_nmaps = s.chunks;
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_mnmajor(&p.b_map[j], dZ[j], s.h, s.Tc, &p.b_mn3d)) return TPMLP_ERR_UNSUPPORTED;
        p.b_part = PART_KSEG;
        p.a_rows_per_map = p.b_rows_per_map = 0;
        for (int i = 0; i < s.t; ++i)
            if (!encode_out(&p.out_map[i], dB_shards[i], s.h, s.fi, true))
                return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_GROUP;
        p.out_rows_per_part = 0;
        if (!attach_split(p, R)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_WGRAD_B, 1, st,
                         [&] { return launch_wgrad(p, st); }));
    }
    // dA_i = X^T.dY_i: t groups, M = h, N = fi, K = Tc per chunk segment
    {
        GemmParams p;
        base_params(p, *dev, s.h, s.fi, s.Tc, s.t, s.chunks);
        for (int j = 0; j < s.chunks; ++j)
            if (!encode_mnmajor(&p.a_map[j], X[j], s.h, s.Tc, &p.a_mn3d)) return TPMLP_ERR_UNSUPPORTED;
        p.a_part = PART_KSEG;
        p.a_nmaps = s.chunks;
        p.b_nmaps = s.t;
        for (int i = 0; i < s.t; ++i)
            if (!encode_mnmajor(&p.b_map[i], shard_ptr(dY, i, s), s.fi, s.T, &p.b_mn3d))
                return TPMLP_ERR_UNSUPPORTED;
        p.b_part = PART_GROUP;
        p.a_rows_per_map = p.b_rows_per_map = 0;
        for (int i = 0; i < s.t; ++i)
            if (!encode_out(&p.out_map[i], dA_shards[i], s.fi, s.h, true))
                return TPMLP_ERR_UNSUPPORTED;
        p.out_part = PART_GROUP;
        p.out_rows_per_part = 0;
        if (!attach_split(p, R)) return TPMLP_ERR_UNSUPPORTED;
        TPMLP_CUDA(timed(TPMLP_KERNEL_WGRAD_A, 1, st,
                         [&] { return launch_wgrad(p, st); }));
    }
    // db1 = column sums of dY: the dH GEMM's epilogue summed each 32-row group
    // of its fp32 output; here the groups are added.  db2 = column sums of dZ.
    {
        const long long groups = (s.T + 31) / 32;
        TPMLP_CUDA(timed(TPMLP_KERNEL_BIAS_GRAD, 1, st, [&] {
            return launch_colsum_f32(reinterpret_cast<const float*>(R.part1), groups, s.f, s.f,
                                     static_cast<float*>(db1), st);
        }));

        if (db2_given) return TPMLP_OK;
        ColsumParams c2;
        std::memset(&c2, 0, sizeof(c2));
        for (int j = 0; j < s.chunks; ++j) c2.src[j] = dZ[j];
        c2.nparts = s.chunks;
        c2.rows_per_part = s.Tc;
        c2.ncols = s.h;
        c2.mode = CS_ROWS_CONCAT;
        c2.out = static_cast<float*>(db2);
        c2.partial = reinterpret_cast<float*>(R.part2);
        const dim3 g2 = colsum_plan(c2, dev->sm_count);
        TPMLP_CUDA(timed(TPMLP_KERNEL_BIAS_GRAD, c2.splits > 1 ? 2 : 1, st,
                         [&] { return launch_colsum(c2, g2, st, nullptr); }));
    }
    return TPMLP_OK;
}

}  // namespace block
}  // namespace tpmlp

using namespace tpmlp;
using namespace tpmlp::abi;
using namespace tpmlp::block;

// =========================================================================================
TPMLP_API const char* tpmlp_status_string(tpmlp_status s) {
    switch (s) {
        case TPMLP_OK: return "ok";
        case TPMLP_ERR_INVALID_ARG: return "invalid argument";
        case TPMLP_ERR_UNSUPPORTED: return "unsupported shape, alignment or device";
        case TPMLP_ERR_CUDA: return "CUDA error";
        case TPMLP_ERR_TIMEOUT: return "bounded device wait expired";
    }
    return "unknown status";
}

TPMLP_API size_t tpmlp_workspace_bytes(const tpmlp_dims* dims) {
    if (check_dims(dims) != TPMLP_OK) return 0;
    return layout_of(*dims).total;
}

TPMLP_API tpmlp_status tpmlp_workspace_layout(const tpmlp_dims* dims, size_t* y_offset,
                                              size_t* h_offset, size_t* dy_offset) {
    TPMLP_TRY(check_dims(dims));
    const Layout L = layout_of(*dims);
    if (y_offset) *y_offset = L.y;
    if (h_offset) *h_offset = L.h;
    if (dy_offset) *dy_offset = L.dy;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_set_split_min_kblocks(int kblocks) {
    if (kblocks < 0) return TPMLP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_split_min_kblocks = kblocks;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_set_head_prefetch(int kblocks) {
    if (kblocks < 0 || kblocks > 64) return TPMLP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_head_prefetch = kblocks;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_set_wide_tiles(int mode) {
    if (mode < 0 || mode > WIDE_TILES_DEEP_K) return TPMLP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_wide_tiles = mode;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_map_cache_stats(uint64_t* hits, uint64_t* misses,
                                              uint64_t* entries) {
    g_maps.stats(hits, misses, entries);
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_selftest_map_cache(uint64_t* out, int n) {
    // A private cache of capacity 4 with a stand-in encoder (no driver, no
    // GPU): the map's bytes are a function of its key, and each encoder call
    // is counted.
    if (!out || n < 8) return TPMLP_ERR_INVALID_ARG;
    MapCache cache(4);
    uint64_t calls = 0;
    auto fake = [&](const MapKey& k, CUtensorMap* m) {
        return cache.get(k, m, [&](CUtensorMap* o) {
            ++calls;
            std::memset(o, 0, sizeof(*o));
            std::memcpy(o, &k, sizeof(k) < sizeof(*o) ? sizeof(k) : sizeof(*o));
            return true;
        });
    };
    alignas(64) static char buf[4096];
    cuuint64_t dims[2] = {1024, 512};
    cuuint64_t strides[1] = {2048};
    cuuint32_t box[2] = {64, 128};
    const MapKey a = make_map_key(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf, dims, strides, box,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    const MapKey a_moved = make_map_key(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf + 256, dims,
                                        strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    cuuint32_t box2[2] = {64, 256};
    const MapKey a_box = make_map_key(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf, dims, strides, box2,
                                      CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    CUtensorMap m1, m2, m3, m4;
    fake(a, &m1);                                  // miss: encoded
    fake(a, &m2);                                  // hit: same key, not encoded again
    const bool same = std::memcmp(&m1, &m2, sizeof(m1)) == 0;
    fake(a_moved, &m3);                            // miss: new address
    fake(a_box, &m4);                              // miss: new box
    const bool moved_differs = std::memcmp(&m1, &m3, sizeof(m1)) != 0;
    for (int i = 0; i < 6; ++i) {                  // more keys than the capacity
        const MapKey k = make_map_key(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf + 512 + 16 * i,
                                      dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        CUtensorMap m;
        fake(k, &m);
    }
    uint64_t hits = 0, misses = 0, entries = 0;
    cache.stats(&hits, &misses, &entries);
    out[0] = hits;
    out[1] = misses;
    out[2] = calls;
    out[3] = entries;
    out[4] = same ? 1 : 0;
    out[5] = moved_differs ? 1 : 0;
    out[6] = 4;  // capacity
    out[7] = sizeof(MapKey);
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_set_wait_timeout_ns(uint64_t ns) {
    if (ns == 0) return TPMLP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    g_timeout_ns = ns;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_forward(const tpmlp_dims* dims, const void* const* X,
                                     const void* const* A_shards, const void* b1,
                                     const void* const* B_shards, const void* b2, int t,
                                     void* const* Z, void* workspace, void* stream) {
    TPMLP_TRY(check_dims(dims));
    if (t != dims->t) return TPMLP_ERR_INVALID_ARG;
    const Shapes s = shapes_of(*dims);
    TPMLP_TRY(check_ptrs(A_shards, s.t));
    TPMLP_TRY(check_ptrs(B_shards, s.t));
    TPMLP_TRY(check_ptr(b1));
    TPMLP_TRY(check_ptr(b2));
    if (s.T > 0) {
        TPMLP_TRY(check_ptrs(X, s.chunks));
        TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(Z), s.chunks));
        TPMLP_TRY(check_ptr(workspace));
    }
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    if (s.T == 0) return TPMLP_OK;
    return run_forward(s, dev, X, A_shards, b1, B_shards, b2, Z,
                       regions_of(static_cast<uint8_t*>(workspace), layout_of(*dims)),
                       static_cast<cudaStream_t>(stream), nullptr);
}

TPMLP_API tpmlp_status tpmlp_backward(const tpmlp_dims* dims, const void* const* dZ,
                                      const void* const* X, const void* const* A_shards,
                                      const void* const* B_shards, void* workspace,
                                      void* const* dX, void* const* dA_shards, void* db1,
                                      void* const* dB_shards, void* db2, void* stream) {
    TPMLP_TRY(check_dims(dims));
    const Shapes s = shapes_of(*dims);
    TPMLP_TRY(check_ptrs(A_shards, s.t));
    TPMLP_TRY(check_ptrs(B_shards, s.t));
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dA_shards), s.t));
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dB_shards), s.t));
    TPMLP_TRY(check_ptr(db1));
    TPMLP_TRY(check_ptr(db2));
    if (s.T > 0) {
        TPMLP_TRY(check_ptrs(dZ, s.chunks));
        TPMLP_TRY(check_ptrs(X, s.chunks));
        TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dX), s.chunks));
        TPMLP_TRY(check_ptr(workspace));
    }
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s.T == 0) return zero_weight_grads(s, dA_shards, db1, dB_shards, db2, st);
    return run_backward(s, dev, dZ, X, A_shards, B_shards, dX, dA_shards, db1, dB_shards, db2,
                        regions_of(static_cast<uint8_t*>(workspace), layout_of(*dims)), false, st);
}

TPMLP_API tpmlp_status tpmlp_recompute_workspace_bytes(const tpmlp_dims* dims, size_t* saved_bytes,
                                                       size_t* scratch_bytes) {
    TPMLP_TRY(check_dims(dims));
    const Layout L = layout_of(*dims);
    if (saved_bytes) *saved_bytes = L.h;            // the Y shards
    if (scratch_bytes) *scratch_bytes = L.total - L.h;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_forward_recompute(const tpmlp_dims* dims, const void* const* X,
                                               const void* const* A_shards, const void* b1,
                                               const void* const* B_shards, const void* b2,
                                               int t, void* const* Z, void* saved, void* scratch,
                                               void* stream) {
    TPMLP_TRY(check_dims(dims));
    if (t != dims->t) return TPMLP_ERR_INVALID_ARG;
    const Shapes s = shapes_of(*dims);
    TPMLP_TRY(check_ptrs(A_shards, s.t));
    TPMLP_TRY(check_ptrs(B_shards, s.t));
    TPMLP_TRY(check_ptr(b1));
    TPMLP_TRY(check_ptr(b2));
    if (s.T > 0) {
        TPMLP_TRY(check_ptrs(X, s.chunks));
        TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(Z), s.chunks));
        TPMLP_TRY(check_ptr(saved));
        TPMLP_TRY(check_ptr(scratch));
    }
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    if (s.T == 0) return TPMLP_OK;
    return run_forward(s, dev, X, A_shards, b1, B_shards, b2, Z,
                       recompute_regions(static_cast<uint8_t*>(saved),
                                         static_cast<uint8_t*>(scratch), layout_of(*dims)),
                       static_cast<cudaStream_t>(stream), nullptr);
}

TPMLP_API tpmlp_status tpmlp_backward_recompute(const tpmlp_dims* dims, const void* const* dZ,
                                                const void* const* X,
                                                const void* const* A_shards,
                                                const void* const* B_shards, void* saved,
                                                void* scratch, void* const* dX,
                                                void* const* dA_shards, void* db1,
                                                void* const* dB_shards, void* db2,
                                                void* stream) {
    TPMLP_TRY(check_dims(dims));
    const Shapes s = shapes_of(*dims);
    TPMLP_TRY(check_ptrs(A_shards, s.t));
    TPMLP_TRY(check_ptrs(B_shards, s.t));
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dA_shards), s.t));
    TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dB_shards), s.t));
    TPMLP_TRY(check_ptr(db1));
    TPMLP_TRY(check_ptr(db2));
    if (s.T > 0) {
        TPMLP_TRY(check_ptrs(dZ, s.chunks));
        TPMLP_TRY(check_ptrs(X, s.chunks));
        TPMLP_TRY(check_ptrs(reinterpret_cast<const void* const*>(dX), s.chunks));
        TPMLP_TRY(check_ptr(saved));
        TPMLP_TRY(check_ptr(scratch));
    }
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s.T == 0) return zero_weight_grads(s, dA_shards, db1, dB_shards, db2, st);
    return run_backward(s, dev, dZ, X, A_shards, B_shards, dX, dA_shards, db1, dB_shards, db2,
                        recompute_regions(static_cast<uint8_t*>(saved),
                                          static_cast<uint8_t*>(scratch), layout_of(*dims)),
                        true, st);
}

TPMLP_API tpmlp_status tpmlp_sync_check(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return TPMLP_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return TPMLP_ERR_CUDA;
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    unsigned int word = 0;
    if (cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TPMLP_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(dev->err, 0, sizeof(word)) != cudaSuccess) return TPMLP_ERR_CUDA;
        return TPMLP_ERR_TIMEOUT;
    }
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_selftest_stalled_gemm(const void* a, const void* b, void* c,
                                                   uint64_t timeout_ns, void* stream) {
    TPMLP_TRY(check_ptr(a));
    TPMLP_TRY(check_ptr(b));
    TPMLP_TRY(check_ptr(c));
    if (timeout_ns == 0) return TPMLP_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    TPMLP_TRY(device_info(&dev));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    GemmParams p;
    base_params(p, *dev, BM, BN, BK, 1, 1);
    if (!encode_kmajor(&p.a_map[0], a, BK, BM, BM)) return TPMLP_ERR_UNSUPPORTED;
    if (!encode_kmajor(&p.b_map[0], b, BK, BN, B_ROWS)) return TPMLP_ERR_UNSUPPORTED;
    p.a_part = p.b_part = PART_SINGLE;
    p.a_rows_per_map = p.b_rows_per_map = 0;
    if (!encode_out(&p.out_map[0], c, BN, BM, false)) return TPMLP_ERR_UNSUPPORTED;
    p.out_part = PART_GROUP;
    p.out_rows_per_part = 0;
    p.timeout_ns = timeout_ns;
    p.stall_producer = 1;
    TPMLP_CUDA(launch_dgrad_x(p, st));
    return tpmlp_sync_check(stream);
}

TPMLP_API tpmlp_status tpmlp_profile_begin_kinds(int capacity, uint32_t kinds) {
    if (capacity <= 0 || kinds == 0 || (kinds >> TPMLP_KERNEL_KINDS) != 0)
        return TPMLP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_kinds = kinds;
    for (auto& r : g_prof_pool) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_prof_pool.assign(static_cast<size_t>(capacity), ProfRec{0, 0, nullptr, nullptr});
    for (auto& r : g_prof_pool) {
        if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess)
            return TPMLP_ERR_CUDA;
    }
    g_prof_used = 0;
    g_prof_on = true;
    return TPMLP_OK;
}

TPMLP_API tpmlp_status tpmlp_profile_begin(int capacity) {
    return tpmlp_profile_begin_kinds(capacity, (1u << TPMLP_KERNEL_KINDS) - 1u);
}

TPMLP_API int tpmlp_profile_end(double* ms, int* launches, int nkinds) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return -1;
    g_prof_on = false;
    for (int k = 0; k < nkinds; ++k) {
        if (ms) ms[k] = 0.0;
        if (launches) launches[k] = 0;
    }
    int n = 0;
    bool ok = true;
    for (size_t i = 0; i < g_prof_used; ++i) {
        ProfRec& r = g_prof_pool[i];
        if (cudaEventSynchronize(r.b) != cudaSuccess) {
            ok = false;
            continue;
        }
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
            ok = false;
            continue;
        }
        if (r.kind >= 0 && r.kind < nkinds) {
            if (ms) ms[r.kind] += t;
            if (launches) launches[r.kind] += r.kernels;
        }
        ++n;
    }
    for (auto& r : g_prof_pool) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_prof_pool.clear();
    g_prof_used = 0;
    return ok ? n : -1;
}

TPMLP_API const char* tpmlp_kernel_name(int kind) {
    switch (kind) {
        case TPMLP_KERNEL_COLUMN_FWD: return "column_fwd";
        case TPMLP_KERNEL_ROW_FWD: return "row_fwd";
        case TPMLP_KERNEL_DGRAD_H: return "dgrad_h";
        case TPMLP_KERNEL_DGRAD_X: return "dgrad_x";
        case TPMLP_KERNEL_WGRAD_B: return "wgrad_b";
        case TPMLP_KERNEL_WGRAD_A: return "wgrad_a";
        case TPMLP_KERNEL_BIAS_GRAD: return "bias_grad";
        case TPMLP_KERNEL_LINEAR_FWD: return "linear_fwd";
        case TPMLP_KERNEL_LINEAR_DGRAD: return "linear_dgrad";
        case TPMLP_KERNEL_LINEAR_WGRAD: return "linear_wgrad";
        case TPMLP_KERNEL_LAYERNORM_FWD: return "layernorm_fwd";
        case TPMLP_KERNEL_LAYERNORM_BWD: return "layernorm_bwd";
        case TPMLP_KERNEL_DROPOUT_BWD: return "dropout_bwd";
        case TPMLP_KERNEL_SP_COPY: return "sp_copy";
    }
    return "unknown";
}
