// abi_internal.h -- host-side helpers shared by the C-ABI translation units:
// tpmlp.cu (the MLP block) and linear.cu (the column- and row-parallel linear
// layers).  Device lookup, TMA tensor-map encoding, argument checks, GEMM
// parameter set-up and the per-kernel profiling events.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "gemm_params.h"
#include "tpmlp.h"

namespace tpmlp {
namespace abi {

constexpr int kMaxShards = 8;
constexpr int kBand = 8;  // cluster M-tiles (256 rows each) per raster band

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    unsigned int* err = nullptr;  // the device error word
};

// The current device's record (looked up once per device): TPMLP_ERR_UNSUPPORTED
// on anything but an sm_103 device.
tpmlp_status device_info(DeviceInfo** out);

// ---- tensor maps (bf16 row-major operands, 128-byte swizzle) -------------------------
//   K-major operand [rows, K]: box {BK, box_rows}
//   MN-major operand [K, rows]: box {64, BK}
//   output [rows, cols], bf16 or fp32: box 32 x 32 for the epilogue's stores
bool encode_kmajor(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, int box_rows);
// MN-major maps are 3-D {64, K, rows / 64} when rows is a multiple of 64 (one
// copy per box of box_rows rows), else 2-D; *mn3d (the operand's GemmParams
// flag) says which.
bool encode_mnmajor(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t K, int* mn3d,
                    int box_rows = BM);
// Both tile widths stage B in boxes of B_ROWS rows (a wide tile's two halves
// are two such boxes), so the operand maps do not depend on the tile width.
bool encode_out(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, bool f32);

// ---- workspace pieces ------------------------------------------------------------------
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
// tail-split partial tiles: fp32 [MAX_SPLIT_UNITS * CLUSTER_M, BN]
inline size_t split_part_bytes() {
    return align256(static_cast<size_t>(MAX_SPLIT_UNITS) * CLUSTER_M * BN * 4);
}
// tail-split arrival counters: int [MAX_SPLIT_UNITS][2]
inline size_t split_cnt_bytes() {
    return align256(static_cast<size_t>(MAX_SPLIT_UNITS) * 2 * sizeof(int));
}

// ---- validation ------------------------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Each of the n pointers non-null (else INVALID_ARG) and 16-byte aligned (else UNSUPPORTED).
tpmlp_status check_ptrs(const void* const* arr, int n);
tpmlp_status check_ptr(const void* p);

#define TPMLP_TRY(expr)                \
    do {                               \
        tpmlp_status _s = (expr);      \
        if (_s != TPMLP_OK) return _s; \
    } while (0)

#define TPMLP_CUDA(expr)                                  \
    do {                                                  \
        if ((expr) != cudaSuccess) return TPMLP_ERR_CUDA; \
    } while (0)

// ---- GEMM set-up -----------------------------------------------------------------------
// Zeroed parameters for an M x N x K GEMM over `groups` groups and `ksegs`
// K segments, with the device's error word and the current wait limit.
void base_params(GemmParams& p, const DeviceInfo& dev, int M, int N, int K, int groups,
                 int ksegs);
// Chooses the tile width of a GEMM with a bf16 output by the policy of
// tpmlp_set_wide_tiles (by default wide tiles for GEMMs of at least
// WIDE_MIN_KSTEPS K steps; K and ksegs must be set) and sets tn, ntiles and
// total_tiles.  The B maps are encoded after this.
void choose_tile_width(GemmParams& p, const DeviceInfo& dev);
// Points the tail split at its workspace buffers (split_part_bytes() and
// split_cnt_bytes() long).
bool attach_split(GemmParams& p, void* split_part, void* split_cnt);

// ---- profiling events ------------------------------------------------------------------
struct ProfRec {
    int kind;
    int kernels;  // kernel launches between the two events
    cudaEvent_t a, b;
};
// The next free event pair while profiling is on, else nullptr.
ProfRec* prof_next(int kind, int kernels);

template <typename F>
cudaError_t timed(int kind, int kernels, cudaStream_t s, F&& launch) {
    ProfRec* r = prof_next(kind, kernels);
    if (r) cudaEventRecord(r->a, s);
    cudaError_t e = launch();
    if (r) cudaEventRecord(r->b, s);
    return e;
}

}  // namespace abi
}  // namespace tpmlp
