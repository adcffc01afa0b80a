"""ctypes binding of libtpmlp (include/tpmlp.h), same names as the C ABI.

Argument marshalling only: torch tensors become device pointers, lists become
host pointer arrays, a non-OK status becomes a :class:`TpmlpError`.  Every step
of the MLP block and of the linear layers runs in the library's CUDA kernels.  There is no fallback: if
the library has not been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libtpmlp.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libtpmlp.so is not built ({_LIB_PATH}); run "
        "`python -m tensor_transformer_mlp_gemm_gb300.build` (nvcc, sm_103a)")

_lib = ctypes.CDLL(_LIB_PATH)

TPMLP_OK = 0
TPMLP_ERR_INVALID_ARG = 1
TPMLP_ERR_UNSUPPORTED = 2
TPMLP_ERR_CUDA = 3
TPMLP_ERR_TIMEOUT = 4

KERNEL_KINDS = 14

# every symbol include/tpmlp.h declares
EXPORTED = (
    "tpmlp_workspace_bytes", "tpmlp_workspace_layout", "tpmlp_forward", "tpmlp_backward",
    "tpmlp_status_string", "tpmlp_sync_check", "tpmlp_set_wait_timeout_ns",
    "tpmlp_selftest_stalled_gemm", "tpmlp_profile_begin", "tpmlp_profile_begin_kinds",
    "tpmlp_profile_end",
    "tpmlp_kernel_name", "tpmlp_column_sums_noalloc", "tpmlp_set_split_min_kblocks",
    "tpmlp_recompute_workspace_bytes", "tpmlp_forward_recompute", "tpmlp_backward_recompute",
    "tpmlp_linear_workspace_bytes", "tpmlp_column_linear_forward", "tpmlp_column_linear_backward",
    "tpmlp_row_linear_forward", "tpmlp_row_linear_backward",
    "tpmlp_sp_workspace_bytes", "tpmlp_sp_workspace_layout", "tpmlp_sp_forward", "tpmlp_sp_backward",
    "tpmlp_set_head_prefetch", "tpmlp_map_cache_stats", "tpmlp_selftest_map_cache",
    "tpmlp_set_wide_tiles", "tpmlp_sp_gather", "tpmlp_sp_scatter",
)


class tpmlp_dims(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("t", ctypes.c_int32), ("seq_chunks", ctypes.c_int32)]


class tpmlp_linear_dims(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("in_features", ctypes.c_int64),
                ("out_features", ctypes.c_int64), ("t", ctypes.c_int32),
                ("seq_chunks", ctypes.c_int32)]


class tpmlp_sp_params(ctypes.Structure):
    _fields_ = [("eps", ctypes.c_float), ("dropout_p", ctypes.c_double),
                ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64)]


class TpmlpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tpmlp_status_string(status)} (status {status})")


_vp = ctypes.c_void_p
_vpp = ctypes.POINTER(ctypes.c_void_p)
_dims_p = ctypes.POINTER(tpmlp_dims)
_sz_p = ctypes.POINTER(ctypes.c_size_t)
_ldims_p = ctypes.POINTER(tpmlp_linear_dims)
_sp_p = ctypes.POINTER(tpmlp_sp_params)

_lib.tpmlp_workspace_bytes.restype = ctypes.c_size_t
_lib.tpmlp_workspace_bytes.argtypes = [_dims_p]
_lib.tpmlp_workspace_layout.restype = ctypes.c_int
_lib.tpmlp_workspace_layout.argtypes = [_dims_p, _sz_p, _sz_p, _sz_p]
_lib.tpmlp_forward.restype = ctypes.c_int
_lib.tpmlp_forward.argtypes = [_dims_p, _vpp, _vpp, _vp, _vpp, _vp, ctypes.c_int, _vpp, _vp, _vp]
_lib.tpmlp_backward.restype = ctypes.c_int
_lib.tpmlp_backward.argtypes = [_dims_p, _vpp, _vpp, _vpp, _vpp, _vp, _vpp, _vpp, _vp, _vpp, _vp, _vp]
_lib.tpmlp_recompute_workspace_bytes.restype = ctypes.c_int
_lib.tpmlp_recompute_workspace_bytes.argtypes = [_dims_p, _sz_p, _sz_p]
_lib.tpmlp_forward_recompute.restype = ctypes.c_int
_lib.tpmlp_forward_recompute.argtypes = [_dims_p, _vpp, _vpp, _vp, _vpp, _vp, ctypes.c_int, _vpp,
                                         _vp, _vp, _vp]
_lib.tpmlp_backward_recompute.restype = ctypes.c_int
_lib.tpmlp_backward_recompute.argtypes = [_dims_p, _vpp, _vpp, _vpp, _vpp, _vp, _vp, _vpp, _vpp,
                                          _vp, _vpp, _vp, _vp]
_u64p = ctypes.POINTER(ctypes.c_uint64)
_lib.tpmlp_map_cache_stats.restype = ctypes.c_int
_lib.tpmlp_map_cache_stats.argtypes = [_u64p, _u64p, _u64p]
_lib.tpmlp_selftest_map_cache.restype = ctypes.c_int
_lib.tpmlp_selftest_map_cache.argtypes = [_u64p, ctypes.c_int]
_lib.tpmlp_sp_gather.restype = ctypes.c_int
_lib.tpmlp_sp_gather.argtypes = [_dims_p, _vpp, ctypes.c_int64, _vp, _vp]
_lib.tpmlp_sp_scatter.restype = ctypes.c_int
_lib.tpmlp_sp_scatter.argtypes = [_dims_p, _vp, ctypes.c_int64, _vpp, _vp]
_lib.tpmlp_status_string.restype = ctypes.c_char_p
_lib.tpmlp_status_string.argtypes = [ctypes.c_int]
_lib.tpmlp_sync_check.restype = ctypes.c_int
_lib.tpmlp_sync_check.argtypes = [_vp]
_lib.tpmlp_set_split_min_kblocks.restype = ctypes.c_int
_lib.tpmlp_set_split_min_kblocks.argtypes = [ctypes.c_int]
_lib.tpmlp_set_head_prefetch.restype = ctypes.c_int
_lib.tpmlp_set_head_prefetch.argtypes = [ctypes.c_int]
_lib.tpmlp_set_wait_timeout_ns.restype = ctypes.c_int
_lib.tpmlp_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
_lib.tpmlp_selftest_stalled_gemm.restype = ctypes.c_int
_lib.tpmlp_selftest_stalled_gemm.argtypes = [_vp, _vp, _vp, ctypes.c_uint64, _vp]
_lib.tpmlp_profile_begin.restype = ctypes.c_int
_lib.tpmlp_profile_begin.argtypes = [ctypes.c_int]
_lib.tpmlp_profile_begin_kinds.restype = ctypes.c_int
_lib.tpmlp_profile_begin_kinds.argtypes = [ctypes.c_int, ctypes.c_uint32]
_lib.tpmlp_profile_end.restype = ctypes.c_int
_lib.tpmlp_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int),
                                   ctypes.c_int]
_lib.tpmlp_kernel_name.restype = ctypes.c_char_p
_lib.tpmlp_kernel_name.argtypes = [ctypes.c_int]
_lib.tpmlp_column_sums_noalloc.restype = ctypes.c_int
_lib.tpmlp_column_sums_noalloc.argtypes = [_vp, ctypes.c_int64, ctypes.c_int64, _vp, _vp]
_lib.tpmlp_sp_workspace_bytes.restype = ctypes.c_size_t
_lib.tpmlp_sp_workspace_bytes.argtypes = [_dims_p]
_lib.tpmlp_sp_workspace_layout.restype = ctypes.c_int
_lib.tpmlp_sp_workspace_layout.argtypes = [_dims_p, _sz_p, _sz_p]
_lib.tpmlp_sp_forward.restype = ctypes.c_int
_lib.tpmlp_sp_forward.argtypes = [_dims_p, _sp_p, _vpp, _vp, _vp, _vpp, _vp, _vpp, _vp, ctypes.c_int,
                                  _vpp, _vp, _vp]
_lib.tpmlp_sp_backward.restype = ctypes.c_int
_lib.tpmlp_sp_backward.argtypes = [_dims_p, _sp_p, _vpp, _vpp, _vp, _vpp, _vpp, _vp, _vpp, _vp, _vp,
                                   _vpp, _vp, _vpp, _vp, _vp]
_lib.tpmlp_linear_workspace_bytes.restype = ctypes.c_size_t
_lib.tpmlp_linear_workspace_bytes.argtypes = [_ldims_p]
for _name in ("tpmlp_column_linear_forward", "tpmlp_row_linear_forward"):
    getattr(_lib, _name).restype = ctypes.c_int
    getattr(_lib, _name).argtypes = [_ldims_p, _vpp, _vpp, _vp, _vpp, _vp, _vp]
for _name in ("tpmlp_column_linear_backward", "tpmlp_row_linear_backward"):
    getattr(_lib, _name).restype = ctypes.c_int
    getattr(_lib, _name).argtypes = [_ldims_p, _vpp, _vpp, _vpp, _vpp, _vpp, _vp, _vp, _vp]


def library_path() -> str:
    return _LIB_PATH


def library():
    return _lib


def make_dims(tokens: int, hidden: int, ffn: int, t: int, seq_chunks: int = 1) -> tpmlp_dims:
    return tpmlp_dims(int(tokens), int(hidden), int(ffn), int(t), int(seq_chunks))


def make_linear_dims(tokens: int, in_features: int, out_features: int, t: int,
                     seq_chunks: int = 1) -> tpmlp_linear_dims:
    return tpmlp_linear_dims(int(tokens), int(in_features), int(out_features), int(t),
                             int(seq_chunks))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _arr(xs):
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != TPMLP_OK:
        raise TpmlpError(status, where)


def tpmlp_status_string(status: int) -> str:
    return _lib.tpmlp_status_string(int(status)).decode()


def tpmlp_kernel_name(kind: int) -> str:
    return _lib.tpmlp_kernel_name(int(kind)).decode()


def tpmlp_workspace_bytes(dims: tpmlp_dims) -> int:
    return int(_lib.tpmlp_workspace_bytes(ctypes.byref(dims)))


def tpmlp_workspace_layout(dims: tpmlp_dims) -> tuple[int, int, int]:
    y, h, dy = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.tpmlp_workspace_layout(ctypes.byref(dims), ctypes.byref(y), ctypes.byref(h),
                                       ctypes.byref(dy)), "tpmlp_workspace_layout")
    return y.value, h.value, dy.value


def tpmlp_forward(dims, X, A_shards, b1, B_shards, b2, t, Z, workspace, stream=None) -> None:
    """X, Z: lists of seq_chunks tensors; A_shards, B_shards: lists of t tensors."""
    _check(_lib.tpmlp_forward(ctypes.byref(dims), _arr(X), _arr(A_shards), _ptr(b1),
                              _arr(B_shards), _ptr(b2), int(t), _arr(Z), _ptr(workspace),
                              _stream(stream)), "tpmlp_forward")


def tpmlp_backward(dims, dZ, X, A_shards, B_shards, workspace, dX, dA_shards, db1, dB_shards,
                   db2, stream=None) -> None:
    _check(_lib.tpmlp_backward(ctypes.byref(dims), _arr(dZ), _arr(X), _arr(A_shards),
                               _arr(B_shards), _ptr(workspace), _arr(dX), _arr(dA_shards),
                               _ptr(db1), _arr(dB_shards), _ptr(db2), _stream(stream)),
           "tpmlp_backward")


def tpmlp_recompute_workspace_bytes(dims: tpmlp_dims) -> tuple[int, int]:
    """(saved bytes kept from forward to backward, scratch bytes used during a call)."""
    sv, sc = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.tpmlp_recompute_workspace_bytes(ctypes.byref(dims), ctypes.byref(sv),
                                                ctypes.byref(sc)), "tpmlp_recompute_workspace_bytes")
    return sv.value, sc.value


def tpmlp_forward_recompute(dims, X, A_shards, b1, B_shards, b2, t, Z, saved, scratch,
                            stream=None) -> None:
    _check(_lib.tpmlp_forward_recompute(ctypes.byref(dims), _arr(X), _arr(A_shards), _ptr(b1),
                                        _arr(B_shards), _ptr(b2), int(t), _arr(Z), _ptr(saved),
                                        _ptr(scratch), _stream(stream)),
           "tpmlp_forward_recompute")


def tpmlp_backward_recompute(dims, dZ, X, A_shards, B_shards, saved, scratch, dX, dA_shards,
                             db1, dB_shards, db2, stream=None) -> None:
    _check(_lib.tpmlp_backward_recompute(ctypes.byref(dims), _arr(dZ), _arr(X), _arr(A_shards),
                                         _arr(B_shards), _ptr(saved), _ptr(scratch), _arr(dX),
                                         _arr(dA_shards), _ptr(db1), _arr(dB_shards), _ptr(db2),
                                         _stream(stream)),
           "tpmlp_backward_recompute")


def tpmlp_sync_check(stream=None) -> int:
    """Returns the status (does not raise), so callers can test for TIMEOUT."""
    return int(_lib.tpmlp_sync_check(_stream(stream)))


def tpmlp_set_split_min_kblocks(kblocks: int) -> None:
    _check(_lib.tpmlp_set_split_min_kblocks(int(kblocks)), "tpmlp_set_split_min_kblocks")


def tpmlp_set_head_prefetch(kblocks: int) -> None:
    _check(_lib.tpmlp_set_head_prefetch(int(kblocks)), "tpmlp_set_head_prefetch")


WIDE_TILES_DEFAULT = 3


def tpmlp_set_wide_tiles(mode: int) -> None:
    """0: 256-wide GEMM tiles; 1: 512-wide where they fill the waves as well;
    2: 512-wide wherever allowed; 3 (default): 512-wide for GEMMs of at least
    256 K steps."""
    _check(_lib.tpmlp_set_wide_tiles(int(mode)), "tpmlp_set_wide_tiles")


def tpmlp_map_cache_stats() -> dict:
    """Hits, misses (encodings) and entries of the library's tensor-map cache."""
    v = [ctypes.c_uint64() for _ in range(3)]
    _check(_lib.tpmlp_map_cache_stats(*[ctypes.byref(x) for x in v]), "tpmlp_map_cache_stats")
    return {"hits": v[0].value, "misses": v[1].value, "entries": v[2].value}


def tpmlp_selftest_map_cache() -> dict:
    """The cache logic's host self-test (see include/tpmlp.h)."""
    out = (ctypes.c_uint64 * 8)()
    _check(_lib.tpmlp_selftest_map_cache(out, 8), "tpmlp_selftest_map_cache")
    keys = ("hits", "misses", "encoder_calls", "entries", "hit_same_bytes", "new_address_differs",
            "capacity", "key_bytes")
    return dict(zip(keys, [int(x) for x in out]))


def tpmlp_set_wait_timeout_ns(ns: int) -> None:
    _check(_lib.tpmlp_set_wait_timeout_ns(int(ns)), "tpmlp_set_wait_timeout_ns")


def tpmlp_selftest_stalled_gemm(a, b, c, timeout_ns: int, stream=None) -> int:
    return int(_lib.tpmlp_selftest_stalled_gemm(_ptr(a), _ptr(b), _ptr(c), int(timeout_ns),
                                                _stream(stream)))


def tpmlp_profile_begin(capacity: int) -> None:
    _check(_lib.tpmlp_profile_begin(int(capacity)), "tpmlp_profile_begin")


def tpmlp_profile_begin_kinds(capacity: int, kinds) -> None:
    """Profile only the named kernel kinds (names as tpmlp_kernel_name)."""
    names = [tpmlp_kernel_name(k) for k in range(KERNEL_KINDS)]
    mask = 0
    for k in kinds:
        mask |= 1 << names.index(k)
    _check(_lib.tpmlp_profile_begin_kinds(int(capacity), mask), "tpmlp_profile_begin_kinds")


def tpmlp_profile_end() -> tuple[dict, dict]:
    ms = (ctypes.c_double * KERNEL_KINDS)()
    cnt = (ctypes.c_int * KERNEL_KINDS)()
    n = _lib.tpmlp_profile_end(ms, cnt, KERNEL_KINDS)
    if n < 0:
        raise TpmlpError(TPMLP_ERR_CUDA, "tpmlp_profile_end")
    names = [tpmlp_kernel_name(k) for k in range(KERNEL_KINDS)]
    return ({names[k]: ms[k] for k in range(KERNEL_KINDS)},
            {names[k]: cnt[k] for k in range(KERNEL_KINDS)})


def tpmlp_sp_gather(dims, chunks, cols: int, out, stream=None) -> None:
    """out [T, cols] = the seq_chunks chunks concatenated along tokens."""
    _check(_lib.tpmlp_sp_gather(ctypes.byref(dims), _arr(chunks), int(cols), _ptr(out),
                                _stream(stream)), "tpmlp_sp_gather")


def tpmlp_sp_scatter(dims, src, cols: int, chunks, stream=None) -> None:
    """The seq_chunks chunks = the token-row blocks of src [T, cols]."""
    _check(_lib.tpmlp_sp_scatter(ctypes.byref(dims), _ptr(src), int(cols), _arr(chunks),
                                 _stream(stream)), "tpmlp_sp_scatter")


def tpmlp_column_sums_noalloc(src, rows: int, cols: int, out, stream=None) -> int:
    """Column sums of bf16 src [rows, cols] into fp32 out [cols] with no device
    allocation (library-owned static scratch).  Returns the status."""
    return int(_lib.tpmlp_column_sums_noalloc(_ptr(src), int(rows), int(cols), _ptr(out),
                                              _stream(stream)))


def tpmlp_linear_workspace_bytes(dims: tpmlp_linear_dims) -> int:
    """Scratch bytes of any linear-layer call with these dims (0 if invalid)."""
    return int(_lib.tpmlp_linear_workspace_bytes(ctypes.byref(dims)))


def tpmlp_column_linear_forward(dims, X, W_shards, b, Y_shards, workspace, stream=None) -> None:
    """X: seq_chunks tensors [Tc, in]; W_shards, Y_shards: t tensors."""
    _check(_lib.tpmlp_column_linear_forward(ctypes.byref(dims), _arr(X), _arr(W_shards), _ptr(b),
                                            _arr(Y_shards), _ptr(workspace), _stream(stream)),
           "tpmlp_column_linear_forward")


def tpmlp_column_linear_backward(dims, dY_shards, X, W_shards, dX, dW_shards, db, workspace,
                                 stream=None) -> None:
    _check(_lib.tpmlp_column_linear_backward(ctypes.byref(dims), _arr(dY_shards), _arr(X),
                                             _arr(W_shards), _arr(dX), _arr(dW_shards), _ptr(db),
                                             _ptr(workspace), _stream(stream)),
           "tpmlp_column_linear_backward")


def tpmlp_row_linear_forward(dims, X_shards, W_shards, b, Z, workspace, stream=None) -> None:
    """X_shards, W_shards: t tensors; Z: seq_chunks tensors [Tc, out]."""
    _check(_lib.tpmlp_row_linear_forward(ctypes.byref(dims), _arr(X_shards), _arr(W_shards),
                                         _ptr(b), _arr(Z), _ptr(workspace), _stream(stream)),
           "tpmlp_row_linear_forward")


def tpmlp_row_linear_backward(dims, dZ, X_shards, W_shards, dX_shards, dW_shards, db, workspace,
                              stream=None) -> None:
    _check(_lib.tpmlp_row_linear_backward(ctypes.byref(dims), _arr(dZ), _arr(X_shards),
                                          _arr(W_shards), _arr(dX_shards), _arr(dW_shards),
                                          _ptr(db), _ptr(workspace), _stream(stream)),
           "tpmlp_row_linear_backward")


def make_sp_params(eps: float = 1e-5, dropout_p: float = 0.1, seed: int = 0,
                   offset: int = 0) -> tpmlp_sp_params:
    return tpmlp_sp_params(float(eps), float(dropout_p), int(seed) & (2**64 - 1),
                           int(offset) & (2**64 - 1))


def tpmlp_sp_workspace_bytes(dims: tpmlp_dims) -> int:
    return int(_lib.tpmlp_sp_workspace_bytes(ctypes.byref(dims)))


def tpmlp_sp_workspace_layout(dims: tpmlp_dims) -> tuple[int, int]:
    xn, dz = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.tpmlp_sp_workspace_layout(ctypes.byref(dims), ctypes.byref(xn), ctypes.byref(dz)),
           "tpmlp_sp_workspace_layout")
    return xn.value, dz.value


def tpmlp_sp_forward(dims, sp, X, gamma, beta, A_shards, b1, B_shards, b2, t, Out, workspace,
                     stream=None) -> None:
    """X, Out: lists of seq_chunks tensors; A_shards, B_shards: lists of t tensors."""
    _check(_lib.tpmlp_sp_forward(ctypes.byref(dims), ctypes.byref(sp), _arr(X), _ptr(gamma),
                                 _ptr(beta), _arr(A_shards), _ptr(b1), _arr(B_shards), _ptr(b2),
                                 int(t), _arr(Out), _ptr(workspace), _stream(stream)),
           "tpmlp_sp_forward")


def tpmlp_sp_backward(dims, sp, dOut, X, gamma, A_shards, B_shards, workspace, dX, dgamma, dbeta,
                      dA_shards, db1, dB_shards, db2, stream=None) -> None:
    _check(_lib.tpmlp_sp_backward(ctypes.byref(dims), ctypes.byref(sp), _arr(dOut), _arr(X),
                                  _ptr(gamma), _arr(A_shards), _arr(B_shards), _ptr(workspace),
                                  _arr(dX), _ptr(dgamma), _ptr(dbeta), _arr(dA_shards), _ptr(db1),
                                  _arr(dB_shards), _ptr(db2), _stream(stream)),
           "tpmlp_sp_backward")
