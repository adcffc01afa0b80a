"""fp64 CPU oracle for the tensor-parallel Transformer MLP block, the
column- and row-parallel linear layers it is built from, and the
sequence-parallel LayerNorm / Dropout sublayer around it.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports it, and it never
imports the product path.

The arithmetic lives in ``oracle.c`` (plain fp64 loops, OpenMP over output
rows); this module only compiles it with the host C compiler, converts arrays
to contiguous float64 and passes pointers.  The sequence-parallel helpers
concatenate and split along the token dimension, which is the definition of
the sequence-parallel gather / reduce-scatter ("并行训练范式 / 序列并行" on
"Megatron-LM：NVIDIA 的大规模并行训练方案").
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_dpp = ctypes.POINTER(_dp)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with the host C compiler."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    lib.oracle_gelu.restype = ctypes.c_double
    lib.oracle_gelu.argtypes = [ctypes.c_double]
    lib.oracle_gelu_grad.restype = ctypes.c_double
    lib.oracle_gelu_grad.argtypes = [ctypes.c_double]
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_get_threads.restype = ctypes.c_int
    dims = [_i64, _i64, _i64, ctypes.c_int]
    lib.oracle_forward.argtypes = dims + [_dp, _dpp, _dp, _dpp, _dp, _dpp, _dpp, _dp]
    lib.oracle_backward.argtypes = dims + [_dp, _dpp, _dpp, _dpp, _dpp, _dp,
                                           _dpp, _dp, _dpp, _dp, _dpp, _dp]
    lib.oracle_rows.argtypes = dims + [_dp, _dpp, _dp, _dpp, _dp, _dp,
                                       _i64, ctypes.POINTER(_i64), _dp, _dp, _dp, _dp, _dp]
    lib.oracle_sp_rows.argtypes = dims + [_dp, _dp, _dp, ctypes.c_double, _dpp, _dp, _dpp, _dp,
                                          ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_double, _dp, _i64, ctypes.POINTER(_i64),
                                          _dp, _dp]
    lib.oracle_cols.argtypes = dims + [_dp, _dpp, _dp, _dpp, _dp,
                                       _i64, ctypes.POINTER(_i64), _dp, _dp, _dp]
    lib.oracle_db2.argtypes = [_i64, _i64, _dp, _dp]
    lib.oracle_column_linear_forward.argtypes = dims + [_dp, _dpp, _dp, _dpp]
    lib.oracle_column_linear_backward.argtypes = dims + [_dp, _dpp, _dpp, _dp, _dpp, _dp]
    lib.oracle_row_linear_forward.argtypes = dims + [_dpp, _dpp, _dp, _dp]
    lib.oracle_row_linear_backward.argtypes = dims + [_dpp, _dpp, _dp, _dpp, _dpp, _dp]
    u32p = ctypes.POINTER(ctypes.c_uint32)
    lib.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
    lib.oracle_dropout_keep.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, _i64,
                                        _i64, ctypes.POINTER(ctypes.c_uint8)]
    lib.oracle_layernorm_forward.argtypes = [_i64, _i64, _dp, _dp, _dp, ctypes.c_double, _dp,
                                             _dp, _dp]
    lib.oracle_layernorm_backward.argtypes = [_i64, _i64, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


@contextlib.contextmanager
def _library(path: str):
    """Route every call through another build of oracle.c for the duration of
    the block (the planted-mistake test compiles mutated copies)."""
    global _lib
    _load()
    with _lock:
        saved, _lib = _lib, _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _f64(a) -> np.ndarray:
    """Contiguous float64 copy/view of an array-like (torch tensors included)."""
    if hasattr(a, "detach"):  # torch tensor: exact upcast on the host
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _ptrs(arrs):
    arr = (_dp * len(arrs))(*[_ptr(a) for a in arrs])
    return ctypes.cast(arr, _dpp), arr


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def gelu(x: float) -> float:
    return float(_load().oracle_gelu(float(x)))


def gelu_grad(x: float) -> float:
    return float(_load().oracle_gelu_grad(float(x)))


def _check_shards(X, A, b1, B, b2):
    t = len(A)
    if t < 1 or len(B) != t:
        raise ValueError("A and B must hold the same number (>=1) of shards")
    T, h = X.shape
    fi = A[0].shape[1]
    for a, b in zip(A, B):
        if a.shape != (h, fi) or b.shape != (fi, h):
            raise ValueError("shard shapes must be A_i [h, f/t] and B_i [f/t, h]")
    if b1.shape != (t * fi,) or b2.shape != (h,):
        raise ValueError("b1 must be [f], b2 must be [h]")
    return T, h, t * fi, t, fi


def forward(X, A_shards, b1, B_shards, b2):
    """Z = (sum_i GeLU(X.A_i + b1_i).B_i) + b2.  Returns dict Y, H (lists of
    [T, f/t] shards) and Z [T, h], all float64."""
    lib = _load()
    X = _f64(X); b1 = _f64(b1); b2 = _f64(b2)
    A = [_f64(a) for a in A_shards]; B = [_f64(b) for b in B_shards]
    T, h, f, t, fi = _check_shards(X, A, b1, B, b2)
    Y = [np.empty((T, fi)) for _ in range(t)]
    H = [np.empty((T, fi)) for _ in range(t)]
    Z = np.empty((T, h))
    pA, _ka = _ptrs(A); pB, _kb = _ptrs(B); pY, _ky = _ptrs(Y); pH, _kh = _ptrs(H)
    lib.oracle_forward(T, h, f, t, _ptr(X), pA, _ptr(b1), pB, _ptr(b2), pY, pH, _ptr(Z))
    return {"Y": Y, "H": H, "Z": Z}


def backward(X, A_shards, B_shards, Y, H, dZ):
    """Chain rule of :func:`forward` for upstream gradient dZ.  Returns dict
    dY (list), dX, dA (list of [h, f/t]), db1 [f], dB (list of [f/t, h]), db2 [h]."""
    lib = _load()
    X = _f64(X); dZ = _f64(dZ)
    A = [_f64(a) for a in A_shards]; B = [_f64(b) for b in B_shards]
    Y = [_f64(y) for y in Y]; H = [_f64(x) for x in H]
    t = len(A); T, h = X.shape; fi = A[0].shape[1]; f = t * fi
    dY = [np.empty((T, fi)) for _ in range(t)]
    dX = np.empty((T, h))
    dA = [np.empty((h, fi)) for _ in range(t)]
    dB = [np.empty((fi, h)) for _ in range(t)]
    db1 = np.empty(f); db2 = np.empty(h)
    keep = []
    def P(lst):
        p, k = _ptrs(lst); keep.append(k); return p
    lib.oracle_backward(T, h, f, t, _ptr(X), P(A), P(B), P(Y), P(H), _ptr(dZ),
                        P(dY), _ptr(dX), P(dA), _ptr(db1), P(dB), _ptr(db2))
    return {"dY": dY, "dX": dX, "dA": dA, "db1": db1, "dB": dB, "db2": db2}


def forward_backward(X, A_shards, b1, B_shards, b2, dZ):
    fw = forward(X, A_shards, b1, B_shards, b2)
    bw = backward(X, A_shards, B_shards, fw["Y"], fw["H"], dZ)
    return {**fw, **bw}


def rows(X, A_shards, b1, B_shards, b2, dZ, row_idx, activations=False):
    """Z[r, :] and dX[r, :] for the selected token rows only; with
    activations=True also their rows of Y, H and dY ([len(rows), f] each, the
    t shards side by side)."""
    lib = _load()
    X = _f64(X); dZ = _f64(dZ); b1 = _f64(b1); b2 = _f64(b2)
    A = [_f64(a) for a in A_shards]; B = [_f64(b) for b in B_shards]
    T, h, f, t, fi = _check_shards(X, A, b1, B, b2)
    idx = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64))
    if idx.size and (idx.min() < 0 or idx.max() >= T):
        raise IndexError("row index out of range")
    Zr = np.empty((idx.size, h)); dXr = np.empty((idx.size, h))
    act = [np.empty((idx.size, f)) for _ in range(3)] if activations else None
    null = ctypes.cast(None, _dp)
    pA, _ka = _ptrs(A); pB, _kb = _ptrs(B)
    lib.oracle_rows(T, h, f, t, _ptr(X), pA, _ptr(b1), pB, _ptr(b2), _ptr(dZ),
                    idx.size, idx.ctypes.data_as(ctypes.POINTER(_i64)), _ptr(Zr), _ptr(dXr),
                    *([_ptr(a) for a in act] if act else [null, null, null]))
    out = {"Z": Zr, "dX": dXr}
    if act:
        out.update(Y=act[0], H=act[1], dY=act[2])
    return out


def cols(X, A_shards, b1, B_shards, dZ, col_idx):
    """dA[:, c], dB[c, :] and db1[c] for the selected global ffn columns c."""
    lib = _load()
    X = _f64(X); dZ = _f64(dZ); b1 = _f64(b1)
    A = [_f64(a) for a in A_shards]; B = [_f64(b) for b in B_shards]
    t = len(A); T, h = X.shape; fi = A[0].shape[1]; f = t * fi
    idx = np.ascontiguousarray(np.asarray(col_idx, dtype=np.int64))
    if idx.size and (idx.min() < 0 or idx.max() >= f):
        raise IndexError("column index out of range")
    dAc = np.empty((idx.size, h)); dBc = np.empty((idx.size, h)); db1c = np.empty(idx.size)
    pA, _ka = _ptrs(A); pB, _kb = _ptrs(B)
    lib.oracle_cols(T, h, f, t, _ptr(X), pA, _ptr(b1), pB, _ptr(dZ),
                    idx.size, idx.ctypes.data_as(ctypes.POINTER(_i64)),
                    _ptr(dAc), _ptr(dBc), _ptr(db1c))
    return {"dA_cols": dAc, "dB_rows": dBc, "db1": db1c}


def db2(dZ):
    lib = _load()
    dZ = _f64(dZ)
    T, h = dZ.shape
    out = np.empty(h)
    lib.oracle_db2(T, h, _ptr(dZ), _ptr(out))
    return out


# ---- sequence-parallel variant ----------------------------------------------
# The sequence-parallel block takes X and dZ as seq_chunks token chunks and
# returns Z and dX in the same chunking: gather = concatenation along tokens
# before the column-parallel linear, reduce-scatter = the shard sum followed by
# a split along tokens after the row-parallel linear.

def sp_gather(chunks):
    return np.concatenate([_f64(c) for c in chunks], axis=0)


def sp_scatter(full, n):
    T = full.shape[0]
    if T % n:
        raise ValueError("token count must divide evenly into chunks")
    return [np.ascontiguousarray(x) for x in np.split(full, n, axis=0)]


def forward_backward_sp(X_chunks, A_shards, b1, B_shards, b2, dZ_chunks):
    n = len(X_chunks)
    out = forward_backward(sp_gather(X_chunks), A_shards, b1, B_shards, b2, sp_gather(dZ_chunks))
    out["Z_chunks"] = sp_scatter(out["Z"], n)
    out["dX_chunks"] = sp_scatter(out["dX"], n)
    return out


# ---- tensor-parallel linear layers (attention projections) -------------------
# Column parallel: Y_i = X.W_i + b_i; row parallel: Z = sum_i X_i.W_i + b
# ("2、分布式训练基础…", 2.2 模型并行 —— 张量并行 / 核心原理).

def column_linear(X, W_shards, b, dY_shards=None):
    """Forward Y_i (list), and with dY_i given the backward dX, dW_i, db."""
    lib = _load()
    X = _f64(X); b = _f64(b); W = [_f64(w) for w in W_shards]
    t = len(W); T, din = X.shape; oi = W[0].shape[1]; dout = t * oi
    if any(w.shape != (din, oi) for w in W) or b.shape != (dout,):
        raise ValueError("W_i must be [in, out/t] and b [out]")
    Y = [np.empty((T, oi)) for _ in range(t)]
    keep = []
    def P(lst):
        p, k = _ptrs(lst); keep.append(k); return p
    lib.oracle_column_linear_forward(T, din, dout, t, _ptr(X), P(W), _ptr(b), P(Y))
    out = {"Y": Y}
    if dY_shards is not None:
        dY = [_f64(d) for d in dY_shards]
        dX = np.empty((T, din)); dW = [np.empty((din, oi)) for _ in range(t)]; db = np.empty(dout)
        lib.oracle_column_linear_backward(T, din, dout, t, _ptr(X), P(W), P(dY), _ptr(dX),
                                          P(dW), _ptr(db))
        out.update(dX=dX, dW=dW, db=db)
    return out


def row_linear(X_shards, W_shards, b, dZ=None):
    """Forward Z, and with dZ given the backward dX_i (list), dW_i, db."""
    lib = _load()
    X = [_f64(x) for x in X_shards]; W = [_f64(w) for w in W_shards]; b = _f64(b)
    t = len(W); T, ii = X[0].shape; dout = W[0].shape[1]; din = t * ii
    if any(w.shape != (ii, dout) for w in W) or any(x.shape != (T, ii) for x in X):
        raise ValueError("X_i must be [T, in/t] and W_i [in/t, out]")
    Z = np.empty((T, dout))
    keep = []
    def P(lst):
        p, k = _ptrs(lst); keep.append(k); return p
    lib.oracle_row_linear_forward(T, din, dout, t, P(X), P(W), _ptr(b), _ptr(Z))
    out = {"Z": Z}
    if dZ is not None:
        dZ = _f64(dZ)
        dX = [np.empty((T, ii)) for _ in range(t)]; dW = [np.empty((ii, dout)) for _ in range(t)]
        db = np.empty(dout)
        lib.oracle_row_linear_backward(T, din, dout, t, P(X), P(W), _ptr(dZ), P(dX), P(dW),
                                       _ptr(db))
        out.update(dX=dX, dW=dW, db=db)
    return out


# ---- sequence-parallel LayerNorm / Dropout sublayer ---------------------------
# Out = X + Dropout(MLP(LN(X))), LayerNorm and Dropout per token chunk
# ("Megatron-LM：NVIDIA 的大规模并行训练方案", 并行训练范式 / 序列并行); the
# composition is the usual pre-LayerNorm residual block (a reading).

def philox4x32_10(counter, key):
    """Philox4x32-10 (Salmon et al., SC'11): 4 output words for a 4-word counter
    and a 2-word key."""
    lib = _load()
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in counter])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib.oracle_philox4x32_10(c, k, o)
    return [int(x) for x in o]


def dropout_threshold(p: float) -> int:
    """keep iff the Philox word is below floor((1 - p) * 2^32)."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return int(np.floor((1.0 - float(p)) * 4294967296.0))


def dropout_keep(T: int, h: int, p: float, seed: int, offset: int = 0, e0: int = 0,
                 count: int | None = None) -> np.ndarray:
    """0/1 keep mask of elements [e0, e0 + count) of a [T, h] tensor (all by default)."""
    lib = _load()
    n = T * h - e0 if count is None else count
    out = np.empty(max(n, 0), dtype=np.uint8)
    if n > 0:
        lib.oracle_dropout_keep(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                dropout_threshold(p), int(e0), int(n),
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return out


def layernorm(X, gamma, beta, eps: float, dXn=None):
    """LayerNorm over the last dimension: Xn, mean, rstd; with dXn the backward
    dX, dgamma, dbeta too."""
    lib = _load()
    X = _f64(X); gamma = _f64(gamma); beta = _f64(beta)
    T, h = X.shape
    if gamma.shape != (h,) or beta.shape != (h,):
        raise ValueError("gamma and beta must be [h]")
    Xn = np.empty((T, h)); mean = np.empty(T); rstd = np.empty(T)
    lib.oracle_layernorm_forward(T, h, _ptr(X), _ptr(gamma), _ptr(beta), float(eps), _ptr(Xn),
                                 _ptr(mean), _ptr(rstd))
    out = {"Xn": Xn, "mean": mean, "rstd": rstd}
    if dXn is not None:
        dXn = _f64(dXn)
        dX = np.empty((T, h)); dg = np.empty(h); db = np.empty(h)
        lib.oracle_layernorm_backward(T, h, _ptr(X), _ptr(gamma), _ptr(mean), _ptr(rstd),
                                      _ptr(dXn), _ptr(dX), _ptr(dg), _ptr(db))
        out.update(dX=dX, dgamma=dg, dbeta=db)
    return out


def sp_block_inputs(X, gamma, beta, eps, p, seed, offset=0, dOut=None):
    """The MLP block's inputs inside the sublayer: Xn = LN(X) (with the row
    mean and rstd), the 0/1 keep mask as float64 [T, h], scale = 1 / (1 - p),
    and with dOut given the block's upstream gradient dZ = dOut * keep * scale
    (dropout backward)."""
    X = _f64(X)
    T, h = X.shape
    ln = layernorm(X, gamma, beta, eps)
    keep = dropout_keep(T, h, p, seed, offset).reshape(T, h).astype(np.float64)
    scale = 1.0 / (1.0 - float(p))
    out = {"Xn": ln["Xn"], "mean": ln["mean"], "rstd": ln["rstd"], "keep": keep, "scale": scale}
    if dOut is not None:
        out["dZ"] = _f64(dOut) * keep * scale
    return out


def sp_layer(X, gamma, beta, eps, A_shards, b1, B_shards, b2, p, seed, offset=0, dOut=None):
    """Out = X + Dropout(MLP(LN(X))); with dOut the backward of every input:
    dX (through both paths), dgamma, dbeta, dA_i, db1, dB_i, db2.  Also returns
    the intermediates Xn, Z, keep."""
    X = _f64(X)
    bi = sp_block_inputs(X, gamma, beta, eps, p, seed, offset, dOut)
    keep, scale = bi["keep"], bi["scale"]
    if dOut is None:
        blk = forward(bi["Xn"], A_shards, b1, B_shards, b2)
        Out = X + keep * scale * blk["Z"]
        return {"Out": Out, "Xn": bi["Xn"], "Z": blk["Z"], "keep": keep, "mean": bi["mean"],
                "rstd": bi["rstd"]}
    dOut = _f64(dOut)
    dZ = bi["dZ"]                                 # dropout backward
    blk = forward_backward(bi["Xn"], A_shards, b1, B_shards, b2, dZ)
    lnb = layernorm(X, gamma, beta, eps, dXn=blk["dX"])
    Out = X + keep * scale * blk["Z"]
    return {"Out": Out, "Xn": bi["Xn"], "Z": blk["Z"], "keep": keep, "dZ": dZ,
            "dXn": blk["dX"], "dX": lnb["dX"] + dOut, "dgamma": lnb["dgamma"],
            "dbeta": lnb["dbeta"], "dA": blk["dA"], "db1": blk["db1"], "dB": blk["dB"],
            "db2": blk["db2"], "mean": bi["mean"], "rstd": bi["rstd"]}


def sp_rows(X, gamma, beta, eps, A_shards, b1, B_shards, b2, p, seed, offset, dOut, row_idx):
    """Out[r, :] and dX[r, :] of :func:`sp_layer` for the selected token rows
    only (each row of the sublayer depends only on that row's inputs; the mask
    of element (r, n) is fixed by its index r * h + n)."""
    lib = _load()
    X = _f64(X); gamma = _f64(gamma); beta = _f64(beta); dOut = _f64(dOut)
    b1 = _f64(b1); b2 = _f64(b2)
    A = [_f64(a) for a in A_shards]; B = [_f64(b) for b in B_shards]
    T, h, f, t, fi = _check_shards(X, A, b1, B, b2)
    if gamma.shape != (h,) or beta.shape != (h,) or dOut.shape != (T, h):
        raise ValueError("gamma, beta must be [h] and dOut [T, h]")
    idx = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64))
    if idx.size and (idx.min() < 0 or idx.max() >= T):
        raise IndexError("row index out of range")
    scale = 1.0 / (1.0 - float(p))
    Outr = np.empty((idx.size, h)); dXr = np.empty((idx.size, h))
    pA, _ka = _ptrs(A); pB, _kb = _ptrs(B)
    lib.oracle_sp_rows(T, h, f, t, _ptr(X), _ptr(gamma), _ptr(beta), float(eps), pA, _ptr(b1),
                       pB, _ptr(b2), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                       dropout_threshold(p), scale, _ptr(dOut), idx.size,
                       idx.ctypes.data_as(ctypes.POINTER(_i64)), _ptr(Outr), _ptr(dXr))
    return {"Out": Outr, "dX": dXr}
