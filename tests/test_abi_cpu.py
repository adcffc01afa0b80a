"""Host-side checks of the C ABI (no GPU): the library builds and loads, it
exports every function include/tpmlp.h declares, argument validation returns
the documented status codes before touching the device, and the product path
never reaches the oracle."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpmlp.h")
PKG = os.path.join(ROOT, "tensor_transformer_mlp_gemm_gb300")


@pytest.fixture(scope="module")
def binding():
    from tensor_transformer_mlp_gemm_gb300.build import build
    build()
    from tensor_transformer_mlp_gemm_gb300 import binding as b
    return b


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tpmlp_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_calls():
    names = _declared_functions()
    for must in ("tpmlp_forward", "tpmlp_backward", "tpmlp_workspace_bytes", "tpmlp_sync_check"):
        assert must in names


def test_library_exports_every_declared_symbol(binding):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (tpmlp_\w+)", out))
    declared = set(_declared_functions())
    assert declared <= exported, declared - exported
    # nothing else leaks from the library's C surface
    assert exported == declared
    assert set(binding.EXPORTED) == declared
    lib = binding.library()
    for name in declared:
        assert getattr(lib, name) is not None


def test_status_strings(binding):
    for s in range(5):
        assert binding.tpmlp_status_string(s)
    assert binding.tpmlp_status_string(99) == "unknown status"
    assert [binding.tpmlp_kernel_name(k) for k in range(binding.KERNEL_KINDS)] == [
        "column_fwd", "row_fwd", "dgrad_h", "dgrad_x", "wgrad_b", "wgrad_a", "bias_grad",
        "linear_fwd", "linear_dgrad", "linear_wgrad", "layernorm_fwd", "layernorm_bwd",
        "dropout_bwd", "sp_copy"]


def test_workspace_bytes(binding):
    d = binding.make_dims(2048, 12288, 49152, 8, 1)
    n = binding.tpmlp_workspace_bytes(d)
    act = 2048 * 49152 * 2
    assert n >= 3 * act
    y, h, dy = binding.tpmlp_workspace_layout(d)
    assert (y, h, dy) == (0, act, 2 * act)
    assert binding.tpmlp_workspace_bytes(binding.make_dims(128, 100, 256, 2)) == 0  # invalid
    assert binding.tpmlp_workspace_bytes(binding.make_dims(0, 64, 256, 2)) > 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def _fwd(binding, dims, t=None, X=None, A=None, b1=FAKE, B=None, b2=FAKE, Z=None, ws=FAKE):
    n, tt = dims.seq_chunks, dims.t
    X = X if X is not None else [FAKE] * n
    Z = Z if Z is not None else [FAKE] * n
    A = A if A is not None else [FAKE] * tt
    B = B if B is not None else [FAKE] * tt
    lib = binding.library()
    arr = lambda xs: (ctypes.c_void_p * max(len(xs), 1))(*xs)
    return lib.tpmlp_forward(ctypes.byref(dims), arr(X), arr(A), b1, arr(B), b2,
                             dims.t if t is None else t, arr(Z), ws, None)


def test_forward_validation_codes(binding):
    mk = binding.make_dims
    INV, UNS = binding.TPMLP_ERR_INVALID_ARG, binding.TPMLP_ERR_UNSUPPORTED
    assert _fwd(binding, mk(256, 256, 1024, 2), t=4) == INV          # t mismatch
    assert _fwd(binding, mk(256, 256, 1000, 3)) == INV              # t does not divide f
    assert _fwd(binding, mk(-1, 256, 1024, 2)) == INV               # negative tokens
    assert _fwd(binding, mk(256, 0, 1024, 2)) == INV                # empty hidden
    assert _fwd(binding, mk(256, 100, 1024, 2)) == UNS              # h not a multiple of 8
    assert _fwd(binding, mk(256, 256, 1044, 2)) == UNS              # fi not a multiple of 8
    assert _fwd(binding, mk(256, 256, 1024, 16)) == UNS             # more than 8 shards
    assert _fwd(binding, mk(384, 256, 1024, 2, 2)) == UNS           # chunk of 192 rows
    assert _fwd(binding, mk(302, 256, 1024, 2, 4)) == INV           # chunks do not divide T
    assert _fwd(binding, mk(256, 256, 1024, 2), b1=None) == INV     # null bias
    assert _fwd(binding, mk(256, 256, 1024, 2), b1=FAKE + 2) == UNS  # misaligned bias
    assert _fwd(binding, mk(256, 256, 1024, 2), A=[FAKE, None]) == INV
    assert _fwd(binding, mk(256, 256, 1024, 2), B=[FAKE, FAKE + 8]) == UNS
    assert _fwd(binding, mk(256, 256, 1024, 2), ws=None) == INV
    assert _fwd(binding, mk(256, 256, 1024, 2), Z=[None]) == INV
    assert binding.library().tpmlp_forward(None, None, None, None, None, None, 1, None, None,
                                           None) == INV


def test_backward_validation_codes(binding):
    lib = binding.library()
    d = binding.make_dims(256, 256, 1024, 2)
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
    two, one = [FAKE, FAKE], [FAKE]
    INV, UNS = binding.TPMLP_ERR_INVALID_ARG, binding.TPMLP_ERR_UNSUPPORTED
    assert lib.tpmlp_backward(ctypes.byref(d), arr(one), arr(one), arr(two), arr(two), FAKE,
                              arr(one), arr([FAKE, None]), FAKE, arr(two), FAKE, None) == INV
    assert lib.tpmlp_backward(ctypes.byref(d), arr(one), arr(one), arr(two), arr(two), FAKE,
                              arr(one), arr(two), FAKE + 4, arr(two), FAKE, None) == UNS
    assert lib.tpmlp_backward(ctypes.byref(d), arr([None]), arr(one), arr(two), arr(two), FAKE,
                              arr(one), arr(two), FAKE, arr(two), FAKE, None) == INV


def test_recompute_workspace_and_validation(binding):
    d = binding.make_dims(2048, 12288, 49152, 8)
    saved, scratch = binding.tpmlp_recompute_workspace_bytes(d)
    assert saved == 2048 * 49152 * 2                     # Y only
    assert saved + scratch == binding.tpmlp_workspace_bytes(d)
    lib = binding.library()
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
    d = binding.make_dims(256, 256, 1024, 2)
    two, one = [FAKE, FAKE], [FAKE]
    INV = binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_forward_recompute(ctypes.byref(d), arr(one), arr(two), FAKE, arr(two), FAKE,
                                       2, arr(one), None, FAKE, None) == INV  # no saved buffer
    assert lib.tpmlp_forward_recompute(ctypes.byref(d), arr(one), arr(two), FAKE, arr(two), FAKE,
                                       2, arr(one), FAKE, None, None) == INV  # no scratch
    assert lib.tpmlp_backward_recompute(ctypes.byref(d), arr(one), arr(one), arr(two), arr(two),
                                        FAKE, FAKE + 8, arr(one), arr(two), FAKE, arr(two), FAKE,
                                        None) == binding.TPMLP_ERR_UNSUPPORTED  # misaligned


def test_linear_workspace_bytes(binding):
    mk = binding.make_linear_dims
    n = binding.tpmlp_linear_workspace_bytes(mk(2048, 12288, 36864, 8))
    assert n >= 64 * 36864 * 4 + 128 * 256 * 256 * 4   # bias partials + split tiles
    assert binding.tpmlp_linear_workspace_bytes(mk(128, 256, 264, 2)) > 0   # valid as a row split
    assert binding.tpmlp_linear_workspace_bytes(mk(128, 100, 256, 2)) == 0  # valid as neither
    assert binding.tpmlp_linear_workspace_bytes(mk(0, 64, 64, 1)) > 0


def _lin(binding, fn, dims, nin=None, W=None, b=FAKE, nout=None, ws=FAKE):
    lib = binding.library()
    arr = lambda xs: (ctypes.c_void_p * max(len(xs), 1))(*xs)
    W = W if W is not None else [FAKE] * dims.t
    if fn in ("tpmlp_column_linear_forward", "tpmlp_row_linear_forward"):
        col = fn.startswith("tpmlp_column")
        ins = nin if nin is not None else [FAKE] * (dims.seq_chunks if col else dims.t)
        outs = nout if nout is not None else [FAKE] * (dims.t if col else dims.seq_chunks)
        return getattr(lib, fn)(ctypes.byref(dims), arr(ins), arr(W), b, arr(outs), ws, None)
    n = max(dims.t, dims.seq_chunks)
    ins = nin if nin is not None else [FAKE] * n
    outs = nout if nout is not None else [FAKE] * n
    return getattr(lib, fn)(ctypes.byref(dims), arr(ins), arr([FAKE] * n), arr(W), arr(outs),
                            arr([FAKE] * dims.t), b, ws, None)


def test_linear_validation_codes(binding):
    mk = binding.make_linear_dims
    INV, UNS = binding.TPMLP_ERR_INVALID_ARG, binding.TPMLP_ERR_UNSUPPORTED
    colf, rowf = "tpmlp_column_linear_forward", "tpmlp_row_linear_forward"
    colb, rowb = "tpmlp_column_linear_backward", "tpmlp_row_linear_backward"
    for fn in (colf, colb, rowf, rowb):
        assert _lin(binding, fn, mk(-1, 256, 256, 2)) == INV             # negative tokens
        assert _lin(binding, fn, mk(256, 256, 256, 0)) == INV            # no shards
        assert _lin(binding, fn, mk(256, 256, 256, 16)) == UNS           # more than 8 shards
        assert _lin(binding, fn, mk(384, 256, 256, 2, 2)) == UNS         # chunk of 192 rows
        assert _lin(binding, fn, mk(256, 256, 256, 2), ws=None) == INV   # no workspace
        assert _lin(binding, fn, mk(256, 256, 256, 2), b=FAKE + 4) == UNS
        assert _lin(binding, fn, mk(256, 256, 256, 2), W=[FAKE, None]) == INV
    assert _lin(binding, colf, mk(256, 256, 300, 7)) == INV   # t does not divide out
    assert _lin(binding, colf, mk(256, 300, 256, 2)) == UNS   # in not a multiple of 8
    assert _lin(binding, colf, mk(256, 256, 260, 2)) == UNS   # oi = 130 not a multiple of 8
    assert _lin(binding, rowf, mk(256, 300, 256, 7)) == INV   # t does not divide in
    assert _lin(binding, rowf, mk(256, 260, 256, 2)) == UNS   # ii = 130
    assert _lin(binding, rowf, mk(256, 256, 300, 2)) == UNS   # out not a multiple of 8
    assert _lin(binding, colf, mk(256, 256, 256, 2), nout=[FAKE, FAKE + 2]) == UNS
    assert _lin(binding, rowf, mk(256, 256, 256, 2), nin=[None, FAKE]) == INV
    assert binding.library().tpmlp_row_linear_forward(None, None, None, None, None, None,
                                                      None) == INV


def test_sp_workspace_and_validation(binding):
    mk = binding.make_dims
    d = mk(16384, 4096, 16384, 8, 8)
    n = binding.tpmlp_sp_workspace_bytes(d)
    assert n >= binding.tpmlp_workspace_bytes(d) + 3 * 16384 * 4096 * 2
    xn, dz = binding.tpmlp_sp_workspace_layout(d)
    assert binding.tpmlp_workspace_bytes(d) <= xn < dz < n
    assert binding.tpmlp_sp_workspace_bytes(mk(128, 32768, 1024, 2)) == 0  # h above 16384
    lib = binding.library()
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
    INV, UNS = binding.TPMLP_ERR_INVALID_ARG, binding.TPMLP_ERR_UNSUPPORTED
    d = mk(256, 256, 1024, 2)
    two, one = [FAKE, FAKE], [FAKE]

    def fwd(sp, **kw):
        a = dict(X=one, gamma=FAKE, beta=FAKE, A=two, b1=FAKE, B=two, b2=FAKE, t=2, Out=one,
                 ws=FAKE)
        a.update(kw)
        return lib.tpmlp_sp_forward(ctypes.byref(d), sp, arr(a["X"]), a["gamma"], a["beta"],
                                    arr(a["A"]), a["b1"], arr(a["B"]), a["b2"], a["t"],
                                    arr(a["Out"]), a["ws"], None)
    ok = ctypes.byref(binding.make_sp_params(1e-5, 0.1, 7))
    assert fwd(None) == INV
    assert fwd(ctypes.byref(binding.make_sp_params(1e-5, 1.0, 7))) == INV   # p = 1
    assert fwd(ctypes.byref(binding.make_sp_params(1e-5, -0.1, 7))) == INV
    assert fwd(ctypes.byref(binding.make_sp_params(-1.0, 0.1, 7))) == INV   # eps < 0
    assert fwd(ok, gamma=None) == INV
    assert fwd(ok, beta=FAKE + 2) == UNS
    assert fwd(ok, t=4) == INV
    assert lib.tpmlp_sp_backward(ctypes.byref(d), ok, arr(one), arr(one), FAKE, arr(two), arr(two),
                                 FAKE, arr(one), FAKE, None, arr(two), FAKE, arr(two), FAKE,
                                 None) == INV  # no dbeta


def test_set_timeout_and_profile_args(binding):
    lib = binding.library()
    assert lib.tpmlp_set_wait_timeout_ns(0) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_set_split_min_kblocks(-1) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_set_head_prefetch(-1) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_set_head_prefetch(65) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_set_wide_tiles(4) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_set_wide_tiles(-1) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_profile_begin(0) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_profile_begin_kinds(0, 1) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_profile_begin_kinds(16, 0) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_profile_begin_kinds(16, 1 << binding.KERNEL_KINDS) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_profile_end(None, None, 0) == -1  # not profiling


def test_product_path_never_imports_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), fn
                assert "liboracle" not in text and "oracle.c" not in text, fn


def test_tensor_map_cache_logic(binding):
    """The tensor-map cache on the host: a repeated key is a hit with the same
    bytes and no new encoding; a new address or box is a miss; the cache never
    holds more than its capacity."""
    r = binding.tpmlp_selftest_map_cache()
    assert r["key_bytes"] == 80
    # a, a (hit), a at a new address, a with a new box, then six new keys
    assert r["hits"] == 1 and r["misses"] == 9 and r["encoder_calls"] == 9
    assert r["hit_same_bytes"] == 1 and r["new_address_differs"] == 1
    assert 1 <= r["entries"] <= r["capacity"]
    lib = binding.library()
    assert lib.tpmlp_selftest_map_cache(None, 8) == binding.TPMLP_ERR_INVALID_ARG
    st = binding.tpmlp_map_cache_stats()
    assert set(st) == {"hits", "misses", "entries"}


def test_sp_copy_validation(binding):
    """Argument checks of the explicit sequence-parallel gather / scatter
    (before any device work)."""
    lib = binding.library()
    arr = lambda n: (ctypes.c_void_p * n)(*([0x1000] * n))
    d = binding.make_dims(512, 256, 1024, 4, 4)
    assert lib.tpmlp_sp_gather(None, arr(4), 256, 0x1000, None) == binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_sp_gather(ctypes.byref(d), arr(4), 0, 0x1000, None) == \
        binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_sp_gather(ctypes.byref(d), arr(4), 12, 0x1000, None) == \
        binding.TPMLP_ERR_UNSUPPORTED                      # cols not a multiple of 8
    assert lib.tpmlp_sp_gather(ctypes.byref(d), None, 256, 0x1000, None) == \
        binding.TPMLP_ERR_INVALID_ARG
    assert lib.tpmlp_sp_scatter(ctypes.byref(d), 0x1002, 256, arr(4), None) == \
        binding.TPMLP_ERR_UNSUPPORTED                      # misaligned
    d9 = binding.make_dims(512, 256, 1024, 4, 9)
    assert lib.tpmlp_sp_scatter(ctypes.byref(d9), 0x1000, 256, arr(9), None) == \
        binding.TPMLP_ERR_UNSUPPORTED                      # more than 8 chunks
