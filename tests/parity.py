"""Parity gate between the CUDA path and the fp64 oracle.

Per output and gradient tensor:
    relative Frobenius error  ||got - ref|| / ||ref||        <= 5e-3
    max |got - ref| - q(ref)  <=  3e-2 * max(1, RMS(ref))
The weight and bias gradients are sums over all tokens, so their size (and
the error that bf16 rounding of the saved activations puts in them) grows
with RMS(ref); tensors with RMS <= 1 (Z, dX) keep the plain 3e-2 absolute
bound.  q(ref) is the rounding a bf16 output cannot avoid: half the bf16
spacing at the reference element (2^(e - 8) for |ref| in [2^e, 2^(e+1)),
so 0.0625 from 16 up), zero for fp32 outputs.  A bf16 element of 8 or more
is otherwise held to less than its own half spacing.  The raw max-abs is
reported alongside.
"""
from __future__ import annotations

import numpy as np
import torch

REL_FRO = 5e-3
MAX_ABS = 3e-2


def _np(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def bf16_half_spacing(r: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 values (8 significant bits) at |r|:
    2^(e - 8) for |r| in [2^e, 2^(e+1)); 0 at r = 0."""
    m, k = np.frexp(np.abs(r))          # |r| = m * 2^k, m in [0.5, 1)
    return np.where(r == 0, 0.0, np.ldexp(1.0, k - 9))


def measure(got, ref) -> dict:
    g, r = _np(got), _np(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return {"rel_fro": 0.0, "max_abs": 0.0, "max_excess": 0.0, "rms": 0.0, "bound": MAX_ABS}
    d = g - r
    nr = np.linalg.norm(r)
    rel = float(np.linalg.norm(d) / nr) if nr > 0 else float(np.linalg.norm(d))
    rms = float(np.sqrt(np.mean(r * r)))
    is_bf16 = isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16
    excess = np.abs(d) - bf16_half_spacing(r) if is_bf16 else np.abs(d)
    return {"rel_fro": rel, "max_abs": float(np.abs(d).max()),
            "max_excess": float(excess.max()), "rms": rms,
            "bound": MAX_ABS * max(1.0, rms), "finite": bool(np.isfinite(g).all())}


def gate(name: str, got, ref, report: dict | None = None) -> dict:
    m = measure(got, ref)
    if report is not None:
        report[name] = m
    assert m.get("finite", True), f"{name}: non-finite values"
    assert m["rel_fro"] <= REL_FRO, f"{name}: relative Frobenius error {m['rel_fro']:.3e} > {REL_FRO}"
    assert m["max_excess"] <= m["bound"], (
        f"{name}: max abs error beyond bf16 rounding {m['max_excess']:.3e} > {m['bound']:.3e} "
        f"(max abs {m['max_abs']:.3e}, RMS {m['rms']:.3g})")
    return m


def cat(lst, axis):
    return torch.cat([x.cpu() for x in lst], dim=axis) if isinstance(lst[0], torch.Tensor) \
        else np.concatenate(lst, axis=axis)


def compare_full(block, ref: dict, report: dict | None = None, intermediates: bool = True):
    """Element-by-element comparison of every output against the full oracle."""
    torch.cuda.synchronize()
    if intermediates:
        sv = block.saved()
        gate("Y", cat(sv["Y"], 1), cat(ref["Y"], 1), report)
        gate("H", cat(sv["H"], 1), cat(ref["H"], 1), report)
        gate("dY", cat(sv["dY"], 1), cat(ref["dY"], 1), report)
    gate("Z", cat(block.Z, 0), ref["Z"], report)
    gate("dX", cat(block.dX, 0), ref["dX"], report)
    gate("dA", cat(block.dA, 1), cat(ref["dA"], 1), report)
    gate("dB", cat(block.dB, 0), cat(ref["dB"], 0), report)
    gate("db1", block.db1, ref["db1"], report)
    gate("db2", block.db2, ref["db2"], report)


def tile_samples(n: int, seed: int, tile: int = 256, half: int = 128) -> np.ndarray:
    """Indices in [0, n) that reach every tile of the GEMMs along one axis:
    one seeded index in each `half`-wide half of every `tile`-wide tile (the
    two CTAs of a pair tile, or the two halves of an output tile's columns),
    plus the first and the last index."""
    rng = np.random.default_rng(seed)
    pick = {0, n - 1} if n > 0 else set()
    for lo in range(0, n, half):
        hi = min(n, lo + half)
        pick.add(int(rng.integers(lo, hi)))
    return np.array(sorted(pick), dtype=np.int64)


def shard_tile_samples(f: int, t: int, seed: int) -> np.ndarray:
    """Global ffn columns that reach every 256-wide tile of every shard's
    [*, f/t] GEMM outputs (one in each 128-wide half), as i * f/t + j."""
    fi = f // t
    out = [i * fi + tile_samples(fi, seed + i) for i in range(t)]
    return np.concatenate(out).astype(np.int64)


def compare_sampled(block, inputs: dict, w, oracle_mod, rows: np.ndarray, cols: np.ndarray,
                    report: dict | None = None, intermediates: bool = True):
    """Sampled outputs computed one by one by the oracle: rows of Z, dX and
    (intermediates=True) of the saved Y, H, dY; dA columns, dB rows and db1
    entries at the sampled ffn columns; db2 in full."""
    from tensor_transformer_mlp_gemm_gb300.inputs import column_shards, row_shards
    torch.cuda.synchronize()
    A = column_shards(inputs["A"], w.t)
    B = row_shards(inputs["B"], w.t)
    r = oracle_mod.rows(inputs["X"], A, inputs["b1"], B, inputs["b2"], inputs["dZ"], rows,
                        activations=intermediates)
    c = oracle_mod.cols(inputs["X"], A, inputs["b1"], B, inputs["dZ"], cols)
    ridx = torch.from_numpy(rows)
    Z = cat(block.Z, 0)
    dX = cat(block.dX, 0)
    gate("Z[rows]", Z[ridx], r["Z"], report)
    gate("dX[rows]", dX[ridx], r["dX"], report)
    if intermediates:
        sv = block.saved()
        dev = sv["Y"][0].device
        gidx = ridx.to(dev)
        for name in ("Y", "H", "dY"):
            got = torch.cat([x.index_select(0, gidx).cpu() for x in sv[name]], dim=1)
            gate(f"{name}[rows]", got, r[name], report)
    fi = w.ffn // w.t
    dA_cols = torch.stack([block.dA[int(q) // fi][:, int(q) % fi].cpu() for q in cols])
    dB_rows = torch.stack([block.dB[int(q) // fi][int(q) % fi, :].cpu() for q in cols])
    gate("dA[:,cols]", dA_cols, c["dA_cols"], report)
    gate("dB[cols,:]", dB_rows, c["dB_rows"], report)
    gate("db1[cols]", block.db1.cpu()[cols], c["db1"], report)
    gate("db2", block.db2, oracle_mod.db2(inputs["dZ"]), report)
