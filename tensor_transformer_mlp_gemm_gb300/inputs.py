"""Seeded synthetic inputs for the tensor-parallel MLP block and the
tensor-parallel linear layers (the attention projections).

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It draws random numbers and lays them out (shards, sequence chunks);
it holds none of the block's arithmetic.

Recipe (every workload): a CPU ``torch.Generator`` seeded with ``seed`` draws,
in this order, X [T, h], A [h, f], b1 [f], B [f, h], b2 [h], dZ [T, h] with
``torch.randn`` in fp32; each draw is multiplied by its standard deviation and
rounded to bf16 (round to nearest even).  X and dZ have std 1, the weights
``sigma_w``, the biases 0.02.

Linear layers (``make_linear_inputs``): the same kind of generator draws, in
this order, X [T, in], W [in, out], b [out], dY [T, out] (dY is the upstream
gradient of the layer's output), with the same standard deviations.

Sequence-parallel sublayer (``make_sp_inputs``): the block's tensors as
above (dZ serving as dOut, the sublayer's upstream gradient), then a second
CPU generator seeded with seed + 0x5EED draws gamma = 1 + 0.1 N(0, 1) and
beta = 0.02 N(0, 1), both [h], rounded to bf16.

Token rows are ordered sequence-major ([seq, micro-batch] flattened, the usual
[s, b, h] activation layout), so sequence chunk j is the contiguous row range
[j*T/n, (j+1)*T/n): a span of sequence positions for every sample.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    micro_batch: int
    seq: int
    hidden: int          # h
    ffn: int             # f
    t: int               # tensor-parallel shards
    sigma_w: float       # weight std
    seq_chunks: int = 1  # sequence-parallel chunks (1 = off, else t)
    sigma_b: float = 0.02

    @property
    def tokens(self) -> int:
        return self.micro_batch * self.seq

    @property
    def flops(self) -> int:
        """fwd+bwd FLOPs: six GEMMs of 2*T*h*f each."""
        return 12 * self.tokens * self.hidden * self.ffn

    def with_tokens(self, tokens: int) -> "Workload":
        """Same layer with a different token count (micro_batch=1, seq=tokens)."""
        return replace(self, name=f"{self.name}[T={tokens}]", micro_batch=1, seq=tokens,
                       seq_chunks=1)


# The five workloads: shapes and distributions of the pages' 1.3B-class and
# 175B-class examples plus a tiny and a small case and the sequence-parallel one.
WORKLOADS = {
    "tiny": Workload("tiny", 2, 64, 256, 1024, 2, 0.02),
    "small_gpt": Workload("small_gpt", 4, 1024, 1024, 4096, 2, 0.02),
    "gpt_1p3b_t1": Workload("gpt_1p3b_t1", 4, 1024, 2048, 8192, 1, 0.02),
    "gpt_1p3b_t4": Workload("gpt_1p3b_t4", 4, 1024, 2048, 8192, 4, 0.02),
    "gpt_175b": Workload("gpt_175b", 1, 2048, 12288, 49152, 8, 0.006),
    "sp_h4096": Workload("sp_h4096", 8, 2048, 4096, 16384, 8, 0.02, seq_chunks=8),
}


def custom(tokens: int, hidden: int, ffn: int, t: int, sigma_w: float = 0.02,
           seq_chunks: int = 1, name: str = "custom") -> Workload:
    return Workload(name, 1, tokens, hidden, ffn, t, sigma_w, seq_chunks)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Full (unsharded) bf16 CPU tensors X, A, b1, B, b2, dZ for workload w."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    T, h, f = w.tokens, w.hidden, w.ffn

    def draw(shape, std):
        x = torch.randn(*shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    X = draw((T, h), 1.0)
    A = draw((h, f), w.sigma_w)
    b1 = draw((f,), w.sigma_b)
    B = draw((f, h), w.sigma_w)
    b2 = draw((h,), w.sigma_b)
    dZ = draw((T, h), 1.0)
    return {"X": X, "A": A, "b1": b1, "B": B, "b2": b2, "dZ": dZ}


def column_shards(A: torch.Tensor, t: int) -> list:
    """A [h, f] -> t contiguous column blocks [h, f/t] (own allocations)."""
    f = A.shape[1]
    if f % t:
        raise ValueError("f must be divisible by t")
    fi = f // t
    return [A[:, i * fi:(i + 1) * fi].contiguous() for i in range(t)]


def row_shards(B: torch.Tensor, t: int) -> list:
    """B [f, h] -> t contiguous row blocks [f/t, h] (own allocations)."""
    f = B.shape[0]
    if f % t:
        raise ValueError("f must be divisible by t")
    fi = f // t
    return [B[i * fi:(i + 1) * fi, :].contiguous() for i in range(t)]


def seq_chunks(X: torch.Tensor, n: int) -> list:
    """X [T, h] -> n contiguous token chunks [T/n, h] (own allocations)."""
    T = X.shape[0]
    if T % n:
        raise ValueError("T must be divisible by the number of chunks")
    r = T // n
    return [X[j * r:(j + 1) * r, :].contiguous() for j in range(n)]


@dataclass(frozen=True)
class LinearWorkload:
    """One tensor-parallel linear layer: W [in, out] split by columns
    (split="column": Y_i = X.W_i + b_i) or by rows (split="row":
    Z = sum_i X_i.W_i + b)."""
    name: str
    tokens: int
    in_features: int
    out_features: int
    t: int
    split: str            # "column" or "row"
    sigma_w: float
    seq_chunks: int = 1
    sigma_b: float = 0.02

    @property
    def flops(self) -> int:
        """fwd+bwd FLOPs: three GEMMs (forward, input gradient, weight gradient)
        of 2*T*in*out each."""
        return 6 * self.tokens * self.in_features * self.out_features

    @property
    def shard(self) -> int:
        """out / t (column split) or in / t (row split)."""
        return (self.out_features if self.split == "column" else self.in_features) // self.t


# Attention projections of the pages' 175B-class layer: hidden 12288, the QKV
# weight 12288 x 36864 split 8 ways into 12288 x 4608 (column parallel), the
# output projection 12288 x 12288 split 8 ways by rows; 2048 tokens as in the
# MLP workload.  Plus small cases.
LINEAR_WORKLOADS = {
    "qkv_tiny": LinearWorkload("qkv_tiny", 128, 256, 768, 2, "column", 0.02),
    "attn_out_tiny": LinearWorkload("attn_out_tiny", 128, 256, 256, 2, "row", 0.02),
    "qkv_175b": LinearWorkload("qkv_175b", 2048, 12288, 36864, 8, "column", 0.006),
    "attn_out_175b": LinearWorkload("attn_out_175b", 2048, 12288, 12288, 8, "row", 0.006),
    "qkv_sp_h4096": LinearWorkload("qkv_sp_h4096", 16384, 4096, 12288, 8, "column", 0.02,
                                   seq_chunks=8),
    "attn_out_sp_h4096": LinearWorkload("attn_out_sp_h4096", 16384, 4096, 4096, 8, "row", 0.02,
                                        seq_chunks=8),
}


def custom_linear(tokens: int, in_features: int, out_features: int, t: int, split: str,
                  sigma_w: float = 0.02, seq_chunks: int = 1,
                  name: str = "custom_linear") -> LinearWorkload:
    return LinearWorkload(name, tokens, in_features, out_features, t, split, sigma_w, seq_chunks)


def make_linear_inputs(w: LinearWorkload, seed: int = 0) -> dict:
    """Full (unsharded) bf16 CPU tensors X [T, in], W [in, out], b [out],
    dY [T, out] for linear workload w."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))

    def draw(shape, std):
        x = torch.randn(*shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    X = draw((w.tokens, w.in_features), 1.0)
    W = draw((w.in_features, w.out_features), w.sigma_w)
    b = draw((w.out_features,), w.sigma_b)
    dY = draw((w.tokens, w.out_features), 1.0)
    return {"X": X, "W": W, "b": b, "dY": dY}


def make_sp_inputs(w: Workload, seed: int = 0) -> dict:
    """The block's inputs plus the LayerNorm parameters gamma, beta [h] (bf16);
    "dZ" is the sublayer's upstream gradient dOut."""
    d = make_inputs(w, seed)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 0x5EED)
    gamma = (1.0 + 0.1 * torch.randn(w.hidden, generator=g, dtype=torch.float32))
    beta = 0.02 * torch.randn(w.hidden, generator=g, dtype=torch.float32)
    d["gamma"] = gamma.to(torch.bfloat16)
    d["beta"] = beta.to(torch.bfloat16)
    return d
