"""Device buffers for the sequence-parallel sublayer Out = X + Dropout(MLP(LN(X)))
and the calls that run it.

PyTorch is used for device memory and streams only; both passes run in
libtpmlp through :mod:`binding`.  Layouts follow the C ABI: X, Out, dOut, dX
as seq_chunks token chunks [T/chunks, h]; A/B as t column/row shards; gamma,
beta [h] bf16; fp32 weight, bias and LayerNorm-parameter gradients.
"""
from __future__ import annotations

import torch

from . import binding
from .inputs import Workload, column_shards, row_shards, seq_chunks


class DeviceSPLayer:
    def __init__(self, w: Workload, inputs: dict, device="cuda:0", eps: float = 1e-5,
                 dropout_p: float = 0.1, seed: int = 1234, offset: int = 0):
        """inputs: make_sp_inputs(w); inputs["dZ"] is the upstream gradient dOut."""
        dev = torch.device(device)
        self.w = w
        T, h, f, t, n = w.tokens, w.hidden, w.ffn, w.t, w.seq_chunks
        fi = f // t
        self.dims = binding.make_dims(T, h, f, t, n)
        self.sp = binding.make_sp_params(eps, dropout_p, seed, offset)
        bf, f32 = torch.bfloat16, torch.float32
        self.X = [c.to(dev) for c in seq_chunks(inputs["X"], n)]
        self.dOut = [c.to(dev) for c in seq_chunks(inputs["dZ"], n)]
        self.A = [a.to(dev) for a in column_shards(inputs["A"], t)]
        self.B = [b.to(dev) for b in row_shards(inputs["B"], t)]
        self.b1 = inputs["b1"].to(dev)
        self.b2 = inputs["b2"].to(dev)
        self.gamma = inputs["gamma"].to(dev)
        self.beta = inputs["beta"].to(dev)
        self.Out = [torch.empty(T // n, h, dtype=bf, device=dev) for _ in range(n)]
        self.dX = [torch.empty(T // n, h, dtype=bf, device=dev) for _ in range(n)]
        self.dA = [torch.empty(h, fi, dtype=f32, device=dev) for _ in range(t)]
        self.dB = [torch.empty(fi, h, dtype=f32, device=dev) for _ in range(t)]
        self.db1 = torch.empty(f, dtype=f32, device=dev)
        self.db2 = torch.empty(h, dtype=f32, device=dev)
        self.dgamma = torch.empty(h, dtype=f32, device=dev)
        self.dbeta = torch.empty(h, dtype=f32, device=dev)
        self.ws = torch.empty(max(binding.tpmlp_sp_workspace_bytes(self.dims), 256),
                              dtype=torch.uint8, device=dev)

    def forward(self, stream=None, X=None, Out=None) -> None:
        binding.tpmlp_sp_forward(self.dims, self.sp, self.X if X is None else X, self.gamma,
                                 self.beta, self.A, self.b1, self.B, self.b2, self.w.t,
                                 self.Out if Out is None else Out, self.ws, stream)

    def backward(self, stream=None, dOut=None, X=None, dX=None) -> None:
        binding.tpmlp_sp_backward(self.dims, self.sp, self.dOut if dOut is None else dOut,
                                  self.X if X is None else X, self.gamma, self.A, self.B, self.ws,
                                  self.dX if dX is None else dX, self.dgamma, self.dbeta, self.dA,
                                  self.db1, self.dB, self.db2, stream)

    def step(self, stream=None) -> None:
        self.forward(stream)
        self.backward(stream)

    def workspace_tensor(self, which: str) -> torch.Tensor:
        """LN(X) ("xn") or dZ ("dz") as a [T, h] bf16 view of the workspace."""
        xn, dz = binding.tpmlp_sp_workspace_layout(self.dims)
        off = xn if which == "xn" else dz
        T, h = self.w.tokens, self.w.hidden
        return self.ws[off:off + T * h * 2].view(torch.bfloat16).view(T, h)
