"""Device buffers for one MLP block and the calls that run it.

PyTorch is used for device memory and streams only; both passes run in
libtpmlp through :mod:`binding`.  Buffers follow the C ABI's layouts: X, Z,
dZ, dX as seq_chunks token chunks, A/B as t column/row shards, fp32 weight
and bias gradients.
"""
from __future__ import annotations

import torch

from . import binding
from .inputs import Workload, column_shards, row_shards, seq_chunks


class DeviceBlock:
    def __init__(self, w: Workload, inputs: dict, device="cuda:0"):
        dev = torch.device(device)
        self.w = w
        self.device = dev
        T, h, f, t, n = w.tokens, w.hidden, w.ffn, w.t, w.seq_chunks
        fi = f // t
        self.dims = binding.make_dims(T, h, f, t, n)
        bf = torch.bfloat16
        self.X = [c.to(dev) for c in seq_chunks(inputs["X"], n)]
        self.dZ = [c.to(dev) for c in seq_chunks(inputs["dZ"], n)]
        self.A = [a.to(dev) for a in column_shards(inputs["A"], t)]
        self.B = [b.to(dev) for b in row_shards(inputs["B"], t)]
        self.b1 = inputs["b1"].to(dev)
        self.b2 = inputs["b2"].to(dev)
        self.Z = [torch.empty(T // n, h, dtype=bf, device=dev) for _ in range(n)]
        self.dX = [torch.empty(T // n, h, dtype=bf, device=dev) for _ in range(n)]
        self.dA = [torch.empty(h, fi, dtype=torch.float32, device=dev) for _ in range(t)]
        self.dB = [torch.empty(fi, h, dtype=torch.float32, device=dev) for _ in range(t)]
        self.db1 = torch.empty(f, dtype=torch.float32, device=dev)
        self.db2 = torch.empty(h, dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(binding.tpmlp_workspace_bytes(self.dims), 256),
                              dtype=torch.uint8, device=dev)

    def forward(self, stream=None) -> None:
        binding.tpmlp_forward(self.dims, self.X, self.A, self.b1, self.B, self.b2, self.w.t,
                              self.Z, self.ws, stream)

    def backward(self, stream=None) -> None:
        binding.tpmlp_backward(self.dims, self.dZ, self.X, self.A, self.B, self.ws, self.dX,
                               self.dA, self.db1, self.dB, self.db2, stream)

    def step(self, stream=None) -> None:
        self.forward(stream)
        self.backward(stream)

    def saved(self) -> dict:
        """Views of the workspace's Y, H, dY as lists of t [T, fi] bf16 tensors."""
        T, fi, t = self.w.tokens, self.w.ffn // self.w.t, self.w.t
        y, h, dy = binding.tpmlp_workspace_layout(self.dims)
        n = T * fi * 2

        def view(off):
            return [self.ws[off + i * n: off + (i + 1) * n].view(torch.bfloat16).view(T, fi)
                    for i in range(t)]
        return {"Y": view(y), "H": view(h), "dY": view(dy)}
