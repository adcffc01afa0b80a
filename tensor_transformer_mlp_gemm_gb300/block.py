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
    def __init__(self, w: Workload, inputs: dict, device="cuda:0", recompute: bool = False,
                 scratch: torch.Tensor | None = None):
        """recompute=True runs the selective-recompute calls: only Y is kept
        between forward and backward (self.saved_y); H and dY live in a
        scratch buffer that several blocks on one stream may share."""
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
        self.recompute = recompute
        if recompute:
            sv, sc = binding.tpmlp_recompute_workspace_bytes(self.dims)
            self.saved_y = torch.empty(max(sv, 256), dtype=torch.uint8, device=dev)
            self.scratch = scratch if scratch is not None else torch.empty(
                max(sc, 256), dtype=torch.uint8, device=dev)
            self.ws = None
        else:
            self.ws = torch.empty(max(binding.tpmlp_workspace_bytes(self.dims), 256),
                                  dtype=torch.uint8, device=dev)

    def forward(self, stream=None) -> None:
        if self.recompute:
            binding.tpmlp_forward_recompute(self.dims, self.X, self.A, self.b1, self.B, self.b2,
                                            self.w.t, self.Z, self.saved_y, self.scratch, stream)
        else:
            binding.tpmlp_forward(self.dims, self.X, self.A, self.b1, self.B, self.b2, self.w.t,
                                  self.Z, self.ws, stream)

    def backward(self, stream=None) -> None:
        if self.recompute:
            binding.tpmlp_backward_recompute(self.dims, self.dZ, self.X, self.A, self.B,
                                             self.saved_y, self.scratch, self.dX, self.dA,
                                             self.db1, self.dB, self.db2, stream)
        else:
            binding.tpmlp_backward(self.dims, self.dZ, self.X, self.A, self.B, self.ws, self.dX,
                                   self.dA, self.db1, self.dB, self.db2, stream)

    def step(self, stream=None) -> None:
        self.forward(stream)
        self.backward(stream)

    def saved(self) -> dict:
        """Views of Y, H, dY as lists of t [T, fi] bf16 tensors (with recompute:
        Y in the saved buffer, H and dY in the scratch buffer)."""
        T, fi, t = self.w.tokens, self.w.ffn // self.w.t, self.w.t
        y, h, dy = binding.tpmlp_workspace_layout(self.dims)
        n = T * fi * 2

        def view(buf, off):
            return [buf[off + i * n: off + (i + 1) * n].view(torch.bfloat16).view(T, fi)
                    for i in range(t)]
        if self.recompute:
            return {"Y": view(self.saved_y, 0), "H": view(self.scratch, 0),
                    "dY": view(self.scratch, dy - h)}
        return {"Y": view(self.ws, y), "H": view(self.ws, h), "dY": view(self.ws, dy)}
