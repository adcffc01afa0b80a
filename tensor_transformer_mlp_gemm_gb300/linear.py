"""Device buffers for one tensor-parallel linear layer and the calls that run
it (the attention projections: QKV column parallel, output projection row
parallel).

PyTorch is used for device memory and streams only; both passes run in
libtpmlp through :mod:`binding`.  Layouts follow the C ABI:
  column: X, dX as seq_chunks token chunks [Tc, in]; W_i [in, oi];
          Y_i, dY_i [T, oi]
  row:    X_i, dX_i [T, ii]; W_i [ii, out]; Z, dZ as seq_chunks chunks [Tc, out]
with fp32 weight and bias gradients.
"""
from __future__ import annotations

import torch

from . import binding
from .inputs import LinearWorkload, column_shards, row_shards, seq_chunks


class DeviceLinear:
    def __init__(self, w: LinearWorkload, inputs: dict, device="cuda:0",
                 workspace: torch.Tensor | None = None):
        """inputs: make_linear_inputs(w).  For a row split the input X is
        handed to the layer as its t column blocks X_i and the upstream
        gradient dY (the gradient of Z) as token chunks."""
        if w.split not in ("column", "row"):
            raise ValueError("split must be 'column' or 'row'")
        dev = torch.device(device)
        self.w = w
        T, din, dout, t, n = w.tokens, w.in_features, w.out_features, w.t, w.seq_chunks
        s = w.shard
        self.dims = binding.make_linear_dims(T, din, dout, t, n)
        bf, f32 = torch.bfloat16, torch.float32
        self.b = inputs["b"].to(dev)
        self.db = torch.empty(dout, dtype=f32, device=dev)
        if w.split == "column":
            self.X = [c.to(dev) for c in seq_chunks(inputs["X"], n)]
            self.W = [x.to(dev) for x in column_shards(inputs["W"], t)]
            self.dY = [x.to(dev) for x in column_shards(inputs["dY"], t)]
            self.Y = [torch.empty(T, s, dtype=bf, device=dev) for _ in range(t)]
            self.dX = [torch.empty(T // n, din, dtype=bf, device=dev) for _ in range(n)]
            self.dW = [torch.empty(din, s, dtype=f32, device=dev) for _ in range(t)]
        else:
            self.X = [x.to(dev) for x in column_shards(inputs["X"], t)]
            self.W = [x.to(dev) for x in row_shards(inputs["W"], t)]
            self.dY = [c.to(dev) for c in seq_chunks(inputs["dY"], n)]
            self.Y = [torch.empty(T // n, dout, dtype=bf, device=dev) for _ in range(n)]
            self.dX = [torch.empty(T, s, dtype=bf, device=dev) for _ in range(t)]
            self.dW = [torch.empty(s, dout, dtype=f32, device=dev) for _ in range(t)]
        need = max(binding.tpmlp_linear_workspace_bytes(self.dims), 256)
        if workspace is not None and workspace.numel() >= need:
            self.ws = workspace
        else:
            self.ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def forward(self, stream=None, X=None, Y=None) -> None:
        """Y = layer(X); X and Y default to the layer's own buffers (a caller
        may pass other device buffers of the same layout)."""
        X = self.X if X is None else X
        Y = self.Y if Y is None else Y
        fn = (binding.tpmlp_column_linear_forward if self.w.split == "column"
              else binding.tpmlp_row_linear_forward)
        fn(self.dims, X, self.W, self.b, Y, self.ws, stream)

    def backward(self, stream=None, dY=None, X=None, dX=None) -> None:
        dY = self.dY if dY is None else dY
        X = self.X if X is None else X
        dX = self.dX if dX is None else dX
        fn = (binding.tpmlp_column_linear_backward if self.w.split == "column"
              else binding.tpmlp_row_linear_backward)
        fn(self.dims, dY, X, self.W, dX, self.dW, self.db, self.ws, stream)

    def step(self, stream=None) -> None:
        self.forward(stream)
        self.backward(stream)
