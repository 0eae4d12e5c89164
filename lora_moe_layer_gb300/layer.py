"""Device-resident layer: owns torch device copies of one layer's tensors and
a workspace, and calls the C ABI through ``binding``.  No arithmetic of the
layer happens here (argument marshalling and memory plumbing only)."""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import binding as B


def _dev_bf16(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


class DeviceLayer:
    """Weights and one batch of a ``workloads.Layer`` copied to a CUDA device."""

    def __init__(self, layer, device="cuda", block_m: int = 0, options: int = 0):
        self.layer = layer
        self.device = torch.device(device)
        self.d = B.dims(layer.T, layer.H, layer.I, layer.E, layer.k, layer.L, layer.r, block_m, options)
        dev = self.device
        self.W1 = _dev_bf16(layer.W1, dev)
        self.W2 = _dev_bf16(layer.W2, dev)
        has = layer.A1 is not None and layer.L > 0
        self.A1 = _dev_bf16(layer.A1, dev) if has else None
        self.B1 = _dev_bf16(layer.B1, dev) if has else None
        self.A2 = _dev_bf16(layer.A2, dev) if has else None
        self.B2 = _dev_bf16(layer.B2, dev) if has else None
        # FP8 base weights (E4M3 codes and per-row scales), when the layer has them
        q = getattr(layer, "w8", None)
        if q is not None:
            self.W1q = torch.from_numpy(np.ascontiguousarray(q.W1q, dtype=np.uint8)).to(dev)
            self.W2q = torch.from_numpy(np.ascontiguousarray(q.W2q, dtype=np.uint8)).to(dev)
            self.W1s = torch.from_numpy(np.ascontiguousarray(q.W1s, dtype=np.float32)).to(dev)
            self.W2s = torch.from_numpy(np.ascontiguousarray(q.W2s, dtype=np.float32)).to(dev)
        self.set_batch(layer.x, layer.topk_ids, layer.topk_weights, layer.lora_ids)
        self.ws_bytes = B.moe_lora_workspace_bytes(self.d)
        if self.ws_bytes == 0:
            raise B.MoeLoraError(B.MOELORA_EINVAL, "moe_lora_workspace_bytes")
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty((layer.T, layer.H), dtype=torch.bfloat16, device=dev)

    def set_batch(self, x_bits, topk_ids, topk_weights, lora_ids):
        dev = self.device
        self.x = _dev_bf16(x_bits, dev)
        self.topk_ids = torch.from_numpy(np.ascontiguousarray(topk_ids, dtype=np.int32)).to(dev)
        self.topk_weights = torch.from_numpy(np.ascontiguousarray(topk_weights, dtype=np.float32)).to(dev)
        self.lora_ids = torch.from_numpy(np.ascontiguousarray(lora_ids, dtype=np.int32)).to(dev)

    def forward(self, stream=None, out: Optional[torch.Tensor] = None) -> int:
        """Launch moe_lora_forward; returns the host-side status (no sync)."""
        o = self.out if out is None else out
        return B.moe_lora_forward(self.d, self.x, self.topk_ids, self.topk_weights, self.lora_ids,
                                  self.W1, self.W2, self.A1, self.B1, self.A2, self.B2, o,
                                  self.workspace, stream)

    def forward_w8(self, stream=None, out: Optional[torch.Tensor] = None) -> int:
        """Launch moe_lora_forward_w8 with the layer's FP8 base weights."""
        o = self.out if out is None else out
        return B.moe_lora_forward_w8(self.d, self.x, self.topk_ids, self.topk_weights, self.lora_ids,
                                     self.W1q, self.W1s, self.W2q, self.W2s, self.A1, self.B1, self.A2, self.B2,
                                     o, self.workspace, stream)

    def forward_traced(self, events, stream=None, w8: bool = False) -> int:
        """The forward (FP8 weights when w8) with an event recorded before each
        kernel slot and after the last (MOELORA_TRACE_EVENTS events)."""
        if w8:
            return B.moe_lora_forward_w8_traced(self.d, self.x, self.topk_ids, self.topk_weights, self.lora_ids,
                                                self.W1q, self.W1s, self.W2q, self.W2s, self.A1, self.B1, self.A2,
                                                self.B2, self.out, self.workspace, events, stream)
        return B.moe_lora_forward_traced(self.d, self.x, self.topk_ids, self.topk_weights, self.lora_ids, self.W1,
                                         self.W2, self.A1, self.B1, self.A2, self.B2, self.out, self.workspace, events,
                                         stream)

    def status(self, stream=None) -> int:
        return B.moe_lora_get_status(self.workspace, stream)

    def out_f64(self) -> np.ndarray:
        """The bf16 output widened to float64 (exact)."""
        bits = self.out.view(torch.int16).cpu().numpy().view(np.uint16)
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def workspace_view(self, name: str, dtype: torch.dtype, shape) -> torch.Tensor:
        """A view of one intermediate of the last forward (see moe_lora_ws_layout)."""
        lay = B.moe_lora_workspace_layout(self.d)
        off = lay[name]
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        return self.workspace[off:off + n].view(dtype).view(*shape)

    def pair_outputs(self) -> np.ndarray:
        """w * d per pair id of the last forward as fp64 [P][H]: the bf16 per-pair
        outputs, or the sum of the fp32 K-split slabs when the down GEMM split K."""
        lay = B.moe_lora_workspace_layout(self.d)
        P, H = self.d.T * self.d.k, self.d.H
        if lay["pair_out_bf16"]:
            bits = self.workspace_view("pair_out", torch.int16, (P, H)).cpu().numpy().view(np.uint16)
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        s = lay["down_splits"]
        return self.workspace_view("pair_out", torch.float32, (s, P, H)).cpu().numpy().astype(np.float64).sum(0)
