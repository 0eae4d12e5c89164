"""Shared helpers for the GPU parity tests (CUDA path via the C ABI vs the oracle)."""
import numpy as np
import torch

from lora_moe_layer_gb300 import binding as B

# max|gpu - ref| / max|ref| on layer outputs, bf16 I/O with fp32 accumulation
TOL = 1e-2


def norm_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(gpu - ref)) / max(float(np.max(np.abs(ref))), 1e-30))


def gpu_align(topk_ids: np.ndarray, lora_ids: np.ndarray, E: int, L: int, bm: int, H: int = 8, I: int = 8,
              r: int = 8):
    """Run moe_lora_align on cuda:0; returns (dict of numpy outputs, status)."""
    dev = torch.device("cuda")
    topk = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, k = topk.shape
    d = B.dims(T, H, I, E, k, L, r, bm)
    cap = B.moe_lora_align_capacity(d)
    assert cap >= 0, cap
    NB = E * (L + 1)
    poison = -12345
    sorted_ids = torch.full((max(cap, 1),), poison, dtype=torch.int32, device=dev)
    tiles = max(cap // bm, 1)
    tile_expert = torch.full((tiles,), poison, dtype=torch.int32, device=dev)
    tile_lora = torch.full((tiles,), poison, dtype=torch.int32, device=dev)
    npp = torch.full((1,), poison, dtype=torch.int32, device=dev)
    cnt = torch.full((NB,), poison, dtype=torch.int32, device=dev)
    off = torch.full((NB + 1,), poison, dtype=torch.int32, device=dev)
    ws = torch.empty(B.moe_lora_workspace_bytes(d), dtype=torch.uint8, device=dev)
    t_topk = torch.from_numpy(topk).to(dev)
    t_lora = torch.from_numpy(np.ascontiguousarray(lora_ids, dtype=np.int32)).to(dev)
    B.check(B.moe_lora_align(d, t_topk, t_lora, sorted_ids, tile_expert, tile_lora, npp, cnt, off, ws),
            "moe_lora_align")
    status = B.moe_lora_get_status(ws)
    n = int(npp.item())
    res = dict(sorted_ids=sorted_ids[:n].cpu().numpy(), tile_expert=tile_expert[:n // bm].cpu().numpy(),
               tile_lora=tile_lora[:n // bm].cpu().numpy(), num_post_padded=n,
               bucket_count=cnt.cpu().numpy(), bucket_offset=off.cpu().numpy(),
               tail=sorted_ids[n:].cpu().numpy())
    return res, status
