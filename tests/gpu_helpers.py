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


def _chain_rows(rows, cap, mult):
    n = (rows + cap - 1) // cap
    return ((rows + n - 1) // n + mult - 1) // mult * mult


def pair_chunk_modes(layer, gate_up=True):
    """The chunk mode the CTA-pair kernel picks for each active expert of a
    layer, from the rule it states: chunks of 256 pairs with chains of nu rows
    (mode 0), or of 256 + 128 pairs with chains of nu_t rows (mode 1),
    whichever copies fewer rows per K step over the expert's tasks.  Returns
    [(pairs, mode)] per expert with pairs; used by tests to show that their
    shapes reach both modes and tails of every size."""
    ids = layer.topk_ids.ravel()
    ids = ids[(ids >= 0) & (ids < layer.E)]
    counts = np.bincount(ids, minlength=layer.E)
    out_rows = layer.I if gate_up else layer.H
    chain = layer.I if gate_up else (layer.H + 1) // 2
    nu0, nu1 = _chain_rows(chain, 256, 16), _chain_rows(chain, 160, 32)
    tr0, tr1 = (nu0, nu1) if gate_up else (2 * nu0, 2 * nu1)
    nt0, nt1 = -(-out_rows // tr0), -(-out_rows // tr1)
    res = []
    for m in counts[counts > 0]:
        m = int(m)
        rows0 = -(-m // 256) * nt0 * (128 + nu0)
        tails = m // 384 + (1 if m % 384 > 256 else 0)
        rows1 = nt1 * (-(-m // 384) * (128 + nu1) + tails * 64)
        res.append((m, 1 if rows1 < rows0 else 0))
    return res
