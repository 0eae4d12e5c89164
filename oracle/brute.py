"""Brute-force numpy restatements used to pin the C oracle -- TEST INFRASTRUCTURE.

Written independently of ``oracle.c``: dense fp64 matrices per (token, slot)
pair with numpy matmuls as the only library step.  Three forms:

* ``forward``          -- shrink-then-expand, y = x W + (x A) B, per pair;
* ``forward_merged``   -- the same layer with each adapter folded into dense
                          weights W' = W + A B, then base-only (the rank-r
                          delta must equal the dense update: associativity of
                          the blog's y = xW + xAB, "Efficiently serve dozens of
                          fine-tuned models with vLLM ...", section
                          "Implementing multi-LoRA inference for MoE models in
                          vLLM");
* ``align_sorted``     -- expert x adapter bucketing via Python's stable sort.

Arrays follow the layouts of ``lora_moe_layer_gb300.workloads`` ([out][in]).
"""
from __future__ import annotations

import numpy as np


def f64(bits) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(u: np.ndarray) -> np.ndarray:
    return u / (1.0 + np.exp(-u))


def _pair_valid(layer, e: int, l: int) -> bool:
    return 0 <= e < layer.E and -1 <= l < layer.L


def forward(layer) -> np.ndarray:
    """[T][H] fp64: out[t] = sum_j w[t,j] * FFN_{e(t,j), l(t)}(x[t])."""
    out = np.zeros((layer.T, layer.H))
    I = layer.I
    has_lora = layer.A1 is not None
    for t in range(layer.T):
        xt = f64(layer.x[t])
        l = int(layer.lora_ids[t])
        for j in range(layer.k):
            e = int(layer.topk_ids[t, j])
            if not _pair_valid(layer, e, l):
                continue
            g = f64(layer.W1[e]) @ xt
            if l >= 0 and has_lora:
                z1 = f64(layer.A1[l, e]) @ xt
                g = g + f64(layer.B1[l, e]) @ z1
            act = silu(g[:I]) * g[I:]
            d = f64(layer.W2[e]) @ act
            if l >= 0 and has_lora:
                z2 = f64(layer.A2[l, e]) @ act
                d = d + f64(layer.B2[l, e]) @ z2
            out[t] += float(layer.topk_weights[t, j]) * d
    return out


def forward_merged(layer) -> np.ndarray:
    """Same layer, each adapter folded into dense expert weights first."""
    out = np.zeros((layer.T, layer.H))
    I = layer.I
    has_lora = layer.A1 is not None
    cache = {}
    for t in range(layer.T):
        xt = f64(layer.x[t])
        l = int(layer.lora_ids[t])
        for j in range(layer.k):
            e = int(layer.topk_ids[t, j])
            if not _pair_valid(layer, e, l):
                continue
            key = (e, l)
            if key not in cache:
                W1 = f64(layer.W1[e])
                W2 = f64(layer.W2[e])
                if l >= 0 and has_lora:
                    # [2I][r] @ [r][H] and [H][r] @ [r][I]: the dense update B.A in [out][in] form
                    W1 = W1 + f64(layer.B1[l, e]) @ f64(layer.A1[l, e])
                    W2 = W2 + f64(layer.B2[l, e]) @ f64(layer.A2[l, e])
                cache[key] = (W1, W2)
            W1, W2 = cache[key]
            g = W1 @ xt
            act = silu(g[:I]) * g[I:]
            out[t] += float(layer.topk_weights[t, j]) * (W2 @ act)
    return out


def align_sorted(topk_ids, lora_ids, E: int, L: int, bm: int) -> dict:
    """Bucketing by Python's (stable) sort on key (expert, adapter)."""
    topk = np.asarray(topk_ids)
    T, k = topk.shape
    P = T * k
    valid = [p for p in range(P)
             if 0 <= int(topk.flat[p]) < E and -1 <= int(lora_ids[p // k]) < L]
    key = {p: (int(topk.flat[p]), int(lora_ids[p // k])) for p in valid}
    order = sorted(valid, key=lambda p: key[p])
    sorted_ids, tile_expert, tile_lora = [], [], []
    counts = np.zeros(E * (L + 1), dtype=np.int64)
    offsets = np.zeros(E * (L + 1) + 1, dtype=np.int64)
    i = 0
    for e in range(E):
        for l in range(-1, L):
            b = e * (L + 1) + (l + 1)
            offsets[b] = len(sorted_ids)
            members = []
            while i < len(order) and key[order[i]] == (e, l):
                members.append(order[i])
                i += 1
            counts[b] = len(members)
            if members:
                n_pad = -(-len(members) // bm) * bm
                sorted_ids.extend(members + [P] * (n_pad - len(members)))
                tile_expert.extend([e] * (n_pad // bm))
                tile_lora.extend([l] * (n_pad // bm))
    offsets[-1] = len(sorted_ids)
    return dict(sorted_ids=np.array(sorted_ids, dtype=np.int32),
                tile_expert=np.array(tile_expert, dtype=np.int32),
                tile_lora=np.array(tile_lora, dtype=np.int32),
                num_post_padded=len(sorted_ids), bucket_count=counts.astype(np.int32),
                bucket_offset=offsets.astype(np.int32), invalid=P - len(valid))
