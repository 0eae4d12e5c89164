"""Seeded synthetic inputs for the multi-LoRA fused MoE layer.

This module only draws numbers: activations, base expert weights, LoRA
adapters, per-token adapter ids and the upstream router's top-k choice.  It
holds none of the layer's own arithmetic (no gate_up, activation, down or
aggregation), so both the CUDA path and the CPU oracle may consume what it
builds without sharing any of the method.

Layouts (all row-major, "[out][in]", i.e. the reduction dimension is the
contiguous one).  The pages write a projection as ``y = xW + xAB`` with W of
shape h_in x h_out, A h_in x r and B r x h_out ("Efficiently serve dozens of
fine-tuned models with vLLM on Amazon SageMaker AI and Amazon Bedrock", section
"Implementing multi-LoRA inference for MoE models in vLLM", around Figure 1);
the arrays here store the transposes of those matrices:

    x        [T][H]          bf16 bits (uint16)
    W1       [E][2I][H]      gate rows [0, I), up rows [I, 2I)
    W2       [E][H][I]
    A1       [L][E][r][H]    B1 [L][E][2I][r]
    A2       [L][E][r][I]    B2 [L][E][H][r]
    topk_ids [T][k] int32, topk_weights [T][k] float32, lora_ids [T] int32

Every tensor has its own PCG64 stream keyed by (seed, tensor tag[, expert]),
so a tensor's values do not depend on the shape of any other tensor (the dense
workload keeps its weights while only the token count changes).
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Optional

import numpy as np

# stream tags: one independent PCG64 stream per tensor
_TAG = {"x": 0, "Wr": 1, "W1": 2, "W2": 3, "A1": 4, "B1": 5, "A2": 6, "B2": 7,
        "lora": 8, "base_mask": 9}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if not np.isfinite(a).all():
        raise ValueError("bf16_bits expects finite values")
    u = a.view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    # slabs bound the temporaries on multi-GB weights; for finite inputs the
    # uint32 sum below cannot wrap (largest finite 0xFF7FFFFF + 0x8000 < 2^32)
    step = 1 << 24
    for s in range(0, u.size, step):
        v = u[s:s + step]
        lsb = (v >> 16) & np.uint32(1)
        lsb += v
        lsb += np.uint32(0x7FFF)
        lsb >>= 16
        out[s:s + step] = lsb
    return out.reshape(a.shape)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(seed: int, tag: str, shape, std: float, sub: Optional[int] = None) -> np.ndarray:
    key = [seed, _TAG[tag]] if sub is None else [seed, _TAG[tag], sub]
    rng = np.random.default_rng(key)
    a = rng.standard_normal(int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return bf16_bits(a).reshape(shape)


def _normal_bf16_per_expert(seed: int, tag: str, lead: tuple, shape_rest: tuple, std: float) -> np.ndarray:
    """Draw a [*lead, *shape_rest] tensor with one stream per flattened lead index."""
    n_lead = int(np.prod(lead)) if lead else 1
    out = np.empty((n_lead,) + tuple(shape_rest), dtype=np.uint16)

    def fill(i):
        out[i] = _normal_bf16(seed, tag, shape_rest, std, sub=i)

    # each slice has its own stream, so the fill order (and thread count) cannot change values
    if n_lead * int(np.prod(shape_rest)) >= (1 << 22) and n_lead > 1:
        with concurrent.futures.ThreadPoolExecutor(max_workers=_threads()) as ex:
            list(ex.map(fill, range(n_lead)))
    else:
        for i in range(n_lead):
            fill(i)
    return out.reshape(tuple(lead) + tuple(shape_rest))


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


@dataclasses.dataclass
class Layer:
    """One synthetic MoE-LoRA layer plus one batch of routed tokens."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    L: int
    r: int
    x: np.ndarray
    W1: np.ndarray
    W2: np.ndarray
    A1: Optional[np.ndarray]
    B1: Optional[np.ndarray]
    A2: Optional[np.ndarray]
    B2: Optional[np.ndarray]
    topk_ids: np.ndarray
    topk_weights: np.ndarray
    lora_ids: np.ndarray
    meta: dict = dataclasses.field(default_factory=dict)
    # FP8 base expert weights (see quantize_e4m3), or None
    w8: Optional["W8Weights"] = None

    @property
    def P(self) -> int:
        return self.T * self.k

    def dims(self) -> dict:
        return dict(T=self.T, H=self.H, I=self.I, E=self.E, k=self.k, L=self.L, r=self.r)


# ----------------------------------------------------------------------------
# router (upstream of the layer: its output is an input of the layer)
# ----------------------------------------------------------------------------

def router_logits(x_bits: np.ndarray, Wr_bits: np.ndarray) -> np.ndarray:
    """fp64 logits x.Wr from bf16 x [T][H] and bf16 Wr [E][H]."""
    x = bf16_to_f32(x_bits).astype(np.float64)
    w = bf16_to_f32(Wr_bits).astype(np.float64)
    return x @ w.T


def route_topk(logits: np.ndarray, k: int):
    """Top-k by descending logit (ties to the lower expert id); weights are the
    softmax over the k chosen logits, which equals the renormalised full softmax."""
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    wts = np.empty((T, k), dtype=np.float32)
    # a stable sort of the negated logits keeps equal logits in ascending expert order
    order_all = np.argsort(-logits, axis=1, kind="stable")
    for t in range(T):
        order = order_all[t, :k]
        sel = logits[t, order]
        m = sel.max()
        ex = np.exp(sel - m)
        ids[t] = order
        wts[t] = (ex / ex.sum()).astype(np.float32)
    return ids, wts


def _hot_share(logits: np.ndarray, k: int, beta: float, n_hot: int) -> float:
    sk = logits.copy()
    sk[:, :n_hot] += beta
    ids, _ = route_topk(sk, k)
    return float((ids < n_hot).mean())


# ----------------------------------------------------------------------------
# generic builder
# ----------------------------------------------------------------------------

def make_layer(name: str, T: int, H: int, I: int, E: int, k: int, L: int, r: int,
               lora_ids: np.ndarray, seed: int = 0, skew_hot: int = 0,
               skew_target: float = 0.5, with_lora: bool = True) -> Layer:
    x = _normal_bf16(seed, "x", (T, H), 1.0)
    Wr = _normal_bf16(seed, "Wr", (E, H), 1.0 / math.sqrt(H))
    W1 = _normal_bf16_per_expert(seed, "W1", (E,), (2 * I, H), 1.0 / math.sqrt(H))
    W2 = _normal_bf16_per_expert(seed, "W2", (E,), (H, I), 1.0 / math.sqrt(I))
    if with_lora and L > 0:
        A1 = _normal_bf16_per_expert(seed, "A1", (L, E), (r, H), 1.0 / math.sqrt(H))
        B1 = _normal_bf16_per_expert(seed, "B1", (L, E), (2 * I, r), 0.02)
        A2 = _normal_bf16_per_expert(seed, "A2", (L, E), (r, I), 1.0 / math.sqrt(I))
        B2 = _normal_bf16_per_expert(seed, "B2", (L, E), (H, r), 0.02)
    else:
        A1 = B1 = A2 = B2 = None
    logits = router_logits(x, Wr)
    meta = {}
    if skew_hot:
        lo, hi = 0.0, 8.0
        beta = 0.0
        for _ in range(40):
            beta = 0.5 * (lo + hi)
            s = _hot_share(logits, k, beta, skew_hot)
            if abs(s - skew_target) < 0.01:
                break
            if s < skew_target:
                lo = beta
            else:
                hi = beta
        logits = logits.copy()
        logits[:, :skew_hot] += beta
        meta["skew_beta"] = beta
    topk_ids, topk_weights = route_topk(logits, k)
    if skew_hot:
        meta["hot_share"] = float((topk_ids < skew_hot).mean())
    return Layer(name, T, H, I, E, k, L, r, x, W1, W2, A1, B1, A2, B2,
                 topk_ids, topk_weights, np.ascontiguousarray(lora_ids, dtype=np.int32), meta)


def _lora_rng(seed: int, tag: str = "lora"):
    return np.random.default_rng([seed, _TAG[tag]])


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

CONFIG_NAMES = {
    0: "tiny T=8 H=256 I=512 E=8 k=2 L=2 r=8",
    1: "GPT-OSS-20B-shaped decode T=16 H=2880 I=2880 E=32 k=4 L=8 r=32",
    2: "GPT-OSS-20B-shaped prefill T=2048 (16x128) H=2880 I=2880 E=32 k=4 L=8 r=32",
    3: "Qwen3-MoE-30B-A3B-shaped mixed T=256 H=2048 I=768 E=128 k=8 L=16 r=16 zipf",
    4: "dense Llama-3.3-70B-shaped MLP E=1 k=1 H=8192 I=28672 L=32 r=64",
}


def config_shape(idx: int, T: Optional[int] = None) -> dict:
    if idx == 0:
        return dict(T=8, H=256, I=512, E=8, k=2, L=2, r=8)
    if idx == 1:
        return dict(T=16, H=2880, I=2880, E=32, k=4, L=8, r=32)
    if idx == 2:
        return dict(T=2048, H=2880, I=2880, E=32, k=4, L=8, r=32)
    if idx == 3:
        return dict(T=256, H=2048, I=768, E=128, k=8, L=16, r=16)
    if idx == 4:
        return dict(T=T if T is not None else 16, H=8192, I=28672, E=1, k=1, L=32, r=64)
    raise ValueError(idx)


def config_lora_ids(idx: int, T: int, L: int, seed: int = 0) -> np.ndarray:
    rng = _lora_rng(seed)
    if idx == 0:
        return rng.integers(-1, L, size=T).astype(np.int32)           # uniform {-1, 0, 1}
    if idx == 1:
        return rng.integers(0, L, size=T).astype(np.int32)            # uniform 0..7
    if idx == 2:
        seq_len = 128
        n_seq = (T + seq_len - 1) // seq_len
        per_seq = rng.integers(-1, L, size=n_seq).astype(np.int32)   # uniform {-1, 0..7}
        return np.repeat(per_seq, seq_len)[:T]
    if idx == 3:
        probs = np.array([(i + 1) ** -1.1 for i in range(L)], dtype=np.float64)
        probs /= probs.sum()
        ids = rng.choice(L, size=T, p=probs).astype(np.int32)          # Zipf(1.1) popularity
        base = _lora_rng(seed, "base_mask").random(T) < 0.1           # 10% base-only
        ids[base] = -1
        return ids
    if idx == 4:
        return rng.integers(0, L, size=T).astype(np.int32)            # uniform 0..31
    raise ValueError(idx)


def make_config(idx: int, T: Optional[int] = None, seed: int = 0, with_lora: bool = True) -> Layer:
    s = config_shape(idx, T)
    lora = config_lora_ids(idx, s["T"], s["L"], seed)
    return make_layer(f"config{idx}", s["T"], s["H"], s["I"], s["E"], s["k"], s["L"], s["r"],
                      lora, seed=seed, skew_hot=16 if idx == 3 else 0, with_lora=with_lora)


def make_random(T: int, H: int, I: int, E: int, k: int, L: int, r: int, seed: int = 1,
                p_base: float = 0.3) -> Layer:
    """A small random layer for tests: adapter ids uniform over {-1..L-1}-ish."""
    rng = np.random.default_rng([seed, 99])
    lora = rng.integers(0, max(L, 1), size=T).astype(np.int32) if L > 0 else np.full(T, -1, np.int32)
    if L > 0:
        lora[rng.random(T) < p_base] = -1
    return make_layer(f"random_T{T}_H{H}_I{I}_E{E}_k{k}_L{L}_r{r}", T, H, I, E, k, L, r, lora,
                      seed=seed, with_lora=L > 0)


# ---------------------------------------------------------------------------- FP8 weights

@dataclasses.dataclass
class W8Weights:
    """E4M3 codes of the base expert weights with one fp32 scale per output
    row: W1q [E][2I][H] uint8, W1s [E][2I] float32, W2q [E][H][I], W2s [E][H];
    weight = scale * value(code)."""
    W1q: np.ndarray
    W1s: np.ndarray
    W2q: np.ndarray
    W2s: np.ndarray


def _e4m3_rows(bits: np.ndarray):
    """Per-row symmetric quantisation of bf16 rows (last axis) to E4M3: scale =
    max |row| / 448 (the largest finite E4M3 value), codes = the row / scale
    rounded to nearest by torch's float8_e4m3fn conversion."""
    import torch
    w = bf16_to_f32(bits).astype(np.float32)
    amax = np.max(np.abs(w), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = torch.from_numpy(np.ascontiguousarray(w / scale[..., None])).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy().copy(), scale


def quantize_e4m3(layer: Layer) -> Layer:
    """The layer with its base expert weights W1, W2 replaced by E4M3 codes and
    per-output-row scales (the LoRA matrices stay bf16).  The bf16 W1 and W2
    are kept for reference; the FP8 forward reads only layer.w8."""
    W1q, W1s = _e4m3_rows(layer.W1)
    W2q, W2s = _e4m3_rows(layer.W2)
    return dataclasses.replace(layer, name=layer.name + "_e4m3", w8=W8Weights(W1q, W1s, W2q, W2s))

