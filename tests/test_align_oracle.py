"""Pins of the oracle's expert x adapter bucketing (CPU only).

The pages describe the fused_moe_lora kernel as the fused_moe logic plus one
more grid dimension over the active adapters, and name the two sparsities it
combines: expert routing and adapter selection ("Efficiently serve dozens of
fine-tuned models with vLLM ...", section "Implementing multi-LoRA inference for
MoE models in vLLM"); one BLOCK_SIZE_M is shared by the four LoRA ops (section
"Tuning kernel configurations").  The bucketing contract is the stable sort by
(expert, adapter) with each bucket padded to the tile height; it has exactly one
correct output, checked here by hand and by Python's stable sort.
"""
import numpy as np
import pytest

import oracle
from oracle import brute
from lora_moe_layer_gb300 import workloads as wl


def test_hand_worked_align():
    # pairs p = t*k + j: p0 (e2,l0) p1 (e0,l0) p2 (e0,l-1) p3 (e1,l-1) p4 (e2,l0) p5 (e0,l0)
    topk = np.array([[2, 0], [0, 1], [2, 0]], np.int32)
    lora = np.array([0, -1, 0], np.int32)
    # bucket b = e*(L+1) + (l+1) with L = 1:
    #   p0 -> 5, p1 -> 1, p2 -> 0, p3 -> 2, p4 -> 5, p5 -> 1
    # sorted, stable: b0 [p2], b1 [p1 p5], b2 [p3], b5 [p0 p4]; pad to 2 with 6
    a = oracle.align(topk, lora, E=3, L=1, bm=2)
    assert a["sorted_ids"].tolist() == [2, 6, 1, 5, 3, 6, 0, 4]
    assert a["num_post_padded"] == 8
    assert a["tile_expert"].tolist() == [0, 0, 1, 2]
    assert a["tile_lora"].tolist() == [-1, 0, -1, 0]
    assert a["bucket_count"].tolist() == [1, 2, 1, 0, 0, 2]
    assert a["bucket_offset"].tolist() == [0, 2, 4, 6, 6, 6, 8]
    assert a["invalid"] == 0


def _check_invariants(a, topk, lora, E, L, bm):
    T, k = topk.shape
    P = T * k
    s = a["sorted_ids"]
    n = a["num_post_padded"]
    assert n % bm == 0 and len(s) == n
    real = s[s != P]
    valid = [p for p in range(P) if 0 <= topk.flat[p] < E and -1 <= lora[p // k] < L]
    assert sorted(real.tolist()) == valid                  # a permutation of the valid pairs
    assert a["bucket_count"].sum() == len(valid)
    for q in range(n // bm):                               # every tile is one (expert, adapter)
        tile = s[q * bm:(q + 1) * bm]
        members = tile[tile != P]
        assert len(members) > 0
        for p in members:
            assert topk.flat[p] == a["tile_expert"][q]
            assert lora[p // k] == a["tile_lora"][q]
        # padding only at the end of a tile, and ascending pairs within it
        assert (np.diff(members) > 0).all()
    assert n <= a["capacity"]


@pytest.mark.parametrize("bm", [1, 2, 8, 16, 64, 128])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_align_matches_python_stable_sort(bm, seed):
    rng = np.random.default_rng([seed, 77])
    T, k, E, L = int(rng.integers(1, 200)), int(rng.integers(1, 9)), int(rng.integers(1, 40)), int(rng.integers(0, 9))
    topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
    lora = rng.integers(-1, L, size=T).astype(np.int32) if L > 0 else np.full(T, -1, np.int32)
    a = oracle.align(topk, lora, E, L, bm)
    b = brute.align_sorted(topk, lora, E, L, bm)
    for key in ("sorted_ids", "tile_expert", "tile_lora", "bucket_count", "bucket_offset"):
        assert np.array_equal(a[key], b[key]), key
    assert a["num_post_padded"] == b["num_post_padded"]
    _check_invariants(a, topk, lora, E, L, bm)


@pytest.mark.parametrize("cfg", [0, 1])
@pytest.mark.parametrize("bm", [8, 16, 64, 128])
def test_align_configs(cfg, bm):
    s = wl.config_shape(cfg)
    lora = wl.config_lora_ids(cfg, s["T"], s["L"])
    # routing only: the router needs x and Wr, not the expert weights
    x = wl._normal_bf16(0, "x", (s["T"], s["H"]), 1.0)
    Wr = wl._normal_bf16(0, "Wr", (s["E"], s["H"]), 1.0 / np.sqrt(s["H"]))
    topk, _ = wl.route_topk(wl.router_logits(x, Wr), s["k"])
    a = oracle.align(topk, lora, s["E"], s["L"], bm)
    b = brute.align_sorted(topk, lora, s["E"], s["L"], bm)
    assert np.array_equal(a["sorted_ids"], b["sorted_ids"])
    _check_invariants(a, topk, lora, s["E"], s["L"], bm)


def test_align_degenerate_cases():
    # all pairs on one expert, all base-only
    topk = np.zeros((10, 1), np.int32)
    lora = np.full(10, -1, np.int32)
    a = oracle.align(topk, lora, E=4, L=2, bm=4)
    assert a["sorted_ids"].tolist() == list(range(10)) + [10, 10]
    assert a["tile_expert"].tolist() == [0, 0, 0] and a["tile_lora"].tolist() == [-1, -1, -1]
    # a single pair
    a = oracle.align(np.array([[3]], np.int32), np.array([1], np.int32), E=4, L=2, bm=16)
    assert a["sorted_ids"].tolist() == [0] + [1] * 15
    assert a["tile_expert"].tolist() == [3] and a["tile_lora"].tolist() == [1]
    # no adapters at all (L = 0)
    a = oracle.align(np.array([[1, 0]], np.int32), np.array([-1], np.int32), E=2, L=0, bm=1)
    assert a["sorted_ids"].tolist() == [1, 0]
    # no tokens
    a = oracle.align(np.zeros((0, 2), np.int32), np.zeros(0, np.int32), E=2, L=1, bm=8)
    assert a["num_post_padded"] == 0 and a["bucket_count"].sum() == 0


def test_align_invalid_ids_left_out():
    topk = np.array([[0, 5], [1, -1], [1, 0]], np.int32)
    lora = np.array([0, 0, 7], np.int32)   # token 2's adapter is out of range
    a = oracle.align(topk, lora, E=2, L=1, bm=2)
    assert a["invalid"] == 4
    assert a["sorted_ids"].tolist() == [0, 6, 2, 6]
    b = brute.align_sorted(topk, lora, 2, 1, 2)
    assert np.array_equal(a["sorted_ids"], b["sorted_ids"]) and b["invalid"] == 4
