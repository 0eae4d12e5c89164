"""moe_lora_align on the GPU is bit-exact with the oracle's bucketing."""
import numpy as np
import pytest

import oracle
from lora_moe_layer_gb300 import workloads as wl

from gpu_helpers import gpu_align

pytestmark = pytest.mark.gpu

KEYS = ("sorted_ids", "tile_expert", "tile_lora", "bucket_count", "bucket_offset")


def _compare(topk, lora, E, L, bm):
    got, status = gpu_align(topk, lora, E, L, bm)
    ref = oracle.align(topk, lora, E, L, bm)
    assert got["num_post_padded"] == ref["num_post_padded"]
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), key
    # entries past num_post_padded are left untouched
    assert (got["tail"] == -12345).all()
    return status, ref


@pytest.mark.parametrize("bm", [1, 8, 16, 64, 128])
@pytest.mark.parametrize("seed", range(4))
def test_random_grid(bm, seed):
    rng = np.random.default_rng([seed, 123])
    T = int(rng.integers(1, 3000))
    k = int(rng.integers(1, 9))
    E = int(rng.integers(1, 160))
    L = int(rng.integers(0, 20))
    topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
    lora = rng.integers(-1, L, size=T).astype(np.int32) if L else np.full(T, -1, np.int32)
    status, _ = _compare(topk, lora, E, L, bm)
    assert status == 0


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
@pytest.mark.parametrize("bm", [8, 16, 64, 128])
def test_config_routing(cfg, bm):
    s = wl.config_shape(cfg)
    lora = wl.config_lora_ids(cfg, s["T"], s["L"])
    x = wl._normal_bf16(0, "x", (s["T"], s["H"]), 1.0)
    Wr = wl._normal_bf16(0, "Wr", (s["E"], s["H"]), 1.0 / np.sqrt(s["H"]))
    logits = wl.router_logits(x, Wr)
    if cfg == 3:
        logits[:, :16] += 1.09375
    topk, _ = wl.route_topk(logits, s["k"])
    status, _ = _compare(topk, lora, s["E"], s["L"], bm)
    assert status == 0


@pytest.mark.parametrize("T", [1, 16, 256])
def test_dense_routing(T):
    lora = wl.config_lora_ids(4, T, 32)
    status, _ = _compare(np.zeros((T, 1), np.int32), lora, 1, 32, 16)
    assert status == 0


def test_adversarial():
    # everything on one expert, all base-only
    s, _ = _compare(np.full((4096, 8), 3, np.int32), np.full(4096, -1, np.int32), 8, 4, 16)
    assert s == 0
    # a single pair
    s, _ = _compare(np.array([[2]], np.int32), np.array([0], np.int32), 4, 1, 128)
    assert s == 0
    # L = 0
    s, _ = _compare(np.array([[1, 0], [0, 1]], np.int32), np.array([-1, -1], np.int32), 2, 0, 8)
    assert s == 0
    # many buckets: histogram does not fit in shared memory (E * (L+1) * 16 ints > 160 KiB)
    rng = np.random.default_rng(5)
    topk = rng.integers(0, 256, size=(3000, 8)).astype(np.int32)
    lora = rng.integers(-1, 63, size=3000).astype(np.int32)
    s, _ = _compare(topk, lora, 256, 63, 16)
    assert s == 0


def test_out_of_range_ids_flagged_and_left_out():
    topk = np.array([[0, 5], [1, -1], [1, 0], [2, 2]], np.int32)
    lora = np.array([0, 0, 7, -1], np.int32)
    status, ref = _compare(topk, lora, 3, 1, 2)
    # t0 slot 1, t1 slot 1, and both slots of t2 (adapter 7 of 1)
    assert status == -5 and ref["invalid"] == 4


def test_status_resets_on_next_call():
    status, _ = _compare(np.array([[9]], np.int32), np.array([0], np.int32), 2, 1, 4)
    assert status == -5
    status, _ = _compare(np.array([[1]], np.int32), np.array([0], np.int32), 2, 1, 4)
    assert status == 0


def test_empty_batch():
    status, ref = _compare(np.zeros((0, 2), np.int32), np.zeros(0, np.int32), 4, 2, 16)
    assert status == 0 and ref["num_post_padded"] == 0
