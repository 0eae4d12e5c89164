"""The seeded input recipe (workloads.py) against its stated rules, on the CPU.

Both sides of every parity test consume these inputs, so a mistake here would
not show up as a disagreement between the CUDA path and the oracle.  These
tests pin the recipe itself:
- bf16 rounding against values fixed by the format;
- the router's top-k order and weights against a brute-force full softmax;
- the per-workload adapter-id rules;
- the hot-expert skew;
- stream independence across shapes.
"""
import math

import numpy as np
import pytest

from lora_moe_layer_gb300 import workloads as wl


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 1.0 and the next value 1 + 2^-7: ties go to the even mantissa
    cases = [
        (1.0, 0x3F80),
        (-2.0, 0xC000),
        (1.0 + 2.0 ** -8, 0x3F80),                  # tie, even neighbour is 1.0
        (1.0 + 3 * 2.0 ** -8, 0x3F82),              # tie between 0x3F81 and 0x3F82: even wins
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),     # just above the tie: rounds up
        (3.140625, 0x4049),                         # exactly representable
        (0.0, 0x0000),
        (-0.0, 0x8000),                             # the sign of zero is kept
    ]
    vals = np.array([v for v, _ in cases], dtype=np.float32)
    got = wl.bf16_bits(vals)
    assert [int(v) for v in got] == [b for _, b in cases]
    # the round trip is exact on bf16 values and within half an ulp otherwise:
    # 8 significand bits give a relative error below the unit roundoff 2^-8
    back = wl.bf16_to_f32(got)
    assert back[0] == 1.0 and back[5] == np.float32(3.140625)
    rng = np.random.default_rng(5)
    x = rng.standard_normal(10000).astype(np.float32)
    err = np.abs(wl.bf16_to_f32(wl.bf16_bits(x)).astype(np.float64) - x) / np.abs(x)
    assert err.max() < 2.0 ** -8
    assert err.max() > 2.0 ** -9                  # and the bound is nearly reached on 10^4 draws


def test_route_topk_order_ties_and_weights():
    logits = np.array([[0.5, 2.0, 2.0, -1.0, 2.0],
                       [1.0, 1.0, 1.0, 1.0, 1.0],
                       [-3.0, 4.0, 0.0, 3.5, 1.0]])
    ids, w = wl.route_topk(logits, 3)
    # descending logit, equal logits in ascending expert order
    assert ids.tolist() == [[1, 2, 4], [0, 1, 2], [1, 3, 4]]
    # weights: the full softmax restricted to the chosen experts, renormalised
    for t in range(logits.shape[0]):
        full = np.exp(logits[t] - logits[t].max())
        full /= full.sum()
        sel = full[ids[t]] / full[ids[t]].sum()
        assert np.allclose(w[t], sel, rtol=1e-6, atol=0)
        assert abs(float(w[t].sum()) - 1.0) < 1e-6
        assert np.all(np.diff(w[t]) <= 0)          # non-increasing, like the logits


def test_adapter_ids_follow_each_workload_rule():
    ids0 = wl.config_lora_ids(0, 4096, 2)
    assert set(np.unique(ids0).tolist()) == {-1, 0, 1}
    ids1 = wl.config_lora_ids(1, 4096, 8)
    assert set(np.unique(ids1).tolist()) == set(range(8))
    # prefill: one id per 128-token sequence, drawn from {-1, 0..7}
    ids2 = wl.config_lora_ids(2, 2048, 8)
    seqs = ids2.reshape(16, 128)
    assert np.all(seqs == seqs[:, :1])
    assert set(np.unique(ids2).tolist()) <= set(range(-1, 8))
    ids4 = wl.config_lora_ids(4, 4096, 32)
    assert ids4.min() >= 0 and ids4.max() <= 31
    assert len(np.unique(ids4)) == 32


def test_mixed_workload_adapters_are_zipf_with_a_base_only_tenth():
    T, L = 200000, 16
    ids = wl.config_lora_ids(3, T, L)
    base = float((ids == -1).mean())
    assert abs(base - 0.1) < 0.005
    counts = np.bincount(ids[ids >= 0], minlength=L).astype(np.float64)
    expect = np.array([(i + 1) ** -1.1 for i in range(L)])
    expect /= expect.sum()
    freq = counts / counts.sum()
    # each adapter within 5% (relative) of its Zipf(1.1) share at this sample size
    assert np.all(np.abs(freq - expect) <= 0.05 * expect)
    assert np.all(np.diff(counts) < 0)             # strictly decreasing popularity


def test_hot_expert_skew_reaches_its_target_share():
    # the mixed workload's skew on a small layer: a bisection on the logit offset
    # of the first 4 experts brings their share of slots to about one half
    lay = wl.make_layer("skew", 512, 64, 32, 16, 4, 2, 8, np.zeros(512, dtype=np.int32),
                        seed=3, skew_hot=4, with_lora=False)
    share = lay.meta["hot_share"]
    assert 0.45 <= share <= 0.55
    assert lay.meta["skew_beta"] > 0
    assert abs(float((lay.topk_ids < 4).mean()) - share) < 1e-12
    # without the skew the same layer routes far fewer slots to those experts
    plain = wl.make_layer("plain", 512, 64, 32, 16, 4, 2, 8, np.zeros(512, dtype=np.int32), seed=3,
                          with_lora=False)
    assert float((plain.topk_ids < 4).mean()) < 0.4


def test_streams_are_per_tensor_and_shape_independent():
    # the dense workload keeps its weights when only T changes, and x's rows do not depend on T
    a = wl.make_layer("a", 4, 64, 32, 2, 1, 2, 8, np.zeros(4, dtype=np.int32), seed=7)
    b = wl.make_layer("b", 9, 64, 32, 2, 1, 2, 8, np.zeros(9, dtype=np.int32), seed=7)
    for name in ("W1", "W2", "A1", "B1", "A2", "B2"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    assert np.array_equal(a.x, b.x[:4])
    # one stream per expert: expert 0's W1 does not change with the expert count
    c = wl.make_layer("c", 4, 64, 32, 3, 1, 2, 8, np.zeros(4, dtype=np.int32), seed=7)
    assert np.array_equal(a.W1[0], c.W1[0]) and np.array_equal(a.W1[1], c.W1[1])
    # another seed gives other values
    d = wl.make_layer("d", 4, 64, 32, 2, 1, 2, 8, np.zeros(4, dtype=np.int32), seed=8)
    assert not np.array_equal(a.W1, d.W1)


@pytest.mark.parametrize("name, fan_in, std_expect", [("W1", 64, 1 / 8), ("W2", 32, 1 / math.sqrt(32)),
                                                     ("B1", None, 0.02)])
def test_weight_scales_follow_the_recipe(name, fan_in, std_expect):
    lay = wl.make_layer("s", 4, 64, 32, 8, 1, 4, 8, np.zeros(4, dtype=np.int32), seed=11)
    vals = wl.bf16_to_f32(getattr(lay, name)).astype(np.float64).ravel()
    assert abs(vals.mean()) < 0.05 * std_expect
    assert abs(vals.std() / std_expect - 1.0) < 0.03
