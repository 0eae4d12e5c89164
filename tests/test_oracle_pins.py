"""Pins of the fp64 oracle against things other than itself (CPU only).

The pages print no worked example and no intermediate value, so the pins are:
a hand-worked closed form, a second independent numpy implementation, the
associativity of the blog's y = xW + xAB (rank-r delta == dense update), the
textbook dense LoRA MLP for one expert (torch float64 routines), and
invariants (zero B, base-only tokens, weight linearity, adapter swap).
Source: "Efficiently serve dozens of fine-tuned models with vLLM on Amazon
SageMaker AI and Amazon Bedrock", section "Implementing multi-LoRA inference
for MoE models in vLLM" (the expert FFN, the LoRA shrink/expand and the router
aggregation) and Figure 1.
"""
import dataclasses
import math

import numpy as np
import pytest

import oracle
from oracle import brute
from lora_moe_layer_gb300 import workloads as wl


def _bits(a):
    return wl.bf16_bits(np.asarray(a, dtype=np.float32))


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def silu(u):
    return u / (1.0 + math.exp(-u))


def hand_layer(lora_id):
    """T=1, H=2, I=1, E=2, k=2, L=1, r=1: every number small and exact in bf16."""
    x = _bits([[1, 2]])
    W1 = _bits([[[1, 0], [0, 1]],            # expert 0: gate row, up row
                [[0, 1], [1, 1]]])           # expert 1
    W2 = _bits([[[1], [2]],                  # expert 0: [H=2][I=1]
                [[-1], [1]]])                # expert 1
    A1 = _bits([[[[1, 1]], [[1, -1]]]])      # [L=1][E=2][r=1][H=2]
    B1 = _bits([[[[0.5], [-1]], [[1], [2]]]])  # [L][E][2I=2][r=1]
    A2 = _bits([[[[2]], [[1]]]])             # [L][E][r=1][I=1]
    B2 = _bits([[[[1], [0.25]], [[0.5], [0.5]]]])  # [L][E][H=2][r=1]
    return wl.Layer("hand", 1, 2, 1, 2, 2, 1, 1, x, W1, W2, A1, B1, A2, B2,
                    np.array([[0, 1]], np.int32), np.array([[0.75, 0.25]], np.float32),
                    np.array([lora_id], np.int32))


def test_hand_example_with_adapter():
    # expert 0: gate = 1 + 0.5*3 = 2.5, up = 2 - 3 = -1  (z1 = x.[1,1] = 3)
    #   act0 = silu(2.5) * -1; d0 = [act0, 2 act0] + [1, 0.25] * (2 act0) = [3 act0, 2.5 act0]
    # expert 1: z1 = x.[1,-1] = -1; gate = 2 - 1 = 1, up = 3 - 2 = 1
    #   act1 = silu(1); d1 = [-act1, act1] + [0.5, 0.5] * act1 = [-0.5 act1, 1.5 act1]
    # out = 0.75 d0 + 0.25 d1
    act0 = -silu(2.5)
    act1 = silu(1.0)
    expect = np.array([0.75 * 3 * act0 + 0.25 * -0.5 * act1, 0.75 * 2.5 * act0 + 0.25 * 1.5 * act1])
    out, inv = oracle.forward(hand_layer(0))
    assert inv == 0
    np.testing.assert_allclose(out[0], expect, rtol=1e-15, atol=1e-15)
    p0 = oracle.pair(hand_layer(0), 0)
    np.testing.assert_allclose(p0["z1"], [3.0])
    np.testing.assert_allclose(p0["g"], [2.5, -1.0])
    np.testing.assert_allclose(p0["z2"], [2 * act0], rtol=1e-15)
    np.testing.assert_allclose(p0["d"], [3 * act0, 2.5 * act0], rtol=1e-15)


def test_hand_example_base_only():
    # l = -1: expert 0 gate 1 up 2 -> act0 = 2 silu(1); expert 1 gate 2 up 3 -> act1 = 3 silu(2)
    act0 = 2 * silu(1.0)
    act1 = 3 * silu(2.0)
    expect = np.array([0.75 * act0 - 0.25 * act1, 0.75 * 2 * act0 + 0.25 * act1])
    out, inv = oracle.forward(hand_layer(-1))
    assert inv == 0
    np.testing.assert_allclose(out[0], expect, rtol=1e-15, atol=1e-15)


SHAPES = [
    # T, H, I, E, k, L, r
    (5, 16, 8, 3, 2, 2, 4),
    (7, 24, 16, 4, 3, 3, 8),
    (4, 8, 24, 2, 1, 1, 2),
    (6, 32, 16, 5, 4, 0, 0),
    (3, 16, 16, 1, 1, 2, 8),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_oracle_matches_brute_force(shape):
    layer = wl.make_random(*shape, seed=3)
    out, inv = oracle.forward(layer)
    assert inv == 0
    ref = brute.forward(layer)
    assert _rel(out, ref) < 1e-12


def test_oracle_matches_brute_force_config0():
    layer = wl.make_config(0)
    out, _ = oracle.forward(layer)
    assert _rel(out, brute.forward(layer)) < 1e-12


@pytest.mark.parametrize("shape", SHAPES[:3] + SHAPES[4:])
def test_rank_r_delta_equals_dense_update(shape):
    layer = wl.make_random(*shape, seed=5)
    out, _ = oracle.forward(layer)
    assert _rel(out, brute.forward_merged(layer)) < 1e-12


def test_rank_r_delta_equals_dense_update_config0():
    layer = wl.make_config(0)
    out, _ = oracle.forward(layer)
    assert _rel(out, brute.forward_merged(layer)) < 1e-12


def test_zero_B_is_exactly_base():
    layer = wl.make_config(0)
    zb = dataclasses.replace(layer, B1=np.zeros_like(layer.B1), B2=np.zeros_like(layer.B2))
    base = dataclasses.replace(layer, lora_ids=np.full_like(layer.lora_ids, -1))
    a, _ = oracle.forward(zb)
    b, _ = oracle.forward(base)
    assert np.array_equal(a, b)
    # and the delta is not trivially zero with the real B
    c, _ = oracle.forward(layer)
    assert not np.array_equal(c, b)


def test_base_only_tokens_equal_base_model():
    layer = wl.make_config(0)
    out, _ = oracle.forward(layer)
    nolora = dataclasses.replace(layer, L=0, A1=None, B1=None, A2=None, B2=None,
                                 lora_ids=np.full_like(layer.lora_ids, -1))
    base, _ = oracle.forward(nolora)
    m = layer.lora_ids == -1
    assert m.any() and (~m).any()
    assert np.array_equal(out[m], base[m])
    assert not np.array_equal(out[~m], base[~m])


def test_adapter_swap_swaps_deltas():
    layer = wl.make_random(4, 16, 8, 3, 2, 2, 4, seed=9)
    x = layer.x.copy()
    x[1] = x[0]
    tk = layer.topk_ids.copy()
    tk[1] = tk[0]
    tw = layer.topk_weights.copy()
    tw[1] = tw[0]
    lo = layer.lora_ids.copy()
    lo[0], lo[1] = 0, 1
    a_layer = dataclasses.replace(layer, x=x, topk_ids=tk, topk_weights=tw, lora_ids=lo)
    lo2 = lo.copy()
    lo2[0], lo2[1] = 1, 0
    b_layer = dataclasses.replace(a_layer, lora_ids=lo2)
    a, _ = oracle.forward(a_layer)
    b, _ = oracle.forward(b_layer)
    assert np.array_equal(a[0], b[1]) and np.array_equal(a[1], b[0])
    assert not np.array_equal(a[0], a[1])


def test_weight_linearity_exact():
    layer = wl.make_config(0)
    out, _ = oracle.forward(layer)
    twice, _ = oracle.forward(dataclasses.replace(layer, topk_weights=layer.topk_weights * 2))
    assert np.array_equal(twice, 2 * out)


def test_single_expert_unit_weight_is_that_experts_ffn():
    layer = wl.make_config(0)
    one = dataclasses.replace(layer, k=1, topk_ids=layer.topk_ids[:, :1].copy(),
                              topk_weights=np.ones((layer.T, 1), np.float32))
    out, _ = oracle.forward(one)
    for t in range(layer.T):
        assert np.array_equal(out[t], oracle.pair(one, t)["d"])


def test_dense_single_expert_is_textbook_lora_mlp():
    """E = 1, k = 1, weight 1: the dense multi-LoRA MLP written with torch float64
    in the pages' orientation (W h_in x h_out, A h_in x r, B r x h_out)."""
    torch = pytest.importorskip("torch")
    T, H, I, L, r = 6, 32, 48, 3, 8
    lora = np.array([0, 1, 2, -1, 1, 0], np.int32)
    layer = wl.make_layer("dense", T, H, I, 1, 1, L, r, lora, seed=11)
    out, _ = oracle.forward(layer)

    def t64(bits):
        return torch.from_numpy(brute.f64(bits))

    x = t64(layer.x)
    W_gu = t64(layer.W1[0]).T            # H x 2I
    W_d = t64(layer.W2[0]).T             # I x H
    ref = torch.zeros(T, H, dtype=torch.float64)
    for t in range(T):
        xt = x[t:t + 1]
        y = xt @ W_gu
        l = int(lora[t])
        if l >= 0:
            y = y + (xt @ t64(layer.A1[l, 0]).T) @ t64(layer.B1[l, 0]).T
        act = torch.nn.functional.silu(y[:, :I]) * y[:, I:]
        o = act @ W_d
        if l >= 0:
            o = o + (act @ t64(layer.A2[l, 0]).T) @ t64(layer.B2[l, 0]).T
        ref[t] = o[0] * float(layer.topk_weights[t, 0])
    assert np.all(layer.topk_weights == 1.0)
    assert _rel(out, ref.numpy()) < 1e-12


def test_intermediates_match_brute_force():
    layer = wl.make_config(0)
    I = layer.I
    for p in range(layer.P):
        t = p // layer.k
        e = int(layer.topk_ids.flat[p])
        l = int(layer.lora_ids[t])
        res = oracle.pair(layer, p)
        xt = brute.f64(layer.x[t])
        g = brute.f64(layer.W1[e]) @ xt
        if l >= 0:
            z1 = brute.f64(layer.A1[l, e]) @ xt
            assert _rel(res["z1"], z1) < 1e-12
            g = g + brute.f64(layer.B1[l, e]) @ z1
        assert _rel(res["g"], g) < 1e-12
        act = brute.silu(g[:I]) * g[I:]
        assert _rel(res["act"], act) < 1e-12


def test_invalid_ids_contribute_nothing():
    layer = wl.make_config(0)
    bad = layer.topk_ids.copy()
    bad[2, 1] = layer.E          # expert out of range
    bad[5, 0] = -3
    lo = layer.lora_ids.copy()
    lo[7] = layer.L              # adapter out of range: all k pairs of token 7
    bl = dataclasses.replace(layer, topk_ids=bad, lora_ids=lo)
    out, inv = oracle.forward(bl)
    assert inv == 2 + layer.k
    assert np.array_equal(out[7], np.zeros(layer.H))
    ref = brute.forward(bl)
    assert _rel(out, ref) < 1e-12


def test_silu_matches_closed_forms():
    # one expert, H = I = 1, gate = up = u: act = silu(u) * u
    for u in [-20.0, -3.5, -1.0, 0.0, 0.5, 1.0, 7.25, 20.0]:
        x = _bits([[u]])
        W1 = _bits([[[1], [1]]])         # gate row and up row both pick x
        layer = wl.Layer("silu", 1, 1, 1, 1, 1, 0, 0, x, W1, _bits([[[1]]]), None, None, None, None,
                         np.array([[0]], np.int32), np.array([[1.0]], np.float32),
                         np.array([-1], np.int32))
        ub = float(brute.f64(x)[0, 0])
        res = oracle.pair(layer, 0)
        # act = silu(u) * u (up row is also 1 * x = u)
        assert res["act"][0] == pytest.approx(ub * ub / (1 + math.exp(-ub)), rel=1e-15, abs=1e-300)
    # symmetry of SiLU: silu(u) - silu(-u) = u
    for u in [0.25, 1.5, 3.0]:
        assert silu(u) - silu(-u) == pytest.approx(u, rel=1e-14)
