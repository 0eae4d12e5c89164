"""moe_lora_forward_w8 (FP8 E4M3 base expert weights with per-row fp32 scales,
bf16 LoRA) on the GPU against the oracle's FP8 forward.

Bar: max|gpu - ref| / max|ref| <= 1e-2 over every output, where ref is the
fp64 layer on the exact weights scale * value(code).  The kernel rounds each
row's scale to bf16 precision (a per-row factor within 2^-9 of 1) and each
scaled weight to bf16 before its bf16 MMA: a relative error of at most about
2^-8 per weight, well inside the bar.  With power-of-two scales every scaled
weight is a bf16 value, so the FP8 forward must equal the bf16 forward on those
weights bit for bit (same kernel, same MMAs, same bf16 operands).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from lora_moe_layer_gb300 import binding as B
from lora_moe_layer_gb300 import workloads as wl
from lora_moe_layer_gb300.layer import DeviceLayer

from gpu_helpers import TOL, norm_err

pytestmark = pytest.mark.gpu


def run_w8(layer, options=0):
    dl = DeviceLayer(layer, "cuda", options=options)
    B.check(dl.forward_w8(), "moe_lora_forward_w8")
    return dl, dl.status()


def check_w8(layer):
    dl, st = run_w8(layer)
    assert st == 0
    ref, inv = oracle.forward_w8(layer)
    assert inv == 0
    err = norm_err(dl.out_f64(), ref)
    assert err <= TOL, err
    return dl, err


# H and I multiples of 16 (byte rows of the codes); ragged against the 240-row
# chains, narrow and wide chunks, many experts, r = 8 .. 64, no adapters
W8_SHAPES = [
    (37, 272, 144, 5, 3, 3, 24),
    (9, 512, 208, 7, 2, 2, 64),
    (64, 128, 80, 3, 2, 4, 8),
    (300, 256, 528, 2, 2, 0, 0),
    (600, 128, 144, 2, 2, 5, 32),
    (24, 272, 144, 40, 2, 3, 24),
    (2, 2048, 512, 2, 1, 1, 64),
    (160, 128, 96, 2, 2, 11, 16),
    (256, 512, 1024, 1, 1, 4, 16),
]


@pytest.mark.parametrize("shape", W8_SHAPES)
def test_w8_shapes(shape):
    check_w8(wl.quantize_e4m3(wl.make_random(*shape, seed=17)))


def test_w8_config0():
    check_w8(wl.quantize_e4m3(wl.make_config(0)))


def test_w8_decode_layer():
    # the GPT-OSS-20B-shaped decode layer (T=16, H=I=2880, E=32, top-4, r=32)
    check_w8(wl.quantize_e4m3(wl.make_config(1)))


@pytest.mark.slow
def test_w8_prefill_chunk_full():
    # every output of the GPT-OSS-20B-shaped prefill chunk (T=2048)
    check_w8(wl.quantize_e4m3(wl.make_config(2)))


def test_w8_power_of_two_scales_equal_the_bf16_forward_bitwise():
    layer = wl.make_random(600, 128, 144, 2, 2, 5, 32, seed=23)   # wide chunks: CTA pairs on both paths
    q = wl.quantize_e4m3(layer).w8
    rng = np.random.default_rng(23)
    W1s = (2.0 ** rng.integers(-10, -4, size=q.W1s.shape)).astype(np.float32)
    W2s = (2.0 ** rng.integers(-10, -4, size=q.W2s.shape)).astype(np.float32)
    vals1 = torch.from_numpy(q.W1q).view(torch.float8_e4m3fn).to(torch.float32).numpy() * W1s[..., None]
    vals2 = torch.from_numpy(q.W2q).view(torch.float8_e4m3fn).to(torch.float32).numpy() * W2s[..., None]
    bf = dataclasses.replace(layer, W1=wl.bf16_bits(vals1), W2=wl.bf16_bits(vals2))
    assert np.array_equal(wl.bf16_to_f32(bf.W1), vals1) and np.array_equal(wl.bf16_to_f32(bf.W2), vals2)
    l8 = dataclasses.replace(bf, w8=wl.W8Weights(q.W1q, W1s, q.W2q, W2s))
    a, st = run_w8(l8)
    assert st == 0
    b = DeviceLayer(bf, "cuda")
    B.check(b.forward())
    assert B.moe_lora_workspace_layout(b.d)["gemm_ctas"] == 2
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_w8_subnormal_codes():
    """Weights made only of subnormal E4M3 codes (exponent field 0): the
    conversion must keep them (value m / 8 * 2^-6 times the scale), not
    flush them to zero."""
    layer = wl.make_random(40, 128, 96, 3, 2, 2, 16, seed=29)
    q = wl.quantize_e4m3(layer).w8
    rng = np.random.default_rng(29)
    sub = lambda shape: (rng.integers(1, 8, size=shape) | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)
    W1q, W2q = sub(q.W1q.shape), sub(q.W2q.shape)
    W1s = np.full(q.W1s.shape, 64.0, np.float32)
    W2s = np.full(q.W2s.shape, 64.0, np.float32)
    l8 = dataclasses.replace(layer, w8=wl.W8Weights(W1q, W1s, W2q, W2s))
    dl, err = check_w8(l8)
    assert np.max(np.abs(dl.out_f64())) > 0


def test_w8_rejects_rows_that_are_not_16_byte_multiples():
    layer = wl.quantize_e4m3(wl.make_random(8, 264, 136, 3, 2, 2, 8, seed=2))
    dl = DeviceLayer(layer, "cuda")
    assert dl.forward_w8() == B.MOELORA_EUNSUPPORTED


def test_w8_out_of_range_ids_flagged():
    layer = wl.quantize_e4m3(wl.make_config(0))
    tk = layer.topk_ids.copy()
    tk[3, 1] = layer.E
    bad = dataclasses.replace(layer, topk_ids=tk)
    dl, st = run_w8(bad)
    assert st == B.MOELORA_EDEVICE_ID
    ref, inv = oracle.forward_w8(bad)
    assert inv == 1
    assert norm_err(dl.out_f64(), ref) <= TOL
