"""Pins of the oracle's FP8 (E4M3) base-weight forward, on the CPU.

The format is OCP 8-bit floating point E4M3 in its finite "fn" form: sign,
4-bit exponent with bias 7, 3-bit mantissa, subnormals at exponent 0, one NaN
pattern per sign and no infinities (largest value 448).  A weight is its
row's fp32 scale times the value of its code.  Pins:
  - every one of the 256 codes against torch's float8_e4m3fn conversion (a
    library decoder written independently of the oracle);
  - values the format definition fixes by hand (one, two, 448, the smallest
    normal and subnormal values, negative zero, NaN);
  - power-of-two scales make every dequantised weight a bf16 value, so the
    FP8 forward must equal the bf16 forward on those weights bit for bit;
  - a hand-worked one-token layer with mixed scales;
  - planted mistakes (wrong exponent bias, subnormals decoded as normals, a
    scale taken from the wrong row) that these pins must reject.
"""
import dataclasses
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from lora_moe_layer_gb300 import workloads as wl

torch = pytest.importorskip("torch")
SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def silu(u):
    return u / (1.0 + math.exp(-u))


def torch_e4m3(codes):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _decode_matches_torch(lib) -> bool:
    mine = np.array([float(lib.oracle_e4m3(c)) for c in range(256)])
    ref = torch_e4m3(np.arange(256))
    if not np.array_equal(np.isnan(mine), np.isnan(ref)):
        return False
    ok = ~np.isnan(ref)
    return np.array_equal(mine[ok], ref[ok]) and np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))


# code -> value, from the format definition
FIXED = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0xC0: -2.0, 0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6,
         0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x3C: 1.5, 0x30: 0.5, 0x77: 240.0}


def _fixed_values_hold(lib) -> bool:
    for code, v in FIXED.items():
        if float(lib.oracle_e4m3(code)) != v:
            return False
    neg_zero = float(lib.oracle_e4m3(0x80))
    return neg_zero == 0.0 and math.copysign(1.0, neg_zero) < 0 and math.isnan(lib.oracle_e4m3(0x7F)) \
        and math.isnan(lib.oracle_e4m3(0xFF))


def _pow2_layer(seed=5):
    """Random layer quantised to E4M3 with power-of-two row scales, and the
    same layer with bf16 weights equal to the dequantised values."""
    layer = wl.make_random(13, 64, 48, 3, 2, 2, 8, seed=seed)
    q = wl.quantize_e4m3(layer).w8
    rng = np.random.default_rng(seed)
    W1s = (2.0 ** rng.integers(-9, -3, size=q.W1s.shape)).astype(np.float32)
    W2s = (2.0 ** rng.integers(-9, -3, size=q.W2s.shape)).astype(np.float32)
    w8 = wl.W8Weights(q.W1q, W1s, q.W2q, W2s)
    dq1 = torch_e4m3(q.W1q) * W1s[..., None]
    dq2 = torch_e4m3(q.W2q) * W2s[..., None]
    bits1, bits2 = wl.bf16_bits(dq1.astype(np.float32)), wl.bf16_bits(dq2.astype(np.float32))
    assert np.array_equal(wl.bf16_to_f32(bits1).astype(np.float64), dq1)  # exactly representable
    assert np.array_equal(wl.bf16_to_f32(bits2).astype(np.float64), dq2)
    return dataclasses.replace(layer, w8=w8), dataclasses.replace(layer, W1=bits1, W2=bits2)


def _pow2_identity_holds(lib) -> bool:
    l8, lbf = _pow2_layer()
    a, _ = oracle.forward_w8(l8, lib=lib, n_threads=2)
    b, _ = oracle.forward(lbf, lib=lib, n_threads=2)
    return np.array_equal(a, b)


def hand_w8_layer():
    """T=1, H=2, I=1, E=1, top-1, no adapters; x = (1.5, 0.25).
    W1 rows: gate codes (1.0, -2.0) scale 0.5, up codes (2.0, 0.5) scale 3;
    W2 rows: (1.5) scale 2, (-1.0) scale 0.25."""
    b = wl.bf16_bits
    x = b(np.array([[1.5, 0.25]], np.float32))
    W1q = np.array([[[0x38, 0xC0], [0x40, 0x30]]], np.uint8)
    W1s = np.array([[0.5, 3.0]], np.float32)
    W2q = np.array([[[0x3C], [0xB8]]], np.uint8)
    W2s = np.array([[2.0, 0.25]], np.float32)
    zeros1 = np.zeros((1, 2, 2), np.uint16)
    zeros2 = np.zeros((1, 2, 1), np.uint16)
    return wl.Layer("hand_w8", 1, 2, 1, 1, 1, 0, 0, x, zeros1, zeros2, None, None, None, None,
                    np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), np.full(1, -1, np.int32),
                    w8=wl.W8Weights(W1q, W1s, W2q, W2s))


def _hand_layer_holds(lib) -> bool:
    gate = 0.5 * (1.0 * 1.5 + (-2.0) * 0.25)      # 0.5
    up = 3.0 * (2.0 * 1.5 + 0.5 * 0.25)           # 9.375
    act = silu(gate) * up
    expect = np.array([2.0 * 1.5 * act, 0.25 * (-1.0) * act])
    out, _ = oracle.forward_w8(hand_w8_layer(), lib=lib, n_threads=1)
    return np.allclose(out[0], expect, rtol=1e-15, atol=0)


def _w8_pins_pass(lib) -> bool:
    return _decode_matches_torch(lib) and _fixed_values_hold(lib) and _pow2_identity_holds(lib) \
        and _hand_layer_holds(lib)


def test_decoder_matches_torch_on_all_codes():
    assert _decode_matches_torch(oracle._load())


def test_decoder_fixed_values():
    assert _fixed_values_hold(oracle._load())


def test_power_of_two_scales_equal_the_bf16_forward_exactly():
    assert _pow2_identity_holds(oracle._load())


def test_hand_worked_fp8_layer():
    assert _hand_layer_holds(oracle._load())


def test_fp8_forward_close_to_bf16_forward_of_the_source_weights():
    # the quantisation error of E4M3 (3 mantissa bits) is a few per cent of the
    # output; a broken decoder or scale axis would be far off
    layer = wl.quantize_e4m3(wl.make_config(0))
    a, _ = oracle.forward_w8(layer)
    b, _ = oracle.forward(layer)
    err = np.max(np.abs(a - b)) / np.max(np.abs(b))
    assert 1e-3 < err < 0.1, err


W8_MUTANTS = {
    "exponent_bias_8": ("v = ldexp(1.0 + (double)m / 8.0, f - 7);", "v = ldexp(1.0 + (double)m / 8.0, f - 8);"),
    "subnormal_as_normal": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp(1.0 + (double)m / 8.0, -7);"),
    "W1_scale_of_other_row": ("q->W1s[(long)e * 2 * I + o]", "q->W1s[(long)e * 2 * I + (o + 1) % (2 * I)]"),
    "W2_scale_of_other_expert": ("q->W2s[(long)e * H + h]", "q->W2s[(long)((e + 1) % E) * H + h]"),
}


@pytest.mark.parametrize("name", sorted(W8_MUTANTS))
def test_planted_fp8_mistake_is_caught(tmp_path, name):
    before, after = W8_MUTANTS[name]
    text = open(SRC).read()
    assert before in text, f"mutant {name}: target text not found in oracle.c"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(text.replace(before, after))
    lib_path = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    str(src), "-o", str(lib_path), "-lm"], check=True)
    lib = oracle.load_library(str(lib_path))
    assert not _w8_pins_pass(lib), f"planted mistake {name} slipped through every FP8 pin"


def test_clean_oracle_passes_fp8_pins():
    assert _w8_pins_pass(oracle._load())
