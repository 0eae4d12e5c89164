"""Pin strength: plant one plausible mistake at a time in a copy of the oracle's
C source, build it on the CPU, and check that the pins reject it.

Each mutant is a textual edit of ``oracle/oracle.c`` (the test first checks the
edited text is present, so a refactor of the oracle cannot silently turn a
mutant into a no-op).  A mutant passes the pins only if the pins are too weak.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import brute
from lora_moe_layer_gb300 import workloads as wl

from test_oracle_pins import hand_layer, silu, SHAPES

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "drop_up_factor": ("act[i] = silu(g[i]) * g[I + i];", "act[i] = silu(g[i]);"),
    "swap_gate_up": ("act[i] = silu(g[i]) * g[I + i];", "act[i] = silu(g[I + i]) * g[i];"),
    "silu_sign": ("return u / (1.0 + exp(-u));", "return u / (1.0 + exp(u));"),
    "transpose_B1": (
        "g[o] += dot_bf(B1 + (((long)l * E + e) * 2 * I + o) * r, z1, r);",
        "{ double s_ = 0; for (long q = 0; q < r; q++) "
        "s_ += bf(B1[((long)l * E + e) * 2 * I * r + q * 2 * I + o]) * z1[q]; g[o] += s_; }"),
    "transpose_W2": (
        "dv[h] = dot_bf(W2 + ((long)e * H + h) * I, act, I);",
        "{ double s_ = 0; for (long i = 0; i < I; i++) "
        "s_ += bf(W2[(long)e * H * I + i * H + h]) * act[i]; dv[h] = s_; }"),
    "drop_down_delta": ("dv[h] += dot_bf(B2 + (((long)l * E + e) * H + h) * r, z2, r);", "(void)0;"),
    "drop_gate_up_delta": ("g[o] += dot_bf(B1 + (((long)l * E + e) * 2 * I + o) * r, z1, r);", "(void)0;"),
    "ignore_topk_weight": ("acc[h] += w * dv[h];", "acc[h] += dv[h];"),
    "A1_wrong_expert": ("z1[q] = dot_bf(A1 + (((long)l * E + e) * r + q) * H, xd, H);",
                        "z1[q] = dot_bf(A1 + (((long)l * E + (e + 1) % E) * r + q) * H, xd, H);"),
    "adapter_of_other_token": ("const int l = lora_ids[t];", "const int l = lora_ids[(t + 1) % d->T];"),
    "A2_on_gate_up_output": ("z2[q] = dot_bf(A2 + (((long)l * E + e) * r + q) * I, act, I);",
                             "z2[q] = dot_bf(A2 + (((long)l * E + e) * r + q) * I, g, I);"),
}


def _build_mutant(tmp_path, name):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert before in text, f"mutant {name}: target text not found in oracle.c"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(text.replace(before, after))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    str(src), "-o", str(lib), "-lm"], check=True)
    return oracle.load_library(str(lib))


def _pins_pass(lib) -> bool:
    """Run the forward pins with the given oracle build; True iff all hold."""
    # hand-worked closed forms
    act0, act1 = -silu(2.5), silu(1.0)
    expect = np.array([0.75 * 3 * act0 - 0.125 * act1, 0.75 * 2.5 * act0 + 0.375 * act1])
    out, _ = oracle.forward(hand_layer(0), lib=lib, n_threads=1)
    if not np.allclose(out[0], expect, rtol=1e-14, atol=1e-14):
        return False
    b0, b1 = 2 * silu(1.0), 3 * silu(2.0)
    out, _ = oracle.forward(hand_layer(-1), lib=lib, n_threads=1)
    if not np.allclose(out[0], [0.75 * b0 - 0.25 * b1, 1.5 * b0 + 0.25 * b1], rtol=1e-14, atol=1e-14):
        return False
    # independent brute force and the dense-update identity
    for shape in SHAPES:
        layer = wl.make_random(*shape, seed=3)
        out, _ = oracle.forward(layer, lib=lib, n_threads=2)
        ref = brute.forward(layer)
        if np.max(np.abs(out - ref)) > 1e-12 * np.max(np.abs(ref)):
            return False
        if layer.L > 0:
            merged = brute.forward_merged(layer)
            if np.max(np.abs(out - merged)) > 1e-12 * np.max(np.abs(merged)):
                return False
    return True


def test_clean_oracle_passes_pins():
    assert _pins_pass(oracle._load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    assert not _pins_pass(lib), f"planted mistake {name} slipped through every pin"
