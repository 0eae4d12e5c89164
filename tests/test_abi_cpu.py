"""The C-ABI library builds, loads and exports every declared symbol; its
host-only entry points answer without a GPU (CPU only, no compute calls)."""
import ctypes
import os
import re

import pytest

from lora_moe_layer_gb300 import binding as B
from lora_moe_layer_gb300 import build as build_mod

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe_lora.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOELORA_API\s+[\w\s\*]+?\b(moe_lora_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(B.library_path())
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_strerror_and_version(lib):
    for code in (0, -1, -2, -3, -4, -5, 99):
        assert isinstance(B.moe_lora_strerror(code), str) and B.moe_lora_strerror(code)
    assert B.moe_lora_version() >= 100


def test_align_capacity_formula(lib):
    for (T, k, E, L, bm) in [(16, 4, 32, 8, 16), (2048, 4, 32, 8, 128), (1, 1, 1, 0, 1), (256, 8, 128, 16, 8)]:
        d = B.dims(T, 64, 64, E, k, L, 8, bm)
        P, NB = T * k, E * (L + 1)
        assert B.moe_lora_align_capacity(d) == P + min(NB, P) * (bm - 1)


def test_workspace_bytes_and_layout(lib):
    d = B.dims(16, 2880, 2880, 32, 4, 8, 32)
    n = B.moe_lora_workspace_bytes(d)
    lay = B.moe_lora_workspace_layout(d)
    assert n == lay["total"] > 0
    P = 64
    # the shrinks split K across CTAs (a decode batch has too few adapter
    # buckets to fill the SMs), keeping at least two 64-wide K steps per split
    for s in (lay["s1"], lay["s2"]):
        assert 1 < s <= min(32, (2880 // 64) // 2)
    # regions are disjoint and inside the workspace
    assert lay["down_splits"] == 1 and lay["pair_out_bf16"] == 1
    assert lay["launches"] == 5  # align, gather, gate_up, down, reduce
    regions = sorted([(lay["compact_ids"], 4 * P), (lay["z1"], 4 * P * 32),
                      (lay["act"], 2 * P * 2880), (lay["z2"], 4 * P * 32),
                      (lay["pair_out"], pair_bytes(lay, P, 2880))])
    for (a, na), (b, _) in zip(regions, regions[1:]):
        assert a + na <= b
    assert regions[-1][0] + regions[-1][1] <= n
    assert all(off % 256 == 0 for off, _ in regions)


def pair_bytes(lay, P, H):
    """pair_out's size: bf16 [P][H] without a down K-split, else fp32 [splits][P][H]."""
    assert lay["pair_out_bf16"] == (1 if lay["down_splits"] == 1 else 0)
    return 2 * P * H if lay["pair_out_bf16"] else 4 * P * H * lay["down_splits"]


def test_layout_of_split_and_expand_workloads(lib):
    # one expert with few weight tiles: the down GEMM splits K, one fp32
    # pair_out slab per split
    d = B.dims(256, 8192, 28672, 1, 1, 32, 64)
    lay = B.moe_lora_workspace_layout(d)
    assert 1 < lay["down_splits"] <= 8 and lay["pair_out_bf16"] == 0
    assert lay["pair_out"] + pair_bytes(lay, 256, 8192) <= lay["total"]


def test_split_plan_follows_the_sm_count(lib):
    """K-split and shrink-split choices are planned for dims.sm_count SMs (0:
    the current device's count; 152, a GB300, with no device visible): fewer
    SMs need fewer splits to fill their waves, more need more.  Each count's
    workspace holds its own plan's regions."""
    def lay(sms, *shape):
        d = B.dims(*shape, sm_count=sms)
        out = B.moe_lora_workspace_layout(d)
        assert out["total"] == B.moe_lora_workspace_bytes(d)
        return out

    decode = (16, 2880, 2880, 32, 4, 8, 32)
    dense = (256, 8192, 28672, 1, 1, 32, 64, 0, B.MOELORA_OPT_SINGLE_CTA)  # one-CTA GEMM plan
    s = {n: lay(n, *decode) for n in (1, 38, 76, 152, 304)}
    assert s[1]["s1"] == s[1]["s2"] == 1
    assert s[1]["s1"] <= s[38]["s1"] <= s[76]["s1"] <= s[152]["s1"] <= s[304]["s1"]
    assert s[76]["s1"] < s[152]["s1"] < s[304]["s1"]
    dn = {n: lay(n, *dense)["down_splits"] for n in (1, 38, 152)}
    assert dn[1] == 1 and 1 < dn[38] < dn[152] <= 8
    for n in (1, 38, 76, 152, 304):
        L = lay(n, *dense)
        assert L["pair_out"] + pair_bytes(L, 256, 8192) <= L["total"]
        L = lay(n, *decode)
        assert L["pair_out"] + pair_bytes(L, 64, 2880) <= L["total"]
    assert B.moe_lora_workspace_bytes(B.dims(*decode, sm_count=-1)) == 0
    assert B.moe_lora_workspace_bytes(B.dims(*decode, sm_count=5000)) == 0


@pytest.mark.parametrize("bad", [
    dict(H=0), dict(E=0), dict(k=0), dict(T=-1), dict(L=-1), dict(block_m=3), dict(block_m=512),
])
def test_invalid_dims(lib, bad):
    base = dict(T=4, H=64, I=64, E=4, k=2, L=2, r=8, block_m=0)
    base.update(bad)
    d = B.moe_lora_dims(*[base[n] for n in ("T", "H", "I", "E", "k", "L", "r", "block_m")])
    assert B.moe_lora_workspace_bytes(d) == 0
    assert B.moe_lora_align_capacity(d) == B.MOELORA_EINVAL


@pytest.mark.parametrize("bad", [dict(H=60), dict(I=12), dict(r=12), dict(r=72)])
def test_unsupported_dims(lib, bad):
    base = dict(T=4, H=64, I=64, E=4, k=2, L=2, r=8, block_m=0)
    base.update(bad)
    d = B.moe_lora_dims(*[base[n] for n in ("T", "H", "I", "E", "k", "L", "r", "block_m")])
    assert B.moe_lora_align_capacity(d) == B.MOELORA_EUNSUPPORTED


def test_host_checks_return_before_any_launch(lib):
    """Null pointers, a short workspace and misalignment are refused on the host
    (fake addresses below are never dereferenced)."""
    d = B.dims(4, 64, 64, 4, 2, 2, 8)
    need = B.moe_lora_workspace_bytes(d)
    f = 1 << 20  # an aligned fake address
    args = [f] * 12
    # x .. B2, out, workspace
    def fwd(ptrs, wb):
        return B.load().moe_lora_forward(ctypes.byref(d), *ptrs, wb, None)
    assert fwd([f] * 5 + [None] + [f] * 6, need) == B.MOELORA_EINVAL          # W1 null
    assert fwd([f] * 7 + [None] + [f] * 4, need) == B.MOELORA_EINVAL          # A1 null with L > 0
    assert fwd(args, need - 1) == B.MOELORA_ENOSPC
    assert fwd([f + 8] + [f] * 11, need) == B.MOELORA_EUNSUPPORTED            # misaligned x
    assert B.load().moe_lora_align(ctypes.byref(d), f, f, None, f, f, f, f, f, f, need, None) == B.MOELORA_EINVAL
    assert B.load().moe_lora_align(ctypes.byref(d), f, f, f, f, f, f, f, f, f, need - 1, None) == B.MOELORA_ENOSPC
    assert B.load().moe_lora_get_status(None, None) == B.MOELORA_EINVAL


def test_no_device_is_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = B.dims(4, 64, 64, 4, 2, 0, 0)
    f = 1 << 20
    st = B.load().moe_lora_forward(ctypes.byref(d), f, f, f, f, f, f, None, None, None, None, f, f,
                                   B.moe_lora_workspace_bytes(d), None)
    assert st == B.MOELORA_ECUDA


def test_gemm_plan_cta_pairs_for_wide_chunks(lib):
    """Wide chunks (more than 48 pairs per expert) run on CTA pairs by default,
    with chains of at most 256 weight rows (a multiple of 16, as few chains as
    possible); MOELORA_OPT_SINGLE_CTA, decode-sized chunks and more adapters
    than a chunk mask holds keep one CTA per task; unknown option bits are
    rejected."""
    wide = B.dims(2048, 2880, 2880, 32, 4, 8, 32)
    lay = B.moe_lora_workspace_layout(wide)
    assert lay["gemm_ctas"] == 2 and lay["tc_expand"] == 1
    single = B.dims(2048, 2880, 2880, 32, 4, 8, 32, 0, B.MOELORA_OPT_SINGLE_CTA)
    assert B.moe_lora_workspace_layout(single)["gemm_ctas"] == 1
    assert B.moe_lora_workspace_layout(B.dims(16, 2880, 2880, 32, 4, 8, 32))["gemm_ctas"] == 1
    # the dense T=256 MLP: one 256-pair chunk; the down GEMM splits K into slabs
    dense = B.moe_lora_workspace_layout(B.dims(256, 8192, 28672, 1, 1, 32, 64))
    assert dense["gemm_ctas"] == 2 and dense["down_splits"] > 1
    # a layer without adapters, and one with few adapters (the pair kernel
    # takes the tensor-core expand whatever the adapter mix)
    assert B.moe_lora_workspace_layout(B.dims(2048, 2880, 2880, 32, 4, 0, 0))["gemm_ctas"] == 2
    few = B.moe_lora_workspace_layout(B.dims(600, 128, 136, 2, 2, 1, 8))
    assert few["gemm_ctas"] == 2 and few["tc_expand"] == 1
    # more adapters than a chunk mask holds: the pair kernel does not cover it
    many = B.dims(2048, 2880, 2880, 32, 4, 80, 32)
    assert B.moe_lora_workspace_layout(many)["gemm_ctas"] == 1
    with pytest.raises(B.MoeLoraError):
        B.moe_lora_workspace_layout(B.dims(16, 64, 64, 2, 1, 0, 0, 0, 2))


def test_noalloc_refuses_oversized_problems_on_the_host(lib):
    """moe_lora_forward_noalloc checks the problem against its built-in scratch
    size before touching the GPU: a workspace one token over the limit is
    refused with ENOSPC, also on a host without a device."""
    shape = (520, 200, 5, 3, 3, 24)
    lim = B.MOELORA_NOALLOC_SCRATCH_BYTES
    T = 1
    while B.moe_lora_workspace_bytes(B.dims(T * 2, *shape)) <= lim:
        T *= 2
    while B.moe_lora_workspace_bytes(B.dims(T + 1, *shape)) <= lim:
        T += 1
    f = 1 << 20  # never dereferenced; stream 0 (no torch stream on a host without a device)
    st = B.moe_lora_forward_noalloc(B.dims(T + 1, *shape), f, f, f, f, f, f, f, f, f, f, f, stream=0)
    assert st == B.MOELORA_ENOSPC


def test_pair_shapes_reach_both_chunk_modes():
    """The CTA-pair parity shapes put experts in both chunk modes, with tails
    of every kind: a single pair, only the first CTA's tail rows, both CTAs'
    partly and fully, and a tail-less chunk after a full one."""
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    from gpu_helpers import pair_chunk_modes
    from lora_moe_layer_gb300 import workloads as wl
    from test_forward_gpu import PAIR_SHAPES
    modes = {0: set(), 1: set()}
    for gate_up in (True, False):
        for shape in PAIR_SHAPES:
            for m, md in pair_chunk_modes(wl.make_random(*shape, seed=7), gate_up):
                modes[md].add(m)
    tails = {m % 384 - 256 for m in modes[1] if m % 384 > 256} | {128 for m in modes[1] if m >= 384}
    assert modes[0] and modes[1]
    assert 1 in tails and any(t <= 64 for t in tails) and any(64 < t < 128 for t in tails) and 128 in tails
    assert any(m > 384 and m % 384 <= 256 for m in modes[1])   # a chunk without a tail after a full one
    # the prefill layer's experts with 257 - 285 pairs take mode 1, the others mode 0
    for m, md in pair_chunk_modes(wl.make_config(2)):
        assert md == (1 if m > 256 else 0)
