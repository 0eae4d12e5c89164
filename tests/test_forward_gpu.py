"""moe_lora_forward on the GPU against the fp64 oracle.

Bar: max|gpu - ref| / max|ref| <= 1e-2 on the layer output (bf16 I/O, fp32
accumulation), per-kernel intermediates against the oracle's, and the exact
invariants that hold for the GPU arithmetic too (zero B, weight scaling by 2,
determinism, block_m independence, adapter swap).
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


def run(layer, block_m=0, options=0):
    dl = DeviceLayer(layer, "cuda", block_m=block_m, options=options)
    B.check(dl.forward(), "moe_lora_forward")
    st = dl.status()
    return dl, st


def check_layer(layer, tokens=None, block_m=0, tol=TOL, options=0):
    dl, st = run(layer, block_m, options)
    assert st == 0
    got = dl.out_f64()
    ref, inv = oracle.forward(layer, tokens=tokens)
    assert inv == 0
    sel = got if tokens is None else got[np.asarray(tokens)]
    err = norm_err(sel, ref)
    assert err <= tol, err
    return dl, err


# ------------------------------------------------------------------ small cases

RAGGED = [
    # T, H, I, E, k, L, r   -- H, I not multiples of the 256-element step; units not multiples of a CTA block
    (37, 264, 136, 5, 3, 3, 24),
    (9, 520, 200, 7, 2, 2, 64),
    (64, 128, 72, 3, 2, 4, 8),
    (5, 96, 1032, 4, 4, 1, 16),
    (40, 256, 512, 9, 1, 0, 0),
    (1, 64, 64, 2, 1, 1, 8),
    (130, 200, 48, 1, 1, 3, 32),
    # many experts, few pairs each: the LoRA shrink runs inside the GEMMs
    (24, 264, 136, 40, 2, 3, 24),
    (30, 520, 200, 24, 3, 2, 64),
    (16, 128, 96, 64, 4, 5, 8),
    # one expert, few weight tiles: the GEMMs split K across CTAs
    (3, 1024, 2048, 1, 1, 4, 16),
    (5, 1032, 1544, 1, 1, 2, 8),
    (2, 2048, 512, 2, 1, 1, 64),
    # more than 64 adapters: the tensor-core expand runs without per-expert adapter masks
    (40, 128, 96, 3, 2, 70, 8),
    # pairs x adapter slots beyond the zexp bound: the expand falls back to CUDA cores
    (2100, 64, 64, 4, 1, 64, 64),
    # r = 8 and r = 16: eight and four adapters packed per expand K block
    (160, 128, 96, 2, 2, 11, 8),
    (160, 128, 96, 2, 2, 7, 16),
    # wide chunks mixing several adapters (prefill-like): 64-row pair boxes, the
    # LoRA expand as tensor-core K blocks (r not a power of two; r = 64 with ragged I)
    (600, 128, 136, 2, 2, 5, 32),
    (200, 264, 136, 3, 2, 6, 24),
    (300, 96, 1032, 2, 1, 8, 64),
    # one expert, K split across CTAs, packed expand blocks (four adapters of
    # r = 16 per block) dealt to the splits
    (64, 1024, 2048, 1, 1, 12, 16),
    # many (expert, adapter) buckets: the forward's align keeps its histogram
    # and work lists in the workspace instead of shared memory
    (300, 64, 64, 256, 4, 63, 8),
    # wide chunks on CTA pairs: no adapters, two chunks per expert
    (300, 256, 520, 2, 2, 0, 0),
    # CTA pairs with the down GEMM's K split into slabs, both shrinks split, and
    # shrink items whose buckets all sit in the first CTA of the pair
    (256, 512, 1024, 1, 1, 4, 16),
]


@pytest.mark.parametrize("shape", RAGGED)
def test_ragged_shapes(shape):
    layer = wl.make_random(*shape, seed=7)
    check_layer(layer)


# wide chunks on CTA pairs (the default for more than 48 pairs per expert):
# ragged intermediate and hidden sizes (chains of 16-multiples beyond I or H),
# r_pad 16 / 32 / 64 with one, two or four adapters per expand block, shrink
# items in one or both CTAs of a pair and split over K, the down GEMM split
# over K into slabs, chunks with a tail of a few pairs, a layer without
# adapters, and one with a single adapter (the tensor-core expand on a
# one-adapter mix); experts in chunks of 256 + 128 pairs (mode 1) with tails
# of 1, 19, 44, 94 and 128 pairs (only the first CTA's tail rows valid, both
# partly, both full), a mode-1 chunk without a tail after a full one, both
# modes in one layer and one GEMM in each mode
PAIR_SHAPES = [
    (300, 256, 520, 2, 2, 0, 0),
    (256, 512, 1024, 1, 1, 4, 16),
    (600, 128, 136, 2, 2, 5, 32),
    (200, 264, 136, 3, 2, 6, 24),
    (300, 96, 1032, 2, 1, 8, 64),
    (160, 128, 96, 2, 2, 11, 8),
    (130, 200, 48, 1, 1, 3, 32),
    (600, 128, 136, 2, 2, 1, 8),
    (520, 264, 200, 2, 1, 9, 16),
    (100, 2048, 512, 1, 1, 7, 24),
    (257, 128, 96, 1, 1, 3, 16),
    (384, 256, 160, 1, 1, 2, 32),
    (350, 192, 272, 1, 1, 4, 8),
    (385, 128, 128, 1, 1, 0, 0),
    (700, 136, 200, 1, 1, 5, 64),
]


@pytest.mark.parametrize("shape", PAIR_SHAPES)
def test_cta_pair_kernel(shape):
    layer = wl.make_random(*shape, seed=7)
    dl, err = check_layer(layer)
    assert B.moe_lora_workspace_layout(dl.d)["gemm_ctas"] == 2
    # the one-CTA kernels on the same layer agree within rounding
    one, _ = check_layer(layer, options=B.MOELORA_OPT_SINGLE_CTA)
    assert B.moe_lora_workspace_layout(one.d)["gemm_ctas"] == 1
    assert norm_err(dl.out_f64(), one.out_f64()) <= TOL


@pytest.mark.slow
def test_single_cta_option_prefill():
    # every output of the prefill chunk on the one-CTA kernels (128- and
    # 256-pair chunks, K-split slabs, expand blocks)
    check_layer(wl.make_config(2), options=B.MOELORA_OPT_SINGLE_CTA)


def test_config0():
    check_layer(wl.make_config(0))


@pytest.mark.parametrize("bm", [1, 8, 64, 128])
def test_block_m_does_not_change_the_result(bm):
    layer = wl.make_config(0)
    a, _ = run(layer, 16)
    b, _ = run(layer, bm)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_intermediates_config0():
    layer = wl.make_config(0)
    dl, st = run(layer)
    assert st == 0
    lay = B.moe_lora_workspace_layout(dl.d)
    P, r, I, H = layer.P, layer.r, layer.I, layer.H
    rows = dl.workspace_view("compact_ids", torch.int32, (P,)).cpu().numpy()
    z1 = dl.workspace_view("z1", torch.float32, (P, r)).cpu().numpy().astype(np.float64)
    act_bits = dl.workspace_view("act", torch.int16, (P, I)).cpu().numpy().view(np.uint16)
    act = (act_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    pair_out = dl.pair_outputs()
    for row, p in enumerate(rows):
        ref = oracle.pair(layer, int(p))
        t = p // layer.k
        if layer.lora_ids[t] >= 0:
            assert norm_err(z1[row], ref["z1"]) < 1e-5
        assert norm_err(act[row], ref["act"]) < 8e-3
        w = float(layer.topk_weights.flat[p])
        assert norm_err(pair_out[p], w * ref["d"]) < 1e-2


@pytest.mark.parametrize("which", ["config0", "config3", "config2"])
def test_forward_groups_pairs_by_bucket(which):
    """The forward's own bucketing (compact order in the workspace): bucket b's
    rows hold exactly the pairs with key e*(L+1)+(l+1), in any order (the
    standalone align's ascending order is checked bit-exact elsewhere).  The
    prefill layer (8192 pairs, 288 buckets) takes the multi-CTA align, the
    others the single-CTA one."""
    layer = wl.make_config({"config0": 0, "config3": 3, "config2": 2}[which])
    dl, st = run(layer)
    assert st == 0
    P, L1 = layer.P, layer.L + 1
    nb = layer.E * L1
    rows = dl.workspace_view("compact_ids", torch.int32, (P,)).cpu().numpy()
    off = dl.workspace_view("compact_offset", torch.int32, (nb + 1,)).cpu().numpy()
    key = layer.topk_ids.reshape(-1).astype(np.int64) * L1 + np.repeat(layer.lora_ids, layer.k) + 1
    assert off[0] == 0 and off[-1] == P
    expect = np.bincount(key, minlength=nb)
    assert np.array_equal(np.diff(off), expect)
    for b in np.nonzero(expect)[0]:
        got = np.sort(rows[off[b]:off[b + 1]])
        assert np.array_equal(got, np.nonzero(key == b)[0])


# ------------------------------------------------------------------ invariants

def test_zero_B_bit_identical_to_base_only():
    layer = wl.make_config(0)
    zb = dataclasses.replace(layer, B1=np.zeros_like(layer.B1), B2=np.zeros_like(layer.B2))
    base = dataclasses.replace(layer, lora_ids=np.full_like(layer.lora_ids, -1))
    a, _ = run(zb)
    b, _ = run(base)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_base_only_tokens_match_a_layer_without_adapters():
    layer = wl.make_config(0)
    a, _ = run(layer)
    nolora = dataclasses.replace(layer, L=0, r=0, A1=None, B1=None, A2=None, B2=None,
                                 lora_ids=np.full_like(layer.lora_ids, -1))
    b, _ = run(nolora)
    m = torch.from_numpy(layer.lora_ids == -1).cuda()
    assert torch.equal(a.out[m].view(torch.int16), b.out[m].view(torch.int16))


def test_weights_times_two_doubles_output_exactly():
    layer = wl.make_config(0)
    a, _ = run(layer)
    b, _ = run(dataclasses.replace(layer, topk_weights=layer.topk_weights * 2))
    assert torch.equal(b.out.float(), 2 * a.out.float())


def test_deterministic():
    layer = wl.make_config(0)
    dl, _ = run(layer)
    first = dl.out.clone()
    for _ in range(3):
        B.check(dl.forward())
        assert torch.equal(first.view(torch.int16), dl.out.view(torch.int16))


def test_adapter_swap_swaps_outputs():
    layer = wl.make_random(6, 64, 32, 3, 2, 2, 8, seed=21)
    x, tk, tw, lo = layer.x.copy(), layer.topk_ids.copy(), layer.topk_weights.copy(), layer.lora_ids.copy()
    x[1], tk[1], tw[1] = x[0], tk[0], tw[0]
    lo[0], lo[1] = 0, 1
    a, _ = run(dataclasses.replace(layer, x=x, topk_ids=tk, topk_weights=tw, lora_ids=lo))
    lo2 = lo.copy()
    lo2[0], lo2[1] = 1, 0
    b, _ = run(dataclasses.replace(layer, x=x, topk_ids=tk, topk_weights=tw, lora_ids=lo2))
    assert torch.equal(a.out[0].view(torch.int16), b.out[1].view(torch.int16))
    assert torch.equal(a.out[1].view(torch.int16), b.out[0].view(torch.int16))


@pytest.mark.parametrize("which", ["config0", "many_experts", "mixed_chunks"])
def test_lora_delta_matches_oracle_delta(which):
    """The adapter delta alone (forward minus the zero-B forward) against the
    oracle's delta: a broken expand could hide under the 1e-2 output bar.  The
    first two layers take the CUDA-core expand, the third (several adapters
    per expert chunk) the tensor-core one.

    Each GPU output carries bf16 roundings (every per-pair output and the
    final sum, each within 2^-9 of its value), so the difference of two
    outputs is off by a few 2^-9 of the outputs' magnitude: the bar is 2^-6 of
    max |out|.  The delta is 10-20% of max |out| here, so the bar stays under
    half of it and a broken expand (an error of the delta's own size) fails."""
    if which == "config0":
        layer = wl.make_config(0)
    elif which == "many_experts":
        layer = wl.make_random(24, 264, 136, 40, 2, 3, 24, seed=8)
    else:
        layer = wl.make_random(300, 128, 136, 2, 2, 6, 32, seed=9)
    zb = dataclasses.replace(layer, B1=np.zeros_like(layer.B1), B2=np.zeros_like(layer.B2))
    a, _ = run(layer)
    b, _ = run(zb)
    d_gpu = a.out_f64() - b.out_f64()
    r1, _ = oracle.forward(layer)
    r0, _ = oracle.forward(zb)
    d_ref = r1 - r0
    bar = 2.0 ** -6 * np.max(np.abs(r1))
    assert bar < 0.5 * np.max(np.abs(d_ref))
    assert np.max(np.abs(d_gpu - d_ref)) <= bar


# ------------------------------------------------------------------ edge cases

def test_out_of_range_ids_are_flagged_and_left_out():
    layer = wl.make_config(0)
    tk = layer.topk_ids.copy()
    tk[2, 1] = layer.E
    tk[5, 0] = -2
    lo = layer.lora_ids.copy()
    lo[7] = layer.L
    bad = dataclasses.replace(layer, topk_ids=tk, lora_ids=lo)
    dl, st = run(bad)
    assert st == B.MOELORA_EDEVICE_ID
    ref, inv = oracle.forward(bad)
    assert inv == 2 + layer.k
    got = dl.out_f64()
    assert norm_err(got, ref) <= TOL
    assert np.all(got[7] == 0)
    # the next clean forward on the same workspace reports OK again
    dl.set_batch(layer.x, layer.topk_ids, layer.topk_weights, layer.lora_ids)
    B.check(dl.forward())
    assert dl.status() == 0


def test_out_of_range_ids_flagged_by_the_multi_cta_align():
    """A batch of 1200 pairs in 12 buckets takes the multi-CTA align: bad
    ids seen by any of its CTAs reach the status word, their pairs are left
    out, and a clean batch afterwards reports OK."""
    layer = wl.make_random(600, 128, 136, 2, 2, 5, 32, seed=7)
    tk = layer.topk_ids.copy()
    tk[3, 1] = layer.E          # first CTA's pairs
    tk[590, 0] = -1             # last CTA's pairs
    lo = layer.lora_ids.copy()
    lo[300] = layer.L           # a middle CTA's token
    bad = dataclasses.replace(layer, topk_ids=tk, lora_ids=lo)
    dl, st = run(bad)
    assert st == B.MOELORA_EDEVICE_ID
    ref, inv = oracle.forward(bad)
    assert inv == 2 + layer.k
    got = dl.out_f64()
    assert norm_err(got, ref) <= TOL
    assert np.all(got[300] == 0)
    dl.set_batch(layer.x, layer.topk_ids, layer.topk_weights, layer.lora_ids)
    B.check(dl.forward())
    assert dl.status() == 0
    ref, _ = oracle.forward(layer)
    assert norm_err(dl.out_f64(), ref) <= TOL


def test_all_pairs_on_one_expert_and_all_base_only():
    layer = wl.make_random(50, 128, 64, 6, 3, 2, 16, seed=4)
    tk = np.tile(np.array([[5, 2, 0]], np.int32), (50, 1))
    check_layer(dataclasses.replace(layer, topk_ids=tk))
    check_layer(dataclasses.replace(layer, lora_ids=np.full(50, -1, np.int32)))


@pytest.mark.parametrize("adapters", [False, True])
def test_duplicate_experts_in_one_tokens_top_k(adapters):
    """A token may name the same expert in several of its top-k slots (a
    router cannot produce it, but the input format allows it): each slot is a
    pair of its own, computed and weighted separately.  Mixed duplicates
    (two and three slots), all-duplicate tokens, with and without adapters
    (the same (expert, adapter) bucket then holds several pairs of one token)."""
    layer = wl.make_random(48, 264, 136, 6, 4, 3 if adapters else 0, 16 if adapters else 0, seed=31)
    tk = layer.topk_ids.copy()
    tk[0] = [2, 2, 2, 2]
    tk[1] = [5, 1, 5, 1]
    tk[7] = [3, 3, 0, 4]
    tk[20:30, 1] = tk[20:30, 0]
    tk[40:, :] = 1
    lo = layer.lora_ids.copy()
    if not adapters:
        lo[:] = -1
    dup = dataclasses.replace(layer, topk_ids=tk, lora_ids=lo)
    dl, err = check_layer(dup)
    # a token whose k slots name one expert equals that expert's FFN scaled by
    # the sum of its weights: check it against the oracle on one slot of weight 1
    one = dataclasses.replace(dup, T=1, k=1, x=dup.x[:1], topk_ids=np.array([[2]], np.int32),
                              topk_weights=np.array([[float(dup.topk_weights[0].sum())]], np.float32),
                              lora_ids=dup.lora_ids[:1])
    ref_one, _ = oracle.forward(one)
    assert norm_err(dl.out_f64()[:1], ref_one) <= TOL


def test_no_adapters_null_pointers():
    layer = wl.make_random(12, 64, 64, 4, 2, 0, 0, seed=2)
    assert layer.A1 is None
    check_layer(layer)


def test_empty_batch_is_ok():
    layer = wl.make_random(3, 64, 64, 4, 2, 1, 8, seed=2)
    dl = DeviceLayer(layer, "cuda")
    d0 = B.dims(0, 64, 64, 4, 2, 1, 8)
    ws = torch.empty(B.moe_lora_workspace_bytes(d0), dtype=torch.uint8, device="cuda")
    st = B.moe_lora_forward(d0, None, None, None, None, dl.W1, dl.W2, dl.A1, dl.B1, dl.A2, dl.B2, None, ws)
    assert st == 0 and B.moe_lora_get_status(ws) == 0


def test_output_guard_bytes_untouched():
    layer = wl.make_config(0)
    dl = DeviceLayer(layer, "cuda")
    buf = torch.full((layer.T * layer.H + 64,), 7, dtype=torch.int16, device="cuda")
    out = buf[:layer.T * layer.H].view(torch.bfloat16).view(layer.T, layer.H)
    B.check(dl.forward(out=out))
    torch.cuda.synchronize()
    assert (buf[layer.T * layer.H:] == 7).all()


# ------------------------------------------------------------------ named workloads at full size

@pytest.fixture(scope="module")
def config1():
    return wl.make_config(1)


def test_config1_decode_full(config1):
    check_layer(config1)


def test_intermediates_config1(config1):
    """z1, z2, act and the weighted pair outputs of the decode layer against the
    oracle (its shrinks split K across CTAs and finish in the last split)."""
    dl, st = run(config1)
    P, I, H, r = config1.P, config1.I, config1.H, config1.r
    rows = dl.workspace_view("compact_ids", torch.int32, (P,)).cpu().numpy()
    z1 = dl.workspace_view("z1", torch.float32, (P, r)).cpu().numpy().astype(np.float64)
    z2 = dl.workspace_view("z2", torch.float32, (P, r)).cpu().numpy().astype(np.float64)
    act_bits = dl.workspace_view("act", torch.int16, (P, I)).cpu().numpy().view(np.uint16)
    act = (act_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    pair_out = dl.pair_outputs()
    for row in range(0, P, 7):
        p = int(rows[row])
        ref = oracle.pair(config1, p)
        assert norm_err(z1[row], ref["z1"]) < 1e-5
        # z2 is A2 applied to the bf16 act of the GPU, so it inherits act's rounding
        assert norm_err(z2[row], ref["z2"]) < 8e-3
        assert norm_err(act[row], ref["act"]) < 8e-3
        assert norm_err(pair_out[p], float(config1.topk_weights.flat[p]) * ref["d"]) < 1e-2


@pytest.mark.slow
def test_config2_prefill_full():
    # all 2048 x 2880 outputs: 128- and 256-pair chunks, each expert's last
    # partial chunk, the tensor-core expand blocks of every adapter mix
    check_layer(wl.make_config(2))


@pytest.mark.slow
def test_config3_mixed_full():
    layer = wl.make_config(3)
    assert 0.45 <= layer.meta["hot_share"] <= 0.55
    check_layer(layer)


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 16, 256])
def test_config4_dense(T):
    check_layer(wl.make_config(4, T=T))


def _silu_probe_layer(u, adapters: bool, experts: int):
    """Experts (all alike) whose first gate unit copies feature 0 of x, whose
    first up unit copies the constant feature 1, and whose first output
    copies act unit 0: out[t][0] = bf16(SiLU(u_t)) with every product and sum
    exact.  Token t goes to expert t mod `experts`: many experts keep the
    chunks decode-sized (one-CTA kernels), one expert makes them wide (CTA
    pairs).  With `adapters`, every token carries adapter 0 of a rank-8 LoRA
    whose A and B are zero: its delta adds exact zeros, and the activation
    goes through the epilogue that follows a LoRA expand."""
    T, H, I, E = len(u), 64, 64, experts
    x = np.zeros((T, H), np.float32)
    x[:, 0] = u
    x[:, 1] = 1.0
    W1 = np.zeros((E, 2 * I, H), np.float32)
    W1[:, 0, 0] = 1.0          # gate unit 0 <- x[:, 0]
    W1[:, I, 1] = 1.0          # up unit 0 <- 1
    W2 = np.zeros((E, H, I), np.float32)
    W2[:, 0, 0] = 1.0          # out[:, 0] <- act unit 0
    b = wl.bf16_bits
    L, r = (1, 8) if adapters else (0, 0)
    A1 = B1 = A2 = B2 = None
    if adapters:
        A1 = np.zeros((L, E, r, H), np.uint16)
        B1 = np.zeros((L, E, 2 * I, r), np.uint16)
        A2 = np.zeros((L, E, r, I), np.uint16)
        B2 = np.zeros((L, E, H, r), np.uint16)
    lora = np.zeros(T, np.int32) if adapters else np.full(T, -1, np.int32)
    ids = (np.arange(T, dtype=np.int32) % E).reshape(T, 1)
    return wl.Layer("silu_probe", T, H, I, E, 1, L, r, b(x), b(W1), b(W2), A1, B1, A2, B2,
                    ids, np.ones((T, 1), np.float32), lora)


# (adapters, wide chunks) -> the epilogue that computes SiLU(gate) * up
SILU_PATHS = {
    "one_cta_lean": (False, False),
    "one_cta_cuda_core_expand": (True, False),
    "cta_pair": (False, True),
    "cta_pair_tc_expand": (True, True),
}


@pytest.mark.parametrize("path", list(SILU_PATHS))
def test_silu_sweep_against_fp64(path):
    """The GPU's SiLU(u) = u / (1 + exp(-u)), rounded once to bf16, against the
    fp64 definition over every bf16 value of u in [-120, 120] on a grid, in
    every epilogue that computes it: the one-CTA kernel's lean epilogue and
    its CUDA-core LoRA expand epilogue, and the CTA-pair kernel's (without
    and after the tensor-core expand).  Past |u| ~ 88 the exponential of -u
    leaves the fp32 range (overflow to infinity for u < 0, underflow to zero
    for u > 0): SiLU must then give 0 (at most 1e-30 away from the true,
    tiny value) or u itself.  One bf16 ulp (2^-8 relative) is allowed
    elsewhere."""
    adapters, wide = SILU_PATHS[path]
    grid = np.concatenate([np.linspace(-120.0, 120.0, 3001), [-88.7, -88.0, -87.3, 87.3, 88.0, 88.7]])
    u = np.unique(wl.bf16_to_f32(wl.bf16_bits(grid.astype(np.float32))).astype(np.float64))
    experts = 1 if wide else (len(u) + 39) // 40
    dl, st = run(_silu_probe_layer(u.astype(np.float32), adapters, experts))
    assert st == 0
    lay = B.moe_lora_workspace_layout(dl.d)
    assert lay["gemm_ctas"] == (2 if wide else 1)
    assert lay["tc_expand"] == (1 if (adapters and wide) else 0)
    got = dl.out_f64()[:, 0]
    ref = u / (1.0 + np.exp(-u))
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)
    # saturated ends: exactly u for large positive u, zero for large negative u
    assert np.all(got[u >= 90.0] == u[u >= 90.0])
    assert np.all(got[u <= -104.0] == 0.0)
    # every other output column is exactly zero (no other unit leaks in)
    assert np.all(dl.out_f64()[:, 1:] == 0.0)
