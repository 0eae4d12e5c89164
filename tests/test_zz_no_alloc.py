"""moe_lora_forward_noalloc: the forward for callers that cannot allocate device
memory (code that must not call cudaMalloc, plugins without access to their
host's allocator), running on the library's own built-in scratch buffer.

Checked through the C ABI against moe_lora_forward with a caller workspace, on
two calls in a row with different problems (the second call reuses the buffer
the first one left behind).  Collected last (file name) so that a stop at the
first failure has already run every other test; it also passes alone.
"""
import numpy as np
import pytest
import torch

from lora_moe_layer_gb300 import binding as B
from lora_moe_layer_gb300 import workloads as wl
from lora_moe_layer_gb300.layer import DeviceLayer

from gpu_helpers import TOL, norm_err

pytestmark = pytest.mark.gpu


def _noalloc(dl, out):
    return B.moe_lora_forward_noalloc(dl.d, dl.x, dl.topk_ids, dl.topk_weights, dl.lora_ids, dl.W1, dl.W2,
                                      dl.A1, dl.B1, dl.A2, dl.B2, out)


def _bits_to_f64(t):
    bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    layers = [wl.make_config(0), wl.make_random(37, 264, 136, 5, 3, 3, 24, seed=7)]
    for layer in layers:  # call 1 and call 2 share the library's scratch buffer
        dl = DeviceLayer(layer, "cuda")
        B.check(dl.forward(), "moe_lora_forward")
        ref = dl.out.clone()
        out = torch.full_like(dl.out, float("nan"))
        B.check(_noalloc(dl, out), "moe_lora_forward_noalloc")
        torch.cuda.synchronize()
        got, want = _bits_to_f64(out), _bits_to_f64(ref)
        assert norm_err(got, want) <= TOL
        # same kernels on the same inputs: the results agree bit for bit as well
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def _largest_fitting_T(shape):
    """The largest token count whose workspace still fits the built-in scratch
    (host-only size queries: the layout grows with T)."""
    lim = B.MOELORA_NOALLOC_SCRATCH_BYTES
    lo, hi = 1, 1 << 17
    assert B.moe_lora_workspace_bytes(B.dims(lo, *shape)) <= lim < B.moe_lora_workspace_bytes(B.dims(hi, *shape))
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if B.moe_lora_workspace_bytes(B.dims(mid, *shape)) <= lim:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_at_the_edge_of_its_scratch():
    """A problem whose workspace takes all but a few KiB of the scratch buffer,
    so its last regions (split-K partials and counters) sit at the end of it,
    matches moe_lora_forward bit for bit; one more token does not fit and is
    refused before any launch."""
    shape = (520, 200, 5, 3, 3, 24)
    T = _largest_fitting_T(shape)
    need = B.moe_lora_workspace_bytes(B.dims(T, *shape))
    assert need > B.MOELORA_NOALLOC_SCRATCH_BYTES - (64 << 10)
    layer = wl.make_random(T, *shape, seed=12)
    dl = DeviceLayer(layer, "cuda")
    B.check(dl.forward(), "moe_lora_forward")
    ref = dl.out.clone()
    out = torch.full_like(dl.out, float("nan"))
    for _ in range(2):
        B.check(_noalloc(dl, out), "moe_lora_forward_noalloc")
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    d = B.dims(T + 1, *shape)
    f = 1 << 20  # never dereferenced: the call returns before any launch
    assert B.moe_lora_forward_noalloc(d, f, f, f, f, f, f, f, f, f, f, f) == B.MOELORA_ENOSPC


def test_noalloc_refuses_problems_larger_than_its_scratch():
    d = B.dims(2048, 2880, 2880, 32, 4, 8, 32)
    assert B.moe_lora_workspace_bytes(d) > B.MOELORA_NOALLOC_SCRATCH_BYTES
    f = 1 << 20  # never dereferenced: the call returns before any launch
    st = B.moe_lora_forward_noalloc(d, f, f, f, f, f, f, f, f, f, f, f)
    assert st == B.MOELORA_ENOSPC
