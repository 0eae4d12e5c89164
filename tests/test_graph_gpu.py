"""The forward is asynchronous on its stream and capturable in a CUDA graph:
captured once, replayed on new inputs written into the same buffers, it gives
bit-for-bit the output of eager calls (the kernels read every size and count
from the device, so one capture serves any routing of the same shape), and
each replayed output matches the fp64 oracle of the routing it was given."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, norm_err

from lora_moe_layer_gb300 import binding as B
from lora_moe_layer_gb300 import workloads as wl
from lora_moe_layer_gb300.layer import DeviceLayer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", ["decode", "wide"])
def test_graph_replay_matches_eager(which):
    if which == "decode":
        layer = wl.make_config(1)
        other = wl.make_random(16, 2880, 2880, 32, 4, 8, 32, seed=11)
    else:
        layer = wl.make_random(300, 128, 136, 2, 2, 6, 32, seed=9)
        other = wl.make_random(300, 128, 136, 2, 2, 6, 32, seed=10)
    dl = DeviceLayer(layer, "cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        B.check(dl.forward(stream=side))            # warm-up: per-device set-up outside the capture
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            B.check(dl.forward(stream=side), "moe_lora_forward under capture")
    torch.cuda.synchronize()

    def eager_out():
        B.check(dl.forward())
        torch.cuda.synchronize()
        assert dl.status() == 0
        return dl.out.clone()

    # replay on the captured inputs
    ref1 = eager_out()
    dl.out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert dl.status() == 0
    assert torch.equal(dl.out.view(torch.int16), ref1.view(torch.int16))
    want1, inv = oracle.forward(layer)
    assert inv == 0 and norm_err(dl.out_f64(), want1) <= TOL

    # new tokens and routing copied into the same buffers: the replay follows them
    dev = dl.x.device
    dl.x.view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(other.x).view(np.int16)).to(dev))
    dl.topk_ids.copy_(torch.from_numpy(np.ascontiguousarray(other.topk_ids, dtype=np.int32)).to(dev))
    dl.topk_weights.copy_(torch.from_numpy(np.ascontiguousarray(other.topk_weights, dtype=np.float32)).to(dev))
    dl.lora_ids.copy_(torch.from_numpy(np.ascontiguousarray(other.lora_ids, dtype=np.int32)).to(dev))
    ref2 = eager_out()
    assert not torch.equal(ref1.view(torch.int16), ref2.view(torch.int16))
    dl.out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert dl.status() == 0
    assert torch.equal(dl.out.view(torch.int16), ref2.view(torch.int16))
    # the second routing with the first layer's weights (only x and the routing were copied in)
    want2, inv = oracle.forward(dataclasses.replace(layer, x=other.x, topk_ids=other.topk_ids,
                                                    topk_weights=other.topk_weights, lora_ids=other.lora_ids))
    assert inv == 0 and norm_err(dl.out_f64(), want2) <= TOL
