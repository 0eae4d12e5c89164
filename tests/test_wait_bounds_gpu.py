"""Device-side waits are bounded: a wait that nothing satisfies ends, the
kernel records the timeout in the workspace status word (read back as
MOELORA_ETIMEOUT), and the context stays usable.  Nothing here faults, traps or
hangs the GPU; each wait gives up after its bounded number of rounds."""
import time

import pytest
import torch

from lora_moe_layer_gb300 import binding as B
from lora_moe_layer_gb300 import workloads as wl

from gpu_helpers import TOL, norm_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier_phase", "global_counter"])
def test_unsatisfied_wait_times_out_and_reports(kind):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    B.check(B.moe_lora_selftest_wait(kind, ws), "moe_lora_selftest_wait")
    assert B.moe_lora_get_status(ws) == B.MOELORA_ETIMEOUT
    elapsed = time.perf_counter() - t0
    assert elapsed < 30.0, elapsed


def test_context_usable_after_a_timeout():
    import oracle
    from lora_moe_layer_gb300.layer import DeviceLayer
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    B.check(B.moe_lora_selftest_wait(1, ws))
    assert B.moe_lora_get_status(ws) == B.MOELORA_ETIMEOUT
    layer = wl.make_config(0)
    dl = DeviceLayer(layer, "cuda")
    B.check(dl.forward())
    assert dl.status() == 0
    ref, _ = oracle.forward(layer)
    assert norm_err(dl.out_f64(), ref) <= TOL


def test_selftest_rejects_bad_arguments():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert B.moe_lora_selftest_wait(2, ws) == B.MOELORA_EINVAL
    assert B.moe_lora_selftest_wait(0, None) == B.MOELORA_EINVAL
