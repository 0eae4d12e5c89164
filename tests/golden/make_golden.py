"""Write the text fixtures in this folder from the oracle alone.

The pages print no worked example and no intermediate value, so these fixtures
are not the pages' numbers: they freeze the oracle's answer on the tiny seeded
workload (T=8, H=256, I=512, E=8, top-2, 2 adapters of rank 8) so that any later
change to the oracle's arithmetic shows up as a diff.  Correctness pins live in
tests/test_oracle_pins.py and tests/test_align_oracle.py.

Run:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from lora_moe_layer_gb300 import workloads as wl  # noqa: E402


def main():
    layer = wl.make_config(0)
    out, inv = oracle.forward(layer, n_threads=1)
    fixture = {
        "workload": wl.CONFIG_NAMES[0] + ", seed 0",
        "source": "oracle/oracle.c via tests/golden/make_golden.py",
        "topk_ids": layer.topk_ids.tolist(),
        "lora_ids": layer.lora_ids.tolist(),
        "invalid_pairs": inv,
        # the first 16 outputs of every token exactly, and a digest of all of them
        "out_head": [[float.hex(float(v)) for v in row[:16]] for row in out],
        "out_sha256": hashlib.sha256(np.ascontiguousarray(out, dtype="<f8").tobytes()).hexdigest(),
        "align": {},
    }
    for bm in (8, 16, 64):
        a = oracle.align(layer.topk_ids, layer.lora_ids, layer.E, layer.L, bm)
        fixture["align"][str(bm)] = {k: (v.tolist() if isinstance(v, np.ndarray) else v)
                                     for k, v in a.items() if k != "capacity"}
    with open(os.path.join(HERE, "config0_oracle.json"), "w") as f:
        # one key per line, values inline
        f.write("{\n" + ",\n".join(f"{json.dumps(k)}: {json.dumps(fixture[k])}"
                                     for k in sorted(fixture)) + "\n}\n")


if __name__ == "__main__":
    main()
