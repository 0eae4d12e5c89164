"""Benchmark of the multi-LoRA fused MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C] [--T T] [--w8]

A step is one full layer forward (align, both LoRA shrinks, gate_up with the
fused expand and SiLU*up, down with the fused expand and top-k weight, top-k
reduce) over one batch of the seeded synthetic workload; by default the
GPT-OSS-20B-shaped prefill chunk (T=2048 tokens from 16 sequences of 128,
H=I=2880, E=32, top-4, 8 adapters of rank 32), the largest of the workloads;
--config 1 selects the decode layer (T=16); --w8 runs the same layer with FP8
(E4M3) base expert weights (moe_lora_forward_w8, parity against the oracle's
FP8 forward).  Rank 0 prints one JSON line.

--impl ours       time the CUDA library (inputs resident in HBM), plus the
                  end-to-end call from pinned host buffers, the roofline of the
                  dominant kernel and the oracle on the host cores.
--impl reference  time the fp64 CPU oracle as it stands on this machine's host
                  cores, each step a bounded sample of the same workload.

Under torchrun each rank runs an independent replica (the layer has no
cross-GPU exchange): value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-LoRA layer tokens/s; achieved HBM GB/s or tensor-pipe % of GB300 peak"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
TOL = 1e-2


# ----------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def algorithmic(layer, w8: bool = False):
    """Layer-level algorithmic bytes and flops from the actual routing (weights
    bf16; with w8, the base expert weights as one-byte codes plus an fp32
    scale per output row)."""
    import numpy as np
    P = layer.P
    e_of = layer.topk_ids.reshape(-1)
    l_of = np.repeat(layer.lora_ids, layer.k)
    experts = len(np.unique(e_of))
    lora_mask = l_of >= 0
    buckets = len({(int(e), int(l)) for e, l in zip(e_of[lora_mask], l_of[lora_mask])})
    H, I, r, T, k = layer.H, layer.I, layer.r, layer.T, layer.k
    wb = 1 if w8 else 2                                  # bytes per base weight
    scales = experts * 4 * (2 * I + H) if w8 else 0      # fp32 row scales of W1, W2
    layer_bytes = (wb * experts * 3 * H * I + scales + 2 * (buckets * r * (2 * H + 3 * I) + 2 * T * H)
                   + 8 * T * k + 4 * T)
    flops = P * 6 * H * I + int(lora_mask.sum()) * 2 * r * (2 * H + 3 * I)
    # per-kernel bytes the two tcgen05 kernels must move: weights of the touched
    # experts (W) and adapter buckets (the expand's B and the shrink's A), the
    # pair rows they read (x in bucket order / act) and what they write
    gate_up = experts * 2 * I * H * wb + buckets * (2 * I * r + r * H) * 2 + P * H * 2 + P * I * 2
    down = experts * H * I * wb + buckets * (H * r + r * I) * 2 + P * I * 2 + P * H * 4
    if w8:
        gate_up += experts * 2 * I * 4
        down += experts * H * 4
    gate_up_flops = P * 2 * H * 2 * I + int(lora_mask.sum()) * 2 * r * (H + 2 * I)
    down_flops = P * 2 * I * H + int(lora_mask.sum()) * 2 * r * (I + H)
    return dict(bytes=layer_bytes, flops=flops, experts_touched=experts, lora_buckets_touched=buckets,
                kernel_bytes={"gate_up_gemm": gate_up, "down_gemm": down},
                kernel_flops={"gate_up_gemm": gate_up_flops, "down_gemm": down_flops})


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.marks = {}
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.perf_counter(), [c.strip() for c in line.split(",")]))

    def mark(self, name):
        self.marks[name] = time.perf_counter()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        t0, t1 = self.marks.get("timed_start", 0), self.marks.get("timed_end", 1e30)
        rows = [r for t, r in self.rows if t0 <= t <= t1]
        window = "timed region"
        if len(rows) < 3:  # a short timed region: use the whole run (warm-up included)
            rows = [r for _, r in self.rows]
            window = "warm-up + timed region"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "window": window}


HBM_NOMINAL_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy peak is the roofline's denominator)


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload_tag: str):
    """dram bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload_tag}.txt")
    if not os.path.exists(path):
        return None, None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith(" "):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    src = vals.get("kernel_sources", "")
    files = [s.strip() for s in src.split(",") if s.strip()]
    try:
        if not files or kernel_source_hash(files) != vals.get("kernel_source_sha256"):
            return None, "kernel changed since the counters were taken"
        return float(vals["dram_bytes_per_launch"]), os.path.relpath(path, ROOT)
    except Exception:
        return None, None


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    from lora_moe_layer_gb300 import binding as B
    from lora_moe_layer_gb300 import build as build_mod
    from lora_moe_layer_gb300 import workloads as wl
    from lora_moe_layer_gb300.layer import DeviceLayer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        build_mod.build()
    if world > 1:
        torch.distributed.barrier()
    B.load()

    layer = wl.make_config(args.config, T=args.T)
    workload = wl.CONFIG_NAMES[args.config] + (f" T={layer.T}" if args.config == 4 else "")
    if args.w8:
        layer = wl.quantize_e4m3(layer)
        workload += ", FP8 (E4M3) base expert weights with per-row scales, bf16 LoRA"
    dl = DeviceLayer(layer, dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # align, [zexp clear], gate_up, down, reduce: as the library reports for these dims
    kernels_per_forward = B.moe_lora_workspace_layout(dl.d)["launches"]

    def fwd():
        st = dl.forward_w8(stream=stream) if args.w8 else dl.forward(stream=stream)
        if st != 0:
            raise B.MoeLoraError(st, "moe_lora_forward_w8" if args.w8 else "moe_lora_forward")

    clocks = ClockSampler(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            fwd()
        stream.synchronize()

        # ---- timed region: K forwards, per-step device events, L2 flushed between steps
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        clocks.mark("timed_start")
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            fwd()
            ends[i].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        clocks.mark("timed_end")
        if world > 1:
            torch.distributed.barrier()
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        dev_s = sum(step_ms) / 1e3

        # ---- beside it: the same forward with L2 left warm (no flush between steps)
        warm = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        fwd()
        warm[0].record(stream)
        for _ in range(args.steps):
            fwd()
        warm[1].record(stream)
        torch.cuda.synchronize()
        warm_ms = warm[0].elapsed_time(warm[1]) / args.steps

        # ---- per-kernel durations: K traced forwards (events between the kernels, same stream)
        n_ev = B.MOELORA_TRACE_EVENTS
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            B.check(dl.forward_traced(evs[i], stream, w8=args.w8), "traced forward")
        torch.cuda.synchronize()
        kern_ms = {name: 0.0 for name in B.KERNEL_SLOTS}
        traced_step_ms = 0.0
        for i in range(args.steps):
            for j, name in enumerate(B.KERNEL_SLOTS):
                kern_ms[name] += evs[i][j].elapsed_time(evs[i][j + 1])
            traced_step_ms += evs[i][0].elapsed_time(evs[i][n_ev - 1])
        kern_ms = {k: v / args.steps for k, v in kern_ms.items()}
        traced_step_ms /= args.steps

        # ---- end to end through the public API: pinned host -> device, forward, result -> host
        x_h = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
        ids_h = torch.from_numpy(layer.topk_ids).pin_memory()
        w_h = torch.from_numpy(layer.topk_weights).pin_memory()
        l_h = torch.from_numpy(layer.lora_ids).pin_memory()
        out_h = torch.empty((layer.T, layer.H), dtype=torch.int16).pin_memory()
        x_d = dl.x.view(torch.int16)
        h2d = sum(t.numel() * t.element_size() for t in (x_h, ids_h, w_h, l_h))
        d2h = out_h.numel() * out_h.element_size()
        e2e_steps = args.steps
        for i in range(args.warmup + e2e_steps):
            if i == args.warmup:
                torch.cuda.synchronize()
                e2e_time = 0.0
            flush.zero_()
            stream.synchronize()
            t0 = time.perf_counter()
            x_d.copy_(x_h, non_blocking=True)
            dl.topk_ids.copy_(ids_h, non_blocking=True)
            dl.topk_weights.copy_(w_h, non_blocking=True)
            dl.lora_ids.copy_(l_h, non_blocking=True)
            fwd()
            out_h.copy_(dl.out.view(torch.int16), non_blocking=True)
            stream.synchronize()
            if i >= args.warmup:
                e2e_time += time.perf_counter() - t0
    clocks.stop()

    # ---- parity of what was timed, against the oracle (full batch)
    parity = None
    status = dl.status(stream)
    if rank == 0 and not args.skip_oracle:
        import oracle
        ref, _ = oracle.forward_w8(layer) if args.w8 else oracle.forward(layer)
        got = dl.out_f64()
        parity = {"norm_err": float(np.max(np.abs(got - ref)) / np.max(np.abs(ref))), "tol": TOL,
                  "status": status, "checked": "all outputs vs fp64 oracle"}

    # max over ranks
    dev_s, e2e_time, value = aggregate_replicas(dev_s, e2e_time, layer.T * args.steps, world, dev)
    if rank != 0:
        return None

    alg = algorithmic(layer, w8=args.w8)
    pk = peaks()
    ms_step = dev_s * 1e3 / args.steps
    dom = max(("gate_up_gemm", "down_gemm"), key=lambda k: kern_ms[k])
    dom_bytes = alg["kernel_bytes"][dom]
    dom_flops = alg["kernel_flops"][dom]
    dom_s = kern_ms[dom] * 1e-3
    dom_gbs = dom_bytes / dom_s / 1e9
    dom_tflops = dom_flops / dom_s / 1e12
    # The bound: tensor when the kernel's algorithmic intensity is at least half
    # the machine balance (measured bf16 burst peak / measured copy bandwidth,
    # ~287 flop/B), i.e. when its flops alone take at least half as long as its
    # bytes at peak (the prefill and dense T=256 GEMMs, gated on the tensor
    # pipe); else HBM (decode-sized batches).  Both fractions are reported.
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    tensor_bound = dom_flops / dom_bytes >= 0.5 * ridge
    tag = f"config{args.config}" + (f"_T{layer.T}" if args.config == 4 else "") + ("_w8" if args.w8 else "")
    traffic, traffic_src = recorded_traffic(dom, tag)

    cpu = None
    if world == 1 and not args.skip_oracle:
        cpu = cpu_baseline(layer, budget_s=args.cpu_seconds, warmed=parity is not None, w8=args.w8)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded PCG64 draws, random-init weights)",
        "config": {"workload": workload, "T": layer.T, "H": layer.H, "I": layer.I, "E": layer.E,
                   "top_k": layer.k, "adapters": layer.L, "rank": layer.r, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({alg['bytes'] / 1e9:.2f} GB/step) and a 256 MiB write "
                         "between steps, outside the step events",
                   "timing": "CUDA events around each forward on its stream; sum over K steps"},
        "layer": {"bytes_alg": alg["bytes"], "flops_alg": alg["flops"], "experts_touched": alg["experts_touched"],
                  "lora_buckets_touched": alg["lora_buckets_touched"],
                  "achieved_gbs": alg["bytes"] / (ms_step * 1e-3) / 1e9,
                  "hbm_frac": alg["bytes"] / (ms_step * 1e-3) / 1e9 / pk["hbm_gbs"],
                  "roof_ms": max(alg["bytes"] / (pk["hbm_gbs"] * 1e9), alg["flops"] / (pk["bf16_tflops"] * 1e12)) * 1e3,
                  "tensor_tflops": alg["flops"] / (ms_step * 1e-3) / 1e12,
                  "tensor_frac": alg["flops"] / (ms_step * 1e-3) / 1e12 / pk["bf16_tflops"],
                  "hbm_frac_nominal": alg["bytes"] / (ms_step * 1e-3) / 1e9 / HBM_NOMINAL_GBS,
                  "warm_l2_ms_per_step": warm_ms},
        "roofline": dict(
            {"kernel": dom, "bound": "tensor", "achieved": dom_tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
             "frac": dom_tflops / pk["bf16_tflops"],
             "peak_source": (pk["source"] + " (MEASURED_PEAKS.json bf16_tflops, cuBLAS bf16 burst)")
             if pk["source"] == "measured" else "fallback"}
            if tensor_bound else
            {"kernel": dom, "bound": "hbm", "achieved": dom_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
             "frac": dom_gbs / pk["hbm_gbs"],
             "peak_source": (pk["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy)")
             if pk["source"] == "measured" else "fallback"},
            traffic=traffic, bytes_per_launch=dom_bytes, flops_per_launch=dom_flops, launch_us=kern_ms[dom] * 1e3,
            hbm_gbs=dom_gbs, hbm_frac=dom_gbs / pk["hbm_gbs"], tensor_tflops=dom_tflops,
            tensor_frac=dom_tflops / pk["bf16_tflops"], intensity_flop_per_byte=dom_flops / dom_bytes,
            ridge_flop_per_byte=ridge,
            timed="kernel events recorded between the kernels over K traced forwards on the launch stream",
            traffic_source=traffic_src),
        "kernels_us": {k: v * 1e3 for k, v in kern_ms.items()},
        "traced_ms_per_step": traced_step_ms,
        "e2e": {"value": layer.T * e2e_steps / e2e_time, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_time * 1e3 / e2e_steps,
                "path": "pinned host -> device copies, moe_lora_forward, out -> pinned host, stream sync (wall clock)"},
        "gpu_launches": kernels_per_forward * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed": t_wall,
        "parity": parity,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def aggregate_replicas(dev_s, e2e_s, tokens_per_rank, world, device):
    """Whole-job numbers of N independent replicas: the slowest rank's device
    and end-to-end times, and tokens of all ranks / that device time."""
    import torch
    t = torch.tensor([dev_s, e2e_s], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    dev_s, e2e_s = float(t[0].item()), float(t[1].item())
    return dev_s, e2e_s, tokens_per_rank * world / dev_s


def _threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(layer, budget_s: float = 12.0, warmed: bool = False, w8: bool = False):
    """The oracle as it stands on the host cores: whole batches until ~budget_s
    of CPU work (at least one; a prefill batch takes several seconds)."""
    import oracle
    nt = _threads()
    run = oracle.forward_w8 if w8 else oracle.forward
    if not warmed:
        run(layer, n_threads=nt)  # warm (page in weights)
    t0 = time.perf_counter()
    n = 0
    while True:
        run(layer, n_threads=nt)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": layer.T * n / dt, "unit": UNIT, "cores": min(nt, layer.T), "kind": "oracle",
            "sample": f"{n} full forwards of the same batch ({layer.T} tokens each), fp64, OpenMP over tokens"}


# ----------------------------------------------------------------------------- reference arm

def _pair_layer(layer, pairs):
    """A layer whose 'tokens' are the given (t, j) pairs, one slot each (same arithmetic per pair)."""
    import numpy as np
    from lora_moe_layer_gb300 import workloads as wl
    ts = np.array([t for t, _ in pairs])
    js = np.array([j for _, j in pairs])
    return wl.Layer(layer.name + "_pairs", len(pairs), layer.H, layer.I, layer.E, 1, layer.L, layer.r,
                    layer.x[ts], layer.W1, layer.W2, layer.A1, layer.B1, layer.A2, layer.B2,
                    layer.topk_ids[ts, js].reshape(-1, 1).astype(np.int32),
                    layer.topk_weights[ts, js].reshape(-1, 1).astype(np.float32),
                    layer.lora_ids[ts].astype(np.int32))


def run_reference(args):
    import oracle
    from lora_moe_layer_gb300 import workloads as wl

    layer = wl.make_config(args.config, T=args.T)
    workload = wl.CONFIG_NAMES[args.config] + (f" T={layer.T}" if args.config == 4 else "")
    nt = _threads()
    all_pairs = [(t, j) for t in range(layer.T) for j in range(layer.k)]
    # calibrate: one pair on one thread
    one = _pair_layer(layer, all_pairs[:1])
    oracle.forward(one, n_threads=1)
    t0 = time.perf_counter()
    oracle.forward(one, n_threads=1)
    t_pair = time.perf_counter() - t0
    budget = min(2.0, max(0.02, args.ref_seconds / max(1, args.steps + args.warmup)))
    n_pairs = max(1, min(len(all_pairs), int(budget * nt / max(t_pair, 1e-6))))
    n_thr = min(nt, n_pairs)
    step_times = []
    cursor = 0
    for i in range(args.warmup + args.steps):
        pairs = [all_pairs[(cursor + q) % len(all_pairs)] for q in range(n_pairs)]
        cursor = (cursor + n_pairs) % len(all_pairs)
        sub = _pair_layer(layer, pairs)
        t0 = time.perf_counter()
        oracle.forward(sub, n_threads=n_thr)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            step_times.append(dt)
    total = sum(step_times)
    tokens = n_pairs * args.steps / layer.k
    value = tokens / total
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded PCG64 draws, random-init weights)", "impl": "reference",
        "config": {"workload": workload, "T": layer.T, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_thr, "kind": "oracle",
                         "sample": f"{n_pairs} (token, slot) pairs per step = {n_pairs / layer.k:g} tokens, "
                                   "cycling through the batch"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", type=int, default=2,
                    help="workload index (default 2: the prefill chunk; 1: the decode layer)")
    ap.add_argument("--T", type=int, default=None, help="token count for the dense workload (config 4)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0)
    ap.add_argument("--skip-oracle", action="store_true", help="no parity check or CPU baseline (profiling runs)")
    ap.add_argument("--w8", action="store_true",
                    help="FP8 (E4M3) base expert weights with per-row scales (moe_lora_forward_w8)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_ours(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
