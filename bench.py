#!/usr/bin/env python3
"""Benchmark of the CosmoFlow conv3d block stack on GB300.

Workload (one step): the five-block stack conv3d k=3 pad 1 -> bias ->
leaky ReLU 0.3 -> 2x2x2 max-pool with C_out 32, 64, 128, 256, 256 on
N = 8 samples of 4 x 128^3 bf16 (x = log(1 + lognormal(0,1))), forward plus
backward (pool/LReLU backward, backward-weight for every block,
backward-data for blocks 2..5), fp32 weight gradients.

Metric: conv3d fwd+bwd TFLOP/s (2 FLOP per multiply-add, every tap counted,
one count per executed fwd / dgrad / wgrad conv) and samples/s, with the
fraction of the measured bf16 tensor peak.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line on rank 0.  With N > 1 (torchrun) every rank runs an
independent replica of the step (the path has no exchange step on one
node here: replicas only); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthdata  # noqa: E402
from cnn_conv3d_gb300 import flops as flops_mod  # noqa: E402

WORKLOAD = dict(n=8, spatial=128, channels=(4, 32, 64, 128, 256, 256), slope=0.3)
METRIC = "conv3d fwd+bwd TFLOP/s and samples/s at 4x128^3, % of GB300 BF16 tensor peak"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def op_table(n, spatial, channels):
    """Every conv op of one step: (key, kind, layer, flops)."""
    ops = []
    s = spatial
    for l in range(len(channels) - 1):
        f = flops_mod.conv_flops(n, channels[l], channels[l + 1], s ** 3)
        ops.append((f"fwd{l + 1}", "fwd", l, f))
        ops.append((f"wgrad{l + 1}", "wgrad", l, f))
        if l > 0:
            ops.append((f"dgrad{l + 1}", "dgrad", l, f))
        s //= 2
    return ops


def csrc_hash():
    h = hashlib.sha1()
    d = os.path.join(ROOT, "cnn_conv3d_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:12]


def traffic_for(key):
    """DRAM bytes per launch of `key` from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = csrc_hash()
    with open(p) as f:
        for line in f:
            t = line.split()
            if len(t) >= 3 and not line.startswith("#") and t[0] == key and t[2] == cur:
                return float(t[1])
    return None


class Clocks:
    """Samples nvidia-smi every 50 ms from the warm-up to the end of the timed
    and end-to-end regions."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{index}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                t = [x.strip() for x in line.split(",")]
                if len(t) < 9:
                    continue
                try:
                    sm.append(float(t[1]))
                    smax.append(float(t[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, t[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- CPU (oracle) leg

def cpu_sample_step(n_threads=None, budget_s=20.0):
    """Times the fp64 oracle on a bounded sample of the step: every conv op of
    the stack evaluated on a slab of one sample (N=1, a few planes of the
    layer's volume), converted to a rate per op; the step's conv FLOPs divided
    by the summed per-op times gives the oracle's TFLOP/s on this workload."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(0)
    ch, s = WORKLOAD["channels"], WORKLOAD["spatial"]
    ops = op_table(WORKLOAD["n"], s, ch)
    per_op_budget = budget_s / len(ops)
    est_time, sampled = 0.0, []
    for key, kind, l, f in ops:
        ci, co = ch[l], ch[l + 1]
        sp = s >> l
        # slab of `planes` planes of one sample; grow until the op takes ~per_op_budget/4
        planes = 1
        while True:
            x = rng.normal(size=(1, planes, sp, sp, ci))
            w = rng.normal(size=(co, 3, 3, 3, ci))
            dz = rng.normal(size=(1, planes, sp, sp, co))
            t0 = time.perf_counter()
            if kind == "fwd":
                oracle.conv3d_fwd(x, w)
            elif kind == "dgrad":
                oracle.conv3d_dgrad(dz, w)
            else:
                oracle.conv3d_wgrad(x, dz)
            dt = time.perf_counter() - t0
            if dt > per_op_budget / 4 or planes >= sp:
                break
            planes = min(sp, planes * 2)
        sflops = 2.0 * co * ci * 27 * planes * sp * sp
        rate = sflops / dt
        est_time += f / rate
        sampled.append(f"{key}:{planes}x{sp}^2")
    total = sum(o[3] for o in ops)
    return total / est_time / 1e12, sampled


def max_over_ranks(value, world, device=None):
    """Largest value of `value` over all ranks (each rank times its own replica;
    the job takes as long as the slowest).  Identity on one rank."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank, world, max_ms):
    """Throughput of the whole job: every rank's work over the slowest rank's time."""
    return world * work_per_rank / (max_ms * 1e-3)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------------------- GPU leg

def run_ours(args, rank, world, local_rank):
    import torch
    from cnn_conv3d_gb300 import build
    build.build()
    from cnn_conv3d_gb300 import cfconv as cf
    from cnn_conv3d_gb300.stack import CosmoStack

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    n, s, ch = WORKLOAD["n"], WORKLOAD["spatial"], WORKLOAD["channels"]
    inp = synthdata.stack_inputs(n, s, ch, seed=20260003 + rank)
    st = CosmoStack(n, s, ch, WORKLOAD["slope"], device=str(dev))
    st.load(inp["x"], inp["w"], inp["b"])
    dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).to(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    ops = op_table(n, s, ch)
    total_flops = sum(o[3] for o in ops)

    # instrumented step: events around the step on the main stream and around
    # every op on the stream it is launched on (the weight gradients run on
    # the stack's second stream, joined before the step's end event); serial:
    # all ops on one stream, so that each op's events time it alone
    def step_with_events(evs, serial=False):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st.forward(stream, evs)
        st.backward(dy, stream, evs, serial)
        e1.record(stream)
        return e0, e1

    clk = Clocks(local_rank).__enter__()
    for _ in range(args.warmup):
        st.step(dy, stream)
    torch.cuda.synchronize(dev)
    if cf.cf_last_device_status(stream) != cf.CF_OK:
        raise RuntimeError("device status word set during warm-up")
    # per-op durations of each op alone: instrumented serial eager steps,
    # outside the timed region; they pick the dominant op
    inst = {}
    for _ in range(3):
        flush.zero_()
        evs = []
        step_with_events(evs, serial=True)
        torch.cuda.synchronize(dev)
        for k, e0, e1 in evs:
            inst.setdefault(k, []).append(e0.elapsed_time(e1))
    conv_keys = {o[0] for o in ops}
    dom = max((k for k in inst if k in conv_keys), key=lambda k: float(np.mean(inst[k])))
    # the timed steps replay a CUDA graph of the step with event nodes around
    # the dominant op only (a node per op would cost the step ~0.1 ms); a torch
    # without graph-recordable events times eager steps
    graph_evs, graph = [], None
    try:
        graph = st.capture(dy, graph_evs, keys={dom})
    except TypeError:
        graph, graph_evs = None, []
    if graph is not None:
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    step_ms, per_op = [], {}
    if True:
        for _ in range(args.steps):
            flush.zero_()  # evict L2 between steps (outside the timed events)
            if graph is not None:
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record(stream)
                graph.replay()
                s1.record(stream)
                evs = graph_evs
            else:
                evs = []
                s0, s1 = step_with_events(evs)
            torch.cuda.synchronize(dev)
            step_ms.append(s0.elapsed_time(s1))
            for k, e0, e1 in evs:
                per_op.setdefault(k, []).append(e0.elapsed_time(e1))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if cf.cf_last_device_status(stream) != cf.CF_OK:
        raise RuntimeError("device status word set during the timed steps")
    ms = max_over_ranks(float(np.mean(step_ms)), world, dev)

    # end-to-end through host buffers: H2D of the step inputs (pinned), the
    # step, D2H of its results (all weight and bias gradients)
    e2e = None
    if not args.no_e2e:
        x_host = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
        dy_host = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).pin_memory()
        dw_host = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in st.dw]
        db_host = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in st.db]
        h2d = x_host.numel() * 2 + dy_host.numel() * 2
        d2h = sum(t.numel() * 4 for t in dw_host) + sum(t.numel() * 4 for t in db_host)

        # the public host-buffer step: the input goes over per sample, each
        # sample's leading blocks starting as it lands; each dW / db leaves as
        # soon as it is final (a CUDA graph of it when the step is graphed)
        host = (x_host, dy_host, dw_host, db_host)
        st.step_host(*host, stream=stream)
        torch.cuda.synchronize(dev)
        e2e_graph = None
        if graph is not None:
            try:
                e2e_graph = st.capture(None, host=host)
            except RuntimeError:
                e2e_graph = None

        def e2e_step():
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                st.step_host(*host, stream=stream)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        e_ms = []
        for _ in range(args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            e_ms.append(e0.elapsed_time(e1))
        em = max_over_ranks(float(np.mean(e_ms)), world, dev)
        e2e = {"value": round(whole_job_rate(total_flops, world, em) / 1e12, 3), "unit": "TFLOP/s",
               "ms_per_step": round(em, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "CosmoStack.step_host (pinned host buffers; input per sample overlapped with the leading "
                      "blocks, gradients copied out as each is final)"
                      + (", CUDA graph" if e2e_graph is not None else ", eager")}

    clk.__exit__(None, None, None)
    # dominant conv op (largest mean duration in the instrumented steps), its
    # duration measured in the timed steps
    op_ms = {k: float(np.mean(v)) for k, v in inst.items()}
    conv_ops = {o[0]: o for o in ops}
    op_ms[dom] = float(np.mean(per_op[dom]))
    pk = peaks()
    dom_flops = conv_ops[dom][3]
    achieved = dom_flops / (op_ms[dom] * 1e-3) / 1e12
    tr = traffic_for(dom)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2),
                "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16_tflops_sustained"], 4), "traffic": tr,
                "peak_kind": f"bf16 sustained ({pk['source']})"}

    value = whole_job_rate(total_flops, world, ms) / 1e12
    res = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "samples_per_s": round(whole_job_rate(n, world, ms), 1),
        "pct_of_bf16_peak": {"measured_burst": round(100 * value / world / pk["bf16_tflops"], 2),
                             "measured_sustained": round(100 * value / world / pk["bf16_tflops_sustained"], 2),
                             "nominal_2250": round(100 * value / world / 2250.0, 2)},
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "cosmoflow 5-block conv3d stack fwd+bwd, N=8 x 4x128^3 bf16, "
                               "C_out 32/64/128/256/256, bias+leaky-ReLU(0.3)+2x2x2 max-pool",
                   "flops_per_step": total_flops, "flop_convention": "executed (layer-1 dgrad skipped)",
                   "l2": "flushed between timed steps (write of 2x L2 outside the timed events)",
                   "execution": ("CUDA graph of the step" if graph is not None else "eager launches")
                                 + ", weight gradients on a second stream",
                   "parallelism": f"replicas x{world}"},
        "per_op_ms": {k: round(v, 4) for k, v in sorted(op_ms.items())},
        "per_op_source": "each op alone (instrumented serial eager steps before the timed ones); "
                         "the dominant op's from the timed steps",
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * st.launches_per_step(),
        "clocks": clk.summary(),
        "csrc": csrc_hash(),
    }
    return res


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the reference arm is the fp64 oracle on the host cores; rank 0 only
        if rank != 0:
            return 0
        import oracle
        oracle.build()
        vals = []
        for _ in range(args.warmup):
            cpu_sample_step(budget_s=4.0)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            v, sample = cpu_sample_step(budget_s=8.0)
            vals.append(v)
        wall = time.perf_counter() - t0
        v = float(np.mean(vals))
        total = sum(o[3] for o in op_table(WORKLOAD["n"], WORKLOAD["spatial"], WORKLOAD["channels"]))
        out = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
               "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": round(total / (v * 1e12) * 1e3, 1),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic",
               "config": {"workload": "cosmoflow 5-block conv3d stack fwd+bwd, N=8 x 4x128^3 (oracle on slabs)"},
               "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": "each conv op on a slab of one sample: " + ", ".join(sample)},
               "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
               "wall_s": round(wall, 1)}
        print(json.dumps(out))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            v, sample = cpu_sample_step(budget_s=15.0)
            res["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                   "sample": "fp64 oracle, each conv op of the step on a slab of one sample: "
                                             + ", ".join(sample)}
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
