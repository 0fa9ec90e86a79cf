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
                       [--sustain-s S] [--no-extra] [--no-cpu-baseline] [--no-e2e]
Prints one JSON line on rank 0.  Besides the K timed steps (the headline,
a burst: each step timed alone after an L2 flush), the line carries a
sustained figure (graph replays back to back for at least S seconds, the
clock and power state a training loop runs in), the other configurations
(the N=4 five-block forward, the 1 x 4 x 512^3 block pair forward +
backward, the single-layer sweep) as extra keys, and the fp64 oracle timed on
the host cores on one seeded sample of the workload.  With N > 1 (torchrun) every rank runs an
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
WORKLOAD_SEED = 20260003
CONFIG2 = dict(n=4, spatial=128, channels=(4, 32, 64, 128, 256, 256), seed=20260002)
CONFIG4 = dict(n=1, spatial=512, channels=(4, 32, 64), seed=20260004)
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
    ap.add_argument("--no-extra", action="store_true", help="skip the other configurations")
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back step replays for the sustained figure (0: skip)")
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

    def __init__(self, index, tag="main"):
        import tempfile
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"cfconv3d_clocks_{os.getpid()}_{index}_{tag}.csv")

    def __enter__(self):
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
            self.proc = False  # samples kept in self.path until summary()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        power = []
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
                    power.append(float(t[3]))
                except ValueError:
                    continue
                for nm, v in zip(names, t[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------- CPU (oracle) leg

def cpu_oracle_sample(inp, sample=0, crop=None):
    """The fp64 oracle as it stands, timed on one sample of the seeded
    workload: the five-block forward chain and the backward chain (pool /
    leaky-ReLU backward, backward-weight of every block, backward-data of
    blocks 2..5) in mirrored mode.  crop: run the chain on the leading crop^3
    corner of the sample instead of its whole 128^3 volume (the same
    computation on 1/(128/crop)^3 of the voxels).  Returns (seconds, conv
    FLOPs of that sample or crop in the step's convention)."""
    import oracle
    oracle.build()
    ch, s = WORKLOAD["channels"], WORKLOAD["spatial"]
    c = s if crop is None else crop
    top = c >> (len(ch) - 1)
    f64 = oracle.bf16_bits_to_f64
    x = f64(inp["x"][sample:sample + 1, :c, :c, :c])
    ws = [f64(w) for w in inp["w"]]
    bs = [b.astype(np.float64) for b in inp["b"]]
    dy = f64(inp["dy"][sample:sample + 1, :top, :top, :top])
    t0 = time.perf_counter()
    xs, _, ys, idxs = oracle.stack_fwd(x, ws, bs, WORKLOAD["slope"], mirrored=True)
    oracle.stack_bwd(xs, ys, idxs, ws, dy, WORKLOAD["slope"], mirrored=True)
    dt = time.perf_counter() - t0
    return dt, sum(o[3] for o in op_table(1, c, ch))


def cpu_sample_step(budget_s=20.0):
    """Times the fp64 oracle on slabs: every conv op of the step on a few
    planes of one sample's layer volume (random N(0,1) data of the layer's
    shape), converted to a rate per op; the step's conv FLOPs divided by the
    summed per-op times gives the oracle's TFLOP/s.  Used for the one-core
    figure, where a whole sample would take minutes."""
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
        rate = 2.0 * co * ci * 27 * planes * sp * sp / dt
        est_time += f / rate
        sampled.append(f"{key}:{planes}x{sp}^2")
    total = sum(o[3] for o in ops)
    return total / est_time / 1e12, sampled


def cpu_one_core_rate(budget_s=8.0):
    """cpu_sample_step on one host core (a child process with OMP_NUM_THREADS=1)."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    code = ("import json, bench; v, s = bench.cpu_sample_step(budget_s=%r); print(json.dumps([v, s]))" % budget_s)
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                             timeout=300)
        v, sampled = json.loads(out.stdout.strip().splitlines()[-1])
        return v, sampled
    except Exception as e:  # noqa: BLE001 -- reported, not fatal
        return None, [f"unavailable: {type(e).__name__}"]


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


def stack_op_bytes(key, n, spatial, channels):
    """Minimum HBM bytes of op `key` ("fwd3", "wgrad1", ...) of the stack step
    (the first block's weight gradient is routed: pooled gradient + codes)."""
    kind = key.rstrip("0123456789")
    l = int(key[len(kind):]) - 1
    s = spatial >> l
    routed = kind == "wgrad" and l == 0 and channels[0] in (1, 4)
    return flops_mod.op_min_bytes(kind, n, s, channels[l], channels[l + 1], routed=routed)


# --------------------------------------------------------------------------- GPU leg

def _timed_replays(torch, graph, stream, flush, steps):
    """Mean ms of `steps` replays, each timed alone (L2 flushed before it,
    outside its events; the host waits for each)."""
    out = []
    for _ in range(steps):
        flush.zero_()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        graph.replay()
        s1.record(stream)
        torch.cuda.synchronize()
        out.append(s0.elapsed_time(s1))
    return float(np.mean(out))


def run_extra_configs(torch, dev, stream, flush, pk):
    """The other configurations, each its own graph: the N=4 five-block forward,
    the 1 x 4 x 512^3 block pair forward + backward, and the single-layer sweep
    (each op alone).  Throughput only; their parity is in the full-size tests."""
    from cnn_conv3d_gb300 import cfconv as cf
    from cnn_conv3d_gb300 import opbench
    from cnn_conv3d_gb300.stack import CosmoStack
    out = {}
    for name, cfg, bwd in (("config2_fwd_n4_128", CONFIG2, False), ("config4_pair_n1_512", CONFIG4, True)):
        inp = synthdata.stack_inputs(cfg["n"], cfg["spatial"], cfg["channels"], seed=cfg["seed"], with_dy=bwd)
        st = CosmoStack(cfg["n"], cfg["spatial"], cfg["channels"], WORKLOAD["slope"], device=str(dev), backward=bwd)
        st.load(inp["x"], inp["w"], inp["b"])
        dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).to(dev) if bwd else None
        for _ in range(2):
            st.step(dy, stream)
        g = st.capture(dy)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        ms = _timed_replays(torch, g, stream, flush, 5)
        if cf.cf_last_device_status(stream) != cf.CF_OK:
            raise RuntimeError(f"device status word set in {name}")
        fl = flops_mod.stack_flops(cfg["n"], cfg["spatial"], cfg["channels"], backward=bwd)
        tf = fl / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "tflops": round(tf, 2), "samples_per_s": round(cfg["n"] / (ms * 1e-3), 1),
                     "flops": fl, "pct_of_bf16_peak": {"nominal_2250": round(100 * tf / 2250.0, 2),
                                                       "measured_burst": round(100 * tf / pk["bf16_tflops"], 2)},
                     "what": ("five-block forward, N=4 x 4x128^3" if not bwd else
                              "blocks 4->32->64 forward + backward, N=1 x 4x512^3")}
        del g, st
        torch.cuda.empty_cache()
    import contextlib
    import io
    with contextlib.redirect_stdout(io.StringIO()):
        recs = opbench.main(["--json", "--warmup", "3", "--iters", "10"])
    out["config5_sweep"] = {f"{r['shape']}_{r['op']}": {"ms": r["ms"], "tflops": r["tflops"],
                                                       "frac_bf16_burst": r["frac_bf16_peak"],
                                                       "frac_hbm_min_bytes": r["frac_hbm"]} for r in recs}
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    from cnn_conv3d_gb300 import build
    build.build()
    from cnn_conv3d_gb300 import cfconv as cf
    from cnn_conv3d_gb300.stack import CosmoStack

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    n, s, ch = WORKLOAD["n"], WORKLOAD["spatial"], WORKLOAD["channels"]
    inp = synthdata.stack_inputs(n, s, ch, seed=WORKLOAD_SEED + rank)
    st = CosmoStack(n, s, ch, WORKLOAD["slope"], device=str(dev))
    st.load(inp["x"], inp["w"], inp["b"])
    dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).to(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    ops = op_table(n, s, ch)
    total_flops = sum(o[3] for o in ops)
    pk = peaks()

    # instrumented step: events around the step on the main stream and around
    # every op on the stream it is launched on (the weight gradients run on
    # the stack's second stream, joined before the step's end event); serial:
    # all ops on one stream, so that each op's events time it alone
    def step_with_events(evs, serial=False):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st.forward(stream, evs, serial=serial)
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
    graphed = graph is not None
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
    clk.__exit__(None, None, None)
    clocks_main = clk.summary()

    # sustained: the step replayed back to back (an L2 flush before each, no
    # host wait in between) for at least --sustain-s seconds, with its own
    # clock record: the clock and power state of a training loop
    sustained = None
    if args.sustain_s > 0 and graph is not None:
        reps = max(10, int(np.ceil(args.sustain_s / (ms * 1e-3))))
        ck = Clocks(local_rank, "sustained").__enter__()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        t0 = time.perf_counter()
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        ck.__exit__(None, None, None)
        if cf.cf_last_device_status(stream) != cf.CF_OK:
            raise RuntimeError("device status word set during the sustained replays")
        sms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in evs])), world, dev)
        sv = whole_job_rate(total_flops, world, sms) / 1e12
        cks = ck.summary()
        sustained = {"value": round(sv, 3), "unit": "TFLOP/s", "ms_per_step": round(sms, 4), "steps": reps,
                     "seconds": round(wall, 2),
                     "pct_of_bf16_peak": {"nominal_2250": round(100 * sv / world / 2250.0, 2),
                                          "measured_sustained": round(
                                              100 * sv / world / pk["bf16_tflops_sustained"], 2)},
                     "clocks": cks,
                     "ms_x_mhz": round(sms * cks["sm_mhz"], 1) if cks.get("sm_mhz") else None}

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

        def timed(fn, steps):
            out = []
            for _ in range(steps):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                out.append(e0.elapsed_time(e1))
            return out

        # (1) the public host-buffer step on its own: the input goes over per
        # sample, each sample's leading blocks starting as it lands; each dW / db
        # leaves as soon as it is final (a CUDA graph of it when the step is graphed)
        host = (x_host, dy_host, dw_host, db_host)
        st.step_host(*host, stream=stream)
        torch.cuda.synchronize(dev)
        e2e_graph = None
        if graph is not None:
            try:
                e2e_graph = st.capture(None, host=host)
            except RuntimeError:
                e2e_graph = None

        def single_step():
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                st.step_host(*host, stream=stream)
        for _ in range(2):
            single_step()
        torch.cuda.synchronize(dev)
        single_ms = max_over_ranks(float(np.mean(timed(single_step, args.steps))), world, dev)
        del e2e_graph

        # (2) the training-loop form: double-buffered input, each step copying the
        # next batch in while it computes on the one the previous step brought
        # (same bytes in and out per step); the pair of graphs alternates
        pipe = None
        if graph is not None:
            try:
                pipe = st.capture_pipelined(*host)
            except RuntimeError:
                pipe = None
        st.prefetch_host(x_host, dy_host, stream=stream)
        turn = [0]

        def pipelined_step():
            if pipe is not None:
                pipe[turn[0]].replay()
                turn[0] ^= 1
            else:
                st.step_host_pipelined(*host, stream=stream)
        for _ in range(4):
            pipelined_step()
        torch.cuda.synchronize(dev)
        em = max_over_ranks(float(np.mean(timed(pipelined_step, args.steps))), world, dev)
        e2e = {"value": round(whole_job_rate(total_flops, world, em) / 1e12, 3), "unit": "TFLOP/s",
               "ms_per_step": round(em, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "CosmoStack.step_host_pipelined (pinned host buffers; double-buffered input, the next "
                      "batch copied in during this step; gradients copied out as each is final)"
                      + (", CUDA graphs" if pipe is not None else ", eager"),
               "single_step": {"ms_per_step": round(single_ms, 4),
                               "value": round(whole_job_rate(total_flops, world, single_ms) / 1e12, 3),
                               "api": "CosmoStack.step_host (input per sample overlapped with the leading "
                                      "blocks of the same step)"}}
        del pipe

    extra = None
    if not args.no_extra and rank == 0:
        del graph
        graph = None
        extra = run_extra_configs(torch, dev, stream, flush, pk)

    # dominant conv op (largest mean duration in the instrumented steps), its
    # duration measured in the timed steps (a burst: each step timed alone at
    # the clocks of a short run, so the burst peak is the denominator)
    op_ms = {k: float(np.mean(v)) for k, v in inst.items()}
    conv_ops = {o[0]: o for o in ops}
    if dom in per_op:
        op_ms[dom] = float(np.mean(per_op[dom]))
    dom_flops = conv_ops[dom][3]
    achieved = dom_flops / (op_ms[dom] * 1e-3) / 1e12
    dom_bytes = stack_op_bytes(dom, n, s, ch)
    tr = traffic_for(dom)
    gbs = dom_bytes / (op_ms[dom] * 1e-3) / 1e9
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": tr,
                "peak_kind": f"bf16 burst ({pk['source']}): the timed steps are a burst",
                "flops_per_launch": dom_flops, "algorithmic_bytes": dom_bytes,
                "hbm": {"achieved_gbs": round(gbs, 1), "peak_gbs": pk["hbm_gbs"],
                        "frac": round(gbs / pk["hbm_gbs"], 4),
                        "traffic_gbs": round(tr / (op_ms[dom] * 1e-3) / 1e9, 1) if tr else None},
                # the launch duration above is the one inside the timed steps, where
                # other kernels of the step may share the GPU with it; the same
                # kernel alone (the instrumented serial steps) for comparison
                "alone": {"ms": round(float(np.mean(inst[dom])), 4),
                          "achieved": round(dom_flops / (float(np.mean(inst[dom])) * 1e-3) / 1e12, 2),
                          "frac": round(dom_flops / (float(np.mean(inst[dom])) * 1e-3) / 1e12 / pk["bf16_tflops"], 4)},
                "timed_ms": round(op_ms[dom], 4)}

    value = whole_job_rate(total_flops, world, ms) / 1e12
    res = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "samples_per_s": round(whole_job_rate(n, world, ms), 1),
        "pct_of_bf16_peak": {"nominal_2250": round(100 * value / world / 2250.0, 2),
                             "measured_burst": round(100 * value / world / pk["bf16_tflops"], 2),
                             "measured_sustained": round(100 * value / world / pk["bf16_tflops_sustained"], 2)},
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "cosmoflow 5-block conv3d stack fwd+bwd, N=8 x 4x128^3 bf16, "
                               "C_out 32/64/128/256/256, bias+leaky-ReLU(0.3)+2x2x2 max-pool",
                   "flops_per_step": total_flops, "flop_convention": "executed (layer-1 dgrad skipped)",
                   "l2": "flushed between timed steps (write of 2x L2 outside the timed events)",
                   "execution": ("CUDA graph of the step" if graphed else "eager launches")
                                 + ", weight gradients on a second stream",
                   "parallelism": f"replicas x{world}"},
        "per_op_ms": {k: round(v, 4) for k, v in sorted(op_ms.items())},
        "per_op_source": "each op alone (instrumented serial eager steps before the timed ones); "
                         "the dominant op's from the timed steps",
        "roofline": roofline,
        "sustained": sustained,
        "e2e": e2e,
        "gpu_launches": args.steps * st.launches_per_step(),
        "clocks": clocks_main,
        "csrc": csrc_hash(),
    }
    if extra is not None:
        res["other_configs"] = extra
    return res, inp


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the reference arm is the fp64 oracle on the host cores; rank 0 only.
        # Each step: one sample of the seeded workload through the oracle's
        # forward and backward chains (a bounded sample: 1 of the 8 samples)
        if rank != 0:
            return 0
        import oracle
        oracle.build()
        inp = synthdata.stack_inputs(WORKLOAD["n"], WORKLOAD["spatial"], WORKLOAD["channels"], seed=WORKLOAD_SEED)
        crop = 64
        for k in range(args.warmup):
            cpu_oracle_sample(inp, sample=k % WORKLOAD["n"], crop=32)
        t0 = time.perf_counter()
        secs, fl = [], 0
        for k in range(args.steps):
            dt, f = cpu_oracle_sample(inp, sample=k % WORKLOAD["n"], crop=crop)
            secs.append(dt)
            fl = f
        wall = time.perf_counter() - t0
        v = fl / float(np.mean(secs)) / 1e12
        total = sum(o[3] for o in op_table(WORKLOAD["n"], WORKLOAD["spatial"], WORKLOAD["channels"]))
        out = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
               "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": round(total / (v * 1e12) * 1e3, 1),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic",
               "config": {"workload": "cosmoflow 5-block conv3d stack fwd+bwd, N=8 x 4x128^3 (the fp64 oracle; "
                                      "each step a 64^3 crop of one of the 8 seeded samples, ms_per_step "
                                      "scaled to the batch at the measured rate)"},
               "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": "per step the 64^3 corner of one seeded sample (of 8) through the full "
                                          "five-block forward and backward chains in fp64, mirrored bf16 "
                                          "rounding (1/512 of the step's conv FLOPs)"},
               "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
               "wall_s": round(wall, 1)}
        print(json.dumps(out))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res, inp = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            dt, fl = cpu_oracle_sample(inp, sample=0)
            v1, sampled1 = cpu_one_core_rate()
            res["cpu_baseline"] = {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(),
                                   "kind": "oracle", "seconds": round(dt, 2),
                                   "sample": "sample 0 of the 8 seeded samples: the fp64 oracle's full five-block "
                                             "forward and backward chains (mirrored bf16 rounding)",
                                   "one_core": {"value": round(v1, 6) if v1 else None, "unit": "TFLOP/s",
                                                "sample": "each conv op on a slab of one sample: "
                                                          + ", ".join(sampled1)}}
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
