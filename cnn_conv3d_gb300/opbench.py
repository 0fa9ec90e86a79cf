"""Per-operation benchmark of the conv3d library (single-layer sweep).

python -m cnn_conv3d_gb300.opbench [--ops fwd,dgrad,wgrad] [--shapes S1,S2,...]
        [--n-scale F] [--pool] [--routed] [--warmup W] [--iters K] [--json]

Shapes S1..S5 are the single-layer sweep (C_in -> C_out, spatial^3, N):
S1 4->32 @128^3 N=8, S2 32->64 @64^3 N=16, S3 64->128 @32^3 N=32,
S4 128->256 @16^3 N=64, S5 256->256 @8^3 N=128 (bf16 N(0,1) activations,
He-normal filters).  A custom shape is "ci:co:spatial:n".  Each op is timed
with CUDA events on the current stream after warm-up, with L2 flushed
between timed launches (outside the events); the FLOP count is 2 * C_out *
C_in * 27 * N * spatial^3 per op.  Reports TFLOP/s, the fraction of the
measured bf16 peak (burst: each op is timed alone), and the minimum-HBM-byte
rate.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SWEEP = {"S1": (4, 32, 128, 8), "S2": (32, 64, 64, 16), "S3": (64, 128, 32, 32), "S4": (128, 256, 16, 64),
         "S5": (256, 256, 8, 128)}


def parse_shape(s):
    if s in SWEEP:
        return s, SWEEP[s]
    ci, co, sp, n = (int(t) for t in s.split(":"))
    return s, (ci, co, sp, n)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--ops", default="fwd,dgrad,wgrad")
    ap.add_argument("--shapes", default="S1,S2,S3,S4,S5")
    ap.add_argument("--n-scale", type=float, default=1.0)
    ap.add_argument("--pool", action="store_true", help="forward with the fused bias/LReLU/max-pool epilogue")
    ap.add_argument("--routed", action="store_true",
                    help="wgrad from the pooled gradient + argmax codes (the fused max-pool backward)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--iters", type=int, default=10)
    ap.add_argument("--json", action="store_true")
    a = ap.parse_args(argv)

    import torch
    from cnn_conv3d_gb300 import build
    build.build()
    from cnn_conv3d_gb300 import cfconv as cf

    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak = json.load(open(pk_path))["bf16_tflops"] if os.path.exists(pk_path) else 1900.0
    hbm = json.load(open(pk_path))["hbm_gbs"] if os.path.exists(pk_path) else 6800.0
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    rng = np.random.default_rng(0)
    out = []
    for name in a.shapes.split(","):
        label, (ci, co, sp, n) = parse_shape(name)
        n = max(1, int(round(n * a.n_scale)))
        desc = cf.cf_conv_desc(n, sp, sp, sp, ci, co)
        x = torch.randn((n, sp, sp, sp, ci), device=dev).to(torch.bfloat16)
        w = (torch.randn((co, 3, 3, 3, ci), device=dev) * np.sqrt(2.0 / (27 * ci))).to(torch.bfloat16)
        dz = torch.randn((n, sp, sp, sp, co), device=dev).to(torch.bfloat16)
        b = torch.zeros((co,), device=dev)
        ws_n = max(cf.cf_workspace_size(cf.CF_OP_WGRAD, desc), cf.cf_workspace_size(cf.CF_OP_DGRAD, desc),
                   cf.cf_workspace_size(cf.CF_OP_WGRAD_ROUTED, desc) if a.routed else 0, 256)
        ws = torch.empty((ws_n,), dtype=torch.uint8, device=dev)
        flops = 2.0 * co * ci * 27 * n * sp ** 3
        for op in a.ops.split(","):
            if op == "fwd":
                if a.pool:
                    y = torch.empty((n, sp // 2, sp // 2, sp // 2, co), dtype=torch.bfloat16, device=dev)
                    idx = torch.empty(y.shape, dtype=torch.uint8, device=dev)
                    fn = lambda: cf.cf_conv3d_fwd(desc, x, w, (b, 0.3, idx), y, None, 0, stream)
                    nbytes = x.numel() * 2 + w.numel() * 2 + y.numel() * 3
                else:
                    y = torch.empty((n, sp, sp, sp, co), dtype=torch.bfloat16, device=dev)
                    fn = lambda: cf.cf_conv3d_fwd(desc, x, w, None, y, None, 0, stream)
                    nbytes = x.numel() * 2 + w.numel() * 2 + y.numel() * 2
            elif op == "dgrad":
                if ci % 16 or co % 32:
                    continue
                dx = torch.empty_like(x)
                fn = lambda: cf.cf_conv3d_dgrad(desc, dz, None, w, x, 0.3, dx, ws, ws_n, stream)
                nbytes = dz.numel() * 2 + w.numel() * 2 + 2 * dx.numel() * 2
            elif op == "wgrad":
                dw = torch.empty((co, 3, 3, 3, ci), dtype=torch.float32, device=dev)
                if a.routed:
                    gp = torch.randn((n, sp // 2, sp // 2, sp // 2, co), device=dev).to(torch.bfloat16)
                    gi = torch.randint(0, 8, gp.shape, dtype=torch.uint8, device=dev)
                    fn = lambda: cf.cf_conv3d_wgrad(desc, x, gp, gi, dw, 0, ws, ws_n, stream)
                    nbytes = x.numel() * 2 + gp.numel() * 3 + dw.numel() * 4
                else:
                    fn = lambda: cf.cf_conv3d_wgrad(desc, x, dz, None, dw, 0, ws, ws_n, stream)
                    nbytes = x.numel() * 2 + dz.numel() * 2 + dw.numel() * 4
            elif op == "poolbwd":
                # the block's pool / leaky-ReLU backward (routed dZ and bias gradient)
                dy = torch.randn((n, sp // 2, sp // 2, sp // 2, co), device=dev).to(torch.bfloat16)
                yp = torch.randn_like(dy)
                ip = torch.randint(0, 8, dy.shape, dtype=torch.uint8, device=dev)
                dzz = torch.empty((n, sp, sp, sp, co), dtype=torch.bfloat16, device=dev)
                dbb = torch.empty((co,), dtype=torch.float32, device=dev)
                pws = max(cf.cf_workspace_size(cf.CF_OP_POOL_BWD, desc), 256)
                pw = torch.empty((pws,), dtype=torch.uint8, device=dev)
                fn = lambda: cf.cf_bias_lrelu_pool_bwd(n, sp, sp, sp, co, dy, yp, ip, 0.3, dzz, None, dbb, pw, pws,
                                                       stream)
                nbytes = dy.numel() * 5 + dzz.numel() * 2
                flops = 0.0
            else:
                raise SystemExit(f"unknown op {op}")
            for _ in range(a.warmup):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(a.iters):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            if cf.cf_last_device_status() != cf.CF_OK:
                raise SystemExit("device status word set")
            ms = float(np.median(ts))
            tf = flops / (ms * 1e-3) / 1e12
            flops = 2.0 * co * ci * 27 * n * sp ** 3
            tag = "+pool" if (op == "fwd" and a.pool) else ("+routed" if (op == "wgrad" and a.routed) else "")
            rec = {"shape": label, "op": op + tag, "n": n, "c_in": ci,
                   "c_out": co, "spatial": sp, "ms": round(ms, 4), "tflops": round(tf, 1),
                   "frac_bf16_peak": round(tf / peak, 3), "min_bytes_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                   "frac_hbm": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 3)}
            out.append(rec)
            if a.json:
                print(json.dumps(rec))
            else:
                print(f"{label:>14} {rec['op']:>9} N={n:<4d} {ms:8.4f} ms {tf:8.1f} TFLOP/s "
                      f"({100 * rec['frac_bf16_peak']:5.1f}% of bf16 peak)  {rec['min_bytes_gbs']:8.1f} GB/s min")
    return out


if __name__ == "__main__":
    main()
