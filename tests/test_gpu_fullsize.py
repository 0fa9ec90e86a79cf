"""Parity at the full sizes of the benchmark configurations, in the launch
configuration bench.py times (the CosmoStack sequence of C-ABI calls).

The fp64 oracle evaluates output elements on the GPU's own bf16 input of
that layer, so every check isolates one kernel: sampled activations and
input gradients (its point routines), and every element of the weight
gradients of the benchmark stack (its per-tap matrix-product form, and for
the first block the routed sum over pooled voxels); the 512^3 pair and the
sweep check at least one weight-gradient element in every (64 output
channels x tap x 32 input channels) tile, 512 or more in all.  Tolerance as elsewhere: |err| <= 1e-2 * S per element
(S = sum of |product| terms) and relative L2 <= 5e-3 over the sample; argmax
codes bit-exact where the window's top-two gap exceeds the tolerance.

Configurations (sizes and seeds from synthdata):
  tiny block   1 x 1 x 16^3 -> 8 channels, pooled (checked in full)
  stack fwd    4 x (4 x 128^3), five blocks 32/64/128/256/256
  stack train  8 x (4 x 128^3), forward + backward (the benchmark workload)
  large pair   1 x (4 x 512^3), blocks 32, 64, forward + backward
  sweep        the five single-layer shapes, fwd / dgrad / wgrad
"""
import numpy as np
import pytest

import synthdata
from tests.gpu_util import assert_close, dev, dev_bf16, empty_bf16, tile_cover_pts

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SLOPE = 0.3


@pytest.fixture(scope="module")
def cf():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_conv3d_gb300 import build
    build.build()
    from cnn_conv3d_gb300 import cfconv
    return cfconv


def u16(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t):
    return (u16(t).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_pts(rng, shape, k):
    return np.stack([rng.integers(0, s, k) for s in shape], 1).astype(np.int64)


def check_pooled_block(oracle_mod, x16, w16, bias, y_gpu16, idx_gpu, rng, k, what):
    """Sampled pooled outputs (n, pd, ph, pw, co) of one block."""
    pts = rand_pts(rng, y_gpu16.shape, k)
    ry, ridx, S, gap = oracle_mod.block_fwd_pts(x16, w16, bias, SLOPE, pts)
    gy = (y_gpu16[tuple(pts.T)].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gi = idx_gpu[tuple(pts.T)]
    notie = gap > 1e-2 * S
    np.testing.assert_array_equal(gi[notie], ridx[notie], err_msg=what)
    assert_close(gy, ry, S, what)
    return int((~notie).sum())


def test_tiny_block_in_full(cf, oracle_mod):
    import torch
    inp = synthdata.tiny_block_inputs()
    y = empty_bf16((1, 8, 8, 8, 8), fill=float("nan"))
    idx = torch.full(y.shape, 255, dtype=torch.uint8, device="cuda")
    cf.cf_conv3d_fwd((1, 16, 16, 16, 1, 8), dev_bf16(inp["x"]), dev_bf16(inp["w"]),
                     (dev(inp["b"]), SLOPE, idx), y)
    x = oracle_mod.bf16_bits_to_f64(inp["x"])
    w = oracle_mod.bf16_bits_to_f64(inp["w"])
    z = oracle_mod.conv3d_fwd(x, w)
    S = oracle_mod.conv3d_fwd(np.abs(x), np.abs(w))
    ry, ridx = oracle_mod.pool_fwd(z, inp["b"].astype(np.float64), SLOPE)
    zw = z.reshape(1, 8, 2, 8, 2, 8, 2, 8).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(1, 8, 8, 8, 8, 8)
    sw = S.reshape(1, 8, 2, 8, 2, 8, 2, 8).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(1, 8, 8, 8, 8, 8)
    srt = np.sort(zw, -1)
    s_at = np.take_along_axis(sw, ridx[..., None].astype(np.int64), -1)[..., 0] + np.abs(inp["b"])
    notie = (srt[..., -1] - srt[..., -2]) > 1e-2 * s_at
    np.testing.assert_array_equal(idx.cpu().numpy()[notie], ridx[notie])
    assert_close(f64(y), ry, s_at, "tiny block")
    # the fp32 input before bf16 rounding: information only, must be close
    z32 = oracle_mod.conv3d_fwd(inp["x32"].astype(np.float64), w)
    y32, _ = oracle_mod.pool_fwd(z32, inp["b"].astype(np.float64), SLOPE)
    assert np.linalg.norm(f64(y) - y32) / np.linalg.norm(y32) < 2e-2


def _stack(cf, n, spatial, channels, seed, backward):
    import torch
    from cnn_conv3d_gb300.stack import CosmoStack
    inp = synthdata.stack_inputs(n, spatial, channels, seed=seed, with_dy=True)
    st = CosmoStack(n, spatial, channels, SLOPE, backward=backward)
    st.load(inp["x"], inp["w"], inp["b"])
    dy = dev_bf16(inp["dy"])
    st.step(dy)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == cf.CF_OK
    return st, inp, dy


def _check_forward(oracle_mod, st, inp, rng, k):
    for l in range(st.L):
        x16 = u16(st.block_input(l))
        check_pooled_block(oracle_mod, x16, inp["w"][l], inp["b"][l], u16(st.y[l]), st.idx[l].cpu().numpy(),
                           rng, k, f"block {l + 1} forward")


def _pool_bwd_checks(oracle_mod, g16, y16, idx, gdb, dz16, rng, what):
    """Bias gradient (oracle over slabs of the pooled tensor) and, when the
    dense dZ was written (dz16 not None), the routed dZ at sampled windows
    (oracle on the extracted windows)."""
    f = oracle_mod.bf16_bits_to_f64
    C = g16.shape[-1]
    db = np.zeros(C)
    sabs = np.zeros(C)
    for n in range(g16.shape[0]):
        for d0 in range(0, g16.shape[1], 8):
            sl = (slice(n, n + 1), slice(d0, d0 + 8))
            _, gp, part = oracle_mod.pool_bwd(f(g16[sl]), None if y16 is None else f(y16[sl]), idx[sl], SLOPE,
                                              want_dz=False)
            db += part
            sabs += np.abs(gp).reshape(-1, C).sum(0)
    assert_close(gdb, db, sabs, f"db {what}")
    if dz16 is None:
        return
    # K sampled windows as K one-channel 2x2x2 windows
    K = 2048
    pw = rand_pts(rng, g16.shape, K)
    n_, pd, ph, pw_, c = pw.T
    gw = f(g16[n_, pd, ph, pw_, c]).reshape(K, 1, 1, 1, 1)
    yw = None if y16 is None else f(y16[n_, pd, ph, pw_, c]).reshape(K, 1, 1, 1, 1)
    dzw, _, _ = oracle_mod.pool_bwd(gw, yw, idx[n_, pd, ph, pw_, c].reshape(K, 1, 1, 1, 1), SLOPE)
    for k in range(8):
        dd, dh, dw = k >> 2, (k >> 1) & 1, k & 1
        got = (dz16[n_, 2 * pd + dd, 2 * ph + dh, 2 * pw_ + dw, c].astype(np.uint32) << 16).view(np.float32)
        np.testing.assert_allclose(got, dzw[:, dd, dh, dw, 0], rtol=2 ** -8, atol=0, err_msg=f"dZ routing {what}")


def _check_dw_dense_full(oracle_mod, x16, dz16, gdw, what, slab=16):
    """The whole weight gradient of one layer, from the GPU's own bf16 input and
    dense dZ: the oracle's per-tap matrix-product form, sample by sample in
    d-slabs (neighbouring planes passed in)."""
    f = oracle_mod.bf16_bits_to_f64
    N, D = x16.shape[:2]
    ref = np.zeros(gdw.shape)
    S = np.zeros(gdw.shape)
    for n in range(N):
        for d0 in range(0, D, slab):
            d1 = min(D, d0 + slab)
            xs, dzs = f(x16[n:n + 1, d0:d1]), f(dz16[n:n + 1, d0:d1])
            below = f(x16[n:n + 1, d0 - 1]) if d0 > 0 else None
            above = f(x16[n:n + 1, d1]) if d1 < D else None
            ref += oracle_mod.conv3d_wgrad_mm(xs, dzs, below, above)
            S += oracle_mod.conv3d_wgrad_mm(np.abs(xs), np.abs(dzs), None if below is None else np.abs(below),
                                            None if above is None else np.abs(above))
    assert_close(gdw, ref, S, what)


def _all_filter_pts(c_out, c_in):
    return np.array([(co, t // 9, (t // 3) % 3, t % 3, ci) for co in range(c_out) for t in range(27)
                     for ci in range(c_in)], dtype=np.int64)


def _check_backward(oracle_mod, st, inp, dy, rng, k_dx, dw_full=True):
    """Every block: bias gradient (full), routed dZ at sampled windows, the
    weight gradient (every element when dw_full, else at least one element per
    split-K / accumulator tile and >= 512 in all), input gradient at k_dx
    sampled elements."""
    L = st.L
    f = oracle_mod.bf16_bits_to_f64
    for l in range(L - 1, -1, -1):
        # pool/LReLU backward: bias gradient and routed dZ
        g16 = u16(dy) if l == L - 1 else u16(st.g[l])
        y16 = u16(st.y[l]) if l == L - 1 else None
        idx = st.idx[l].cpu().numpy()
        dz16 = None if st.routed(l) else u16(st.dz[l])
        _pool_bwd_checks(oracle_mod, g16, y16, idx, st.db[l].cpu().numpy().astype(np.float64), dz16, rng,
                         f"block {l + 1}")
        x16 = u16(st.block_input(l))
        gdw = st.dw[l].cpu().numpy().astype(np.float64)
        co, ci = gdw.shape[0], gdw.shape[4]
        if dz16 is None:
            # routed weight gradient (the first block: g is already the pre-activation
            # gradient): every filter element, summed over the pooled voxels
            assert y16 is None
            pts = _all_filter_pts(co, ci) if dw_full else tile_cover_pts(rng, co, ci)
            ref, S = oracle_mod.conv3d_wgrad_routed_pts(x16, g16, idx, pts)
            assert_close(gdw[tuple(pts.T)], ref, S, f"dW{l + 1} (routed, {len(pts)} elements)")
            continue
        if dw_full:
            _check_dw_dense_full(oracle_mod, x16, dz16, gdw, f"dW{l + 1} (all elements)")
        else:
            pts = tile_cover_pts(rng, co, ci)
            ref, S = oracle_mod.conv3d_wgrad_pts(x16, dz16, pts)
            assert_close(gdw[tuple(pts.T)], ref, S, f"dW{l + 1} ({len(pts)} tile-covering elements)")
        if l > 0:
            # input gradient times the previous block's leaky-ReLU derivative
            pts = rand_pts(rng, x16.shape, k_dx)
            ref, S = oracle_mod.conv3d_dgrad_pts(dz16, inp["w"][l], pts)
            fac = np.where(f(x16[tuple(pts.T)]) > 0, 1.0, SLOPE)
            got = f(u16(st.g[l - 1])[tuple(pts.T)])
            assert_close(got, ref * fac, S * fac, f"dX{l + 1}")
        del dz16


def test_stack_forward_n4(cf, oracle_mod):
    st, inp, _ = _stack(cf, 4, 128, synthdata.STACK_CHANNELS, 20260002, backward=False)
    _check_forward(oracle_mod, st, inp, np.random.default_rng(2), 4096)


def test_stack_train_step_n8(cf, oracle_mod):
    st, inp, dy = _stack(cf, 8, 128, synthdata.STACK_CHANNELS, 20260003, backward=True)
    rng = np.random.default_rng(3)
    _check_forward(oracle_mod, st, inp, rng, 2048)
    _check_backward(oracle_mod, st, inp, dy, rng, k_dx=2048, dw_full=True)


def test_large_sample_pair_512(cf, oracle_mod):
    st, inp, dy = _stack(cf, 1, 512, (4, 32, 64), 20260004, backward=True)
    rng = np.random.default_rng(4)
    _check_forward(oracle_mod, st, inp, rng, 2048)
    _check_backward(oracle_mod, st, inp, dy, rng, k_dx=1024, dw_full=False)


@pytest.mark.parametrize("shape", list(synthdata.SWEEP_SHAPES))
def test_sweep_layer(cf, oracle_mod, shape):
    import torch
    ci, co, sp, n = shape
    inp = synthdata.sweep_inputs(ci, co, sp, n)
    desc = cf.cf_conv_desc(n, sp, sp, sp, ci, co)
    x, w, dz = dev_bf16(inp["x"]), dev_bf16(inp["w"]), dev_bf16(inp["dz"])
    rng = np.random.default_rng(ci * 1000 + co)
    y = empty_bf16((n, sp, sp, sp, co))
    cf.cf_conv3d_fwd(desc, x, w, None, y)
    pts = rand_pts(rng, y.shape, 2048)
    ref, S = oracle_mod.conv3d_fwd_pts(inp["x"], inp["w"], pts)
    assert_close(f64(y)[tuple(pts.T)], ref, S, f"sweep fwd {shape}")
    if ci % 16 == 0 and co % 32 == 0:
        ws = torch.empty((max(cf.cf_workspace_size(cf.CF_OP_DGRAD, desc), 256),), dtype=torch.uint8, device="cuda")
        dx = empty_bf16((n, sp, sp, sp, ci))
        cf.cf_conv3d_dgrad(desc, dz, None, w, None, SLOPE, dx, ws, ws.numel())
        pts = rand_pts(rng, dx.shape, 2048)
        ref, S = oracle_mod.conv3d_dgrad_pts(inp["dz"], inp["w"], pts)
        assert_close(f64(dx)[tuple(pts.T)], ref, S, f"sweep dgrad {shape}")
    ws = torch.empty((max(cf.cf_workspace_size(cf.CF_OP_WGRAD, desc), 256),), dtype=torch.uint8, device="cuda")
    dw = torch.empty((co, 3, 3, 3, ci), dtype=torch.float32, device="cuda")
    cf.cf_conv3d_wgrad(desc, x, dz, None, dw, 0, ws, ws.numel())
    pts = tile_cover_pts(rng, co, ci)
    ref, S = oracle_mod.conv3d_wgrad_pts(inp["x"], inp["dz"], pts)
    assert_close(dw.cpu().numpy()[tuple(pts.T)].astype(np.float64), ref, S,
                 f"sweep wgrad {shape} ({len(pts)} tile-covering elements)")
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == cf.CF_OK


def test_table1_model_128_n4(cf, oracle_mod):
    """The hybrid-parallelism page's Table I model at input width 128 (4 x
    128^3 per sample, N=4): forward + backward through CosmoStack, every
    kernel checked on its own GPU inputs (the three large blocks sampled,
    their weight gradients in full; the rest in full)."""
    from oracle import TABLE1_CHANNELS, table1_specs
    from cnn_conv3d_gb300 import flops
    from tests.test_gpu_chain import check_chain_per_kernel, run_chain
    st, inp, dy16 = run_chain(cf, 4, 128, TABLE1_CHANNELS, table1_specs(128), seed=20260006)
    assert tuple(st.y[-1].shape) == (4, 2, 2, 2, 256)
    check_chain_per_kernel(oracle_mod, st, inp, dy16, big_from=4 * 32 ** 3, rng=np.random.default_rng(6))
    # the executed forward FLOPs of the chain are Table I's per-sample row x N
    fwd = 0
    for l in range(st.L):
        n, d, h, w = st.odims[l]
        fwd += flops.conv_flops(n, TABLE1_CHANNELS[l], TABLE1_CHANNELS[l + 1], d * h * w)
    assert fwd == 4 * flops.p3_table1_forward_flops(128)
