"""The page variants chained through CosmoStack (per-block stride and pooling
kind), checked kernel by kernel: every block's forward on the GPU's own input,
and every backward op (pool / activation backward, backward-weight,
backward-data) on the GPU's own upstream gradient, against the fp64 oracle.

Chains: the hybrid-parallelism page's Table I model (channels 4, 16, 32, 64,
128, 256, 256, 256; the fourth conv stride 2; no pooling after the last two
at this width) at 64^3, and an average-pooling chain (CosmoFlow page, section
III-C) with a stride-2 block and an unpooled top."""
import numpy as np
import pytest

import synthdata
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu

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


def _wins(a):
    N, D, H, W, C = a.shape
    return a.reshape(N, D // 2, 2, H // 2, 2, W // 2, 2, C).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(
        N, D // 2, H // 2, W // 2, C, 8)


def run_chain(cf, n, spatial, channels, specs, seed):
    import torch
    from cnn_conv3d_gb300.stack import CosmoStack
    inp = synthdata.stack_inputs(n, spatial, channels, seed=seed, with_dy=False)
    rng = np.random.default_rng(seed)
    # biases of both signs, so both branches of every derivative are exercised
    inp["b"] = [rng.normal(0, 0.5, size=c).astype(np.float32) for c in channels[1:]]
    st = CosmoStack(n, spatial, channels, SLOPE, backward=True, specs=specs)
    st.load(inp["x"], inp["w"], inp["b"])
    inp["gamma"] = [rng.normal(1.0, 0.5, size=c).astype(np.float32) for c in channels[1:]]
    for l in range(st.L):
        if st.bn(l):
            st.gamma[l].copy_(torch.from_numpy(inp["gamma"][l]))
    dy16 = synthdata.to_bf16_bits(rng.normal(size=tuple(st.y[-1].shape)))
    dy = torch.from_numpy(dy16.view(np.int16)).view(torch.bfloat16).cuda()
    st.step(dy)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == cf.CF_OK
    return st, inp, dy16


def _big(st, l, limit):
    return limit is not None and st.dims[l][0] * st.dims[l][1] ** 3 >= limit


def check_big_block(oracle, st, inp, dy16, l, rng):
    """A stride-1 max-pooled block too large for full fp64 tensors: sampled
    pooled outputs, the bias gradient in full, every weight-gradient element
    (per-tap matrix products, or the routed sum), sampled input gradients."""
    from tests.gpu_util import tile_cover_pts  # noqa: F401
    f = oracle.bf16_bits_to_f64
    assert st.specs[l] == (1, "max")
    x16 = u16(st.block_input(l))
    y16 = u16(st.y[l])
    pts = np.stack([rng.integers(0, s, 2048) for s in y16.shape], 1).astype(np.int64)
    ry, ridx, S, gap = oracle.block_fwd_pts(x16, inp["w"][l], inp["b"][l], SLOPE, pts)
    gy = f(y16[tuple(pts.T)])
    gi = st.idx[l].cpu().numpy()[tuple(pts.T)]
    notie = gap > 1e-2 * S
    np.testing.assert_array_equal(gi[notie], ridx[notie])
    assert_close(gy, ry, S, f"block {l + 1} forward (sampled)")
    top = l == st.L - 1
    g16 = dy16 if top else u16(st.g[l])
    idx = st.idx[l].cpu().numpy()
    _, gp, rdb = oracle.pool_bwd(f(g16), f(y16) if top else None, idx, SLOPE, want_dz=False)
    assert_close(st.db[l].cpu().numpy().astype(np.float64), rdb, np.abs(gp).reshape(-1, gp.shape[-1]).sum(0),
                 f"db block {l + 1}")
    gdw = st.dw[l].cpu().numpy().astype(np.float64)
    if st.routed(l):
        pts = np.array([(co, t // 9, (t // 3) % 3, t % 3, ci) for co in range(gdw.shape[0]) for t in range(27)
                        for ci in range(gdw.shape[4])], dtype=np.int64)
        ref, S = oracle.conv3d_wgrad_routed_pts(x16, g16, idx, pts)
        assert_close(gdw[tuple(pts.T)], ref, S, f"dW block {l + 1} (routed, every element)")
        return
    dz16 = u16(st.dz[l])
    ref = np.zeros(gdw.shape)
    S = np.zeros(gdw.shape)
    for n in range(x16.shape[0]):
        xs, dzs = f(x16[n:n + 1]), f(dz16[n:n + 1])
        ref += oracle.conv3d_wgrad_mm(xs, dzs)
        S += oracle.conv3d_wgrad_mm(np.abs(xs), np.abs(dzs))
    assert_close(gdw, ref, S, f"dW block {l + 1} (every element)")
    if l > 0:
        pts = np.stack([rng.integers(0, s, 2048) for s in x16.shape], 1).astype(np.int64)
        ref, S = oracle.conv3d_dgrad_pts(dz16, inp["w"][l], pts)
        fac = np.where(f(x16[tuple(pts.T)]) > 0, 1.0, SLOPE) if st.specs[l - 1][1] != "avg" else 1.0
        assert_close(f(u16(st.g[l - 1])[tuple(pts.T)]), ref * fac, S * fac, f"dX block {l + 1} (sampled)")


def check_chain_per_kernel(oracle, st, inp, dy16, big_from=None, rng=None):
    """Every kernel of the step against the oracle on the GPU's own inputs;
    blocks whose input has at least `big_from` voxels go through
    check_big_block (sampled / per-element routines)."""
    f = oracle.bf16_bits_to_f64
    L = st.L
    for l in range(L):
        if _big(st, l, big_from):
            check_big_block(oracle, st, inp, dy16, l, rng)
            continue
        stride, pool = st.specs[l][0], st.specs[l][1]
        x = f(u16(st.block_input(l)))
        w = f(inp["w"][l])
        b = inp["b"][l].astype(np.float64)
        conv = oracle.conv3d_fwd if stride == 1 else oracle.conv3d_fwd_s2
        z, S = conv(x, w), conv(np.abs(x), np.abs(w))
        gy = f(u16(st.y[l]))
        what = f"block {l + 1} forward {st.specs[l]}"
        if st.bn(l):
            # the stored conv output, then the normalisation + activation + pooling
            # on that stored bf16 z: u = a*z + c with the batch statistics of z
            zg = f(u16(st.zc[l]))
            assert_close(zg, z, S, f"{what}: conv output")
            gam = inp["gamma"][l].astype(np.float64)
            mean, var = zg.reshape(-1, zg.shape[-1]).mean(0), zg.reshape(-1, zg.shape[-1]).var(0)
            np.testing.assert_allclose(st.stats[l].cpu().numpy()[:zg.shape[-1]] / zg[..., 0].size, mean,
                                       rtol=1e-4, atol=1e-5 * np.abs(zg).max())
            u, _, _ = oracle.bn_fwd(zg, gam, b, st.bn_eps)
            # scale of u's rounding: |a| |z| + |c| (fp32 coefficients, bf16 output)
            a = gam / np.sqrt(var + st.bn_eps)
            Su = np.abs(a) * np.abs(zg) + np.abs(b - a * mean)
            z, S, b = u, Su, np.zeros_like(b)
        if pool == "max":
            ry, ridx = oracle.pool_fwd(z, b, SLOPE)
            zw, sw = _wins(z), _wins(S)
            srt = np.sort(zw, -1)
            s_at = np.take_along_axis(sw, ridx[..., None].astype(np.int64), -1)[..., 0] + np.abs(b)
            notie = (srt[..., -1] - srt[..., -2]) > 1e-2 * s_at
            np.testing.assert_array_equal(st.idx[l].cpu().numpy()[notie], ridx[notie], err_msg=what)
            assert_close(gy, ry, s_at, what)
        elif pool == "avg":
            ry, rmask = oracle.avgpool_fwd(z, b, SLOPE)
            sw = _wins(S + np.abs(b))
            assert_close(gy, ry, sw.mean(-1), what)
            sure = np.abs(_wins(z + b)) > 1e-2 * sw
            gm = st.idx[l].cpu().numpy()
            bits = lambda m: (m[..., None].astype(np.int64) >> np.arange(8)) & 1  # noqa: E731
            np.testing.assert_array_equal(bits(gm)[sure], bits(rmask)[sure], err_msg=what)
        else:
            assert_close(gy, oracle.act_fwd(z, b, SLOPE), S + np.abs(b), what)
    # backward, top down, each op on the GPU's own inputs
    for l in range(L - 1, -1, -1):
        if _big(st, l, big_from):
            continue  # done in check_big_block
        stride, pool = st.specs[l][0], st.specs[l][1]
        x = f(u16(st.block_input(l)))
        w = f(inp["w"][l])
        what = f"block {l + 1} ({stride}, {pool})"
        top = l == L - 1
        g = f(dy16) if top else f(u16(st.g[l]))
        # dZ and db of the pool / activation backward
        if pool == "max":
            rdz, _, rdb = oracle.pool_bwd(g, f(u16(st.y[l])) if top else None, st.idx[l].cpu().numpy(), SLOPE)
        elif pool == "avg":
            rdz, rdb = oracle.avgpool_bwd(g, st.idx[l].cpu().numpy(), SLOPE)
        elif top:
            rdz, rdb = oracle.act_bwd(g, f(u16(st.y[l])), SLOPE)
        else:
            rdz, rdb = g, g.reshape(-1, g.shape[-1]).sum(0)  # the dgrad output is dZ itself
        if st.bn(l):
            # the batch-norm backward of du = the pooling backward above, on the
            # stored z: dz, dgamma, dbeta (db)
            zg = f(u16(st.zc[l]))
            gam = inp["gamma"][l].astype(np.float64)
            du = rdz
            rdz, rdg, rdb = oracle.bn_bwd(zg, du, gam, st.bn_eps)
            C = zg.shape[-1]
            zz = zg.reshape(-1, C)
            inv = 1 / np.sqrt(zz.var(0) + st.bn_eps)
            zh = (zz - zz.mean(0)) * inv
            dd = du.reshape(-1, C)
            assert_close(st.dgamma[l].cpu().numpy().astype(np.float64), rdg, np.abs(dd * zh).sum(0), f"dgamma {what}")
            assert_close(st.db[l].cpu().numpy().astype(np.float64), rdb, np.abs(dd).sum(0), f"dbeta {what}")
            Sdz = np.abs(gam * inv) * (np.abs(dd) + np.abs(dd).mean(0) + np.abs(zh) * np.abs(dd * zh).mean(0))
            dz = f(u16(st.dz[l]))
            assert_close(dz, rdz, Sdz.reshape(dz.shape), f"dZ {what}")
        else:
            assert_close(st.db[l].cpu().numpy().astype(np.float64), rdb,
                         np.abs(rdz).reshape(-1, rdz.shape[-1]).sum(0), f"db {what}")
        if st.bn(l):
            pass
        elif st.routed(l):
            dz = oracle.round_to_bf16(rdz)  # routed on chip from the same bf16 values
        else:
            dz = f(u16(st.dz[l]))
            np.testing.assert_allclose(dz, rdz, rtol=2 ** -8, atol=0, err_msg=f"dZ {what}")
        wg = oracle.conv3d_wgrad if stride == 1 else oracle.conv3d_wgrad_s2
        assert_close(st.dw[l].cpu().numpy().astype(np.float64), wg(x, dz), wg(np.abs(x), np.abs(dz)), f"dW {what}")
        if l > 0:
            if stride == 1:
                rdx, Sx = oracle.conv3d_dgrad(dz, w), oracle.conv3d_dgrad(np.abs(dz), np.abs(w))
            else:
                rdx = oracle.conv3d_dgrad_s2(dz, w, x.shape[1:4])
                Sx = oracle.conv3d_dgrad_s2(np.abs(dz), np.abs(w), x.shape[1:4])
            if st.specs[l - 1][1] != "avg":
                fac = np.where(x > 0, 1.0, SLOPE)
                rdx, Sx = rdx * fac, Sx * fac
            assert_close(f(u16(st.g[l - 1])), rdx, Sx, f"dX {what}")


def test_table1_model_64(cf, oracle_mod):
    """The Table I model (stride-2 c4; c6, c7 unpooled) on 1 x 4 x 64^3."""
    from oracle import TABLE1_CHANNELS, table1_specs
    st, inp, dy16 = run_chain(cf, 1, 64, TABLE1_CHANNELS, table1_specs(128), seed=5151)
    assert tuple(st.y[-1].shape) == (1, 1, 1, 1, 256)
    check_chain_per_kernel(oracle_mod, st, inp, dy16)


@pytest.mark.parametrize("specs,channels", [
    ([(1, "avg"), (1, "avg"), (2, "max"), (1, "none")], (4, 16, 32, 64, 64)),
    ([(1, "max"), (2, "avg"), (1, "none"), (1, "max")], (1, 32, 48, 64, 32)),
])
def test_variant_chain_32(cf, oracle_mod, specs, channels):
    st, inp, dy16 = run_chain(cf, 2, 32, channels, specs, seed=5252)
    check_chain_per_kernel(oracle_mod, st, inp, dy16)


def test_variant_chain_schedules_agree(cf):
    """Serial and two-stream schedules of a variant chain give the same bits."""
    import torch
    from cnn_conv3d_gb300.stack import CosmoStack
    from oracle import TABLE1_CHANNELS, table1_specs
    inp = synthdata.stack_inputs(1, 64, TABLE1_CHANNELS, seed=77, with_dy=False)
    st = CosmoStack(1, 64, TABLE1_CHANNELS, SLOPE, specs=table1_specs(128))
    st.load(inp["x"], inp["w"], inp["b"])
    dy = torch.randn(tuple(st.y[-1].shape), device="cuda").to(torch.bfloat16)
    st.step(dy, serial=True)
    torch.cuda.synchronize()
    ref = [t.clone() for t in st.y + st.dw + st.db]
    st.step(dy)
    g = st.capture(dy)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, st.y + st.dw + st.db):
        assert torch.equal(a, b)


@pytest.mark.parametrize("specs,channels", [
    ([(1, "max", "bn"), (1, "max", "bn"), (1, "none", "bn")], (4, 16, 32, 32)),
    ([(1, "avg", "bn"), (2, "max", "bn"), (1, "none")], (16, 32, 64, 32)),
])
def test_batchnorm_chain_32(cf, oracle_mod, specs, channels):
    """Batch normalisation after every conv (hybrid-parallelism page, section
    IV), chained with max / average / no pooling and a stride-2 block."""
    st, inp, dy16 = run_chain(cf, 2, 32, channels, specs, seed=5353)
    check_chain_per_kernel(oracle_mod, st, inp, dy16)
