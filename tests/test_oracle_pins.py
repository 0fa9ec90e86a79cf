"""Pins for the fp64 oracle: each check compares it with something other than
itself (an independently built dense operator, a library correlation routine,
closed forms, identities, finite differences, the pages' printed numbers).
CPU only."""
import os

import numpy as np
import pytest

import synthdata

RNG = np.random.default_rng(1234)


def _dense_shift(n, k):
    """1D shift matrix S with (S v)[i] = v[i + k - 1] (zero outside)."""
    return np.eye(n, k=k - 1)


def _shift3(D, H, W, kd, kh, kw):
    return np.kron(np.kron(_dense_shift(D, kd), _dense_shift(H, kh)), _dense_shift(W, kw))


def dense_conv_operator(N, D, H, W, w):
    """Matrix A (rows (n,v,co), cols (n,u,ci)) of the pad-1 cross-correlation,
    built from Kronecker products of 1D shift matrices and the per-tap
    channel-mixing blocks w[:, kd, kh, kw, :]."""
    Co, _, _, _, Ci = w.shape
    V = D * H * W
    A = np.zeros((N * V * Co, N * V * Ci))
    for kd in range(3):
        for kh in range(3):
            for kw in range(3):
                S = np.kron(np.eye(N), _shift3(D, H, W, kd, kh, kw))
                A += np.kron(S, w[:, kd, kh, kw, :])
    return A


def dense_weight_jacobian(x, Co):
    """Matrix J with z_flat = J @ w_flat for fixed x (w flat in [Co][3][3][3][Ci])."""
    N, D, H, W, Ci = x.shape
    V = D * H * W
    J = np.zeros((N * V * Co, Co * 27 * Ci))
    xf = x.reshape(N, V, Ci)
    for t in range(27):
        kd, kh, kw = t // 9, (t // 3) % 3, t % 3
        S = _shift3(D, H, W, kd, kh, kw)
        xs = np.einsum("uv,nvc->nuc", S, xf).reshape(N * V, Ci)
        for co in range(Co):
            rows = np.arange(N * V) * Co + co
            cols = co * 27 * Ci + t * Ci + np.arange(Ci)
            J[np.ix_(rows, cols)] = xs
    return J


SHAPES = [
    (1, 2, 3, 4, 1, 1),
    (1, 3, 3, 3, 2, 2),
    (2, 4, 2, 5, 3, 2),
    (1, 5, 4, 3, 2, 3),
]


@pytest.mark.parametrize("N,D,H,W,Ci,Co", SHAPES)
def test_conv_matches_dense_operator(oracle_mod, N, D, H, W, Ci, Co):
    x = RNG.normal(size=(N, D, H, W, Ci))
    w = RNG.normal(size=(Co, 3, 3, 3, Ci))
    dz = RNG.normal(size=(N, D, H, W, Co))
    A = dense_conv_operator(N, D, H, W, w)
    z = oracle_mod.conv3d_fwd(x, w)
    np.testing.assert_allclose(z.ravel(), A @ x.ravel(), rtol=1e-12, atol=1e-12)
    dx = oracle_mod.conv3d_dgrad(dz, w)
    np.testing.assert_allclose(dx.ravel(), A.T @ dz.ravel(), rtol=1e-12, atol=1e-12)
    J = dense_weight_jacobian(x, Co)
    np.testing.assert_allclose(J @ w.ravel(), z.ravel(), rtol=1e-12, atol=1e-12)
    dw = oracle_mod.conv3d_wgrad(x, dz)
    np.testing.assert_allclose(dw.ravel(), J.T @ dz.ravel(), rtol=1e-12, atol=1e-12)


def test_conv_matches_scipy_correlate(oracle_mod):
    from scipy.signal import correlate
    N, D, H, W, Ci, Co = 2, 6, 5, 7, 3, 4
    x = RNG.normal(size=(N, D, H, W, Ci))
    w = RNG.normal(size=(Co, 3, 3, 3, Ci))
    z = oracle_mod.conv3d_fwd(x, w)
    ref = np.zeros_like(z)
    for n in range(N):
        for co in range(Co):
            for ci in range(Ci):
                ref[n, :, :, :, co] += correlate(x[n, :, :, :, ci], w[co, :, :, :, ci],
                                                 mode="same", method="direct")
    np.testing.assert_allclose(z, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("t0", [0, 4, 13, 22, 26])
def test_delta_kernel_shift(oracle_mod, t0):
    N, D, H, W, C = 1, 4, 5, 6, 3
    kd, kh, kw = t0 // 9, (t0 // 3) % 3, t0 % 3
    x = RNG.normal(size=(N, D, H, W, C))
    w = np.zeros((C, 3, 3, 3, C))
    for c in range(C):
        w[c, kd, kh, kw, c] = 1.0
    z = oracle_mod.conv3d_fwd(x, w)
    xp = np.pad(x, ((0, 0), (1, 1), (1, 1), (1, 1), (0, 0)))
    expect = xp[:, kd:kd + D, kh:kh + H, kw:kw + W, :]
    np.testing.assert_array_equal(z, expect)
    if t0 == 13:
        np.testing.assert_array_equal(z, x)


def test_constant_input_tap_counts(oracle_mod):
    N, D, H, W, Ci, Co = 1, 5, 5, 5, 2, 1
    c = 0.75
    x = np.full((N, D, H, W, Ci), c)
    w = np.ones((Co, 3, 3, 3, Ci))
    z = oracle_mod.conv3d_fwd(x, w)[0, :, :, :, 0] / (c * Ci)
    assert z[2, 2, 2] == 27  # interior
    assert z[0, 2, 2] == 18  # face
    assert z[0, 0, 2] == 12  # edge
    assert z[0, 0, 0] == 8   # corner
    assert z[4, 4, 4] == 8
    # with random weights: sum over the valid taps only
    w = RNG.normal(size=(2, 3, 3, 3, Ci))
    z = oracle_mod.conv3d_fwd(x, w)
    np.testing.assert_allclose(z[0, 2, 2, 2], c * w.sum(axis=(1, 2, 3, 4)), rtol=1e-13)
    np.testing.assert_allclose(z[0, 0, 0, 0], c * w[:, 1:, 1:, 1:, :].sum(axis=(1, 2, 3, 4)),
                               rtol=1e-13)


def test_linearity(oracle_mod):
    x1 = RNG.normal(size=(2, 4, 3, 5, 3))
    x2 = RNG.normal(size=x1.shape)
    w = RNG.normal(size=(2, 3, 3, 3, 3))
    a, b = 1.7, -0.4
    lhs = oracle_mod.conv3d_fwd(a * x1 + b * x2, w)
    rhs = a * oracle_mod.conv3d_fwd(x1, w) + b * oracle_mod.conv3d_fwd(x2, w)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-11, atol=1e-11)


def test_adjoint_identities(oracle_mod):
    x = RNG.normal(size=(2, 6, 5, 4, 3))
    w = RNG.normal(size=(4, 3, 3, 3, 3))
    g = RNG.normal(size=(2, 6, 5, 4, 4))
    lhs = np.vdot(oracle_mod.conv3d_fwd(x, w), g)
    mid = np.vdot(x, oracle_mod.conv3d_dgrad(g, w))
    rhs = np.vdot(w, oracle_mod.conv3d_wgrad(x, g))
    assert abs(lhs - mid) <= 1e-10 * abs(lhs)
    assert abs(lhs - rhs) <= 1e-10 * abs(lhs)


def _block_loss(oracle_mod, x, w, b, g, slope):
    z = oracle_mod.conv3d_fwd(x, w)
    y, idx = oracle_mod.pool_fwd(z, b, slope)
    return np.vdot(g, y), z, y, idx


def test_finite_difference_gradients(oracle_mod):
    slope = 0.3
    rng = np.random.default_rng(7)
    # resample until there is no kink: every pre-activation away from 0 and
    # every window's top-two gap above 1e-3
    for _ in range(200):
        x = rng.normal(size=(1, 4, 4, 6, 2))
        w = rng.normal(size=(3, 3, 3, 3, 2))
        b = rng.normal(size=(3,))
        z = oracle_mod.conv3d_fwd(x, w)
        y, idx = oracle_mod.pool_fwd(z, b, slope)
        win = z.reshape(1, 2, 2, 2, 2, 3, 2, 3).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(1, 2, 2, 3, 3, 8)
        srt = np.sort(win, axis=-1)
        pre = srt[..., -1] + b
        if np.min(srt[..., -1] - srt[..., -2]) > 1e-3 and np.min(np.abs(pre)) > 1e-3:
            break
    else:
        pytest.fail("could not draw a kink-free case")
    g = rng.normal(size=y.shape)
    dz, dyp, db = oracle_mod.pool_bwd(g, y, idx, slope)
    dw = oracle_mod.conv3d_wgrad(x, dz)
    dx = oracle_mod.conv3d_dgrad(dz, w)
    h = 1e-6

    def fd(arr, pos, which):
        a = arr.copy(); a[pos] += h
        lp = _block_loss(oracle_mod, *(which(a)), g, slope)[0]
        a = arr.copy(); a[pos] -= h
        lm = _block_loss(oracle_mod, *(which(a)), g, slope)[0]
        return (lp - lm) / (2 * h)

    for _ in range(6):
        pos = tuple(rng.integers(0, s) for s in x.shape)
        num = fd(x, pos, lambda a: (a, w, b))
        assert abs(num - dx[pos]) <= 1e-5 * max(1.0, abs(num)), (pos, num, dx[pos])
        pos = tuple(rng.integers(0, s) for s in w.shape)
        num = fd(w, pos, lambda a: (x, a, b))
        assert abs(num - dw[pos]) <= 1e-5 * max(1.0, abs(num)), (pos, num, dw[pos])
    for c in range(3):
        num = fd(b, (c,), lambda a: (x, w, a))
        assert abs(num - db[c]) <= 1e-5 * max(1.0, abs(num))


def test_pool_closed_forms(oracle_mod):
    N, D, H, W, C = 1, 4, 4, 6, 2
    d, h, w = np.meshgrid(np.arange(D), np.arange(H), np.arange(W), indexing="ij")
    ramp = ((d * H) + h) * W + w
    z = np.repeat(ramp[None, :, :, :, None].astype(float), C, axis=4)
    y, idx = oracle_mod.pool_fwd(z, None, 0.3)
    assert np.all(idx == 7)
    # the maximum of each window is its (1,1,1) corner
    np.testing.assert_array_equal(y, z[:, 1::2, 1::2, 1::2, :])
    y, idx = oracle_mod.pool_fwd(-z, None, 0.3)
    assert np.all(idx == 0)
    np.testing.assert_allclose(y, 0.3 * (-z[:, 0::2, 0::2, 0::2, :]))
    y, idx = oracle_mod.pool_fwd(np.full((1, 2, 2, 2, 1), 5.0), None, 0.3)
    assert idx.item() == 0 and y.item() == 5.0  # ties: first maximum wins
    y, _ = oracle_mod.pool_fwd(np.full((1, 2, 2, 2, 1), -1.0), None, 0.3)
    assert y.item() == pytest.approx(-0.3, abs=1e-15)
    y, _ = oracle_mod.pool_fwd(np.full((1, 2, 2, 2, 1), 2.0), None, 0.3)
    assert y.item() == 2.0
    # bias shifts before the activation
    y, _ = oracle_mod.pool_fwd(np.full((1, 2, 2, 2, 1), 1.0), np.array([-3.0]), 0.3)
    assert y.item() == pytest.approx(-0.6, abs=1e-15)


def test_pool_commutes_with_activation(oracle_mod):
    z = RNG.normal(size=(2, 4, 6, 4, 3))
    y, _ = oracle_mod.pool_fwd(z, None, 0.3)
    act = np.where(z > 0, z, 0.3 * z)
    # pool the activated tensor with a plain numpy window max
    win = act.reshape(2, 2, 2, 3, 2, 2, 2, 3).max(axis=(2, 4, 6))
    np.testing.assert_array_equal(y, win)


def test_pool_bwd_routes_to_argmax(oracle_mod):
    z = RNG.normal(size=(1, 4, 4, 4, 2))
    b = np.array([0.1, -0.2])
    y, idx = oracle_mod.pool_fwd(z, b, 0.3)
    dy = RNG.normal(size=y.shape)
    dz, dyp, db = oracle_mod.pool_bwd(dy, y, idx, 0.3)
    np.testing.assert_allclose(dyp, dy * np.where(y > 0, 1.0, 0.3))
    np.testing.assert_allclose(db, dyp.sum(axis=(0, 1, 2, 3)))
    # exactly one nonzero per window and channel, at the window's argmax of z
    win = dz.reshape(1, 2, 2, 2, 2, 2, 2, 2).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(1, 2, 2, 2, 2, 8)
    zw = z.reshape(1, 2, 2, 2, 2, 2, 2, 2).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(1, 2, 2, 2, 2, 8)
    am = np.argmax(zw, axis=-1)
    np.testing.assert_array_equal(am, idx)
    np.testing.assert_array_equal(np.take_along_axis(win, am[..., None], -1)[..., 0], dyp)
    assert np.count_nonzero(win) == np.count_nonzero(dyp)
    # y=None: dy is taken as the pre-activation gradient
    dz2, dyp2, db2 = oracle_mod.pool_bwd(dyp, None, idx, 0.3)
    np.testing.assert_array_equal(dz2, dz)


def test_point_routines_match_full(oracle_mod):
    c = synthdata.random_case(11, 2, 4, 6, 8, 16, 8)
    x = oracle_mod.bf16_bits_to_f64(c["x"])
    w = oracle_mod.bf16_bits_to_f64(c["w"])
    dz = oracle_mod.bf16_bits_to_f64(c["dz"])
    z = oracle_mod.conv3d_fwd(x, w)
    dx = oracle_mod.conv3d_dgrad(dz, w)
    dw = oracle_mod.conv3d_wgrad(x, dz)
    rng = np.random.default_rng(3)
    pts = np.stack([rng.integers(0, s, 40) for s in z.shape], 1)
    v, s = oracle_mod.conv3d_fwd_pts(c["x"], c["w"], pts)
    np.testing.assert_array_equal(v, z[tuple(pts.T)])
    assert np.all(s >= np.abs(v))
    pts = np.stack([rng.integers(0, s, 40) for s in dx.shape], 1)
    v, s = oracle_mod.conv3d_dgrad_pts(c["dz"], c["w"], pts)
    np.testing.assert_array_equal(v, dx[tuple(pts.T)])
    pts = np.stack([rng.integers(0, s, 40) for s in dw.shape], 1)
    v, s = oracle_mod.conv3d_wgrad_pts(c["x"], c["dz"], pts)
    np.testing.assert_allclose(v, dw[tuple(pts.T)], rtol=1e-12, atol=1e-12)
    # fused block at pooled points
    y, idx = oracle_mod.pool_fwd(z, c["b"].astype(np.float64), 0.3)
    pts = np.stack([rng.integers(0, s, 40) for s in y.shape], 1)
    yv, iv, sv, gap = oracle_mod.block_fwd_pts(c["x"], c["w"], c["b"], 0.3, pts)
    np.testing.assert_array_equal(yv, y[tuple(pts.T)])
    np.testing.assert_array_equal(iv, idx[tuple(pts.T)])
    assert np.all(gap >= 0)


def test_bf16_rounding_agrees_with_torch(oracle_mod):
    torch = pytest.importorskip("torch")
    v = np.concatenate([RNG.normal(size=5000) * 10.0 ** RNG.integers(-8, 8, 5000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, -3.0e38]])
    ref = torch.tensor(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle_mod.round_to_bf16(v), ref)
    np.testing.assert_array_equal(
        synthdata.bf16_bits_to_f32(synthdata.to_bf16_bits(v)).astype(np.float64), ref)


def _golden_rows():
    path = os.path.join(os.path.dirname(__file__), "golden", "p3_table1_flops.txt")
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(t) for t in line.split()])
    return rows


@pytest.mark.parametrize("row", _golden_rows())
def test_flop_convention_reproduces_table1(row):
    from cnn_conv3d_gb300 import flops
    wi, ops, fwd, params = row
    f = flops.p3_table1_forward_flops(int(wi)) / 1e9
    # the page prints 4 significant digits; agree to the printed precision
    assert abs(f - fwd) <= 0.5 * 10 ** (np.floor(np.log10(fwd)) - 3) + 1e-9, (f, fwd)
    assert abs(3 * f - ops) <= 0.5 * 10 ** (np.floor(np.log10(ops)) - 3) + 1e-9, (3 * f, ops)
    assert round(flops.p3_table1_params() / 1e6, 2) == params


def _window_view(a):
    """[N,D,H,W,C] -> [N,D/2,H/2,W/2,C,8], window members in (dd,dh,dw) order."""
    N, D, H, W, C = a.shape
    return a.reshape(N, D // 2, 2, H // 2, 2, W // 2, 2, C).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(
        N, D // 2, H // 2, W // 2, C, 8)


def test_stack_chain_finite_differences(oracle_mod):
    """Two chained blocks through oracle.stack_fwd / stack_bwd (exact mode):
    the weight and bias gradients of both blocks against central differences
    of L = <g, y_top>.  This pins the chaining itself -- the top block's
    gradient through its stored output, the lower block's leaky-ReLU
    derivative taken from its pooled output (the next block's input) -- and
    not only one block."""
    slope = 0.3
    rng = np.random.default_rng(21)
    ch = (2, 3, 2)
    for _ in range(500):
        x = rng.normal(size=(1, 4, 4, 4, ch[0]))
        ws = [rng.normal(size=(ch[l + 1], 3, 3, 3, ch[l])) for l in range(2)]
        # biases that put about half of each block's pooled pre-activations below
        # zero, so that both branches of the leaky-ReLU derivative are exercised
        bs = []
        cur = x
        for l in range(2):
            m = _window_view(oracle_mod.conv3d_fwd(cur, ws[l])).max(axis=-1)
            bs.append(-np.median(m.reshape(-1, ch[l + 1]), axis=0) + rng.choice([-0.5, 0.5], ch[l + 1]))
            cur = oracle_mod.pool_fwd(oracle_mod.conv3d_fwd(cur, ws[l]), bs[l], slope)[0]
        xs, zs, ys, idxs = oracle_mod.stack_fwd(x, ws, bs, slope, mirrored=False)
        ok = True
        for l in range(2):
            srt = np.sort(_window_view(zs[l]), axis=-1)
            pre = srt[..., -1] + bs[l]
            ok &= np.min(srt[..., -1] - srt[..., -2]) > 1e-3 and np.min(np.abs(pre)) > 1e-3
            ok &= np.any(pre < 0) and np.any(pre > 0)
        if ok:
            break
    else:
        pytest.fail("could not draw a kink-free case")
    g = rng.normal(size=ys[-1].shape)
    dws, dbs, _, dxs = oracle_mod.stack_bwd(xs, ys, idxs, ws, g, slope, mirrored=False)
    assert dxs[0] is None and dxs[1].shape == ys[0].shape

    def loss(ws_, bs_):
        return np.vdot(g, oracle_mod.stack_fwd(x, ws_, bs_, slope, mirrored=False)[2][-1])

    h = 1e-6
    for l in range(2):
        for _ in range(5):
            pos = tuple(rng.integers(0, s) for s in ws[l].shape)
            wp = [w.copy() for w in ws]
            wm = [w.copy() for w in ws]
            wp[l][pos] += h
            wm[l][pos] -= h
            num = (loss(wp, bs) - loss(wm, bs)) / (2 * h)
            assert abs(num - dws[l][pos]) <= 1e-5 * max(1.0, abs(num)), (l, pos, num, dws[l][pos])
        for c in range(ch[l + 1]):
            bp = [b.copy() for b in bs]
            bm = [b.copy() for b in bs]
            bp[l][c] += h
            bm[l][c] -= h
            num = (loss(ws, bp) - loss(ws, bm)) / (2 * h)
            assert abs(num - dbs[l][c]) <= 1e-5 * max(1.0, abs(num)), (l, c, num, dbs[l][c])
    # the gradient at the lower block's pooled pre-activation, g1 = dL/d(m1 + b1):
    # shifting b1 by h moves every m1 + b1 of that channel, so its channel sums
    # are db1, already checked above; check them against dxs[1] directly
    np.testing.assert_allclose(dxs[1].reshape(-1, ch[1]).sum(0), dbs[0], rtol=1e-12, atol=1e-12)


def test_stack_mirrored_rounds_at_block_boundaries(oracle_mod):
    """Mirrored mode stores each block output as bf16 (exactly representable)
    and stays within bf16 rounding of the exact chain."""
    rng = np.random.default_rng(22)
    x = oracle_mod.round_to_bf16(rng.normal(size=(1, 8, 8, 8, 4)))
    ws = [oracle_mod.round_to_bf16(rng.normal(0, 0.2, size=(8, 3, 3, 3, 4))),
          oracle_mod.round_to_bf16(rng.normal(0, 0.1, size=(8, 3, 3, 3, 8)))]
    bs = [np.zeros(8), np.zeros(8)]
    xs, _, ys, _ = oracle_mod.stack_fwd(x, ws, bs, 0.3, mirrored=True)
    _, _, ye, _ = oracle_mod.stack_fwd(x, ws, bs, 0.3, mirrored=False)
    for l in range(2):
        np.testing.assert_array_equal(oracle_mod.round_to_bf16(ys[l]), ys[l])
    np.testing.assert_array_equal(xs[1], ys[0])
    assert np.linalg.norm(ys[-1] - ye[-1]) <= 2e-2 * np.linalg.norm(ye[-1])


def test_point_routine_scales_and_gaps(oracle_mod):
    """S (sum of |products|) and the top-two gap returned by the point
    routines, against the full routines on |x|, |w|, |dz| and a numpy sort of
    each window's eight values.  These two numbers set the tolerance and the
    no-tie selection of every full-size GPU check."""
    c = synthdata.random_case(12, 2, 4, 6, 8, 16, 8)
    f = oracle_mod.bf16_bits_to_f64
    x, w, dz = f(c["x"]), f(c["w"]), f(c["dz"])
    rng = np.random.default_rng(4)
    Sf = oracle_mod.conv3d_fwd(np.abs(x), np.abs(w))
    pts = np.stack([rng.integers(0, s, 60) for s in Sf.shape], 1)
    _, s = oracle_mod.conv3d_fwd_pts(c["x"], c["w"], pts)
    np.testing.assert_allclose(s, Sf[tuple(pts.T)], rtol=1e-13)
    Sd = oracle_mod.conv3d_dgrad(np.abs(dz), np.abs(w))
    pts = np.stack([rng.integers(0, s, 60) for s in Sd.shape], 1)
    _, s = oracle_mod.conv3d_dgrad_pts(c["dz"], c["w"], pts)
    np.testing.assert_allclose(s, Sd[tuple(pts.T)], rtol=1e-13)
    Sw = oracle_mod.conv3d_wgrad(np.abs(x), np.abs(dz))
    pts = np.stack([rng.integers(0, s, 60) for s in Sw.shape], 1)
    _, s = oracle_mod.conv3d_wgrad_pts(c["x"], c["dz"], pts)
    np.testing.assert_allclose(s, Sw[tuple(pts.T)], rtol=1e-12)
    # fused block: S at the argmax voxel plus |b|, gap = largest - second largest
    z = oracle_mod.conv3d_fwd(x, w)
    b = c["b"].astype(np.float64)
    zw, sw = _window_view(z), _window_view(Sf)
    pts = np.stack([rng.integers(0, s, 60) for s in zw.shape[:5]], 1)
    _, iv, sv, gap = oracle_mod.block_fwd_pts(c["x"], c["w"], c["b"], 0.3, pts)
    win = zw[tuple(pts.T)]
    srt = np.sort(win, axis=-1)
    np.testing.assert_allclose(gap, srt[:, -1] - srt[:, -2], rtol=1e-12, atol=1e-14)
    s_at = sw[tuple(pts.T)][np.arange(len(pts)), iv.astype(np.int64)] + np.abs(b[pts[:, 4]])
    np.testing.assert_allclose(sv, s_at, rtol=1e-13)
    # an all-zero input: every window is a tie, gap 0 and code 0 (first maximum)
    x0 = np.zeros_like(c["x"])
    _, iv, sv, gap = oracle_mod.block_fwd_pts(x0, c["w"], c["b"], 0.3, pts)
    assert np.all(gap == 0) and np.all(iv == 0)
    np.testing.assert_array_equal(sv, np.abs(b[pts[:, 4]]))


def test_wgrad_matmul_form_and_slabs(oracle_mod):
    """The per-tap matrix-product form of the weight gradient equals the direct
    loops, and summing it over d-slabs (with the neighbouring planes passed in)
    equals the whole volume."""
    rng = np.random.default_rng(31)
    x = rng.normal(size=(2, 6, 5, 4, 3))
    dz = rng.normal(size=(2, 6, 5, 4, 5))
    ref = oracle_mod.conv3d_wgrad(x, dz)
    np.testing.assert_allclose(oracle_mod.conv3d_wgrad_mm(x, dz), ref, rtol=1e-12, atol=1e-12)
    acc = np.zeros_like(ref)
    for d0, d1 in ((0, 2), (2, 5), (5, 6)):
        below = x[:, d0 - 1] if d0 > 0 else None
        above = x[:, d1] if d1 < 6 else None
        acc += oracle_mod.conv3d_wgrad_mm(x[:, d0:d1], dz[:, d0:d1], below, above)
    np.testing.assert_allclose(acc, ref, rtol=1e-12, atol=1e-12)


def test_routed_wgrad_points_match_dense(oracle_mod):
    """Weight gradient from the pooled gradient + argmax codes (summed over
    pooled voxels) equals the weight gradient of the dense routed dZ."""
    rng = np.random.default_rng(32)
    N, D, H, W, Ci, Co = 2, 4, 6, 8, 4, 5
    z = rng.normal(size=(N, D, H, W, Co))
    _, idx = oracle_mod.pool_fwd(z, None, 0.3)
    g16 = synthdata.to_bf16_bits(rng.normal(size=idx.shape))
    x16 = synthdata.to_bf16_bits(rng.normal(size=(N, D, H, W, Ci)))
    f = oracle_mod.bf16_bits_to_f64
    dz, _, _ = oracle_mod.pool_bwd(f(g16), None, idx, 0.3)
    ref = oracle_mod.conv3d_wgrad(f(x16), dz)
    S = oracle_mod.conv3d_wgrad(np.abs(f(x16)), np.abs(dz))
    pts = np.array([[co, kd, kh, kw, ci] for co in range(Co) for kd in range(3) for kh in range(3)
                    for kw in range(3) for ci in range(Ci)])
    v, s = oracle_mod.conv3d_wgrad_routed_pts(x16, g16, idx, pts)
    np.testing.assert_allclose(v, ref[tuple(pts.T)], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s, S[tuple(pts.T)], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- page variants

def test_avgpool_closed_forms(oracle_mod):
    slope = 0.3
    # a constant window: the average of eight equal activations
    y, m = oracle_mod.avgpool_fwd(np.full((1, 2, 2, 2, 1), 2.0), None, slope)
    assert y.item() == 2.0 and m.item() == 0xFF
    y, m = oracle_mod.avgpool_fwd(np.full((1, 2, 2, 2, 1), -1.0), None, slope)
    assert y.item() == pytest.approx(-0.3, abs=1e-15) and m.item() == 0
    # a window with values -4..3 in (dd,dh,dw) order: activations average to
    # (0+1+2+3 + 0.3*(-4-3-2-1)) / 8, mask = the four positive positions (0 is not)
    z = (np.arange(8, dtype=float) - 4).reshape(1, 2, 2, 2, 1)
    y, m = oracle_mod.avgpool_fwd(z, None, slope)
    assert y.item() == pytest.approx((0 + 1 + 2 + 3 + slope * (-10)) / 8, abs=1e-15)
    assert m.item() == 0b11100000
    # bias shifts before the activation
    y, m = oracle_mod.avgpool_fwd(z, np.array([4.5]), slope)
    assert y.item() == pytest.approx(np.mean(np.arange(8) + 0.5), abs=1e-15) and m.item() == 0xFF
    # the average of a ramp equals numpy's window mean of the activation
    zz = RNG.normal(size=(2, 4, 6, 4, 3))
    b = RNG.normal(size=3)
    y, m = oracle_mod.avgpool_fwd(zz, b, slope)
    a = np.where(zz + b > 0, zz + b, slope * (zz + b))
    np.testing.assert_allclose(y, a.reshape(2, 2, 2, 3, 2, 2, 2, 3).mean(axis=(2, 4, 6)), rtol=1e-13, atol=1e-15)
    bits = (_window_view(zz + b) > 0).astype(np.int64) << np.arange(8)
    np.testing.assert_array_equal(m, bits.sum(-1))


def test_act_closed_forms(oracle_mod):
    z = np.array([-2.0, -0.0, 0.0, 1.5]).reshape(1, 1, 1, 4, 1)
    y = oracle_mod.act_fwd(z, np.array([0.5]), 0.3)
    np.testing.assert_allclose(y.ravel(), [0.3 * -1.5, 0.5, 0.5, 2.0])
    dz, db = oracle_mod.act_bwd(np.ones_like(z), y, 0.3)
    np.testing.assert_allclose(dz.ravel(), [0.3, 1, 1, 1])
    assert db.item() == pytest.approx(3.3)


def test_stride2_conv_is_subsampled_stride1(oracle_mod):
    """Stride 2 with padding 1 evaluates the stride-1 output at even positions;
    its backward-data and backward-weight are the stride-1 ones applied to the
    output gradient with zeros inserted at the odd positions; adjoints hold."""
    rng = np.random.default_rng(41)
    for shape in ((1, 4, 6, 8, 3), (2, 5, 3, 7, 2)):
        x = rng.normal(size=shape)
        w = rng.normal(size=(4, 3, 3, 3, shape[4]))
        z2 = oracle_mod.conv3d_fwd_s2(x, w)
        np.testing.assert_allclose(z2, oracle_mod.conv3d_fwd(x, w)[:, ::2, ::2, ::2], rtol=1e-13, atol=1e-13)
        g = rng.normal(size=z2.shape)
        up = oracle_mod._upsample2(g, shape[1:4])
        dx = oracle_mod.conv3d_dgrad_s2(g, w, shape[1:4])
        np.testing.assert_allclose(dx, oracle_mod.conv3d_dgrad(up, w), rtol=1e-12, atol=1e-12)
        dw = oracle_mod.conv3d_wgrad_s2(x, g)
        np.testing.assert_allclose(dw, oracle_mod.conv3d_wgrad(x, up), rtol=1e-12, atol=1e-12)
        lhs = np.vdot(z2, g)
        assert abs(lhs - np.vdot(x, dx)) <= 1e-10 * abs(lhs)
        assert abs(lhs - np.vdot(w, dw)) <= 1e-10 * abs(lhs)


def test_chain_with_variants_finite_differences(oracle_mod):
    """A chain of an average-pooled block, a stride-2 max-pooled block and an
    unpooled block: every dW and db against central differences of <g, y_top>
    (exact mode).  Biases put pre-activations on both sides of zero."""
    slope = 0.3
    specs = [(1, "avg"), (2, "max"), (1, "none")]
    ch = (2, 3, 3, 2)
    rng = np.random.default_rng(42)
    for _ in range(300):
        x = rng.normal(size=(1, 8, 8, 8, ch[0]))
        ws = [rng.normal(size=(ch[l + 1], 3, 3, 3, ch[l])) for l in range(3)]
        bs = [rng.normal(size=(ch[l + 1],)) * 3 for l in range(3)]
        xs, ys, auxs = oracle_mod.chain_fwd(x, ws, bs, slope, specs, mirrored=False)
        # kink-free: every pre-activation away from zero, every max window's gap > 1e-3
        z0 = oracle_mod.conv3d_fwd(xs[0], ws[0]) + bs[0]
        z1 = oracle_mod.conv3d_fwd_s2(xs[1], ws[1])
        z2 = oracle_mod.conv3d_fwd(xs[2], ws[2]) + bs[2]
        srt = np.sort(_window_view(z1), axis=-1)
        ok = (np.min(np.abs(z0)) > 1e-3 and np.min(np.abs(z2)) > 1e-3 and np.min(srt[..., -1] - srt[..., -2]) > 1e-3
              and np.min(np.abs(srt[..., -1] + bs[1])) > 1e-3)
        ok = ok and np.any(z0 < 0) and np.any(z0 > 0) and np.any(srt[..., -1] + bs[1] < 0)
        if ok:
            break
    else:
        pytest.fail("could not draw a kink-free case")
    g = rng.normal(size=ys[-1].shape)
    dws, dbs, _ = oracle_mod.chain_bwd(xs, ys, auxs, ws, g, slope, specs, mirrored=False)

    def loss(ws_, bs_):
        return np.vdot(g, oracle_mod.chain_fwd(x, ws_, bs_, slope, specs, mirrored=False)[1][-1])

    h = 1e-6
    for l in range(3):
        for _ in range(4):
            pos = tuple(rng.integers(0, s) for s in ws[l].shape)
            wp, wm = [w.copy() for w in ws], [w.copy() for w in ws]
            wp[l][pos] += h
            wm[l][pos] -= h
            num = (loss(wp, bs) - loss(wm, bs)) / (2 * h)
            assert abs(num - dws[l][pos]) <= 1e-5 * max(1.0, abs(num)), (l, pos, num, dws[l][pos])
        for c in range(ch[l + 1]):
            bp, bm = [b.copy() for b in bs], [b.copy() for b in bs]
            bp[l][c] += h
            bm[l][c] -= h
            num = (loss(ws, bp) - loss(ws, bm)) / (2 * h)
            assert abs(num - dbs[l][c]) <= 1e-5 * max(1.0, abs(num)), (l, c, num, dbs[l][c])


def test_chain_matches_stack_for_max_blocks(oracle_mod):
    rng = np.random.default_rng(43)
    x = oracle_mod.round_to_bf16(rng.normal(size=(1, 8, 8, 8, 4)))
    ws = [oracle_mod.round_to_bf16(rng.normal(0, 0.2, size=(8, 3, 3, 3, 4))),
          oracle_mod.round_to_bf16(rng.normal(0, 0.1, size=(16, 3, 3, 3, 8)))]
    bs = [rng.normal(size=8), rng.normal(size=16)]
    dy = rng.normal(size=(1, 2, 2, 2, 16))
    specs = [(1, "max"), (1, "max")]
    xs, ys, auxs = oracle_mod.chain_fwd(x, ws, bs, 0.3, specs)
    sx, _, sy, sidx = oracle_mod.stack_fwd(x, ws, bs, 0.3)
    dws, dbs, dzs = oracle_mod.chain_bwd(xs, ys, auxs, ws, dy, 0.3, specs)
    sdw, sdb, sdz, _ = oracle_mod.stack_bwd(sx, sy, sidx, ws, dy, 0.3)
    for a, b in zip(ys + dws + dbs + dzs, sy + sdw + sdb + sdz):
        np.testing.assert_array_equal(a, b)


def test_table1_specs_reproduce_the_flop_rows():
    """The Table I chain specs (stride-2 c4, pooling while the width allows)
    give the printed forward FLOPs per sample."""
    import oracle
    from cnn_conv3d_gb300 import flops
    for wi in (128, 256, 512):
        specs = oracle.table1_specs(wi)
        s, tot = wi, 0
        for l, (stride, pool) in enumerate(specs):
            s //= stride
            tot += flops.conv_flops(1, oracle.TABLE1_CHANNELS[l], oracle.TABLE1_CHANNELS[l + 1], s ** 3)
            if pool != "none":
                s //= 2
        assert tot == flops.p3_table1_forward_flops(wi)
        assert s == 2  # 256 x 2^3 = 2048 inputs of fc1


# ----------------------------------------------------------------------------- batch normalisation

def test_bn_closed_forms(oracle_mod):
    """Normalised output: per-channel mean beta and variance gamma^2 *
    var/(var + eps); the backward's dz sums to zero per channel (shift
    invariance) and its projection on the normalised input is the closed form
    of scale invariance with eps."""
    rng = np.random.default_rng(51)
    z = rng.normal(3.0, 2.0, size=(2, 4, 3, 5, 6))
    g, b, eps = rng.normal(size=6), rng.normal(size=6), 1e-5
    u, mean, var = oracle_mod.bn_fwd(z, g, b, eps)
    zz = z.reshape(-1, 6)
    np.testing.assert_allclose(mean, zz.mean(0), rtol=1e-13)
    np.testing.assert_allclose(var, zz.var(0), rtol=1e-12)
    uu = u.reshape(-1, 6)
    np.testing.assert_allclose(uu.mean(0), b, atol=1e-12)
    np.testing.assert_allclose(uu.var(0), g ** 2 * var / (var + eps), rtol=1e-10)
    du = rng.normal(size=z.shape)
    dz, dg, db = oracle_mod.bn_bwd(z, du, g, eps)
    dzz = dz.reshape(-1, 6)
    np.testing.assert_allclose(dzz.sum(0), 0, atol=1e-10)
    zh = (zz - zz.mean(0)) / np.sqrt(zz.var(0) + eps)
    # scale invariance up to eps: sum(dz * zh) = g * dgamma * eps / ((var + eps) * sqrt(var + eps))
    np.testing.assert_allclose((dzz * zh).sum(0), g * dg * eps / ((var + eps) * np.sqrt(var + eps)),
                               rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(db, du.reshape(-1, 6).sum(0), rtol=1e-12)


def test_bn_chain_finite_differences(oracle_mod):
    """conv -> BN -> leaky ReLU -> max-pool, then conv -> BN -> leaky ReLU
    (unpooled): dW, dgamma, dbeta of both blocks against central differences
    of <g, y_top> (exact mode)."""
    slope = 0.3
    specs = [(1, "max", "bn"), (1, "none", "bn")]
    ch = (2, 3, 2)
    rng = np.random.default_rng(52)
    for _ in range(300):
        x = rng.normal(size=(2, 4, 4, 4, ch[0]))
        ws = [rng.normal(size=(ch[l + 1], 3, 3, 3, ch[l])) for l in range(2)]
        gs = [rng.normal(size=ch[l + 1]) for l in range(2)]
        bs = [rng.normal(size=ch[l + 1]) * 0.5 for l in range(2)]
        state = []
        xs, ys, auxs = oracle_mod.chain_fwd(x, ws, bs, slope, specs, mirrored=False, gammas=gs, bn_state=state)
        u0 = oracle_mod.bn_fwd(state[0][0], gs[0], bs[0])[0]
        u1 = oracle_mod.bn_fwd(state[1][0], gs[1], bs[1])[0]
        srt = np.sort(_window_view(u0), -1)
        if (np.min(srt[..., -1] - srt[..., -2]) > 1e-3 and np.min(np.abs(srt[..., -1])) > 1e-3
                and np.min(np.abs(u1)) > 1e-3 and np.any(u1 < 0) and np.any(srt[..., -1] < 0)):
            break
    else:
        pytest.fail("could not draw a kink-free case")
    g = rng.normal(size=ys[-1].shape)
    dgs = [None, None]
    dws, dbs, _ = oracle_mod.chain_bwd(xs, ys, auxs, ws, g, slope, specs, mirrored=False, gammas=gs,
                                       bn_state=state, dgammas=dgs)

    def loss(ws_, gs_, bs_):
        return np.vdot(g, oracle_mod.chain_fwd(x, ws_, bs_, slope, specs, mirrored=False, gammas=gs_)[1][-1])

    h = 1e-6
    for l in range(2):
        for _ in range(4):
            pos = tuple(rng.integers(0, s) for s in ws[l].shape)
            wp, wm = [w.copy() for w in ws], [w.copy() for w in ws]
            wp[l][pos] += h
            wm[l][pos] -= h
            num = (loss(wp, gs, bs) - loss(wm, gs, bs)) / (2 * h)
            assert abs(num - dws[l][pos]) <= 1e-5 * max(1.0, abs(num)), (l, pos, num, dws[l][pos])
        for c in range(ch[l + 1]):
            for arr, grad in ((gs, dgs[l]), (bs, dbs[l])):
                ap, am = [a.copy() for a in arr], [a.copy() for a in arr]
                ap[l][c] += h
                am[l][c] -= h
                if arr is gs:
                    num = (loss(ws, ap, bs) - loss(ws, am, bs)) / (2 * h)
                else:
                    num = (loss(ws, gs, ap) - loss(ws, gs, am)) / (2 * h)
                assert abs(num - grad[c]) <= 1e-5 * max(1.0, abs(num)), (l, c, num, grad[c])


# ----------------------------------------------------------------------------- rest of the network

def test_head_finite_differences(oracle_mod):
    """fc -> LReLU -> dropout -> fc -> LReLU -> dropout -> fc -> MSE: every
    weight, bias and input gradient against central differences."""
    rng = np.random.default_rng(61)
    M, F, H1, H2, O = 3, 10, 8, 6, 4
    fcs = [(rng.normal(size=(H1, F)), rng.normal(size=H1)), (rng.normal(size=(H2, H1)), rng.normal(size=H2)),
           (rng.normal(size=(O, H2)), rng.normal(size=O))]
    masks = [(rng.random((M, H1)) < 0.8).astype(np.uint8), (rng.random((M, H2)) < 0.8).astype(np.uint8)]
    feat, target = rng.normal(size=(M, F)), rng.normal(size=(M, O))
    keep, slope = 0.8, 0.3

    def loss(fcs_, feat_):
        return oracle_mod.mse(oracle_mod.head_fwd(feat_, fcs_, masks, keep, slope)[1], target)[0]

    hs, pred = oracle_mod.head_fwd(feat, fcs, masks, keep, slope)
    l0, dpred = oracle_mod.mse(pred, target)
    grads, dfeat = oracle_mod.head_bwd(hs, fcs, masks, keep, slope, dpred)
    h = 1e-6
    for i in range(3):
        for j in (0, 1):
            arr = fcs[i][j]
            for _ in range(4):
                pos = tuple(rng.integers(0, s) for s in arr.shape)
                fp = [[a.copy() for a in p] for p in fcs]
                fm = [[a.copy() for a in p] for p in fcs]
                fp[i][j][pos] += h
                fm[i][j][pos] -= h
                num = (loss(fp, feat) - loss(fm, feat)) / (2 * h)
                assert abs(num - grads[i][j][pos]) <= 1e-6 * max(1.0, abs(num)), (i, j, pos)
    for _ in range(5):
        pos = tuple(rng.integers(0, s) for s in feat.shape)
        fp, fm = feat.copy(), feat.copy()
        fp[pos] += h
        fm[pos] -= h
        num = (loss(fcs, fp) - loss(fcs, fm)) / (2 * h)
        assert abs(num - dfeat[pos]) <= 1e-6 * max(1.0, abs(num))


def test_adam_and_decay_closed_forms(oracle_mod):
    """Adam's first step from zero moments moves each weight by lr * g / (|g| +
    eps) (the bias corrections make m_hat = g, v_hat = g^2); with a constant
    gradient every later step moves by the same amount; the linear decay runs
    from lr0 to 0.01 lr0."""
    g = np.array([0.5, -2.0, 1e-3, 0.0])
    w = np.zeros(4)
    w1, m, v = oracle_mod.adam_step(w, g, np.zeros(4), np.zeros(4), lr=0.1, t=1)
    np.testing.assert_allclose(w1, -0.1 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(m, 0.1 * g)
    np.testing.assert_allclose(v, 0.001 * g * g)
    w2, _, _ = oracle_mod.adam_step(w1, g, m, v, lr=0.1, t=2)
    np.testing.assert_allclose(w2 - w1, -0.1 * g / (np.abs(g) + 1e-8), rtol=1e-9, atol=1e-15)
    assert oracle_mod.linear_decay_lr(2.0, 0, 100) == 2.0
    assert oracle_mod.linear_decay_lr(2.0, 100, 100) == pytest.approx(0.02)
    assert oracle_mod.linear_decay_lr(2.0, 50, 100) == pytest.approx(1.01)
    assert oracle_mod.linear_decay_lr(2.0, 500, 100) == pytest.approx(0.02)


def test_mse_closed_form(oracle_mod):
    pred = np.array([[1.0, 2.0], [3.0, 4.0]])
    tgt = np.array([[1.0, 0.0], [0.0, 0.0]])
    loss, d = oracle_mod.mse(pred, tgt)
    assert loss == pytest.approx((0 + 4 + 9 + 16) / 4)
    np.testing.assert_allclose(d, 2 * (pred - tgt) / 4)
