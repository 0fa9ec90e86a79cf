"""GPU parity of every entry point against the fp64 oracle on the same seeded
bf16 inputs, at sizes that span several tiles and a ragged tail.  Calls go
through the C ABI (ctypes binding)."""
import numpy as np
import pytest

import synthdata
from tests.gpu_util import assert_close, dev, dev_bf16, empty_bf16, guarded, host_bf16_f64

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


def _f64(o, u16):
    return o.bf16_bits_to_f64(u16)


def _ws(cf, op, desc):
    import torch
    n = max(cf.cf_workspace_size(op, desc), 256)
    return torch.empty((n,), dtype=torch.uint8, device="cuda"), n


def test_library_loaded_and_symbols(cf):
    import ctypes
    for name in cf.header_symbols():
        assert hasattr(cf._lib, name), name
    assert isinstance(cf._lib, ctypes.CDLL)


def test_wait_timeout_probe_reports_status(cf):
    import torch
    assert cf.cf_last_device_status() == cf.CF_OK
    cf.cf_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        cf.cf_debug_wait_timeout_probe()
        assert cf.cf_last_device_status() == cf.CF_ERR_TIMEOUT
        # the status word is cleared by the read and the context stays usable
        assert cf.cf_last_device_status() == cf.CF_OK
        t = torch.ones(16, device="cuda")
        assert float(t.sum()) == 16.0
    finally:
        cf.cf_set_wait_limit_ns(2_000_000_000)


def test_invalid_arguments_return_codes(cf):
    desc = cf.cf_conv_desc(1, 4, 4, 4, 32, 64)
    assert cf.cf_conv3d_fwd(desc, None, None, None, None, check=False) == cf.CF_ERR_INVALID_ARG
    import torch
    x = torch.empty(1 * 4 * 4 * 4 * 48, dtype=torch.bfloat16, device="cuda")
    w = torch.empty(64 * 27 * 48, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(4 * 4 * 4 * 64, dtype=torch.bfloat16, device="cuda")
    bad = cf.cf_conv_desc(1, 4, 4, 4, 40, 64)  # c_in 40: not 1, 4 or a multiple of 16
    assert cf.cf_conv3d_fwd(bad, x, w, None, y, check=False) == cf.CF_ERR_UNSUPPORTED
    bad = cf.cf_conv_desc(1, 4, 4, 4, 32, 72)  # c_out 72: not a multiple of 16
    assert cf.cf_conv3d_fwd(bad, x, w, None, y, check=False) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_conv3d_wgrad(bad, x, y, None, w, 0, x, 16, check=False) == cf.CF_ERR_UNSUPPORTED
    # misaligned pointer
    assert cf.cf_conv3d_fwd(desc, x.data_ptr() + 2, w, None, y, check=False) == cf.CF_ERR_INVALID_ARG
    # workspace too small
    dz = torch.empty(4 * 4 * 4 * 64, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(64 * 27 * 32, dtype=torch.float32, device="cuda")
    assert cf.cf_conv3d_wgrad(desc, x, dz, None, dw, 0, None, 0, check=False) == cf.CF_ERR_WORKSPACE


# ----------------------------------------------------------------------------- pooling

def test_pool_fwd_standalone(cf, oracle_mod):
    rng = np.random.default_rng(5)
    N, D, H, W, C = 2, 4, 6, 10, 24
    z16 = synthdata.to_bf16_bits(rng.normal(size=(N, D, H, W, C)))
    # plant exact ties in a few windows (the first maximum must win)
    z16[0, 0:2, 0:2, 0:2, 3] = z16[0, 0, 0, 0, 3]
    z16[1, 2:4, 2:4, 4:6, 5] = synthdata.to_bf16_bits(np.array([1.5]))[0]
    b = rng.normal(0, 0.1, size=C).astype(np.float32)
    import torch
    y, ycheck = guarded((N, D // 2, H // 2, W // 2, C), torch.bfloat16)
    idx, icheck = guarded(y.shape, torch.uint8)
    cf.cf_bias_lrelu_pool_fwd(N, D, H, W, C, dev_bf16(z16), dev(b), SLOPE, y, idx)
    ycheck("y")
    icheck("idx")
    ry, ridx = oracle_mod.pool_fwd(_f64(oracle_mod, z16), b.astype(np.float64), SLOPE)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    gy = host_bf16_f64(y)
    np.testing.assert_allclose(gy, ry, rtol=2 ** -8, atol=1e-30)


def test_pool_bwd_standalone(cf, oracle_mod):
    import torch
    rng = np.random.default_rng(6)
    N, D, H, W, C = 2, 4, 6, 10, 16
    z = rng.normal(size=(N, D, H, W, C))
    b = rng.normal(0, 0.1, size=C)
    ry, ridx = oracle_mod.pool_fwd(z, b, SLOPE)
    y16 = synthdata.to_bf16_bits(ry)
    dy16 = synthdata.to_bf16_bits(rng.normal(size=ry.shape))
    dz, dzcheck = guarded((N, D, H, W, C), torch.bfloat16, fill=7.0)
    dyp, dypcheck = guarded(ry.shape, torch.bfloat16)
    db, dbcheck = guarded((C,), torch.float32)
    ws, wsb = _ws(cf, cf.CF_OP_POOL_BWD, cf.cf_conv_desc(N, D, H, W, C, C))
    cf.cf_bias_lrelu_pool_bwd(N, D, H, W, C, dev_bf16(dy16), dev_bf16(y16), dev(ridx), SLOPE, dz, dyp, db, ws, wsb)
    dzcheck("dz")
    dypcheck("dy_pre")
    dbcheck("db")
    rdz, rdyp, rdb = oracle_mod.pool_bwd(_f64(oracle_mod, dy16), _f64(oracle_mod, y16), ridx, SLOPE)
    gdz = host_bf16_f64(dz)
    # same nonzero pattern (zeros everywhere but the argmax), values = bf16(g)
    np.testing.assert_array_equal(gdz == 0, rdz == 0)
    np.testing.assert_allclose(gdz, rdz, rtol=2 ** -8, atol=0)
    np.testing.assert_allclose(host_bf16_f64(dyp), rdyp, rtol=2 ** -8, atol=0)
    assert_close(db.cpu().numpy(), rdb, np.abs(rdyp).sum(axis=(0, 1, 2, 3)), "db")
    # the bias gradient left as per-block partial sums and reduced separately:
    # the same dz, dy_pre and db bits
    rows = cf.cf_pool_bwd_partial_rows()
    assert rows > 0
    part, pcheck = guarded((rows, C), torch.float32, fill=float("nan"))
    dz3, dy3 = empty_bf16((N, D, H, W, C)), empty_bf16(ry.shape)
    cf.cf_bias_lrelu_pool_bwd_partials(N, D, H, W, C, dev_bf16(dy16), dev_bf16(y16), dev(ridx), SLOPE, dz3, dy3, part)
    pcheck("partials")
    db3, db3check = guarded((C,), torch.float32, fill=float("nan"))
    cf.cf_column_sums(rows, C, part, db3)
    db3check("column sums")
    assert torch.equal(dz3, dz) and torch.equal(dy3, dyp) and torch.equal(db3, db)
    # y=None: dy is already the pre-activation gradient; no dbias
    dz2 = empty_bf16((N, D, H, W, C))
    cf.cf_bias_lrelu_pool_bwd(N, D, H, W, C, dyp, None, dev(ridx), SLOPE, dz2, None, None)
    np.testing.assert_array_equal(host_bf16_f64(dz2), gdz)


# ----------------------------------------------------------------------------- forward conv

FWD_SHAPES = [
    # N, D, H, W, Cin, Cout
    (2, 4, 6, 40, 32, 64),     # W ragged (40 = 32 + 8), several tiles in every dim
    (1, 4, 4, 16, 64, 128),
    (1, 2, 8, 8, 128, 256),
    (1, 2, 8, 8, 256, 256),
    (2, 4, 4, 12, 32, 32),
    (1, 2, 2, 8, 64, 16),
    (1, 2, 4, 8, 96, 96),      # three 32-channel K chunks, N tile 96
    (1, 2, 4, 8, 64, 512),     # two N tiles of 256
    (1, 4, 6, 16, 16, 32),     # 16-channel input (Table I c2: 16 -> 32): halo tile, 16-channel chunks
    (1, 2, 4, 24, 16, 48),     # 16-channel chunks, per-tap engine, N tile 48
    (1, 2, 6, 8, 48, 64),      # three 16-channel chunks, halo tile
    (2, 2, 4, 8, 32, 80),      # N tile 80
    (1, 6, 4, 16, 32, 64),     # halo tile: a full and a half tile in depth
    (1, 2, 4, 16, 64, 32),     # halo tile deeper than the volume, two chunks
    (1, 2, 16, 16, 128, 256),  # per-tap engine, N tile 256, several tiles per sample
    (1, 6, 18, 10, 32, 32),    # 4-plane halo tile ragged in d, h and w (pooled: all even)
    (1, 4, 16, 8, 32, 384),    # per-tap engine, two N tiles (256 + 128)
]


def _case(shape, seed):
    N, D, H, W, Ci, Co = shape
    return synthdata.random_case(seed, N, D, H, W, Ci, Co)


@pytest.mark.parametrize("shape", FWD_SHAPES)
def test_conv_fwd_plain(cf, oracle_mod, shape):
    N, D, H, W, Ci, Co = shape
    c = _case(shape, 100 + Ci + Co)
    import torch
    y, check = guarded((N, D, H, W, Co), torch.bfloat16, fill=float("nan"))
    cf.cf_conv3d_fwd(shape, dev_bf16(c["x"]), dev_bf16(c["w"]), None, y)
    check(f"fwd {shape}")
    x, w = _f64(oracle_mod, c["x"]), _f64(oracle_mod, c["w"])
    ref = oracle_mod.conv3d_fwd(x, w)
    S = oracle_mod.conv3d_fwd(np.abs(x), np.abs(w))
    assert_close(host_bf16_f64(y), ref, S, f"fwd {shape}")


def _check_pooled(oracle_mod, x, w, b, gy, gidx, what):
    z = oracle_mod.conv3d_fwd(x, w)
    S = oracle_mod.conv3d_fwd(np.abs(x), np.abs(w))
    ry, ridx = oracle_mod.pool_fwd(z, b, SLOPE)
    N, D, H, W, C = z.shape
    def win(a):
        return a.reshape(N, D // 2, 2, H // 2, 2, W // 2, 2, C).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(
            N, D // 2, H // 2, W // 2, C, 8)
    zw, sw = win(z), win(S)
    srt = np.sort(zw, axis=-1)
    gap = srt[..., -1] - srt[..., -2]
    s_at = np.take_along_axis(sw, ridx[..., None].astype(np.int64), -1)[..., 0] + np.abs(b)
    tol = 1e-2 * s_at
    notie = gap > tol
    np.testing.assert_array_equal(gidx[notie], ridx[notie])
    # where the pick differs (near-tie), the value must still be within tolerance
    assert_close(gy, ry, s_at, what)
    return int((~notie).sum())


@pytest.mark.parametrize("shape", FWD_SHAPES[:6] + FWD_SHAPES[8:])
def test_conv_fwd_pooled(cf, oracle_mod, shape):
    import torch
    N, D, H, W, Ci, Co = shape
    c = _case(shape, 200 + Ci + Co)
    y, ycheck = guarded((N, D // 2, H // 2, W // 2, Co), torch.bfloat16, fill=float("nan"))
    idx, icheck = guarded(y.shape, torch.uint8, fill=255)
    cf.cf_conv3d_fwd(shape, dev_bf16(c["x"]), dev_bf16(c["w"]), (dev(c["b"]), SLOPE, idx), y)
    ycheck(f"pooled y {shape}")
    icheck(f"pooled idx {shape}")
    x, w = _f64(oracle_mod, c["x"]), _f64(oracle_mod, c["w"])
    _check_pooled(oracle_mod, x, w, c["b"].astype(np.float64), host_bf16_f64(y), idx.cpu().numpy(),
                  f"pooled {shape}")


SMALLC_SHAPES = [
    (2, 4, 6, 40, 4, 32),
    (1, 4, 8, 16, 4, 16),
    (1, 2, 8, 8, 4, 64),
    (1, 16, 16, 16, 1, 8),  # the single-block CosmoFlow case: 1 -> 8 channels at 16^3
    (1, 4, 6, 24, 1, 16),
    (2, 2, 4, 10, 4, 32),   # ragged tile in w (10 = 8 + 2)
    # pooled: the first-layer quad-row forward (d even, h % 16 == 0, w % 32 == 0)
    (2, 4, 32, 64, 4, 32),  # several tiles in every dimension
    (1, 2, 16, 32, 4, 16),  # c_out 16: MMA width 64
    (1, 6, 16, 96, 4, 32),  # three tiles along w, three plane pairs
]


def test_smallc_row_alignment_rule(cf):
    import torch
    # c_in = 1 needs w a multiple of 8 (16-byte halo rows): rejected before any launch
    x = torch.empty(4 * 4 * 12, dtype=torch.bfloat16, device="cuda")
    w = torch.empty(16 * 27, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(4 * 4 * 12 * 16, dtype=torch.bfloat16, device="cuda")
    assert cf.cf_conv3d_fwd((1, 4, 4, 12, 1, 16), x, w, None, y, check=False) == cf.CF_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape", SMALLC_SHAPES)
@pytest.mark.parametrize("pooled", [False, True])
def test_conv_fwd_smallc(cf, oracle_mod, shape, pooled):
    import torch
    N, D, H, W, Ci, Co = shape
    c = _case(shape, 300 + Ci + Co)
    x, w = _f64(oracle_mod, c["x"]), _f64(oracle_mod, c["w"])
    if not pooled:
        y, check = guarded((N, D, H, W, Co), torch.bfloat16, fill=float("nan"))
        cf.cf_conv3d_fwd(shape, dev_bf16(c["x"]), dev_bf16(c["w"]), None, y)
        check(f"smallc fwd {shape}")
        ref = oracle_mod.conv3d_fwd(x, w)
        S = oracle_mod.conv3d_fwd(np.abs(x), np.abs(w))
        assert_close(host_bf16_f64(y), ref, S, f"smallc fwd {shape}")
    else:
        y, ycheck = guarded((N, D // 2, H // 2, W // 2, Co), torch.bfloat16, fill=float("nan"))
        idx, icheck = guarded(y.shape, torch.uint8, fill=255)
        cf.cf_conv3d_fwd(shape, dev_bf16(c["x"]), dev_bf16(c["w"]), (dev(c["b"]), SLOPE, idx), y)
        ycheck(f"smallc pooled y {shape}")
        icheck(f"smallc pooled idx {shape}")
        _check_pooled(oracle_mod, x, w, c["b"].astype(np.float64), host_bf16_f64(y), idx.cpu().numpy(),
                      f"smallc pooled {shape}")


# ----------------------------------------------------------------------------- backward data

DGRAD_SHAPES = [
    (2, 4, 6, 40, 32, 64),
    (1, 4, 4, 16, 64, 128),
    (1, 2, 8, 8, 128, 256),
    (1, 2, 8, 8, 256, 256),
    (1, 2, 4, 8, 16, 32),
    (1, 4, 6, 16, 16, 32),     # the Table I c2 layer: dX has 16 channels
    (1, 2, 4, 8, 48, 16),      # dZ has 16 channels: 16-channel K chunks
    (1, 2, 4, 16, 32, 80),     # dZ has 80 channels: five 16-channel chunks, halo tile
    (1, 6, 4, 16, 32, 64),     # halo tile (N 32, two chunks): a full and a half tile in depth
    (1, 6, 4, 8, 64, 128),     # halo tile (N 64, four chunks), ragged in depth
    (1, 2, 16, 8, 256, 64),    # dX has 256 channels: per-tap engine
    (1, 6, 6, 16, 64, 32),     # halo tile with N 64 (dX 64 channels from 32), ragged in depth
    (1, 5, 20, 12, 32, 48),    # 4-plane halo tile (N 32, three 16-channel chunks), ragged in d, h and w
]


@pytest.mark.parametrize("shape", DGRAD_SHAPES)
@pytest.mark.parametrize("with_act", [False, True])
def test_conv_dgrad(cf, oracle_mod, shape, with_act):
    N, D, H, W, Ci, Co = shape
    c = _case(shape, 400 + Ci + Co)
    desc = cf.cf_conv_desc(*shape)
    ws, wsb = _ws(cf, cf.CF_OP_DGRAD, desc)
    import torch
    dx, dxcheck = guarded((N, D, H, W, Ci), torch.bfloat16, fill=float("nan"))
    x_act = dev_bf16(c["x"]) if with_act else None
    dsum, scheck = guarded((Ci,), torch.float32, fill=float("nan"))
    cf.cf_conv3d_dgrad(desc, dev_bf16(c["dz"]), None, dev_bf16(c["w"]), x_act, SLOPE, dx, ws, wsb, dsum=dsum)
    dxcheck(f"dgrad dx {shape}")
    scheck(f"dgrad dsum {shape}")
    # dsum: channel sums of the stored dx (fused in the epilogue for c_in <= 32)
    got_dx = host_bf16_f64(dx)
    ref_sum = got_dx.reshape(-1, Ci).sum(0)
    np.testing.assert_allclose(dsum.cpu().numpy().astype(np.float64), ref_sum,
                               rtol=1e-5, atol=1e-5 * np.abs(got_dx).reshape(-1, Ci).sum(0).max())
    dz, w = _f64(oracle_mod, c["dz"]), _f64(oracle_mod, c["w"])
    ref = oracle_mod.conv3d_dgrad(dz, w)
    S = oracle_mod.conv3d_dgrad(np.abs(dz), np.abs(w))
    if with_act:
        f = np.where(_f64(oracle_mod, c["x"]) > 0, 1.0, SLOPE)
        ref, S = ref * f, S * f
    assert_close(host_bf16_f64(dx), ref, S, f"dgrad {shape} act={with_act}")
    # the filter flipped once (cf_filter_flip) and passed to the pre-flipped entry:
    # the flipped filter is the reversed-tap transpose, and dx and dsum are the same bits
    wt, wtc = guarded((Ci, 3, 3, 3, Co), torch.bfloat16, fill=float("nan"))
    cf.cf_filter_flip(Co, Ci, dev_bf16(c["w"]), wt)
    wtc("flipped filter")
    w16 = c["w"].reshape(Co, 27, Ci)
    want = w16[:, ::-1, :].transpose(2, 1, 0)
    assert np.array_equal(wt.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(Ci, 27, Co), want)
    dxf, dxfc = guarded((N, D, H, W, Ci), torch.bfloat16, fill=float("nan"))
    dsf, dsfc = guarded((Ci,), torch.float32, fill=float("nan"))
    cf.cf_conv3d_dgrad_flipped(desc, dev_bf16(c["dz"]), None, wt, x_act, SLOPE, dxf, ws, wsb, dsum=dsf)
    dxfc("flipped dgrad dx")
    dsfc("flipped dgrad dsum")
    assert torch.equal(dxf, dx) and torch.equal(dsf, dsum)
    if with_act:
        # the previous block's max-pool backward fused into the epilogue: the same
        # dx, and its routing by the codes equals the standalone pool backward's
        pidx = torch.from_numpy(np.random.default_rng(Ci).integers(0, 8, size=(N, D, H, W, Ci)).astype(np.uint8)).cuda()
        dx2, dx2c = guarded((N, D, H, W, Ci), torch.bfloat16, fill=float("nan"))
        pdz, pdzc = guarded((N, 2 * D, 2 * H, 2 * W, Ci), torch.bfloat16, fill=float("nan"))
        cf.cf_conv3d_dgrad_pool_bwd(desc, dev_bf16(c["dz"]), dev_bf16(c["w"]), x_act, SLOPE, dx2, pidx, pdz, ws, wsb)
        dx2c("fused dx")
        pdzc("fused routed dz")
        assert torch.equal(dx2, dx)
        rdz = empty_bf16((N, 2 * D, 2 * H, 2 * W, Ci))
        cf.cf_bias_lrelu_pool_bwd(N, 2 * D, 2 * H, 2 * W, Ci, dx, None, pidx, SLOPE, rdz, None, None)
        assert torch.equal(pdz, rdz)
    # dsum against the oracle: channel sums of the exact dx (each stored element
    # is within 1e-2*S of it, so the sums are within 1e-2 * sum(S))
    assert_close(dsum.cpu().numpy().astype(np.float64), ref.reshape(-1, Ci).sum(0), S.reshape(-1, Ci).sum(0),
                 f"dgrad dsum vs oracle {shape}")


# ----------------------------------------------------------------------------- backward weight

WGRAD_SHAPES = [
    (2, 4, 6, 40, 32, 64),
    (1, 4, 4, 16, 64, 128),
    (1, 2, 8, 8, 128, 256),
    (2, 2, 8, 8, 256, 256),
    (2, 4, 6, 40, 4, 32),
    (1, 4, 8, 16, 4, 16),
    (1, 8, 8, 8, 1, 16),
    (1, 2, 4, 8, 32, 192),
    (1, 2, 4, 16, 4, 128),     # small c_in with A in tensor memory, one accumulator per issuer
    (1, 2, 8, 24, 1, 64),
    (2, 2, 8, 16, 32, 32),     # halo-tile wgrad variants: 32 -> 32, 32 -> 128, 64 -> 64
    (1, 4, 20, 8, 32, 128),
    (1, 2, 4, 24, 64, 64),
    (1, 4, 6, 16, 16, 32),     # 16-channel input rows (Table I c2)
    (1, 2, 4, 8, 48, 48),      # N tile 48
    (1, 2, 4, 16, 32, 80),     # c_out 80 in a 96-wide tile (channels past c_out read as zero)
    (1, 2, 4, 8, 64, 320),     # two N tiles, the second mostly beyond c_out
    (1, 2, 4, 8, 32, 512),     # two full N tiles
    (1, 2, 4, 16, 4, 80),      # small c_in, c_out 80 in a 128-wide tile
    (1, 3, 6, 16, 32, 64),     # depth-stacked halo wgrad (c_in 32): odd depth, the last K block half empty
    (1, 5, 20, 24, 32, 32),    # depth-stacked, one output-channel set, ragged in d, h and w
    (1, 3, 20, 16, 64, 128),   # halo wgrad, 64-channel chunks, ragged in d, h and w
]


@pytest.mark.parametrize("shape", WGRAD_SHAPES)
def test_conv_wgrad(cf, oracle_mod, shape):
    import torch
    N, D, H, W, Ci, Co = shape
    c = _case(shape, 500 + Ci + Co)
    desc = cf.cf_conv_desc(*shape)
    ws, wsb = _ws(cf, cf.CF_OP_WGRAD, desc)
    dw, check = guarded((Co, 3, 3, 3, Ci), torch.float32, fill=float("nan"))
    cf.cf_conv3d_wgrad(desc, dev_bf16(c["x"]), dev_bf16(c["dz"]), None, dw, 0, ws, wsb)
    check(f"wgrad {shape}")
    x, dz = _f64(oracle_mod, c["x"]), _f64(oracle_mod, c["dz"])
    ref = oracle_mod.conv3d_wgrad(x, dz)
    S = oracle_mod.conv3d_wgrad(np.abs(x), np.abs(dz))
    g1 = dw.cpu().numpy().astype(np.float64)
    assert_close(g1, ref, S, f"wgrad {shape}")
    # accumulate=1 adds onto the existing values
    cf.cf_conv3d_wgrad(desc, dev_bf16(c["x"]), dev_bf16(c["dz"]), None, dw, 1, ws, wsb)
    assert_close(dw.cpu().numpy().astype(np.float64), 2 * ref, 2 * S, f"wgrad acc {shape}")


# ----------------------------------------------------------------------------- argmax-routed inputs

ROUTED_SHAPES = [
    (2, 4, 6, 40, 32, 64),
    (1, 4, 4, 16, 4, 32),      # small c_in: dZ expanded on chip by the weight-gradient kernel
    (2, 4, 6, 40, 4, 32),      # ragged box in w (40 = 2.5 boxes of 16)
    (1, 2, 8, 24, 1, 16),
    (1, 2, 4, 16, 4, 64),
    (1, 2, 4, 16, 4, 128),
    (1, 2, 4, 16, 4, 256),
    (1, 2, 4, 16, 4, 48),      # routed small c_in with a padded N tile
    (1, 2, 4, 16, 16, 32),     # 16-channel input, dZ expanded in the workspace
    # the first-layer quad-row weight gradient (c_in 4, c_out 32; h % 16 == 0, w % 32 == 0)
    (2, 4, 32, 64, 4, 32),
    (1, 6, 16, 96, 4, 32),
    (1, 2, 48, 32, 4, 32),
    (3, 16, 64, 96, 4, 32),    # 576 tiles: 3-4 per CTA, all three builder groups, stage and slot reuse
]


@pytest.mark.parametrize("shape", ROUTED_SHAPES)
def test_routed_gradients_match_dense(cf, oracle_mod, shape):
    import torch
    N, D, H, W, Ci, Co = shape
    rng = np.random.default_rng(77)
    c = _case(shape, 600 + Ci)
    z = rng.normal(size=(N, D, H, W, Co))
    _, ridx = oracle_mod.pool_fwd(z, None, SLOPE)
    g16 = synthdata.to_bf16_bits(rng.normal(size=ridx.shape))
    desc = cf.cf_conv_desc(*shape)
    rdz, _, _ = oracle_mod.pool_bwd(_f64(oracle_mod, g16), None, ridx, SLOPE)
    # wgrad from (g, idx)
    ws, wsb = _ws(cf, cf.CF_OP_WGRAD_ROUTED, desc)
    dw, check = guarded((Co, 3, 3, 3, Ci), torch.float32, fill=float("nan"))
    cf.cf_conv3d_wgrad(desc, dev_bf16(c["x"]), dev_bf16(g16), dev(ridx), dw, 0, ws, wsb)
    check("routed wgrad")
    x = _f64(oracle_mod, c["x"])
    ref = oracle_mod.conv3d_wgrad(x, rdz)
    S = oracle_mod.conv3d_wgrad(np.abs(x), np.abs(rdz))
    assert_close(dw.cpu().numpy().astype(np.float64), ref, S, "routed wgrad")
    cf.cf_conv3d_wgrad(desc, dev_bf16(c["x"]), dev_bf16(g16), dev(ridx), dw, 1, ws, wsb)
    assert_close(dw.cpu().numpy().astype(np.float64), 2 * ref, 2 * S, "routed wgrad acc")
    if Ci % 16 == 0 and Co % 32 == 0:
        ws, wsb = _ws(cf, cf.CF_OP_DGRAD_ROUTED, desc)
        dx, check = guarded((N, D, H, W, Ci), torch.bfloat16, fill=float("nan"))
        cf.cf_conv3d_dgrad(desc, dev_bf16(g16), dev(ridx), dev_bf16(c["w"]), None, SLOPE, dx, ws, wsb)
        check("routed dgrad")
        w = _f64(oracle_mod, c["w"])
        ref = oracle_mod.conv3d_dgrad(rdz, w)
        S = oracle_mod.conv3d_dgrad(np.abs(rdz), np.abs(w))
        assert_close(host_bf16_f64(dx), ref, S, "routed dgrad")


# ----------------------------------------------------------------------------- page variants

def _wins(a):
    N, D, H, W, C = a.shape
    return a.reshape(N, D // 2, 2, H // 2, 2, W // 2, 2, C).transpose(0, 1, 3, 5, 7, 2, 4, 6).reshape(
        N, D // 2, H // 2, W // 2, C, 8)


def _check_avgpooled(oracle_mod, z, S, b, gy, gmask, what):
    """Average of the activated window within 1e-2 of the window's mean S (the
    activation is 1-Lipschitz), and every sign bit whose pre-activation is
    farther than 1e-2 * S from zero equal to the oracle's."""
    ry, rmask = oracle_mod.avgpool_fwd(z, b, SLOPE)
    sw = _wins(S + np.abs(b))
    assert_close(gy, ry, sw.mean(-1), what)
    zb = _wins(z + b)
    sure = np.abs(zb) > 1e-2 * sw
    gb = (gmask[..., None].astype(np.int64) >> np.arange(8)) & 1
    rb = (rmask[..., None].astype(np.int64) >> np.arange(8)) & 1
    np.testing.assert_array_equal(gb[sure], rb[sure], err_msg=what)


VARIANT_FWD = [
    (2, 4, 6, 40, 4, 32),      # first-layer kernel (c_in 4)
    (1, 2, 16, 64, 4, 32),     # first-layer quad-row kernel (unpooled: bias + leaky ReLU; average: im2col kernel)
    (1, 4, 6, 16, 32, 64),     # halo tile
    (1, 2, 4, 8, 64, 256),     # per-tap engine
    (1, 4, 8, 16, 16, 32),     # halo tile, 16-channel chunks
]


@pytest.mark.parametrize("shape", VARIANT_FWD)
def test_conv_fwd_avgpool(cf, oracle_mod, shape):
    import torch
    N, D, H, W, Ci, Co = shape
    c = _case(shape, 700 + Ci + Co)
    y, ycheck = guarded((N, D // 2, H // 2, W // 2, Co), torch.bfloat16, fill=float("nan"))
    mask, mcheck = guarded(y.shape, torch.uint8, fill=0)
    cf.cf_conv3d_fwd(shape, dev_bf16(c["x"]), dev_bf16(c["w"]), (dev(c["b"]), SLOPE, mask, cf.CF_POOL_AVG), y)
    ycheck("avg y")
    mcheck("avg mask")
    x, w = _f64(oracle_mod, c["x"]), _f64(oracle_mod, c["w"])
    z = oracle_mod.conv3d_fwd(x, w)
    S = oracle_mod.conv3d_fwd(np.abs(x), np.abs(w))
    _check_avgpooled(oracle_mod, z, S, c["b"].astype(np.float64), host_bf16_f64(y), mask.cpu().numpy(),
                     f"avg-pooled {shape}")


@pytest.mark.parametrize("shape", VARIANT_FWD)
def test_conv_fwd_unpooled_activation(cf, oracle_mod, shape):
    import torch
    N, D, H, W, Ci, Co = shape
    c = _case(shape, 800 + Ci + Co)
    y, ycheck = guarded((N, D, H, W, Co), torch.bfloat16, fill=float("nan"))
    cf.cf_conv3d_fwd(shape, dev_bf16(c["x"]), dev_bf16(c["w"]), (dev(c["b"]), SLOPE, None, cf.CF_POOL_NONE), y)
    ycheck("act y")
    x, w = _f64(oracle_mod, c["x"]), _f64(oracle_mod, c["w"])
    b = c["b"].astype(np.float64)
    ref = oracle_mod.act_fwd(oracle_mod.conv3d_fwd(x, w), b, SLOPE)
    S = oracle_mod.conv3d_fwd(np.abs(x), np.abs(w)) + np.abs(b)
    assert_close(host_bf16_f64(y), ref, S, f"unpooled {shape}")


def test_block_epilogue_variants_standalone(cf, oracle_mod):
    import torch
    rng = np.random.default_rng(9)
    N, D, H, W, C = 2, 4, 6, 10, 24
    z16 = synthdata.to_bf16_bits(rng.normal(size=(N, D, H, W, C)))
    b = rng.normal(0, 0.3, size=C).astype(np.float32)
    z = _f64(oracle_mod, z16)
    bb = b.astype(np.float64)
    # average pooling: forward
    y, yc = guarded((N, D // 2, H // 2, W // 2, C), torch.bfloat16, fill=float("nan"))
    m, mc = guarded(y.shape, torch.uint8)
    cf.cf_block_epilogue_fwd(cf.CF_POOL_AVG, N, D, H, W, C, dev_bf16(z16), dev(b), SLOPE, y, m)
    yc("avg y")
    mc("avg mask")
    _check_avgpooled(oracle_mod, z, np.abs(z), bb, host_bf16_f64(y), m.cpu().numpy(), "standalone avg")
    # average pooling: backward from the GPU's own masks
    dy16 = synthdata.to_bf16_bits(rng.normal(size=y.shape))
    gmask = m.cpu().numpy()
    dz, dzc = guarded((N, D, H, W, C), torch.bfloat16, fill=float("nan"))
    db, dbc = guarded((C,), torch.float32, fill=float("nan"))
    ws, wsb = _ws(cf, cf.CF_OP_POOL_BWD, cf.cf_conv_desc(N, D, H, W, C, C))
    cf.cf_block_epilogue_bwd(cf.CF_POOL_AVG, N, D, H, W, C, dev_bf16(dy16), None, m, SLOPE, dz, None, db, ws, wsb)
    dzc("avg dz")
    dbc("avg db")
    rdz, rdb = oracle_mod.avgpool_bwd(_f64(oracle_mod, dy16), gmask, SLOPE)
    np.testing.assert_allclose(host_bf16_f64(dz), rdz, rtol=2 ** -8, atol=0)
    assert_close(db.cpu().numpy(), rdb, np.abs(rdz).reshape(-1, C).sum(0), "avg db")
    # no pooling: forward and backward (with the output, and with y = NULL)
    ya, yac = guarded((N, D, H, W, C), torch.bfloat16, fill=float("nan"))
    cf.cf_block_epilogue_fwd(cf.CF_POOL_NONE, N, D, H, W, C, dev_bf16(z16), dev(b), SLOPE, ya, None)
    yac("act y")
    ry = oracle_mod.act_fwd(z, bb, SLOPE)
    np.testing.assert_allclose(host_bf16_f64(ya), ry, rtol=2 ** -8, atol=1e-30)
    g16 = synthdata.to_bf16_bits(rng.normal(size=(N, D, H, W, C)))
    dz2, dz2c = guarded((N, D, H, W, C), torch.bfloat16, fill=float("nan"))
    cf.cf_block_epilogue_bwd(cf.CF_POOL_NONE, N, D, H, W, C, dev_bf16(g16), ya, None, SLOPE, dz2, None, db, ws, wsb)
    dz2c("act dz")
    rdz2, rdb2 = oracle_mod.act_bwd(_f64(oracle_mod, g16), host_bf16_f64(ya), SLOPE)
    np.testing.assert_allclose(host_bf16_f64(dz2), rdz2, rtol=2 ** -8, atol=0)
    assert_close(db.cpu().numpy(), rdb2, np.abs(rdz2).reshape(-1, C).sum(0), "act db")
    cf.cf_block_epilogue_bwd(cf.CF_POOL_NONE, N, D, H, W, C, dev_bf16(g16), None, None, SLOPE, dz2, None, None)
    np.testing.assert_array_equal(host_bf16_f64(dz2), _f64(oracle_mod, g16))


STRIDE2_SHAPES = [
    # N, D, H, W (input), Cin, Cout
    (1, 8, 8, 16, 32, 64),
    (2, 6, 10, 8, 16, 48),     # odd output sizes (3, 5, 4)
    (1, 16, 16, 16, 64, 128),  # the Table I c4 layer at batch 1
]


@pytest.mark.parametrize("shape", STRIDE2_SHAPES)
def test_stride2_conv(cf, oracle_mod, shape):
    import torch
    N, D, H, W, Ci, Co = shape
    Do, Ho, Wo = (D + 1) // 2, (H + 1) // 2, (W + 1) // 2
    c = _case(shape, 900 + Ci + Co)
    desc = cf.cf_conv_desc(N, D, H, W, Ci, Co, 2)
    x16, w16 = c["x"], c["w"]
    x, w = _f64(oracle_mod, x16), _f64(oracle_mod, w16)
    # forward, plain
    y, yc = guarded((N, Do, Ho, Wo, Co), torch.bfloat16, fill=float("nan"))
    cf.cf_conv3d_fwd(desc, dev_bf16(x16), dev_bf16(w16), None, y)
    yc("stride-2 y")
    ref = oracle_mod.conv3d_fwd_s2(x, w)
    S = oracle_mod.conv3d_fwd_s2(np.abs(x), np.abs(w))
    assert_close(host_bf16_f64(y), ref, S, f"stride-2 fwd {shape}")
    # forward with the pooled epilogue (even output sizes only)
    if Do % 2 == 0 and Ho % 2 == 0 and Wo % 2 == 0:
        yp, ypc = guarded((N, Do // 2, Ho // 2, Wo // 2, Co), torch.bfloat16, fill=float("nan"))
        idx, ic = guarded(yp.shape, torch.uint8, fill=255)
        cf.cf_conv3d_fwd(desc, dev_bf16(x16), dev_bf16(w16), (dev(c["b"]), SLOPE, idx), yp)
        ypc("stride-2 pooled y")
        ic("stride-2 idx")
        bb = c["b"].astype(np.float64)
        ry, ridx = oracle_mod.pool_fwd(ref, bb, SLOPE)
        zw, sw = _wins(ref), _wins(S)
        srt = np.sort(zw, -1)
        s_at = np.take_along_axis(sw, ridx[..., None].astype(np.int64), -1)[..., 0] + np.abs(bb)
        notie = (srt[..., -1] - srt[..., -2]) > 1e-2 * s_at
        np.testing.assert_array_equal(idx.cpu().numpy()[notie], ridx[notie])
        assert_close(host_bf16_f64(yp), ry, s_at, f"stride-2 pooled {shape}")
    # backward data (with the previous block's leaky-ReLU derivative) and weight
    dz16 = synthdata.to_bf16_bits(np.random.default_rng(Ci).normal(size=(N, Do, Ho, Wo, Co)))
    dzf = _f64(oracle_mod, dz16)
    ws, wsb = _ws(cf, cf.CF_OP_DGRAD, desc)
    dx, dxc = guarded((N, D, H, W, Ci), torch.bfloat16, fill=float("nan"))
    cf.cf_conv3d_dgrad(desc, dev_bf16(dz16), None, dev_bf16(w16), dev_bf16(x16), SLOPE, dx, ws, wsb)
    dxc("stride-2 dx")
    f = np.where(x > 0, 1.0, SLOPE)
    ref = oracle_mod.conv3d_dgrad_s2(dzf, w, (D, H, W)) * f
    S = oracle_mod.conv3d_dgrad_s2(np.abs(dzf), np.abs(w), (D, H, W)) * f
    assert_close(host_bf16_f64(dx), ref, S, f"stride-2 dgrad {shape}")
    ws, wsb = _ws(cf, cf.CF_OP_WGRAD, desc)
    dw, dwc = guarded((Co, 3, 3, 3, Ci), torch.float32, fill=float("nan"))
    cf.cf_conv3d_wgrad(desc, dev_bf16(x16), dev_bf16(dz16), None, dw, 0, ws, wsb)
    dwc("stride-2 dw")
    ref = oracle_mod.conv3d_wgrad_s2(x, dzf)
    S = oracle_mod.conv3d_wgrad_s2(np.abs(x), np.abs(dzf))
    assert_close(dw.cpu().numpy().astype(np.float64), ref, S, f"stride-2 wgrad {shape}")
