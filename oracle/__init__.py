"""fp64 CPU oracle for the CosmoFlow conv3d block -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never links or
calls it, and it imports nothing from the product package.

The arithmetic lives in ``cf_oracle.c`` (direct nested loops in double
precision, see its header for the sources and the readings of the pages).
This module only compiles it with gcc, marshals numpy arrays, and chains the
per-layer routines into the five-block stack ("mirrored" mode rounds the
tensors that cross a block boundary to bf16 at the same points where the GPU
path stores bf16).

Parity of every routine is pinned in ``tests/test_oracle_pins.py`` against
things other than the oracle itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cf_oracle.c")
_LIB = os.path.join(_HERE, "libcforacle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_I64 = ctypes.POINTER(ctypes.c_int64)
_F32 = ctypes.POINTER(ctypes.c_float)
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math).  Returns the path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dims = [_i64, _i64, _i64, _i64, _i32, _i32]
        lib.oracle_conv3d_fwd.argtypes = dims + [_D, _D, _D]
        lib.oracle_conv3d_dgrad.argtypes = dims + [_D, _D, _D]
        lib.oracle_conv3d_wgrad.argtypes = dims + [_D, _D, _D]
        pdims = [_i64, _i64, _i64, _i64, _i32]
        lib.oracle_pool_fwd.argtypes = pdims + [_D, _D, ctypes.c_double, _D, _U8]
        lib.oracle_pool_bwd.argtypes = pdims + [_D, _D, _U8, ctypes.c_double, _D, _D, _D]
        pts = [_i64, _I64, _D, _D]
        lib.oracle_conv3d_fwd_pts_bf16.argtypes = dims + [_U16, _U16] + pts
        lib.oracle_conv3d_dgrad_pts_bf16.argtypes = dims + [_U16, _U16] + pts
        lib.oracle_conv3d_wgrad_pts_bf16.argtypes = dims + [_U16, _U16] + pts
        lib.oracle_block_fwd_pts_bf16.argtypes = dims + [_U16, _U16, _F32, ctypes.c_double,
                                                         _i64, _I64, _D, _U8, _D, _D]
        lib.oracle_conv3d_wgrad_routed_pts_bf16.argtypes = dims + [_U16, _U16, _U8] + pts
        lib.oracle_avgpool_fwd.argtypes = pdims + [_D, _D, ctypes.c_double, _D, _U8]
        lib.oracle_avgpool_bwd.argtypes = pdims + [_D, _U8, ctypes.c_double, _D, _D]
        lib.oracle_act_fwd.argtypes = [_i64, _i32, _D, _D, ctypes.c_double, _D]
        lib.oracle_act_bwd.argtypes = [_i64, _i32, _D, _D, ctypes.c_double, _D, _D]
        lib.oracle_conv3d_fwd_s2.argtypes = dims + [_D, _D, _D]
        lib.oracle_conv3d_dgrad_s2.argtypes = dims + [_D, _D, _D]
        lib.oracle_conv3d_wgrad_s2.argtypes = dims + [_D, _D, _D]
        lib.oracle_bn_fwd.argtypes = [_i64, _i32, _D, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_bn_bwd.argtypes = [_i64, _i32, _D, _D, _D, ctypes.c_double, _D, _D, _D]
        lib.oracle_bn_fwd.restype = lib.oracle_bn_bwd.restype = None
        for f in (lib.oracle_avgpool_fwd, lib.oracle_avgpool_bwd, lib.oracle_act_fwd, lib.oracle_act_bwd,
                  lib.oracle_conv3d_fwd_s2, lib.oracle_conv3d_dgrad_s2, lib.oracle_conv3d_wgrad_s2):
            f.restype = None
        for f in (lib.oracle_conv3d_fwd, lib.oracle_conv3d_dgrad, lib.oracle_conv3d_wgrad,
                  lib.oracle_pool_fwd, lib.oracle_pool_bwd, lib.oracle_conv3d_fwd_pts_bf16,
                  lib.oracle_conv3d_dgrad_pts_bf16, lib.oracle_conv3d_wgrad_pts_bf16,
                  lib.oracle_block_fwd_pts_bf16, lib.oracle_conv3d_wgrad_routed_pts_bf16):
            f.restype = None
        _lib = lib
    return _lib


def _p(a, t):
    return a.ctypes.data_as(t) if a is not None else None


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u = np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (via fp32, round-to-nearest-even at each
    step) and return the rounded values as float64.  Used by mirrored mode."""
    f = np.ascontiguousarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32)
    nan = np.isnan(f)
    r = np.where(nan, (f.view(np.uint32) >> 16) | 0x40, r).astype(np.uint32)
    return (r << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# full-tensor routines (float64 in, float64 out; NDHWC / [Co][3][3][3][Ci])

def conv3d_fwd(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """z = cross-correlation of x [N,D,H,W,Ci] with w [Co,3,3,3,Ci], pad 1."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    N, D, H, W, Ci = x.shape
    Co = w.shape[0]
    assert w.shape == (Co, 3, 3, 3, Ci)
    z = np.empty((N, D, H, W, Co), np.float64)
    lib.oracle_conv3d_fwd(N, D, H, W, Ci, Co, _p(x, _D), _p(w, _D), _p(z, _D))
    return z


def conv3d_dgrad(dz: np.ndarray, w: np.ndarray) -> np.ndarray:
    """dx [N,D,H,W,Ci] from dz [N,D,H,W,Co] and w [Co,3,3,3,Ci]."""
    lib = _load()
    dz, w = _f64(dz), _f64(w)
    N, D, H, W, Co = dz.shape
    Ci = w.shape[4]
    assert w.shape == (Co, 3, 3, 3, Ci)
    dx = np.empty((N, D, H, W, Ci), np.float64)
    lib.oracle_conv3d_dgrad(N, D, H, W, Ci, Co, _p(dz, _D), _p(w, _D), _p(dx, _D))
    return dx


def conv3d_wgrad(x: np.ndarray, dz: np.ndarray) -> np.ndarray:
    """dW [Co,3,3,3,Ci] from x [N,D,H,W,Ci] and dz [N,D,H,W,Co]."""
    lib = _load()
    x, dz = _f64(x), _f64(dz)
    N, D, H, W, Ci = x.shape
    Co = dz.shape[4]
    dw = np.empty((Co, 3, 3, 3, Ci), np.float64)
    lib.oracle_conv3d_wgrad(N, D, H, W, Ci, Co, _p(x, _D), _p(dz, _D), _p(dw, _D))
    return dw


def pool_fwd(z: np.ndarray, bias, slope: float):
    """(y, idx) = bias + leaky ReLU + 2x2x2 max-pool of z [N,D,H,W,C]."""
    lib = _load()
    z = _f64(z)
    N, D, H, W, C = z.shape
    b = None if bias is None else _f64(bias)
    y = np.empty((N, D // 2, H // 2, W // 2, C), np.float64)
    idx = np.empty((N, D // 2, H // 2, W // 2, C), np.uint8)
    lib.oracle_pool_fwd(N, D, H, W, C, _p(z, _D), _p(b, _D), slope, _p(y, _D), _p(idx, _U8))
    return y, idx


def pool_bwd(dy: np.ndarray, y, idx: np.ndarray, slope: float, want_dz: bool = True):
    """(dz, dy_pre, db) of the pool/LReLU stage; y=None means dy is already the
    gradient w.r.t. the pooled pre-activation.  want_dz=False skips the
    full-resolution dz (returned as None)."""
    lib = _load()
    dy = _f64(dy)
    N, D2, H2, W2, C = dy.shape
    yy = None if y is None else _f64(y)
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    dz = np.empty((N, 2 * D2, 2 * H2, 2 * W2, C), np.float64) if want_dz else None
    dyp = np.empty_like(dy)
    db = np.empty((C,), np.float64)
    lib.oracle_pool_bwd(N, 2 * D2, 2 * H2, 2 * W2, C, _p(dy, _D), _p(yy, _D), _p(idx, _U8), slope,
                        _p(dz, _D), _p(dyp, _D), _p(db, _D))
    return dz, dyp, db


def avgpool_fwd(z: np.ndarray, bias, slope: float):
    """(y, mask) = 2x2x2 average of LReLU(z + b) and the per-window bits of
    z + b > 0 (bit dd*4+dh*2+dw)."""
    lib = _load()
    z = _f64(z)
    N, D, H, W, C = z.shape
    b = None if bias is None else _f64(bias)
    y = np.empty((N, D // 2, H // 2, W // 2, C), np.float64)
    mask = np.empty((N, D // 2, H // 2, W // 2, C), np.uint8)
    lib.oracle_avgpool_fwd(N, D, H, W, C, _p(z, _D), _p(b, _D), slope, _p(y, _D), _p(mask, _U8))
    return y, mask


def avgpool_bwd(dy: np.ndarray, mask: np.ndarray, slope: float):
    """(dz, db) of the average-pool block: dz = dy/8 * LReLU'(z+b) per voxel."""
    lib = _load()
    dy = _f64(dy)
    N, D2, H2, W2, C = dy.shape
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    dz = np.empty((N, 2 * D2, 2 * H2, 2 * W2, C), np.float64)
    db = np.empty((C,), np.float64)
    lib.oracle_avgpool_bwd(N, 2 * D2, 2 * H2, 2 * W2, C, _p(dy, _D), _p(mask, _U8), slope, _p(dz, _D), _p(db, _D))
    return dz, db


def act_fwd(z: np.ndarray, bias, slope: float):
    """y = LReLU(z + b) (an unpooled block)."""
    lib = _load()
    z = _f64(z)
    C = z.shape[-1]
    b = None if bias is None else _f64(bias)
    y = np.empty_like(z)
    lib.oracle_act_fwd(z.size, C, _p(z, _D), _p(b, _D), slope, _p(y, _D))
    return y


def act_bwd(dy: np.ndarray, y: np.ndarray, slope: float):
    """(dz, db) of an unpooled block: dz = dy * LReLU'(y)."""
    lib = _load()
    dy, y = _f64(dy), _f64(y)
    C = dy.shape[-1]
    dz = np.empty_like(dy)
    db = np.empty((C,), np.float64)
    lib.oracle_act_bwd(dy.size, C, _p(dy, _D), _p(y, _D), slope, _p(dz, _D), _p(db, _D))
    return dz, db


def bn_fwd(z: np.ndarray, gamma, beta, eps: float = 1e-5):
    """(u, mean, var): batch normalisation of z [..., C] with the batch's
    per-channel statistics (biased variance)."""
    lib = _load()
    z = _f64(z)
    C = z.shape[-1]
    u = np.empty_like(z)
    mean, var = np.empty(C), np.empty(C)
    lib.oracle_bn_fwd(z.size // C, C, _p(z, _D), _p(_f64(gamma), _D), _p(_f64(beta), _D), eps, _p(u, _D),
                      _p(mean, _D), _p(var, _D))
    return u, mean, var


def bn_bwd(z: np.ndarray, du: np.ndarray, gamma, eps: float = 1e-5):
    """(dz, dgamma, dbeta) of bn_fwd (training mode)."""
    lib = _load()
    z, du = _f64(z), _f64(du)
    C = z.shape[-1]
    dz = np.empty_like(z)
    dg, db = np.empty(C), np.empty(C)
    lib.oracle_bn_bwd(z.size // C, C, _p(z, _D), _p(du, _D), _p(_f64(gamma), _D), eps, _p(dz, _D), _p(dg, _D),
                      _p(db, _D))
    return dz, dg, db


def conv3d_fwd_s2(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Stride-2 cross-correlation, pad 1: z [N, (D+1)/2, (H+1)/2, (W+1)/2, Co]."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    N, D, H, W, Ci = x.shape
    Co = w.shape[0]
    z = np.empty((N, (D + 1) // 2, (H + 1) // 2, (W + 1) // 2, Co), np.float64)
    lib.oracle_conv3d_fwd_s2(N, D, H, W, Ci, Co, _p(x, _D), _p(w, _D), _p(z, _D))
    return z


def conv3d_dgrad_s2(dz: np.ndarray, w: np.ndarray, in_shape) -> np.ndarray:
    """dx [N,D,H,W,Ci] of the stride-2 conv (in_shape = (D, H, W) of its input)."""
    lib = _load()
    dz, w = _f64(dz), _f64(w)
    N, Co = dz.shape[0], dz.shape[4]
    D, H, W = in_shape
    Ci = w.shape[4]
    dx = np.empty((N, D, H, W, Ci), np.float64)
    lib.oracle_conv3d_dgrad_s2(N, D, H, W, Ci, Co, _p(dz, _D), _p(w, _D), _p(dx, _D))
    return dx


def conv3d_wgrad_s2(x: np.ndarray, dz: np.ndarray) -> np.ndarray:
    """dW of the stride-2 conv from its input x and output gradient dz."""
    lib = _load()
    x, dz = _f64(x), _f64(dz)
    N, D, H, W, Ci = x.shape
    Co = dz.shape[4]
    dw = np.empty((Co, 3, 3, 3, Ci), np.float64)
    lib.oracle_conv3d_wgrad_s2(N, D, H, W, Ci, Co, _p(x, _D), _p(dz, _D), _p(dw, _D))
    return dw


# ----------------------------------------------------------------------------
# sampled routines on bf16 bit patterns (for sizes too large for full fp64)

def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def conv3d_fwd_pts(x16, w16, pts):
    """Exact z and S = sum|w*x| at points (n,d,h,w,co)."""
    lib = _load()
    x16, w16 = _u16(x16), _u16(w16)
    N, D, H, W, Ci = x16.shape
    Co = w16.shape[0]
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 5)
    out = np.empty(len(pts)); s = np.empty(len(pts))
    lib.oracle_conv3d_fwd_pts_bf16(N, D, H, W, Ci, Co, _p(x16, _U16), _p(w16, _U16), len(pts),
                                   _p(pts, _I64), _p(out, _D), _p(s, _D))
    return out, s


def conv3d_dgrad_pts(dz16, w16, pts):
    """Exact dx and S = sum|w*dz| at points (n,d,h,w,ci)."""
    lib = _load()
    dz16, w16 = _u16(dz16), _u16(w16)
    N, D, H, W, Co = dz16.shape
    Ci = w16.shape[4]
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 5)
    out = np.empty(len(pts)); s = np.empty(len(pts))
    lib.oracle_conv3d_dgrad_pts_bf16(N, D, H, W, Ci, Co, _p(dz16, _U16), _p(w16, _U16), len(pts),
                                     _p(pts, _I64), _p(out, _D), _p(s, _D))
    return out, s


def conv3d_wgrad_pts(x16, dz16, pts):
    """Exact dW and S = sum|dz*x| at points (co,kd,kh,kw,ci)."""
    lib = _load()
    x16, dz16 = _u16(x16), _u16(dz16)
    N, D, H, W, Ci = x16.shape
    Co = dz16.shape[4]
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 5)
    out = np.empty(len(pts)); s = np.empty(len(pts))
    lib.oracle_conv3d_wgrad_pts_bf16(N, D, H, W, Ci, Co, _p(x16, _U16), _p(dz16, _U16), len(pts),
                                     _p(pts, _I64), _p(out, _D), _p(s, _D))
    return out, s


def conv3d_wgrad_routed_pts(x16, g16, idx, pts):
    """Exact dW and S at points (co,kd,kh,kw,ci) when dZ is the argmax-routed
    expansion of the pooled gradient g16 [n][d/2][h/2][w/2][co] by the codes idx."""
    lib = _load()
    x16, g16 = _u16(x16), _u16(g16)
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    N, D, H, W, Ci = x16.shape
    Co = g16.shape[4]
    assert g16.shape == (N, D // 2, H // 2, W // 2, Co) and idx.shape == g16.shape
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 5)
    out = np.empty(len(pts)); s = np.empty(len(pts))
    lib.oracle_conv3d_wgrad_routed_pts_bf16(N, D, H, W, Ci, Co, _p(x16, _U16), _p(g16, _U16), _p(idx, _U8),
                                            len(pts), _p(pts, _I64), _p(out, _D), _p(s, _D))
    return out, s


def conv3d_wgrad_mm(x, dz, x_below=None, x_above=None):
    """dW [Co,3,3,3,Ci] = sum over n and voxels of dz[n,v,co] * x[n,v+t-1,ci],
    one matrix product per tap t (numpy matmul of the flattened dz with the
    tap-shifted x; x zero outside the volume).  x_below / x_above: the plane
    of a taller volume just below / above the d-range of x and dz ([N,H,W,Ci]),
    zero when None, so that slabs of a volume can be summed one at a time."""
    x, dz = _f64(x), _f64(dz)
    N, D, H, W, Ci = x.shape
    Co = dz.shape[4]
    xp = np.zeros((N, D + 2, H + 2, W + 2, Ci))
    xp[:, 1:D + 1, 1:H + 1, 1:W + 1, :] = x
    if x_below is not None:
        xp[:, 0, 1:H + 1, 1:W + 1, :] = x_below
    if x_above is not None:
        xp[:, D + 1, 1:H + 1, 1:W + 1, :] = x_above
    g = dz.reshape(-1, Co).T
    dw = np.empty((Co, 3, 3, 3, Ci))
    for kd in range(3):
        for kh in range(3):
            for kw in range(3):
                xs = np.ascontiguousarray(xp[:, kd:kd + D, kh:kh + H, kw:kw + W, :]).reshape(-1, Ci)
                dw[:, kd, kh, kw, :] = g @ xs
    return dw


def block_fwd_pts(x16, w16, bias, slope, pts):
    """Fused block at pooled points (n,pd,ph,pw,co): (y, idx, S, top-two gap)."""
    lib = _load()
    x16, w16 = _u16(x16), _u16(w16)
    N, D, H, W, Ci = x16.shape
    Co = w16.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 5)
    n = len(pts)
    y = np.empty(n); idx = np.empty(n, np.uint8); s = np.empty(n); gap = np.empty(n)
    lib.oracle_block_fwd_pts_bf16(N, D, H, W, Ci, Co, _p(x16, _U16), _p(w16, _U16), _p(b, _F32),
                                  slope, n, _p(pts, _I64), _p(y, _D), _p(idx, _U8), _p(s, _D),
                                  _p(gap, _D))
    return y, idx, s, gap


# ----------------------------------------------------------------------------
# the stack (config-level chains)

def block_fwd(x, w, bias, slope):
    """One block: z = conv(x, w); (y, idx) = pool(z + b) with LReLU.  Returns
    (z, y, idx)."""
    z = conv3d_fwd(x, w)
    y, idx = pool_fwd(z, bias, slope)
    return z, y, idx


def stack_fwd(x, ws, bs, slope, mirrored=True):
    """Forward through the blocks.  In mirrored mode each block output is
    rounded to bf16 before it feeds the next block (as the GPU stores it).
    Returns lists (xs, zs, ys, idxs) with xs[l] the input of block l."""
    xs, zs, ys, idxs = [], [], [], []
    cur = _f64(x)
    for w, b in zip(ws, bs):
        xs.append(cur)
        z, y, idx = block_fwd(cur, w, b, slope)
        if mirrored:
            y = round_to_bf16(y)
        zs.append(z); ys.append(y); idxs.append(idx)
        cur = y
    return xs, zs, ys, idxs


def stack_bwd(xs, ys, idxs, ws, dy, slope, mirrored=True):
    """Backward through the blocks from dy at the last pooled output.
    Returns per block (dW, db) and the dense dZ of each block, plus the
    gradient w.r.t. each block's input (None for block 0, never computed)."""
    L = len(ws)
    dws, dbs, dzs, dxs = [None] * L, [None] * L, [None] * L, [None] * L
    g = _f64(dy)
    use_y = True
    for l in range(L - 1, -1, -1):
        dz, dyp, db = pool_bwd(g, ys[l] if use_y else None, idxs[l], slope)
        if mirrored:
            dz = round_to_bf16(dz)
        dzs[l], dbs[l] = dz, db
        dws[l] = conv3d_wgrad(xs[l], dz)
        if l > 0:
            dx = conv3d_dgrad(dz, ws[l])
            # LReLU' of the previous block's activation (= this block's input)
            g = dx * np.where(xs[l] > 0, 1.0, slope)
            if mirrored:
                g = round_to_bf16(g)
            dxs[l] = g
            use_y = False
    return dws, dbs, dzs, dxs


# ----------------------------------------------------------------------------
# general chain: per-block stride (1 or 2) and pooling ("max", "avg", "none")

def _upsample2(dz, out_shape):
    """Zero-insertion of a stride-2 output gradient at the even positions of the
    input grid (out_shape = (D, H, W))."""
    N, _, _, _, C = dz.shape
    D, H, W = out_shape
    up = np.zeros((N, D, H, W, C))
    up[:, ::2, ::2, ::2, :] = dz
    return up


def chain_fwd(x, ws, bs, slope, specs, mirrored=True, gammas=None, bn_state=None):
    """Blocks conv (stride s) -> + b -> leaky ReLU -> pooling, one spec
    (stride, pool) per block, pool in {"max", "avg", "none"}.  Max pooling is
    taken before the activation (equal by monotonicity), average pooling after
    it (CosmoFlow page, section III-A/III-C).  A spec (stride, pool, "bn")
    puts batch normalisation between the conv and the activation
    (hybrid-parallelism page, section IV): z = conv(x) (stored bf16 in
    mirrored mode), u = gammas[l] * zh + bs[l] (bs[l] is the BN shift beta),
    then the activation and pooling of u; bn_state (a list) receives (z, mean,
    var) per BN block.  Returns (xs, ys, auxs): block inputs, outputs
    (bf16-rounded in mirrored mode) and the argmax codes (max) or
    pre-activation sign masks (avg) or None."""
    xs, ys, auxs = [], [], []
    cur = _f64(x)
    for l, (spec, w, b) in enumerate(zip(specs, ws, bs)):
        stride, pool = spec[0], spec[1]
        xs.append(cur)
        z = conv3d_fwd(cur, w) if stride == 1 else conv3d_fwd_s2(cur, w)
        if len(spec) > 2 and spec[2] == "bn":
            if mirrored:
                z = round_to_bf16(z)
            zb = z
            z, mean, var = bn_fwd(zb, gammas[l], b)
            if bn_state is not None:
                bn_state.append((zb, mean, var))
            b = None
        elif bn_state is not None:
            bn_state.append(None)
        if pool == "max":
            y, aux = pool_fwd(z, b, slope)
        elif pool == "avg":
            y, aux = avgpool_fwd(z, b, slope)
        else:
            y, aux = act_fwd(z, b, slope), None
        if mirrored:
            y = round_to_bf16(y)
        ys.append(y)
        auxs.append(aux)
        cur = y
    return xs, ys, auxs


def chain_bwd(xs, ys, auxs, ws, dy, slope, specs, mirrored=True, gammas=None, bn_state=None, dgammas=None):
    """Backward of chain_fwd from dy at the last output: per block (dW, db) and
    the dense dZ.  Where the lower block's output derivative is a function of
    that output (max pooling, no pooling), it is applied to the input gradient
    right after backward-data, as the GPU stack stores it; an average-pooled
    block applies the per-voxel derivative itself (from its sign mask).  For a
    BN block, db is dbeta and dgammas[l] receives dgamma; dZ is the batch-norm
    backward of the activation/pooling backward."""
    L = len(ws)
    dws, dbs, dzs = [None] * L, [None] * L, [None] * L
    g = _f64(dy)
    pre = False  # g already carries the output derivative of block l
    for l in range(L - 1, -1, -1):
        stride, pool = specs[l][0], specs[l][1]
        bn = len(specs[l]) > 2 and specs[l][2] == "bn"
        if pool == "max":
            dz, _, db = pool_bwd(g, None if pre else ys[l], auxs[l], slope)
        elif pool == "avg":
            dz, db = avgpool_bwd(g, auxs[l], slope)
        elif pre:
            dz, db = g, g.reshape(-1, g.shape[-1]).sum(0)
        else:
            dz, db = act_bwd(g, ys[l], slope)
        if bn:
            zb = bn_state[l][0]
            dz, dgamma, db = bn_bwd(zb, dz, gammas[l])
            if dgammas is not None:
                dgammas[l] = dgamma
        if mirrored:
            dz = round_to_bf16(dz)
        dzs[l], dbs[l] = dz, db
        dws[l] = conv3d_wgrad(xs[l], dz) if stride == 1 else conv3d_wgrad_s2(xs[l], dz)
        if l > 0:
            dx = conv3d_dgrad(dz, ws[l]) if stride == 1 else conv3d_dgrad_s2(dz, ws[l], xs[l].shape[1:4])
            if specs[l - 1][1] != "avg":
                g, pre = dx * np.where(xs[l] > 0, 1.0, slope), True
            else:
                g, pre = dx, False
            if mirrored:
                g = round_to_bf16(g)
    return dws, dbs, dzs


# The seven-conv model of the hybrid-parallelism page, Table I, for input width
# 128: c4 has stride 2, c6 and c7 are not pooled at this width; pooling is max
# (this build's block), biases present (zero in the synthetic inputs).
TABLE1_CHANNELS = (4, 16, 32, 64, 128, 256, 256, 256)


def table1_specs(wi: int = 128):
    pooled = {128: 5, 256: 6, 512: 7}[wi]
    return [(2 if l == 3 else 1, "max" if l < pooled else "none") for l in range(7)]


# ----------------------------------------------------------------------------
# the rest of the network (hybrid-parallelism page, section IV and Table I:
# fc1 2048 -> fc2 256 -> fc3 4 outputs; leaky ReLU after every layer but the
# last; dropout with keep probability 0.8 after the fully connected layers;
# mean squared error; Adam with beta1 0.9, beta2 0.999, eps 1e-8 and a linear
# learning-rate decay to 0.01x).  Readings: dropout after the two hidden fc
# layers (not on the regression outputs); the dropout draws are inputs (keep
# masks), scaled by 1/keep where kept.

def fc_fwd(x, w, b):
    """y [M,N] = x [M,K] @ w[N,K]^T + b (fp64)."""
    return _f64(x) @ _f64(w).T + _f64(b)


def fc_bwd(x, w, dy):
    """(dx, dw, db) of fc_fwd."""
    x, w, dy = _f64(x), _f64(w), _f64(dy)
    return dy @ w, dy.T @ x, dy.sum(0)


def head_fwd(feat, fcs, masks, keep, slope):
    """feat [M, F] -> predictions [M, 4] through the fc layers fcs = [(w, b)]:
    hidden layers leaky ReLU then dropout (masks[i] of 0/1, scale 1/keep), the
    last layer linear.  Returns (hs, pred): hs[i] = input of layer i."""
    hs = [_f64(feat)]
    cur = hs[0]
    for i, (w, b) in enumerate(fcs):
        z = fc_fwd(cur, w, b)
        if i < len(fcs) - 1:
            z = np.where(z > 0, z, slope * z) * _f64(masks[i]) / keep
            hs.append(z)
        cur = z
    return hs, cur


def head_bwd(hs, fcs, masks, keep, slope, dpred):
    """Backward of head_fwd from dpred: ([(dw, db)], dfeat).  The leaky-ReLU
    derivative of a hidden layer is read from its stored output (its sign is
    the pre-activation's wherever the mask kept it; elsewhere the gradient is
    zero)."""
    grads = [None] * len(fcs)
    g = _f64(dpred)
    for i in range(len(fcs) - 1, -1, -1):
        dx, dw, db = fc_bwd(hs[i], fcs[i][0], g)
        grads[i] = (dw, db)
        if i > 0:
            h = hs[i]
            g = dx * _f64(masks[i - 1]) / keep * np.where(h > 0, 1.0, slope)
        else:
            g = dx
    return grads, g


def mse(pred, target):
    """(loss, dpred): mean over every element of (pred - target)^2 and its gradient."""
    d = _f64(pred) - _f64(target)
    return float(np.mean(d * d)), 2.0 * d / d.size


def adam_step(w, g, m, v, lr, t, beta1=0.9, beta2=0.999, eps=1e-8):
    """One Adam step (bias-corrected moments, step t >= 1); returns (w, m, v)."""
    w, g, m, v = _f64(w), _f64(g), _f64(m), _f64(v)
    m = beta1 * m + (1 - beta1) * g
    v = beta2 * v + (1 - beta2) * g * g
    mh = m / (1 - beta1 ** t)
    vh = v / (1 - beta2 ** t)
    return w - lr * mh / (np.sqrt(vh) + eps), m, v


def linear_decay_lr(lr0, step, total_steps, final_frac=0.01):
    """Linear decay from lr0 to final_frac * lr0 over total_steps, then constant."""
    return lr0 * (1.0 - (1.0 - final_frac) * min(step / total_steps, 1.0))
