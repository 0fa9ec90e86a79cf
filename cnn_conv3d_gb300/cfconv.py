"""ctypes binding of libcfconv3d.so -- argument marshalling only.

Every function has the name of the C entry point it calls (see
include/cf_conv3d.h for arguments, layouts, ownership and errors).  Pointer
arguments accept ``None``, a plain integer device address, or any object with
``data_ptr()`` (a torch tensor); streams accept ``None``, an integer handle,
or a ``torch.cuda.Stream``.  Nothing here computes: there is no fallback, and
importing this module raises if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcfconv3d.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "cf_conv3d.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libcfconv3d.so is not built ({LIB_PATH}); run cnn_conv3d_gb300.build.build()")

_lib = ctypes.CDLL(LIB_PATH)

CF_OK, CF_ERR_INVALID_ARG, CF_ERR_UNSUPPORTED, CF_ERR_WORKSPACE, CF_ERR_CUDA, CF_ERR_TIMEOUT = range(6)
CF_OP_FWD, CF_OP_DGRAD, CF_OP_WGRAD, CF_OP_DGRAD_ROUTED, CF_OP_WGRAD_ROUTED, CF_OP_POOL_BWD, CF_OP_BN = range(7)
CF_POOL_MAX, CF_POOL_AVG, CF_POOL_NONE = range(3)


class cf_conv_desc(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("d", ctypes.c_int64), ("h", ctypes.c_int64), ("w", ctypes.c_int64),
                ("c_in", ctypes.c_int32), ("c_out", ctypes.c_int32), ("stride", ctypes.c_int32)]


class cf_pool_epi(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("slope", ctypes.c_float), ("argmax", ctypes.c_void_p),
                ("pool", ctypes.c_int32)]


class CfError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {cf_status_string(status)} ({status})")
        self.status = status


_vp, _i64, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_DP = ctypes.POINTER(cf_conv_desc)
_EP = ctypes.POINTER(cf_pool_epi)

_SIGS = {
    "cf_conv3d_fwd": ([_DP, _vp, _vp, _EP, _vp, _vp, _sz, _vp], ctypes.c_int),
    "cf_conv3d_dgrad": ([_DP, _vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    "cf_conv3d_dgrad_flipped": ([_DP, _vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    "cf_filter_flip": ([_i32, _i32, _vp, _vp, _vp], ctypes.c_int),
    "cf_bias_lrelu_pool_bwd_partials": ([_i64, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _sz,
                                         _vp], ctypes.c_int),
    "cf_pool_bwd_partial_rows": ([], ctypes.c_int64),
    "cf_column_sums": ([_i64, _i32, _vp, _vp, _vp], ctypes.c_int),
    "cf_conv3d_wgrad": ([_DP, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _sz, _vp], ctypes.c_int),
    "cf_conv3d_dgrad_pool_bwd": ([_DP, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    "cf_bias_lrelu_pool_fwd": ([_i64, _i64, _i64, _i64, _i32, _vp, _vp, _f32, _vp, _vp, _vp], ctypes.c_int),
    "cf_bias_lrelu_pool_bwd": ([_i64, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _sz, _vp],
                               ctypes.c_int),
    "cf_bias_lrelu_pool_bwd_noalloc": ([_i64, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp],
                                       ctypes.c_int),
    "cf_block_epilogue_fwd": ([_i32, _i64, _i64, _i64, _i64, _i32, _vp, _vp, _f32, _vp, _vp, _vp], ctypes.c_int),
    "cf_block_epilogue_bwd": ([_i32, _i64, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _sz,
                               _vp], ctypes.c_int),
    "cf_bn_stats": ([_i64, _i32, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    "cf_bn_act_pool_fwd": ([_i32, _i64, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _f32, _f32, _vp, _vp, _vp],
                           ctypes.c_int),
    "cf_bn_act_pool_bwd": ([_i32, _i64, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _f32, _vp, _vp,
                            _vp, _sz, _vp], ctypes.c_int),
    "cf_fc_fwd": ([_i64, _i32, _i32, _vp, _i32, _vp, _vp, _i32, _f32, _vp, _f32, _vp, _vp], ctypes.c_int),
    "cf_fc_bwd": ([_i64, _i32, _i32, _vp, _i32, _vp, _vp, _f32, _vp, _f32, _vp, _vp, _i32, _vp, _vp, _vp],
                  ctypes.c_int),
    "cf_mse": ([_i64, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "cf_adam_step": ([_i64, _vp, _vp, _vp, _vp, _vp, _f32, _f32, _f32, _f32, _i64, _vp], ctypes.c_int),
    "cf_workspace_size": ([ctypes.c_int, _DP], _sz),
    "cf_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "cf_last_device_status": ([_vp], ctypes.c_int),
    "cf_set_wait_limit_ns": ([ctypes.c_uint64], ctypes.c_int),
    "cf_debug_wait_timeout_probe": ([_vp], ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


def header_symbols():
    """Names of the functions include/cf_conv3d.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(cf_\w+)\s*\(", text, re.M)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _desc(d):
    """cf_conv_desc, or a tuple (n, d, h, w, c_in, c_out[, stride])."""
    if isinstance(d, cf_conv_desc):
        return d
    n, dd, h, w, ci, co = d[:6]
    return cf_conv_desc(n, dd, h, w, ci, co, d[6] if len(d) > 6 else 1)


def _check(st, what):
    if st != CF_OK:
        raise CfError(st, what)
    return st


def cf_status_string(status: int) -> str:
    return _lib.cf_status_string(status).decode()


def cf_workspace_size(op: int, desc) -> int:
    return _lib.cf_workspace_size(op, ctypes.byref(_desc(desc)))


def cf_conv3d_fwd(desc, x, w, epi, y, ws=None, ws_bytes=0, stream=None, check=True):
    """epi: None, or (bias, slope, argmax[, pool]) / cf_pool_epi."""
    e = None
    if epi is not None:
        if not isinstance(epi, cf_pool_epi):
            b, slope, am = epi[:3]
            epi = cf_pool_epi(_ptr(b), float(slope), _ptr(am), epi[3] if len(epi) > 3 else CF_POOL_MAX)
        e = ctypes.byref(epi)
    st = _lib.cf_conv3d_fwd(ctypes.byref(_desc(desc)), _ptr(x), _ptr(w), e, _ptr(y), _ptr(ws), ws_bytes,
                            _stream(stream))
    return _check(st, "cf_conv3d_fwd") if check else st


def cf_conv3d_dgrad(desc, dz, idx, w, x_act, slope, dx, ws=None, ws_bytes=0, stream=None, check=True, dsum=None):
    st = _lib.cf_conv3d_dgrad(ctypes.byref(_desc(desc)), _ptr(dz), _ptr(idx), _ptr(w), _ptr(x_act), float(slope),
                              _ptr(dx), _ptr(dsum), _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "cf_conv3d_dgrad") if check else st


def cf_conv3d_dgrad_flipped(desc, dz, idx, wt, x_act, slope, dx, ws=None, ws_bytes=0, stream=None, check=True,
                            dsum=None):
    st = _lib.cf_conv3d_dgrad_flipped(ctypes.byref(_desc(desc)), _ptr(dz), _ptr(idx), _ptr(wt), _ptr(x_act),
                                      float(slope), _ptr(dx), _ptr(dsum), _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "cf_conv3d_dgrad_flipped") if check else st


def cf_filter_flip(c_out, c_in, w, wt, stream=None, check=True):
    st = _lib.cf_filter_flip(int(c_out), int(c_in), _ptr(w), _ptr(wt), _stream(stream))
    return _check(st, "cf_filter_flip") if check else st


def cf_bias_lrelu_pool_bwd_partials(n, d, h, w, c, dy, y, idx, slope, dz, dy_pre, partial, stream=None, check=True):
    st = _lib.cf_bias_lrelu_pool_bwd_partials(n, d, h, w, c, _ptr(dy), _ptr(y), _ptr(idx), float(slope), _ptr(dz),
                                              _ptr(dy_pre), _ptr(partial), partial.numel() * partial.element_size(),
                                              _stream(stream))
    return _check(st, "cf_bias_lrelu_pool_bwd_partials") if check else st


def cf_pool_bwd_partial_rows():
    return int(_lib.cf_pool_bwd_partial_rows())


def cf_column_sums(rows, c, partial, out, stream=None, check=True):
    st = _lib.cf_column_sums(int(rows), int(c), _ptr(partial), _ptr(out), _stream(stream))
    return _check(st, "cf_column_sums") if check else st


def cf_conv3d_dgrad_pool_bwd(desc, dz, w, x_act, slope, dx, prev_idx, prev_dz, ws=None, ws_bytes=0, stream=None,
                             check=True, dsum=None):
    st = _lib.cf_conv3d_dgrad_pool_bwd(ctypes.byref(_desc(desc)), _ptr(dz), _ptr(w), _ptr(x_act), float(slope),
                                       _ptr(dx), _ptr(dsum), _ptr(prev_idx), _ptr(prev_dz), _ptr(ws), ws_bytes,
                                       _stream(stream))
    return _check(st, "cf_conv3d_dgrad_pool_bwd") if check else st


def cf_conv3d_wgrad(desc, x, dz, idx, dw, accumulate=0, ws=None, ws_bytes=0, stream=None, check=True):
    st = _lib.cf_conv3d_wgrad(ctypes.byref(_desc(desc)), _ptr(x), _ptr(dz), _ptr(idx), _ptr(dw), int(accumulate),
                              _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "cf_conv3d_wgrad") if check else st


def cf_bias_lrelu_pool_fwd(n, d, h, w, c, z, bias, slope, y, idx, stream=None, check=True):
    st = _lib.cf_bias_lrelu_pool_fwd(n, d, h, w, c, _ptr(z), _ptr(bias), float(slope), _ptr(y), _ptr(idx),
                                     _stream(stream))
    return _check(st, "cf_bias_lrelu_pool_fwd") if check else st


def cf_bias_lrelu_pool_bwd(n, d, h, w, c, dy, y, idx, slope, dz, dy_pre, dbias, ws=None, ws_bytes=0, stream=None,
                           check=True):
    st = _lib.cf_bias_lrelu_pool_bwd(n, d, h, w, c, _ptr(dy), _ptr(y), _ptr(idx), float(slope), _ptr(dz),
                                     _ptr(dy_pre), _ptr(dbias), _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "cf_bias_lrelu_pool_bwd") if check else st


def cf_bias_lrelu_pool_bwd_noalloc(n, d, h, w, c, dy, y, idx, slope, dz, dy_pre, dbias, stream=None, check=True):
    st = _lib.cf_bias_lrelu_pool_bwd_noalloc(n, d, h, w, c, _ptr(dy), _ptr(y), _ptr(idx), float(slope), _ptr(dz),
                                             _ptr(dy_pre), _ptr(dbias), _stream(stream))
    return _check(st, "cf_bias_lrelu_pool_bwd_noalloc") if check else st


def cf_block_epilogue_fwd(pool, n, d, h, w, c, z, bias, slope, y, aux, stream=None, check=True):
    st = _lib.cf_block_epilogue_fwd(int(pool), n, d, h, w, c, _ptr(z), _ptr(bias), float(slope), _ptr(y), _ptr(aux),
                                    _stream(stream))
    return _check(st, "cf_block_epilogue_fwd") if check else st


def cf_block_epilogue_bwd(pool, n, d, h, w, c, dy, y, aux, slope, dz, dy_pre, dbias, ws=None, ws_bytes=0,
                          stream=None, check=True):
    st = _lib.cf_block_epilogue_bwd(int(pool), n, d, h, w, c, _ptr(dy), _ptr(y), _ptr(aux), float(slope), _ptr(dz),
                                    _ptr(dy_pre), _ptr(dbias), _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "cf_block_epilogue_bwd") if check else st


def cf_bn_stats(rows, c, z, sums, ws=None, ws_bytes=0, stream=None, check=True):
    st = _lib.cf_bn_stats(rows, c, _ptr(z), _ptr(sums), _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "cf_bn_stats") if check else st


def cf_bn_act_pool_fwd(pool, n, d, h, w, c, z, sums, gamma, beta, eps, slope, y, aux, stream=None, check=True):
    st = _lib.cf_bn_act_pool_fwd(int(pool), n, d, h, w, c, _ptr(z), _ptr(sums), _ptr(gamma), _ptr(beta), float(eps),
                                 float(slope), _ptr(y), _ptr(aux), _stream(stream))
    return _check(st, "cf_bn_act_pool_fwd") if check else st


def cf_bn_act_pool_bwd(pool, n, d, h, w, c, dy, y, aux, z, sums, gamma, eps, slope, dz, dsums, ws=None, ws_bytes=0,
                       stream=None, check=True):
    st = _lib.cf_bn_act_pool_bwd(int(pool), n, d, h, w, c, _ptr(dy), _ptr(y), _ptr(aux), _ptr(z), _ptr(sums),
                                 _ptr(gamma), float(eps), float(slope), _ptr(dz), _ptr(dsums), _ptr(ws), ws_bytes,
                                 _stream(stream))
    return _check(st, "cf_bn_act_pool_bwd") if check else st


def cf_fc_fwd(m, k, n, x, x_is_bf16, w, b, act, slope, keep_mask, keep, y, stream=None, check=True):
    st = _lib.cf_fc_fwd(m, k, n, _ptr(x), int(x_is_bf16), _ptr(w), _ptr(b), int(act), float(slope), _ptr(keep_mask),
                        float(keep), _ptr(y), _stream(stream))
    return _check(st, "cf_fc_fwd") if check else st


def cf_fc_bwd(m, k, n, x, x_is_bf16, w, h, slope, keep_mask, keep, dy, dx, dx_is_bf16, dw, db, stream=None,
              check=True):
    st = _lib.cf_fc_bwd(m, k, n, _ptr(x), int(x_is_bf16), _ptr(w), _ptr(h), float(slope), _ptr(keep_mask),
                        float(keep), _ptr(dy), _ptr(dx), int(dx_is_bf16), _ptr(dw), _ptr(db), _stream(stream))
    return _check(st, "cf_fc_bwd") if check else st


def cf_mse(count, pred, target, loss, dpred, stream=None, check=True):
    st = _lib.cf_mse(count, _ptr(pred), _ptr(target), _ptr(loss), _ptr(dpred), _stream(stream))
    return _check(st, "cf_mse") if check else st


def cf_adam_step(count, w, w_bf16, g, m, v, lr, beta1, beta2, eps, t, stream=None, check=True):
    st = _lib.cf_adam_step(count, _ptr(w), _ptr(w_bf16), _ptr(g), _ptr(m), _ptr(v), float(lr), float(beta1),
                           float(beta2), float(eps), int(t), _stream(stream))
    return _check(st, "cf_adam_step") if check else st


def cf_last_device_status(stream=None) -> int:
    return _lib.cf_last_device_status(_stream(stream))


def cf_set_wait_limit_ns(ns: int):
    return _check(_lib.cf_set_wait_limit_ns(int(ns)), "cf_set_wait_limit_ns")


def cf_debug_wait_timeout_probe(stream=None):
    return _check(_lib.cf_debug_wait_timeout_probe(_stream(stream)), "cf_debug_wait_timeout_probe")
