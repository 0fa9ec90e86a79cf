"""The allocation-free pool backward (cf_bias_lrelu_pool_bwd_noalloc) against
the workspace version, through the C ABI.

It serves callers that cannot allocate device memory: its bias-gradient
partials live in a fixed array inside the library instead of a caller
workspace.  Two calls in a row check that the array's leftover contents from
the first call do not leak into the second.  This file is collected last so
that a stop-at-first-failure run has already run every other test."""
import numpy as np
import pytest

import synthdata
from tests.gpu_util import assert_close, dev, dev_bf16, empty_bf16, host_bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cf():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_conv3d_gb300 import build
    build.build()
    from cnn_conv3d_gb300 import cfconv
    return cfconv


def _case(seed, N, D, H, W, C):
    rng = np.random.default_rng(seed)
    y = synthdata.to_bf16_bits(rng.normal(size=(N, D // 2, H // 2, W // 2, C)))
    dy = synthdata.to_bf16_bits(rng.normal(size=(N, D // 2, H // 2, W // 2, C)))
    idx = rng.integers(0, 8, size=(N, D // 2, H // 2, W // 2, C)).astype(np.uint8)
    return dev_bf16(dy), dev_bf16(y), dev(idx)


def _run(cf, fn, shape, dy, y, idx, ws=None):
    import torch
    N, D, H, W, C = shape
    dz = empty_bf16((N, D, H, W, C), fill=3.0)
    dyp = empty_bf16((N, D // 2, H // 2, W // 2, C), fill=3.0)
    db = torch.full((C,), 7.0, dtype=torch.float32, device="cuda")
    if ws is None:
        fn(N, D, H, W, C, dy, y, idx, 0.3, dz, dyp, db)
    else:
        fn(N, D, H, W, C, dy, y, idx, 0.3, dz, dyp, db, ws, ws.numel())
    torch.cuda.synchronize()
    return host_bf16_f64(dz), host_bf16_f64(dyp), db.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", [(2, 8, 12, 16, 64), (1, 4, 4, 8, 256)])
def test_noalloc_matches_workspace_version_twice(cf, shape):
    import torch
    N, D, H, W, C = shape
    ws = torch.empty((max(cf.cf_workspace_size(cf.CF_OP_POOL_BWD, (N, D, H, W, C, C)), 256),),
                     dtype=torch.uint8, device="cuda")
    for seed in (1, 2):  # two calls in a row, different data
        dy, y, idx = _case(seed * 100 + C, *shape)
        ref = _run(cf, cf.cf_bias_lrelu_pool_bwd, shape, dy, y, idx, ws)
        got = _run(cf, cf.cf_bias_lrelu_pool_bwd_noalloc, shape, dy, y, idx)
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])
        assert_close(got[2], ref[2], np.abs(ref[1]).reshape(-1, C).sum(axis=0), "dbias")
    assert cf.cf_last_device_status() == cf.CF_OK


def test_noalloc_rejects_channels_beyond_scratch(cf):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    C = (65536 // sms + 8) // 8 * 8  # first multiple of 8 beyond the array's capacity
    N, D, H, W = 1, 2, 2, 2
    dy = torch.zeros((N * C,), dtype=torch.bfloat16, device="cuda")
    db = torch.zeros((C,), dtype=torch.float32, device="cuda")
    st = cf.cf_bias_lrelu_pool_bwd_noalloc(N, D, H, W, C, dy, None, None, 0.3, None, None, db, check=False)
    assert st == cf.CF_ERR_WORKSPACE
