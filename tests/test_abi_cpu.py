"""The C-ABI library builds, loads and exports every symbol its header
declares; argument errors come back as status codes (no GPU needed)."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def cf():
    from cnn_conv3d_gb300 import build
    build.build()
    from cnn_conv3d_gb300 import cfconv
    return cfconv


def test_exports_every_header_symbol(cf):
    names = cf.header_symbols()
    expected = {"cf_conv3d_fwd", "cf_conv3d_dgrad", "cf_conv3d_wgrad", "cf_bias_lrelu_pool_fwd",
                "cf_bias_lrelu_pool_bwd", "cf_workspace_size", "cf_status_string", "cf_last_device_status",
                "cf_set_wait_limit_ns", "cf_debug_wait_timeout_probe", "cf_block_epilogue_fwd",
                "cf_block_epilogue_bwd", "cf_bias_lrelu_pool_bwd_noalloc"}
    assert expected <= set(names)
    lib = ctypes.CDLL(cf.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(cf):
    assert cf.cf_status_string(cf.CF_OK) == "ok"
    assert "workspace" in cf.cf_status_string(cf.CF_ERR_WORKSPACE)
    assert cf.cf_status_string(99) == "unknown status"


def test_argument_errors_before_any_launch(cf):
    d = cf.cf_conv_desc(1, 4, 4, 4, 32, 64)
    assert cf.cf_conv3d_fwd(d, None, None, None, None, check=False) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_conv3d_fwd(cf.cf_conv_desc(0, 4, 4, 4, 32, 64), 16, 16, None, 16,
                            check=False) == cf.CF_ERR_INVALID_ARG
    # misaligned pointers are rejected before anything touches the device
    assert cf.cf_conv3d_fwd(d, 18, 32, None, 64, check=False) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_conv3d_dgrad(d, None, None, None, None, 0.3, None, check=False) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_conv3d_wgrad(d, None, None, None, None, check=False) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_bias_lrelu_pool_fwd(1, 4, 4, 4, 8, None, None, 0.3, None, None,
                                     check=False) == cf.CF_ERR_INVALID_ARG
    # dz requested without argmax codes
    assert cf.cf_bias_lrelu_pool_bwd(1, 4, 4, 4, 8, 16, None, None, 0.3, 32, None, None,
                                     check=False) == cf.CF_ERR_INVALID_ARG
    with pytest.raises(cf.CfError):
        cf.cf_set_wait_limit_ns(0)


def test_unsupported_shapes(cf):
    # odd spatial size with pooling, and c_in not in {1, 4} or a multiple of 32
    assert cf.cf_bias_lrelu_pool_fwd(1, 3, 4, 4, 8, 16, None, 0.3, 32, None,
                                     check=False) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_bias_lrelu_pool_fwd(1, 4, 4, 4, 12, 16, None, 0.3, 32, None,
                                     check=False) == cf.CF_ERR_UNSUPPORTED


def test_tile_divider_method():
    """The tile decoders divide by launch-time constants with the unsigned
    multiply-and-shift method of Granlund and Montgomery ("Division by
    Invariant Integers using Multiplication", figure 4.1, N = 32).  The
    method, as the kernels write it, equals floor division for every divisor
    and numerator checked here (all divisors up to 4096 plus large ones, with
    numerators at 0, around multiples of d and at the 32-bit edge)."""
    import random

    def make(d):
        l = 0
        while l < 32 and (1 << l) < d:
            l += 1
        m = ((1 << 32) * ((1 << l) - d)) // d + 1
        assert 0 < m < (1 << 32)
        return m, (1 if l else 0), (l - 1 if l else 0)

    def div(x, mss):
        m, s1, s2 = mss
        t = (x * m) >> 32
        return (t + ((x - t) >> s1)) >> s2

    rng = random.Random(5)
    divisors = list(range(1, 4097)) + [rng.randrange(4097, 1 << 31) for _ in range(200)] + [(1 << 31) - 1]
    for d in divisors:
        mss = make(d)
        xs = [0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, (1 << 32) - 1, (1 << 31) - 1]
        xs += [rng.randrange(0, 1 << 32) for _ in range(40)]
        for x in xs:
            if 0 <= x < (1 << 32):
                assert div(x, mss) == x // d, (x, d)


def test_variant_argument_errors(cf):
    # stride 3, an unknown pooling kind, average-pool backward without masks,
    # dy_pre outside max pooling: all refused before anything is launched
    d = cf.cf_conv_desc(1, 4, 4, 4, 32, 64, 3)
    assert cf.cf_conv3d_fwd(d, 16, 16, None, 16, check=False) == cf.CF_ERR_INVALID_ARG
    d = cf.cf_conv_desc(1, 4, 4, 4, 32, 64, 1)
    assert cf.cf_conv3d_fwd(d, 16, 16, (None, 0.3, None, 7), 16, check=False) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_block_epilogue_fwd(5, 1, 4, 4, 4, 8, 16, None, 0.3, 16, None, check=False) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_block_epilogue_bwd(cf.CF_POOL_AVG, 1, 4, 4, 4, 8, 16, None, None, 0.3, 32, None, None,
                                    check=False) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_block_epilogue_bwd(cf.CF_POOL_NONE, 1, 4, 4, 4, 8, 16, None, None, 0.3, 32, 48, None,
                                    check=False) == cf.CF_ERR_INVALID_ARG
