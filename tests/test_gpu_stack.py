"""The stack's execution schedules compute the same step: every launch on one
stream (serial), the two-stream schedule (weight gradients beside the
backward-data chain), and a CUDA-graph replay of the two-stream step all give
bit-identical outputs and gradients (the kernels' reductions have a fixed
order, so the schedule cannot change any value)."""
import numpy as np
import pytest

import synthdata

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_conv3d_gb300 import build
    build.build()
    return torch


def _snapshot(st):
    return [t.clone() for t in st.y + st.idx + st.dw + st.db] + [g.clone() for g in st.g if g is not None]


@pytest.mark.parametrize("shape", [(2, 32, (4, 32, 64, 128)), (1, 16, (1, 32, 64))])
def test_schedules_agree(torch_cuda, shape):
    torch = torch_cuda
    from cnn_conv3d_gb300 import cfconv as cf
    from cnn_conv3d_gb300.stack import CosmoStack
    n, s, ch = shape
    inp = synthdata.stack_inputs(n, s, ch, seed=4242, with_dy=True)
    dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).cuda()
    st = CosmoStack(n, s, ch, 0.3, backward=True)
    st.load(inp["x"], inp["w"], inp["b"])
    st.step(dy, serial=True)
    torch.cuda.synchronize()
    ref = _snapshot(st)
    for t in st.dw + st.db:
        t.fill_(float("nan"))
    st.step(dy)
    torch.cuda.synchronize()
    two = _snapshot(st)
    g = st.capture(dy)
    for t in st.dw + st.db:
        t.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    graph = _snapshot(st)
    assert cf.cf_last_device_status() == cf.CF_OK
    for a, b, c in zip(ref, two, graph):
        assert torch.equal(a, b)
        assert torch.equal(a, c)
