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


@pytest.mark.parametrize("shape", [(3, 64, (4, 32, 64, 128))])
def test_host_step_matches(torch_cuda, shape):
    """step_host (input copied in per sample range, overlapped with the first
    block; gradients copied out as each is final), eager and as a CUDA graph,
    gives the bits of load + step + copy-back."""
    torch = torch_cuda
    from cnn_conv3d_gb300 import cfconv as cf
    from cnn_conv3d_gb300.stack import CosmoStack
    n, s, ch = shape
    inp = synthdata.stack_inputs(n, s, ch, seed=4343, with_dy=True)
    dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).cuda()
    st = CosmoStack(n, s, ch, 0.3, backward=True)
    st.load(inp["x"], inp["w"], inp["b"])
    st.step(dy)
    torch.cuda.synchronize()
    ref = [t.clone() for t in st.y + st.idx] + [t.cpu() for t in st.dw + st.db]
    x_host = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    dy_host = dy.cpu().pin_memory()
    dw_host = [torch.full(t.shape, float("nan"), dtype=t.dtype).pin_memory() for t in st.dw]
    db_host = [torch.full(t.shape, float("nan"), dtype=t.dtype).pin_memory() for t in st.db]
    st.x.zero_()
    for t in st.y + st.dw + st.db:
        t.zero_()
    st.step_host(x_host, dy_host, dw_host, db_host, chunks=2)
    torch.cuda.synchronize()
    got = [t.clone() for t in st.y + st.idx] + [t.clone() for t in dw_host + db_host]
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    for t in dw_host + db_host:
        t.fill_(float("nan"))
    g = st.capture(None, host=(x_host, dy_host, dw_host, db_host))
    g.replay()
    torch.cuda.synchronize()
    got = [t.clone() for t in st.y + st.idx] + [t.clone() for t in dw_host + db_host]
    assert cf.cf_last_device_status() == cf.CF_OK
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("shape", [(2, 64, (4, 32, 64, 128))])
def test_pipelined_host_steps_match(torch_cuda, shape):
    """step_host_pipelined (the next batch copied in while this one computes,
    two input buffers), eager and as its pair of CUDA graphs, gives each batch
    the gradient bits of load + step."""
    torch = torch_cuda
    from cnn_conv3d_gb300 import cfconv as cf
    from cnn_conv3d_gb300.stack import CosmoStack
    n, s, ch = shape
    st = CosmoStack(n, s, ch, 0.3, backward=True)
    batches, refs = [], []
    for seed in (5151, 5252):
        inp = synthdata.stack_inputs(n, s, ch, seed=seed, with_dy=True)
        if not batches:
            w, b = inp["w"], inp["b"]  # one set of weights for both batches
        st.load(inp["x"], w, b)
        dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).cuda()
        st.step(dy)
        torch.cuda.synchronize()
        refs.append([t.cpu() for t in st.dw + st.db])
        batches.append((torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory(),
                        dy.cpu().pin_memory()))
    dw_host = [torch.full(t.shape, float("nan"), dtype=t.dtype).pin_memory() for t in st.dw]
    db_host = [torch.full(t.shape, float("nan"), dtype=t.dtype).pin_memory() for t in st.db]

    def check(k):
        torch.cuda.synchronize()
        assert cf.cf_last_device_status() == cf.CF_OK
        for a, b in zip(refs[k], dw_host + db_host):
            assert torch.equal(a, b)
        for t in dw_host + db_host:
            t.fill_(float("nan"))

    st.prefetch_host(*batches[0])
    st.step_host_pipelined(*batches[1], dw_host, db_host)
    check(0)
    st.step_host_pipelined(*batches[0], dw_host, db_host)
    check(1)
    # the graphs bind one pinned pair for the next batch; the loop refills it
    xh, dyh = torch.empty_like(batches[0][0]).pin_memory(), torch.empty_like(batches[0][1]).pin_memory()
    graphs = st.capture_pipelined(xh, dyh, dw_host, db_host)
    st.prefetch_host(*batches[1])
    for k, g in enumerate(graphs * 2):
        nxt = batches[k % 2]
        xh.copy_(nxt[0])
        dyh.copy_(nxt[1])
        g.replay()
        check((k + 1) % 2)


@pytest.mark.parametrize("shape", [(2, 32, (4, 32, 64, 128)), (1, 32, (32, 64, 128, 64))])
def test_fused_pool_backward_matches_separate(torch_cuda, shape):
    """Lower blocks' pool backward inside the backward-data epilogue of the
    block above gives the bits of the separate pool-backward launches."""
    torch = torch_cuda
    from cnn_conv3d_gb300 import cfconv as cf
    from cnn_conv3d_gb300.stack import CosmoStack
    n, s, ch = shape
    inp = synthdata.stack_inputs(n, s, ch, seed=4545, with_dy=True)
    dy = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).cuda()
    out = []
    for fuse in (False, True):  # the stack's default, then the fused path
        st = CosmoStack(n, s, ch, 0.3, backward=True)
        st.fuse_pool_bwd = fuse
        st.load(inp["x"], inp["w"], inp["b"])
        st.step(dy)
        torch.cuda.synchronize()
        out.append([t.clone() for t in st.y + st.dw + st.db] + [t.clone() for t in st.dz if t is not None])
    assert cf.cf_last_device_status() == cf.CF_OK
    for a, b in zip(*out):
        assert torch.equal(a, b)
