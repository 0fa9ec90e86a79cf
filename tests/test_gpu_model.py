"""The whole network's training step through the C ABI (CosmoFlowModel): conv
stack, fully connected head with leaky ReLU and dropout, mean squared error,
backward, Adam -- each stage against the fp64 oracle on the GPU's own inputs
of that stage."""
import numpy as np
import pytest

import synthdata
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu

SLOPE, KEEP = 0.3, 0.8


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_conv3d_gb300 import build
    build.build()
    return torch


def _model(torch, n=2, spatial=64, seed=6161):
    from cnn_conv3d_gb300.model import CosmoFlowModel
    from oracle import TABLE1_CHANNELS, table1_specs
    m = CosmoFlowModel(n, spatial, TABLE1_CHANNELS, specs=table1_specs(128))
    inp = synthdata.stack_inputs(n, spatial, TABLE1_CHANNELS, seed=seed, with_dy=False)
    m.stack.load(inp["x"], inp["w"], inp["b"])
    m.sync_master()
    rng = np.random.default_rng(seed)
    fcs = []
    for i in range(len(m.fw)):
        w = rng.normal(0, np.sqrt(2.0 / m.dims[i]), size=m.fw[i].shape).astype(np.float32)
        b = rng.normal(0, 0.05, size=m.fb[i].shape).astype(np.float32)
        m.fw[i].copy_(torch.from_numpy(w))
        m.fb[i].copy_(torch.from_numpy(b))
        fcs.append((w, b))
    masks = [(rng.random(t.shape) < KEEP).astype(np.uint8) for t in m.masks]
    m.set_masks(masks)
    target = rng.uniform(-1, 1, size=m.target.shape).astype(np.float32)
    m.target.copy_(torch.from_numpy(target))
    return m, fcs, masks, target


def test_training_step_stages(torch_cuda, oracle_mod):
    torch = torch_cuda
    from cnn_conv3d_gb300 import cfconv as cf
    m, fcs, masks, target = _model(torch)
    m.forward()
    torch.cuda.synchronize()
    n = m.n
    f = oracle_mod.bf16_bits_to_f64
    feat = f(m.stack.y[-1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)).reshape(n, -1)
    # head forward on the GPU's features, layer by layer on the GPU's own inputs
    x = feat
    for i, (w, b) in enumerate(fcs):
        ref = oracle_mod.fc_fwd(x, w, b)
        S = np.abs(x) @ np.abs(w.astype(np.float64)).T + np.abs(b)
        last = i == len(fcs) - 1
        if not last:
            ref = np.where(ref > 0, ref, SLOPE * ref) * masks[i] / KEEP
            S = S * masks[i] / KEEP
        got = (m.pred if last else m.h[i]).cpu().numpy().astype(np.float64)
        assert_close(got, ref, S + 1e-30, f"fc{i + 1} forward")
        x = got
    loss, dpred = oracle_mod.mse(m.pred.cpu().numpy(), target)
    assert abs(float(m.loss[0]) - loss) <= 1e-5 * max(1.0, loss)
    # backward: every fc gradient and the stack's input gradient, on the GPU's stored activations
    m.backward()
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == cf.CF_OK
    # each layer's backward on its own GPU inputs: stored activations and the
    # gradient the layer above produced; S = sums of |products|
    hs = [feat] + [t.cpu().numpy().astype(np.float64) for t in m.h]
    L = len(fcs)
    for i in range(L - 1, -1, -1):
        dy = (m.dpred if i == L - 1 else m.dh[i]).cpu().numpy().astype(np.float64)
        g = dy if i == L - 1 else dy * masks[i] / KEEP * np.where(hs[i + 1] > 0, 1.0, SLOPE)
        dx, dw, db = oracle_mod.fc_bwd(hs[i], fcs[i][0], g)
        assert_close(m.dfw[i].cpu().numpy(), dw, np.abs(g).T @ np.abs(hs[i]), f"fc{i + 1} dW")
        assert_close(m.dfb[i].cpu().numpy(), db, np.abs(g).sum(0), f"fc{i + 1} db")
        Sx = np.abs(g) @ np.abs(fcs[i][0].astype(np.float64))
        if i > 0:
            assert_close(m.dh[i - 1].cpu().numpy(), dx, Sx, f"fc{i + 1} dx")
        else:
            gdf = f(m.dfeat.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)).reshape(n, -1)
            assert_close(gdf, dx, Sx, "dfeat (bf16)")
    # Adam on every parameter, from the gradients just computed
    before = [(p.cpu().numpy().astype(np.float64), g.cpu().numpy().astype(np.float64)) for p, _, g in m.params()]
    m.update(1e-3)
    torch.cuda.synchronize()
    for (p, p16, _), (w0, g0) in zip(m.params(), before):
        ref, _, _ = oracle_mod.adam_step(w0, g0, np.zeros_like(w0), np.zeros_like(w0), lr=1e-3, t=1)
        got = p.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-7)
        if p16 is not None:  # the conv kernels' bf16 copy follows the fp32 master
            assert torch.equal(p16, p.to(torch.bfloat16))


def test_training_reduces_loss_on_a_fixed_batch(torch_cuda):
    torch = torch_cuda
    from cnn_conv3d_gb300 import cfconv as cf
    m, _, _, _ = _model(torch, seed=6262)
    losses = []
    for _ in range(12):
        m.step(2e-4)
        torch.cuda.synchronize()
        losses.append(float(m.loss[0]))
    assert cf.cf_last_device_status() == cf.CF_OK
    assert np.all(np.isfinite(losses))
    assert losses[-1] < 0.7 * losses[0], losses
