"""The whole CosmoFlow network as one training step through the C ABI: the
conv stack (CosmoStack), the fully connected head, the mean squared error and
Adam (hybrid-parallelism page, section IV and Table I: fc1 2048 -> fc2 256 ->
fc3 4 outputs, leaky ReLU after every layer but the last, dropout with keep
probability 0.8 after the hidden fc layers, MSE loss, Adam with beta1 0.9,
beta2 0.999, eps 1e-8 and a linear learning-rate decay to 0.01x).

Python only owns buffers (torch allocations) and enqueues library calls; every
arithmetic step runs in libcfconv3d's kernels.  Conv weights keep an fp32
master copy that Adam updates; the bf16 copy the conv kernels read is written
by the same Adam launch.  Dropout draws are inputs (keep masks), set per step
by the caller (set_masks).
"""
from __future__ import annotations

import torch

from . import cfconv as cf
from .stack import CosmoStack


class CosmoFlowModel:
    def __init__(self, n: int, spatial: int, channels, specs=None, fc=(2048, 256, 4), slope: float = 0.3,
                 keep: float = 0.8, device: str = "cuda"):
        self.n, self.slope, self.keep, self.device = n, float(slope), float(keep), device
        self.stack = CosmoStack(n, spatial, channels, slope, device, backward=True, specs=specs)
        st = self.stack
        f32, u8 = torch.float32, torch.uint8
        self.feat = int(st.y[-1][0].numel())  # flattened NDHWC top output per sample
        self.dims = [self.feat] + list(fc)
        D = self.dims
        self.fw = [torch.zeros((D[i + 1], D[i]), dtype=f32, device=device) for i in range(len(fc))]
        self.fb = [torch.zeros((D[i + 1],), dtype=f32, device=device) for i in range(len(fc))]
        # hidden outputs (after activation and dropout), predictions, keep masks
        self.h = [torch.empty((n, D[i + 1]), dtype=f32, device=device) for i in range(len(fc) - 1)]
        self.pred = torch.empty((n, D[-1]), dtype=f32, device=device)
        self.masks = [torch.ones((n, D[i + 1]), dtype=u8, device=device) for i in range(len(fc) - 1)]
        self.target = torch.zeros((n, D[-1]), dtype=f32, device=device)
        self.loss = torch.zeros((4,), dtype=f32, device=device)
        # gradients
        self.dpred = torch.empty_like(self.pred)
        self.dh = [torch.empty_like(t) for t in self.h]
        self.dfw = [torch.empty_like(t) for t in self.fw]
        self.dfb = [torch.empty_like(t) for t in self.fb]
        self.dfeat = torch.empty(tuple(st.y[-1].shape), dtype=torch.bfloat16, device=device)
        # conv weights' fp32 master copies (set by sync_master after loading)
        self.w32 = [torch.empty(w.shape, dtype=f32, device=device) for w in st.w]
        self._adam = None
        self.t = 0

    # ---------------------------------------------------------------- set-up
    def sync_master(self):
        """fp32 master copies of the conv weights from their bf16 values."""
        for m, w in zip(self.w32, self.stack.w):
            m.copy_(w.float())

    def set_masks(self, masks):
        for dst, src in zip(self.masks, masks):
            dst.copy_(torch.as_tensor(src, dtype=torch.uint8).reshape(dst.shape))

    def params(self):
        """(fp32 tensor, bf16 copy or None, gradient) of every trained parameter."""
        st = self.stack
        out = []
        for l in range(st.L):
            out.append((self.w32[l], st.w[l], st.dw[l]))
            out.append((st.b[l], None, st.db[l]))
            if st.bn(l):
                out.append((st.gamma[l], None, st.dgamma[l]))
        for i in range(len(self.fw)):
            out.append((self.fw[i], None, self.dfw[i]))
            out.append((self.fb[i], None, self.dfb[i]))
        return out

    # ------------------------------------------------------------------ step
    def forward(self, stream=None):
        """Conv stack, then the head: predictions in self.pred, loss in self.loss[0]."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = self.stack
        st.forward(s)
        n, D = self.n, self.dims
        x, xb = st.y[-1], 1
        for i in range(len(self.fw)):
            last = i == len(self.fw) - 1
            out = self.pred if last else self.h[i]
            cf.cf_fc_fwd(n, D[i], D[i + 1], x, xb, self.fw[i], self.fb[i], 0 if last else 1, self.slope,
                         None if last else self.masks[i], self.keep, out, s)
            x, xb = out, 0
        cf.cf_mse(self.pred.numel(), self.pred, self.target, self.loss, self.dpred, s)

    def backward(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        n, D, L = self.n, self.dims, len(self.fw)
        g = self.dpred
        for i in range(L - 1, -1, -1):
            last = i == L - 1
            x, xb = (self.stack.y[-1], 1) if i == 0 else (self.h[i - 1], 0)
            dx, dxb = (self.dfeat, 1) if i == 0 else (self.dh[i - 1], 0)
            cf.cf_fc_bwd(n, D[i], D[i + 1], x, xb, self.fw[i], None if last else self.h[i], self.slope,
                         None if last else self.masks[i], self.keep, g, dx, dxb, self.dfw[i], self.dfb[i], s)
            g = dx if i > 0 else None
        self.stack.backward(self.dfeat, s)

    def update(self, lr, beta1=0.9, beta2=0.999, eps=1e-8, stream=None):
        """One Adam step of every parameter (step counter t advances)."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        ps = self.params()
        if self._adam is None:
            self._adam = [(torch.zeros_like(p), torch.zeros_like(p)) for p, _, _ in ps]
        self.t += 1
        for (p, p16, g), (m, v) in zip(ps, self._adam):
            cf.cf_adam_step(p.numel(), p, p16, g, m, v, lr, beta1, beta2, eps, self.t, s)

    def step(self, lr, stream=None):
        self.forward(stream)
        self.backward(stream)
        self.update(lr, stream=stream)
