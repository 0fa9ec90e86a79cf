"""The CosmoFlow-shaped block stack on one GPU, sequenced through the C ABI.

A block is conv3d k=3 pad 1 -> + bias -> leaky ReLU -> 2x2x2 max-pool; the
stack chains L blocks, each halving the spatial width (CosmoFlow page,
section III-A; hybrid-parallelism page, Table I).  This class only owns the
device buffers (torch allocations) and enqueues the library's entry points on
one stream; every arithmetic step runs in libcfconv3d's kernels.

One training step of the stack (forward + backward):
  forward : for each block l  cf_conv3d_fwd(x_l, W_l, epi=(b_l, slope, I_l)) -> y_l
  backward: block L-1: cf_bias_lrelu_pool_bwd(dY, y, I) -> dZ, db
            block l < L-1: cf_bias_lrelu_pool_bwd(g_l, None, I_l) -> dZ_l, db_l
            cf_conv3d_wgrad(x_l, dZ_l) -> dW_l
            l > 0: cf_conv3d_dgrad(dZ_l, W_l, x_act = x_l) -> g_{l-1}
            (g_{l-1} already carries the leaky-ReLU derivative of block l-1;
            the first block's input gradient has no consumer and is skipped)
  With fuse_pool_bwd set, a max-pooled block below the top gets its dense dZ
  (and its bias gradient, the channel sums of g) from the backward-data launch
  of the block above (cf_conv3d_dgrad_pool_bwd routes g to the argmax in its
  epilogue) instead of a pool-backward launch.
  The first block, when its input has 1 or 4 channels, needs dZ only for its
  weight gradient: cf_conv3d_wgrad takes the pooled gradient with the argmax
  codes (routed form), expanding dZ on chip, so its dense dZ is never
  allocated, and its bias gradient (the channel sums of that pooled gradient)
  comes from the epilogue of block 2's backward-data conv (dsum): block 1 has
  no pool-backward launch.
  The weight gradients are off the backward critical path (nothing in the
  step reads dW), so by default they run on a second stream, each after its
  block's pool backward (event), with their own workspace; the step ends by
  joining that stream.  Kernels of the two chains overlap where one leaves
  SMs idle (the small deep layers, grid tails).  The first block's weight
  gradient is the exception: it goes on the critical stream right after
  block 2's backward data, so that it does not queue behind block 2's weight
  gradient (measured: 1.426 -> 1.409 ms per step).
"""
from __future__ import annotations

import torch

from . import cfconv as cf


def sample_ranges(n: int, chunks: int):
    """[n0, n1) sample ranges splitting n samples into min(n, chunks) nearly
    equal, non-empty, ascending pieces (at least one)."""
    k = max(1, min(n, chunks))
    return [(i * n // k, (i + 1) * n // k) for i in range(k) if (i + 1) * n // k > i * n // k]


POOL_CODES = {"max": cf.CF_POOL_MAX, "avg": cf.CF_POOL_AVG, "none": cf.CF_POOL_NONE}


class CosmoStack:
    """specs: optional per-block (stride, pool) or (stride, pool, "bn"), stride
    1 or 2, pool "max", "avg" or "none" (default: stride 1 and max-pooling
    everywhere, the CosmoFlow-shaped five-block stack); "bn" puts batch
    normalisation (batch statistics, gamma / beta = self.gamma[l] / self.b[l])
    between the conv and the activation.  The hybrid-parallelism page's Table I
    model is channels (4, 16, 32, 64, 128, 256, 256, 256) with a stride-2
    fourth conv and no pooling after the last two at width 128."""

    # batch-norm epsilon of blocks with spec (stride, pool, "bn")
    bn_eps = 1e-5

    def __init__(self, n: int, spatial: int, channels, slope: float = 0.3, device: str = "cuda",
                 backward: bool = True, overlap: bool = True, specs=None):
        self.n, self.spatial, self.channels, self.slope = n, spatial, tuple(channels), float(slope)
        self.L = len(channels) - 1
        self.specs = [tuple(t) for t in specs] if specs is not None else [(1, "max")] * self.L
        assert len(self.specs) == self.L
        self.device = device
        bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
        s = spatial
        self.dims = []   # (n, d, h, w) of each block's conv input
        self.odims = []  # (n, d, h, w) of each block's conv output
        self.x = torch.empty((n, s, s, s, channels[0]), dtype=bf, device=device)
        self.w, self.b, self.y, self.idx = [], [], [], []
        for l in range(self.L):
            ci, co = channels[l], channels[l + 1]
            stride, pool = self.specs[l][0], self.specs[l][1]
            so = (s + stride - 1) // stride
            sp = so if pool == "none" else so // 2
            self.dims.append((n, s, s, s))
            self.odims.append((n, so, so, so))
            self.w.append(torch.empty((co, 3, 3, 3, ci), dtype=bf, device=device))
            self.b.append(torch.zeros((co,), dtype=f32, device=device))
            self.y.append(torch.empty((n, sp, sp, sp, co), dtype=bf, device=device))
            # argmax codes (max) or sign masks (avg) of the pooled output
            self.idx.append(torch.empty((n, sp, sp, sp, co), dtype=u8, device=device) if pool != "none" else None)
            s = sp
        # batch-norm blocks: the stored conv output, the channel sums (sum z,
        # sum z^2), gamma
        self.zc, self.stats, self.gamma = [None] * self.L, [None] * self.L, [None] * self.L
        for l in range(self.L):
            if self.bn(l):
                n_, d, h, w = self.odims[l]
                co = channels[l + 1]
                self.zc[l] = torch.empty((n_, d, h, w, co), dtype=bf, device=device)
                self.stats[l] = torch.empty((2 * co,), dtype=f32, device=device)
                self.gamma[l] = torch.ones((co,), dtype=f32, device=device)
        self.backward_enabled = backward
        # with overlap: the backward-data chain on a high-priority stream (it is the
        # step's critical path), the weight gradients on a normal-priority one
        self.side = torch.cuda.Stream(device=device) if (backward and overlap) else None
        self.crit = torch.cuda.Stream(device=device, priority=-1) if (backward and overlap) else None
        ws = ws_w = 0
        for l in range(self.L):
            if self.bn(l):
                ws = max(ws, cf.cf_workspace_size(cf.CF_OP_BN, cf.cf_conv_desc(1, 1, 1, 1, 1, channels[l + 1])))
        if backward:
            self.dz, self.dw, self.db, self.g = [], [], [], []
            # per-block partial bias sums of each max-pooled block's pool backward,
            # reduced on the side stream (see backward)
            self.bpart_rows = cf.cf_pool_bwd_partial_rows()
            self.bpart = [torch.empty((self.bpart_rows, channels[l + 1]), dtype=f32, device=device)
                          for l in range(self.L)]
            # backward-data filters of blocks 2..L (cf_filter_flip), see backward
            self.wt = [None] + [torch.empty((channels[l], 3, 3, 3, channels[l + 1]), dtype=bf, device=device)
                                for l in range(1, self.L)]
            self.dgamma = [None] * self.L
            self.dsums = [None] * self.L
            for l in range(self.L):
                n_, d, h, w = self.odims[l]
                co = channels[l + 1]
                self.dz.append(None if self.routed(l) else torch.empty((n_, d, h, w, co), dtype=bf, device=device))
                self.dw.append(torch.empty((co, 3, 3, 3, channels[l]), dtype=f32, device=device))
                if self.bn(l):
                    # (dbeta, dgamma) side by side, as the batch-norm backward writes them
                    self.dsums[l] = torch.empty((2 * co,), dtype=f32, device=device)
                    self.db.append(self.dsums[l][:co])
                    self.dgamma[l] = self.dsums[l][co:]
                else:
                    self.db.append(torch.empty((co,), dtype=f32, device=device))
                # g[l]: the dgrad output of block l+1: the gradient w.r.t. block l's
                # pooled pre-activation (max), its output (avg); an unpooled block's
                # dgrad output is its dZ itself (g[l] aliases dz[l]) unless it is
                # batch-normalised
                pool = self.specs[l][1]
                if pool == "none" and l < self.L - 1 and not self.bn(l):
                    self.g.append(self.dz[l])
                elif l < self.L - 1 or self.routed(l):
                    self.g.append(torch.empty(tuple(self.y[l].shape), dtype=bf, device=device))
                else:
                    self.g.append(None)
            for l in range(self.L):
                desc = self.desc(l)
                ws_w = max(ws_w, cf.cf_workspace_size(
                    cf.CF_OP_WGRAD_ROUTED if self.routed(l) else cf.CF_OP_WGRAD, desc))
                ws = max(ws, cf.cf_workspace_size(cf.CF_OP_POOL_BWD, desc))
                if l > 0:
                    ws = max(ws, cf.cf_workspace_size(cf.CF_OP_DGRAD, desc))
        if self.side is None:
            ws = max(ws, ws_w)
        elif backward and self.first_wgrad_on_main:
            ws = max(ws, cf.cf_workspace_size(cf.CF_OP_WGRAD_ROUTED if self.routed(0) else cf.CF_OP_WGRAD,
                                              self.desc(0)))
        self.ws = torch.empty((max(ws, 256),), dtype=torch.uint8, device=device)
        # the weight gradients' workspace (the main one when they share the stream)
        self.ws_w = torch.empty((max(ws_w, 256),), dtype=torch.uint8, device=device) if self.side else self.ws

    # lower max-pooled blocks take their dZ (and bias gradient) from the
    # backward-data launch of the block above (cf_conv3d_dgrad_pool_bwd) when
    # set.  Off by default: that epilogue's lanes own voxels, so its routed
    # stores scatter over 32 rows per instruction, and measured slower than
    # the separate pool backward whose lanes own channel groups (dgrad3 +
    # routing 0.248 ms against 0.101 + 0.060 ms for N = 8 x 4 x 128^3)
    fuse_pool_bwd = False

    # the max-pool backward leaves its bias gradient as partial sums that the
    # side stream reduces (cf_bias_lrelu_pool_bwd_partials, cf_column_sums):
    # nothing on the critical stream reads it
    defer_bias_sums = True

    # the backward-data filters are flipped once per step on the side stream,
    # during the forward (cf_filter_flip), instead of inside each backward-data
    # call on the critical stream
    preflip = True
    # the first block's weight gradient on the critical stream, right after the
    # backward data of block 2 (its input), with the critical stream's workspace
    first_wgrad_on_main = True

    def routed(self, l) -> bool:
        """Block l's weight gradient takes the pooled gradient + argmax codes."""
        return l == 0 and self.channels[0] in (1, 4) and self.specs[0] == (1, "max")

    def bn(self, l) -> bool:
        """Block l has batch normalisation between its conv and its activation."""
        return len(self.specs[l]) > 2 and self.specs[l][2] == "bn"

    def pool_bwd_fused(self, l) -> bool:
        """Block l's max-pool backward runs in block l+1's backward-data epilogue."""
        return (self.fuse_pool_bwd and l < self.L - 1 and self.specs[l][1] == "max" and not self.routed(l)
                and not self.bn(l) and self.specs[l + 1][0] == 1)

    def desc(self, l):
        n, d, h, w = self.dims[l]
        return cf.cf_conv_desc(n, d, h, w, self.channels[l], self.channels[l + 1], self.specs[l][0])

    def epi(self, l, idx=None):
        """Forward epilogue of block l (bias, slope, codes/masks, pooling kind);
        None for a batch-normalised block (its conv output is stored plain)."""
        if self.bn(l):
            return None
        return (self.b[l], self.slope, self.idx[l] if idx is None else idx, POOL_CODES[self.specs[l][1]])

    def _fwd_block(self, l, stream):
        """Block l's forward launches: the conv with its fused epilogue, or, with
        batch normalisation, the plain conv, the channel sums and the
        normalisation + activation + pooling."""
        if not self.bn(l):
            cf.cf_conv3d_fwd(self.desc(l), self.block_input(l), self.w[l], self.epi(l), self.y[l], None, 0, stream)
            return
        n, d, h, w = self.odims[l]
        co = self.channels[l + 1]
        cf.cf_conv3d_fwd(self.desc(l), self.block_input(l), self.w[l], None, self.zc[l], None, 0, stream)
        cf.cf_bn_stats(n * d * h * w, co, self.zc[l], self.stats[l], self.ws, self.ws.numel(), stream)
        cf.cf_bn_act_pool_fwd(POOL_CODES[self.specs[l][1]], n, d, h, w, co, self.zc[l], self.stats[l], self.gamma[l],
                              self.b[l], self.bn_eps, self.slope, self.y[l], self.idx[l], stream)

    def block_input(self, l):
        return self.x if l == 0 else self.y[l - 1]

    def load(self, x_u16, ws_u16, bs_f32):
        """Copies host inputs (numpy bf16 bit patterns / fp32) into the device buffers."""
        import numpy as np

        def up(dst, a):
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
            dst.copy_(t.reshape(dst.shape))
        up(self.x, x_u16)
        for l in range(self.L):
            up(self.w[l], ws_u16[l])
            self.b[l].copy_(torch.from_numpy(np.ascontiguousarray(bs_f32[l], dtype=np.float32)))

    def _main(self, stream):
        return stream if stream is not None else torch.cuda.current_stream(self.device)

    _capturing = False
    timer_keys = None  # when set, only these ops get events

    def _run(self, key, stream, fn, timer):
        """fn(); with a timer list, CUDA events around it on `stream` are appended
        as (key, start, end) (recorded as graph nodes while capturing)."""
        if timer is None or (self.timer_keys is not None and key not in self.timer_keys):
            fn()
            return
        kw = {"external": True} if self._capturing else {}
        e0, e1 = torch.cuda.Event(enable_timing=True, **kw), torch.cuda.Event(enable_timing=True, **kw)
        e0.record(stream)
        fn()
        e1.record(stream)
        timer.append((key, e0, e1))

    # blocks run per sample range by step_host while the input is still arriving
    # (those whose per-sample volume is at least 32^3 voxels: enough tiles)
    def _chunked_blocks(self) -> int:
        return sum(1 for l in range(self.L) if self.dims[l][1] >= 32)

    def _issue_flips(self, caller, side, timer):
        """The backward-data filters of blocks 2..L (cf_filter_flip) on `side`,
        after the work enqueued on `caller` so far.  Returns the event the
        critical stream waits on before its first backward-data launch (None
        when `side` is `caller`)."""
        if side is not caller:
            ev = torch.cuda.Event()
            ev.record(caller)
            side.wait_event(ev)

        def flips():
            for l in range(1, self.L):
                cf.cf_filter_flip(self.channels[l + 1], self.channels[l], self.w[l], self.wt[l], side)

        self._run("flip", side, flips, timer)
        if side is caller:
            return None
        ev = torch.cuda.Event()
        ev.record(side)
        return ev

    def forward(self, stream=None, timer=None, x_chunks=None, serial=False):
        """timer: optional list receiving (key, start event, end event) per launch.
        x_chunks: optional [(n0, n1, event)]: the leading blocks (those of
        _chunked_blocks) run per sample range [n0, n1), each range after its
        event (its input has landed); a sample's outputs do not depend on the
        others, so the results are the same bits as launches over the batch.
        With the backward enabled, the backward-data filters are flipped on the
        side stream while the forward runs (serial: on the caller's stream)."""
        main = self._main(stream)
        if self.backward_enabled and self.preflip and self.L > 1:
            side = self.side if (self.side is not None and not serial) else main
            self._flips = (self._issue_flips(main, side, timer),)
        first = 0
        if x_chunks is not None:
            first = max(1, self._chunked_blocks())
            if any(self.bn(l) for l in range(first)):
                first = 0  # batch statistics need the whole batch: no per-sample blocks
            for n0, n1, ev in x_chunks:
                main.wait_event(ev)
                for l in range(first):
                    _, d, h, w = self.dims[l]
                    idx = self.idx[l][n0:n1] if self.idx[l] is not None else None
                    cf.cf_conv3d_fwd(cf.cf_conv_desc(n1 - n0, d, h, w, self.channels[l], self.channels[l + 1],
                                                     self.specs[l][0]),
                                     self.block_input(l)[n0:n1], self.w[l], self.epi(l, idx), self.y[l][n0:n1],
                                     None, 0, main)
        if x_chunks is not None and first == 0:
            for _, _, ev in x_chunks:
                main.wait_event(ev)
        for l in range(first, self.L):
            self._run(f"fwd{l + 1}", main, lambda l=l: self._fwd_block(l, main), timer)

    def backward(self, dy, stream=None, timer=None, serial=False, host_out=None):
        """timer: as in forward (keys "poolbwd<l+1>", "wgrad<l+1>", "dgrad<l+1>").
        serial: every op on the caller's stream (each op's events then time it
        alone).  host_out: optional (dw_host, db_host, copy_stream): each dW and
        db is copied to its host tensor on the copy stream as soon as the
        launch that completes it has run (the caller joins the copy stream)."""
        caller = self._main(stream)
        main = self.crit if (self.crit is not None and not serial) else caller
        side = self.side if (self.side is not None and not serial) else caller
        if main is not caller:
            ev = torch.cuda.Event()
            ev.record(caller)
            main.wait_event(ev)
        ws, wsb = self.ws, self.ws.numel()
        wsw, wswb = self.ws_w, self.ws_w.numel()
        # the backward-data filters (flipped, transposed) of blocks 2..L: issued by
        # the forward of this step, else here on the side stream
        flip_ev = None
        flips = self.__dict__.pop("_flips", None)
        if self.preflip and self.L > 1:
            flip_ev = flips[0] if flips is not None else self._issue_flips(caller, side, timer)

        def to_host(src_stream, dst, src):
            if host_out is None:
                return
            cp = host_out[2]
            ev = torch.cuda.Event()
            ev.record(src_stream)
            cp.wait_event(ev)
            with torch.cuda.stream(cp):
                dst.copy_(src, non_blocking=True)

        for l in range(self.L - 1, -1, -1):
            n, d, h, w = self.odims[l]
            co = self.channels[l + 1]
            routed = self.routed(l)
            pool = self.specs[l][1]
            deferred = False  # the bias gradient left as partial sums for the side stream
            if self.bn(l):
                # batch norm (with the activation / pooling backward folded in):
                # dZ, dbeta (db[l]) and dgamma from dy or g
                top = l == self.L - 1
                src = dy if top else self.g[l]
                fn = lambda: cf.cf_bn_act_pool_bwd(POOL_CODES[pool], n, d, h, w, co, src,
                                                   self.y[l] if top else None, self.idx[l], self.zc[l],
                                                   self.stats[l], self.gamma[l], self.bn_eps, self.slope,
                                                   self.dz[l], self.dsums[l], ws, wsb, main)
                self._run(f"poolbwd{l + 1}", main, fn, timer)
                to_host(main, host_out and host_out[1][l], self.db[l])
            elif l == self.L - 1:
                if pool == "max" and self.defer_bias_sums:
                    fn = lambda: cf.cf_bias_lrelu_pool_bwd_partials(n, d, h, w, co, dy, self.y[l], self.idx[l],
                                                                    self.slope, self.dz[l],
                                                                    self.g[l] if routed else None, self.bpart[l],
                                                                    main)
                    deferred = True
                elif pool == "max":
                    fn = lambda: cf.cf_bias_lrelu_pool_bwd(n, d, h, w, co, dy, self.y[l], self.idx[l], self.slope,
                                                           self.dz[l], self.g[l] if routed else None, self.db[l],
                                                           ws, wsb, main)
                else:
                    fn = lambda: cf.cf_block_epilogue_bwd(POOL_CODES[pool], n, d, h, w, co, dy,
                                                          self.y[l] if pool == "none" else None, self.idx[l],
                                                          self.slope, self.dz[l], None, self.db[l], ws, wsb, main)
                self._run(f"poolbwd{l + 1}", main, fn, timer)
                if not deferred:
                    to_host(main, host_out and host_out[1][l], self.db[l])
            elif pool == "max" and not routed and not self.pool_bwd_fused(l):
                if self.defer_bias_sums:
                    fn = lambda: cf.cf_bias_lrelu_pool_bwd_partials(n, d, h, w, co, self.g[l], None, self.idx[l],
                                                                    self.slope, self.dz[l], None, self.bpart[l], main)
                    deferred = True
                else:
                    fn = lambda: cf.cf_bias_lrelu_pool_bwd(n, d, h, w, co, self.g[l], None, self.idx[l], self.slope,
                                                           self.dz[l], None, self.db[l], ws, wsb, main)
                self._run(f"poolbwd{l + 1}", main, fn, timer)
                if not deferred:
                    to_host(main, host_out and host_out[1][l], self.db[l])
            elif pool == "avg":
                fn = lambda: cf.cf_block_epilogue_bwd(cf.CF_POOL_AVG, n, d, h, w, co, self.g[l], None, self.idx[l],
                                                      self.slope, self.dz[l], None, self.db[l], ws, wsb, main)
                self._run(f"poolbwd{l + 1}", main, fn, timer)
                to_host(main, host_out and host_out[1][l], self.db[l])
            # (a routed, unpooled or fused block below the top: db[l] came with g[l]
            # from block l+1's dgrad, as the channel sums of its output; a fused
            # one's dZ too)
            desc = self.desc(l)
            if side is not main:
                ev = torch.cuda.Event()
                ev.record(main)
                side.wait_event(ev)
            if deferred:
                # the bias gradient from the pool backward's partial sums, off the
                # critical stream
                self._run(f"poolbwd{l + 1}_sum", side,
                          lambda: cf.cf_column_sums(self.bpart_rows, co, self.bpart[l], self.db[l], side), timer)
                to_host(side, host_out and host_out[1][l], self.db[l])
            # (the first block's weight gradient: after block 2's backward data, below)
            if l == 0 and self.first_wgrad_on_main and side is not main:
                wst, wws, wwsb = main, ws, wsb
            else:
                wst, wws, wwsb = side, wsw, wswb
            if routed:
                fn = lambda: cf.cf_conv3d_wgrad(desc, self.block_input(l), self.g[l], self.idx[l], self.dw[l], 0,
                                                wws, wwsb, wst)
            else:
                fn = lambda: cf.cf_conv3d_wgrad(desc, self.block_input(l), self.dz[l], None, self.dw[l], 0, wws,
                                                wwsb, wst)
            self._run(f"wgrad{l + 1}", wst, fn, timer)
            to_host(wst, host_out and host_out[0][l], self.dw[l])
            if l > 0:
                below = self.specs[l - 1][1]
                fused = self.pool_bwd_fused(l - 1)
                dsum = self.db[l - 1] if (not self.bn(l - 1) and (self.routed(l - 1) or below == "none" or fused)) \
                    else None
                # the lower block's output derivative rides on the input gradient
                # unless it is average-pooled (its derivative is per voxel, from its masks)
                x_act = self.block_input(l) if below != "avg" else None
                if fused:
                    fn = lambda: cf.cf_conv3d_dgrad_pool_bwd(desc, self.dz[l], self.w[l], x_act, self.slope,
                                                             self.g[l - 1], self.idx[l - 1], self.dz[l - 1], ws, wsb,
                                                             main, dsum=dsum)
                elif self.preflip:
                    if flip_ev is not None:
                        main.wait_event(flip_ev)
                        flip_ev = None
                    fn = lambda: cf.cf_conv3d_dgrad_flipped(desc, self.dz[l], None, self.wt[l], x_act, self.slope,
                                                            self.g[l - 1], ws, wsb, main, dsum=dsum)
                else:
                    fn = lambda: cf.cf_conv3d_dgrad(desc, self.dz[l], None, self.w[l], x_act, self.slope,
                                                    self.g[l - 1], ws, wsb, main, dsum=dsum)
                self._run(f"dgrad{l + 1}", main, fn, timer)
                if dsum is not None:
                    to_host(main, host_out and host_out[1][l - 1], dsum)
        for s in (main, side) + ((host_out[2],) if host_out is not None else ()):
            if s is not caller:
                ev = torch.cuda.Event()
                ev.record(s)
                caller.wait_event(ev)

    def step(self, dy, stream=None, timer=None, serial=False):
        self.forward(stream, timer, serial=serial)
        if self.backward_enabled:
            self.backward(dy, stream, timer, serial)

    def _copy_stream(self):
        if getattr(self, "_cp", None) is None:
            self._cp = torch.cuda.Stream(device=self.device)
        return self._cp

    def step_host(self, x_host, dy_host, dw_host, db_host, stream=None, chunks=None):
        """One training step from host inputs to host results: x_host (the batch,
        [n][d][h][w][c0] bf16) and dy_host (the gradient at the top output) in
        pinned host memory are copied in, every dW[l] and db[l] is copied out to
        the pinned host tensors dw_host[l] / db_host[l].  The copies overlap the
        compute: the input goes over in `chunks` sample ranges (default: one per
        sample, at most 8), the leading blocks running on each range as it
        lands, and each gradient leaves as soon as it is final.  Same results, bit for
        bit, as load + step + copy-back.  The host tensors must stay untouched
        until the caller's stream has passed the step."""
        main = self._main(stream)
        cp = self._copy_stream()
        ev = torch.cuda.Event()
        ev.record(main)
        cp.wait_event(ev)  # after the previous work on the caller's stream (buffer reuse)
        x_chunks = []
        with torch.cuda.stream(cp):
            for n0, n1 in sample_ranges(self.n, chunks if chunks else 8):
                self.x[n0:n1].copy_(x_host.view(self.x.shape)[n0:n1], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cp)
                x_chunks.append((n0, n1, e))
            dy_dev = self._dy_buffer(dy_host)
            dy_dev.copy_(dy_host.view(dy_dev.shape), non_blocking=True)
            e_dy = torch.cuda.Event()
            e_dy.record(cp)
        self.forward(main, None, x_chunks)
        if self.backward_enabled:
            main.wait_event(e_dy)
            self.backward(dy_dev, main, host_out=(dw_host, db_host, cp))
        else:
            ev = torch.cuda.Event()
            ev.record(cp)
            main.wait_event(ev)

    def _input_buffers(self):
        """The two input buffer pairs (x, dY at the top) of step_host_pipelined."""
        if getattr(self, "_xbuf", None) is None:
            dy_shape = tuple(self.y[-1].shape)
            self._xbuf = [self.x, torch.empty_like(self.x)]
            self._dybuf = [torch.empty(dy_shape, dtype=torch.bfloat16, device=self.device) for _ in range(2)]
            self._pf = torch.cuda.Stream(device=self.device)
            self._parity = 0
        return self._xbuf, self._dybuf

    def prefetch_host(self, x_host, dy_host, stream=None):
        """Copies the first batch of a step_host_pipelined loop (pinned host x and
        dY) into the input buffers its next call computes on."""
        main = self._main(stream)
        xs, dys = self._input_buffers()
        p = self._parity
        with torch.cuda.stream(main):
            xs[p].copy_(x_host.view(xs[p].shape), non_blocking=True)
            dys[p].copy_(dy_host.view(dys[p].shape), non_blocking=True)

    def step_host_pipelined(self, x_next, dy_next, dw_host, db_host, stream=None):
        """One step of a host-fed training loop with double-buffered input: the
        step computes on the batch the previous call (or prefetch_host) copied
        in, while the next batch (x_next, dy_next: pinned host) goes over on the
        copy stream into the other buffer pair; every dW[l] and db[l] is copied
        out to dw_host[l] / db_host[l] as soon as it is final.  Per call: one
        batch in, one set of gradients out, like step_host; the results are the
        same bits as load + step + copy-back of the batch computed on.  The host
        tensors must stay untouched until the caller's stream has passed the call."""
        main = self._main(stream)
        cp = self._copy_stream()
        xs, dys = self._input_buffers()
        pf = self._pf  # host-to-device, beside the device-to-host gradient copies on cp
        p = self._parity
        ev = torch.cuda.Event()
        ev.record(main)
        cp.wait_event(ev)
        pf.wait_event(ev)  # the other buffer pair was last read by the previous call
        with torch.cuda.stream(pf):
            xs[1 - p].copy_(x_next.view(xs[1 - p].shape), non_blocking=True)
            dys[1 - p].copy_(dy_next.view(dys[1 - p].shape), non_blocking=True)
        self.x = xs[p]
        try:
            self.forward(main)
            if self.backward_enabled:
                self.backward(dys[p], main, host_out=(dw_host, db_host, cp))
        finally:
            self.x = xs[0]
        for s in (cp, pf):
            ev = torch.cuda.Event()
            ev.record(s)
            main.wait_event(ev)
        self._parity = 1 - p

    def _dy_buffer(self, dy_host):
        """Device buffer of the top-output gradient for step_host."""
        if getattr(self, "_dy", None) is None:
            self._dy = torch.empty(tuple(self.y[-1].shape), dtype=torch.bfloat16, device=self.device)
        return self._dy

    def capture_pipelined(self, x_host, dy_host, dw_host, db_host):
        """The two CUDA graphs of step_host_pipelined (one per input buffer
        pair), to be replayed alternately starting with the first after
        prefetch_host; the parity is back at its value on entry."""
        self._input_buffers()
        self._copy_stream()
        p0 = self._parity
        graphs = [self.capture(None, host=(x_host, dy_host, dw_host, db_host), pipelined=True) for _ in range(2)]
        assert self._parity == p0
        return graphs

    def capture(self, dy, timer=None, keys=None, host=None, pipelined=False):
        """Records one step into a CUDA graph (replay() then re-runs it with no
        per-launch host work).  The buffers, dy included, are bound at capture.
        With a timer list, the events of the ops in `keys` (all if None) become
        event-record nodes.  host: (x_host, dy_host, dw_host, db_host) records
        step_host instead (its copies become graph nodes; dy is unused)."""
        g = torch.cuda.CUDAGraph()
        cur = torch.cuda.current_stream(self.device)
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(cur)
        self._capturing, self.timer_keys = True, keys
        try:
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    if host is not None and pipelined:
                        self.step_host_pipelined(*host, stream=s)
                    elif host is not None:
                        self.step_host(*host, stream=s)
                    else:
                        self.step(dy, s, timer)
        finally:
            self._capturing, self.timer_keys = False, None
        cur.wait_stream(s)
        return g

    def launches_per_step(self) -> int:
        """Kernels one step enqueues: fwd 1 per block; pool-bwd 2 (scatter +
        bias sum) per block except a routed or unpooled block below the top;
        wgrad 2 (split-K + reduce) per block, +1 for a stride-2 block (zero
        insertion); dgrad 2 (filter flip + conv) for blocks 1..L-1 (+1 for
        stride 2), plus the channel sums for a routed or unpooled block below:
        1 (partials reduction) when fused in the halo-tile epilogue, else 2."""
        n = self.L + 3 * sum(1 for l in range(self.L) if self.bn(l))  # BN: sums, reduction, normalisation
        if self.backward_enabled:
            ch = self.channels
            for l in range(self.L):
                s2 = self.specs[l][0] == 2
                n += 2 + s2  # wgrad
                pool = self.specs[l][1]
                if self.bn(l):
                    n += 3  # batch-norm backward: sums, their reduction, dZ
                elif l == self.L - 1 or not (self.routed(l) or pool == "none" or self.pool_bwd_fused(l)):
                    n += 2  # pool backward
                if l > 0:
                    n += 2 + s2  # dgrad
                    if self.bn(l - 1):
                        pass
                    elif self.routed(l - 1) or self.specs[l - 1][1] == "none" or self.pool_bwd_fused(l - 1):
                        fused = (not s2 and ch[l] <= 32 and ch[l] % 16 == 0 and ch[l] in (32, 64, 128)
                                 and ch[l + 1] % 16 == 0)
                        n += 1 if fused else 2
        return n
