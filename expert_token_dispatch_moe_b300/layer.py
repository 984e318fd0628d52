"""MoELayer: the whole single-device hot path as one object.

Holds the layer's weights (with W1/W3 packed once for the grouped FFN) and
every intermediate buffer, allocated once through torch on the current CUDA
device, and runs the C-ABI steps in order on one stream:

    moe_router_logits -> moe_route -> moe_permute -> moe_ep_layout
      -> moe_grouped_ffn -> moe_combine

(the seven steps of an expert-parallel MoE layer forward, with the exchange
steps replaced by the simulated send layout on one device).
"""
from __future__ import annotations

import torch

from . import (MoeCfg, MoeLayerBufs, moe_backward_workspace_bytes, moe_combine, moe_combine_backward,
               moe_ep_layout, moe_grouped_ffn, moe_grouped_ffn_backward, moe_grouped_ffn_gather,
               moe_grouped_ffn_train, moe_grouped_ffn_combine, moe_layer_forward, moe_layer_forward_host,
               moe_grouped_rows, moe_last_launch_count, moe_pack_backward, moe_pack_router,
               moe_pack_w13, moe_permute, moe_permute_backward, moe_route, moe_router_logits,
               moe_workspace_bytes, moe_workspace_init)

# Routers with at least this many experts run on the tensor cores (three-term
# bf16 split of the fp32 weights); smaller ones are bandwidth-bound SIMT dot
# products.
TC_ROUTER_MIN_E = 17


class MoELayer:
    def __init__(self, cfg, W1, W3, W2, W_r=None, logit_bias=None, selection_bias=None,
                 device=None, with_send_buf=True, tc_router=None, gather=False, train=False,
                 combine_in_epilogue=False):
        """gather=True: the permute computes indices only and GEMM 1 gathers its
        rows from x (moe_grouped_ffn_gather); x_sorted is not written.
        train=True: the forward keeps GEMM 1's pre-activations (self.g1) so the
        backward need not recompute them.
        combine_in_epilogue=True: GEMM 2 adds its gated rows into y itself
        (moe_grouped_ffn_combine) and y_sorted is not written; faster on the
        large layers, but with more than two contributions per token the output
        is not bit-reproducible from run to run."""
        self.cfg = cfg if isinstance(cfg, MoeCfg) else MoeCfg.from_layer(cfg)
        c = self.cfg
        if combine_in_epilogue and (gather or train):
            raise ValueError("combine_in_epilogue takes neither gather nor train")
        self.combine_in_epilogue = combine_in_epilogue
        dev = torch.device(device or "cuda")
        self.device = dev
        i32, f32, bf16 = torch.int32, torch.float32, torch.bfloat16
        n_exp = c.E + c.has_shared
        for w, shape in ((W1, (n_exp, c.f, c.d)), (W3, (n_exp, c.f, c.d)), (W2, (n_exp, c.d, c.f))):
            if tuple(w.shape) != shape or w.dtype != bf16 or w.device.type != "cuda":
                raise ValueError(f"expert weight must be bf16 cuda {shape}, got {tuple(w.shape)}")
        self.W_r = W_r
        self.W_r_split = None
        if tc_router is None:
            tc_router = c.E >= TC_ROUTER_MIN_E
        if W_r is not None and tc_router:
            self.W_r_split = torch.empty(3, c.E, c.d, dtype=bf16, device=dev)
            moe_pack_router(c, W_r, self.W_r_split)
        self.logit_bias = logit_bias
        self.selection_bias = selection_bias
        self.W2 = W2.contiguous()
        self.W13 = torch.empty(n_exp, 2 * c.f, c.d, dtype=bf16, device=dev)
        moe_pack_w13(c, W1.contiguous(), W3.contiguous(), self.W13)
        rows = moe_grouped_rows(c)
        self.scores = torch.empty(c.T, c.E, dtype=f32, device=dev)
        self.topk_idx = torch.empty(c.T, c.k, dtype=i32, device=dev)
        self.topk_gate = torch.empty(c.T, c.k, dtype=f32, device=dev)
        self.counts = torch.empty(c.E, dtype=i32, device=dev)
        self.offsets = torch.empty(c.E + 1, dtype=i32, device=dev)
        self.order = torch.empty(c.R, dtype=i32, device=dev)
        self.inv = torch.empty(c.A, dtype=i32, device=dev)
        self.x_sorted = torch.empty(c.R, c.d, dtype=bf16, device=dev)
        self.count_mat = torch.empty(c.n_ep, c.n_ep, dtype=i32, device=dev)
        self.send_off = torch.empty(c.n_ep, c.n_ep, dtype=i32, device=dev)
        self.recv_off = torch.empty(c.n_ep, c.n_ep, dtype=i32, device=dev)
        self.send_idx = torch.empty(c.A, dtype=i32, device=dev)
        self.send_buf = torch.empty(c.A, c.d, dtype=bf16, device=dev) if with_send_buf else None
        self.h = torch.empty(rows, c.f, dtype=bf16, device=dev)
        self.y_sorted = torch.empty(rows, c.d, dtype=bf16, device=dev)
        self.y = torch.empty(c.T, c.d, dtype=bf16, device=dev)
        self.ws = torch.zeros(moe_workspace_bytes(c), dtype=torch.uint8, device=dev)
        moe_workspace_init(c, self.ws)
        self.gather = gather
        self.train = train
        self.g1 = torch.empty(rows, 2 * c.f, dtype=bf16, device=dev) if train else None
        self.launches_per_forward = None
        self.launches_per_backward = None
        self.W13t = None        # backward buffers, allocated on the first backward

    def forward(self, x, scores=None, y=None):
        """Run the layer on device tokens x (bf16 [T, d]); returns self.y, or
        `y` (bf16 [T, d] on the device) when given.

        With `scores` (fp32 [T, E]) the router step is skipped and the given
        scores are routed (used to check routing on exact inputs).  Each C-ABI
        call sits in an NVTX range named after it, for profilers' timelines."""
        c = self.cfg
        n = 0
        push, pop = torch.cuda.nvtx.range_push, torch.cuda.nvtx.range_pop
        if scores is None:
            push("moe_router_logits")
            moe_router_logits(c, x, self.W_r, self.W_r_split, self.logit_bias, self.scores,
                              self.ws)
            pop()
            n += moe_last_launch_count()
            scores = self.scores
        push("moe_route")
        moe_route(c, scores, self.selection_bias, self.topk_idx, self.topk_gate)
        pop()
        n += moe_last_launch_count()
        push("moe_permute")
        if self.gather:
            moe_permute(c, None, self.topk_idx, self.counts, self.offsets, self.order, self.inv,
                        None, self.ws)
        else:
            moe_permute(c, x, self.topk_idx, self.counts, self.offsets, self.order, self.inv,
                        self.x_sorted, self.ws)
        pop()
        n += moe_last_launch_count()
        push("moe_ep_layout")
        moe_ep_layout(c, self.topk_idx, self.offsets, self.inv, self.count_mat, self.send_off,
                      self.recv_off, self.send_idx, x if self.send_buf is not None else None,
                      self.send_buf, self.ws)
        pop()
        n += moe_last_launch_count()
        push("moe_grouped_ffn")
        if self.gather:
            moe_grouped_ffn_gather(c, x, self.order, self.counts, self.offsets, self.W13, self.W2,
                                   self.h, self.y_sorted, self.ws)
        elif self.train:
            moe_grouped_ffn_train(c, self.x_sorted, x if c.has_shared else None, self.counts,
                                  self.offsets, self.W13, self.W2, self.h, self.y_sorted, self.g1,
                                  self.ws)
        elif self.combine_in_epilogue:
            out = self.y if y is None else y
            moe_grouped_ffn_combine(c, self.x_sorted, x if c.has_shared else None, self.counts,
                                    self.offsets, self.W13, self.W2, self.h, self.order,
                                    self.topk_gate, out, self.ws)
            pop()
            n += moe_last_launch_count()
            self.launches_per_forward = n
            return out
        else:
            moe_grouped_ffn(c, self.x_sorted, x if c.has_shared else None, self.counts,
                            self.offsets, self.W13, self.W2, self.h, self.y_sorted, self.ws)
        pop()
        n += moe_last_launch_count()
        out = self.y if y is None else y
        push("moe_combine")
        moe_combine(c, self.y_sorted, self.inv, self.topk_gate, out)
        pop()
        n += moe_last_launch_count()
        self.launches_per_forward = n
        return out

    __call__ = forward

    def _backward_buffers(self):
        c, dev, bf16 = self.cfg, self.device, torch.bfloat16
        n_exp = c.E + c.has_shared
        rows = moe_grouped_rows(c)
        self.W13t = torch.empty(n_exp, c.d, 2 * c.f, dtype=bf16, device=dev)
        self.W2t = torch.empty(n_exp, c.f, c.d, dtype=bf16, device=dev)
        moe_pack_backward(c, self.W13, self.W2, self.W13t, self.W2t)
        self.d_o = torch.empty(rows, c.d, dtype=bf16, device=dev)
        self.dx_sorted = torch.empty(rows, c.d, dtype=bf16, device=dev)
        self.dW13 = torch.empty(n_exp, 2 * c.f, c.d, dtype=bf16, device=dev)
        self.dW2 = torch.empty(n_exp, c.d, c.f, dtype=bf16, device=dev)
        self.dgate = torch.empty(c.T, c.k, dtype=torch.float32, device=dev)
        self.dx = torch.empty(c.T, c.d, dtype=bf16, device=dev)
        self.bws = torch.empty(moe_backward_workspace_bytes(c), dtype=torch.uint8, device=dev)

    def backward(self, x, dy):
        """Gradients of the last forward (rows path) for output gradient dy
        (bf16 [T, d]), routing held fixed: returns self.dx and leaves self.dW13
        (packed like W13), self.dW2 and self.dgate."""
        if self.gather:
            raise RuntimeError("backward needs the forward's x_sorted (gather=False)")
        if self.combine_in_epilogue:
            raise RuntimeError("backward needs the forward's y_sorted (combine_in_epilogue=False)")
        c = self.cfg
        if self.W13t is None:
            self._backward_buffers()
        moe_combine_backward(c, dy, self.y_sorted, self.inv, self.topk_gate, self.d_o, self.dgate)
        n = moe_last_launch_count()
        moe_grouped_ffn_backward(c, self.x_sorted, x if c.has_shared else None, self.counts,
                                 self.offsets, self.W13, self.W13t, self.W2t, self.h, self.g1,
                                 self.d_o, self.dx_sorted, self.dW13, self.dW2, self.bws, self.ws)
        n += moe_last_launch_count()
        moe_permute_backward(c, self.dx_sorted, self.inv, self.dx)
        n += moe_last_launch_count()
        self.launches_per_backward = n
        return self.dx

    def unpacked_dW13(self):
        """(dW1, dW3) [E + has_shared, f, d] from the packed dW13."""
        n, f2, d = self.dW13.shape
        blk = self.dW13.view(n, f2 // 256, 2, 128, d)
        return blk[:, :, 0].reshape(n, f2 // 2, d), blk[:, :, 1].reshape(n, f2 // 2, d)

    def c_bufs(self) -> MoeLayerBufs:
        """This layer's weights and buffers as the C struct moe_layer (the
        router step included when the layer holds router weights)."""
        if getattr(self, "_c_bufs", None) is None:
            self._c_bufs = MoeLayerBufs.of(
                W_r=self.W_r if self.W_r_split is None else None, W_r_split=self.W_r_split,
                logit_bias=self.logit_bias, selection_bias=self.selection_bias, W13=self.W13,
                W2=self.W2, scores=self.scores, topk_idx=self.topk_idx, topk_gate=self.topk_gate,
                counts=self.counts, offsets=self.offsets, order=self.order, inv=self.inv,
                x_sorted=self.x_sorted, count_mat=self.count_mat, send_off=self.send_off,
                recv_off=self.recv_off, send_idx=self.send_idx, send_buf=self.send_buf,
                h=self.h, y_sorted=self.y_sorted, ws=self.ws,
                combine_in_epilogue=self.combine_in_epilogue, gather=self.gather)
        return self._c_bufs

    def forward_c(self, x, y=None):
        """The forward through the library's single entry point
        moe_layer_forward (same steps as forward, issued from C)."""
        if self.train:
            raise RuntimeError("moe_layer_forward runs the inference forward")
        out = self.y if y is None else y
        moe_layer_forward(self.cfg, self.c_bufs(), x, out)
        self.launches_per_forward = moe_last_launch_count()
        return out

    def forward_host_c(self, x_hosts, y_hosts):
        """forward_host_stream done by the library (moe_layer_forward_host):
        pinned host batches in and out, one copy per direction per batch on
        its own stream, double-buffered on the device, the forward issued
        from C.  Returns once enqueued; synchronise the current stream to wait
        for the last result."""
        if self.train:
            raise RuntimeError("moe_layer_forward_host runs the inference forward")
        s_in, s_out = self._copy_streams()
        self._stream_buffers()
        moe_layer_forward_host(self.cfg, self.c_bufs(), x_hosts, y_hosts, self._xbuf,
                               self._ybuf, torch.cuda.current_stream(self.device), s_in, s_out)
        return y_hosts

    def forward_host_stream(self, x_hosts, y_hosts):
        """Runs the layer on a sequence of host batches (pinned bf16 [T, d] each)
        and writes each result into the matching pinned host buffer.  Batch i's
        host-to-device copy and batch i-1's device-to-host copy run on their own
        streams while batch i-1 (resp. i) computes, with two device buffers on
        each side; the compute stream is the caller's current stream.  Returns
        when all copies have been enqueued (synchronise the current stream to
        wait for the last result)."""
        comp = torch.cuda.current_stream(self.device)
        s_in, s_out = self._copy_streams()
        self._stream_buffers()
        graphs = getattr(self, "_graphs", None)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        start = ev()
        start.record(comp)
        s_in.wait_event(start)
        for i, (xh, yh) in enumerate(zip(x_hosts, y_hosts)):
            b = i & 1
            if i >= 2:
                s_in.wait_event(comp_done[b])     # batch i-2 no longer reads xbuf[b]
            with torch.cuda.stream(s_in):
                self._xbuf[b].copy_(xh, non_blocking=True)
            in_done[b].record(s_in)
            comp.wait_event(in_done[b])
            if i >= 2:
                comp.wait_event(out_done[b])      # batch i-2's result has left ybuf[b]
            if graphs:
                graphs[b].replay()
            else:
                self.forward(self._xbuf[b], y=self._ybuf[b])
            comp_done[b].record(comp)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                yh.copy_(self._ybuf[b], non_blocking=True)
            out_done[b].record(s_out)
        n = len(x_hosts)
        for b in range(min(n, 2)):
            comp.wait_event(out_done[b])
        return y_hosts

    def capture_graphs(self):
        """Records the forward on each of forward_host_stream's two device
        buffer pairs as a CUDA graph, after one eager call per pair (one-time
        set-up such as kernel attributes happens there).  forward_host_stream
        then replays one graph per batch instead of issuing about ten calls,
        which matters when a batch computes in less time than the host takes
        to issue it.  The graphs hold this layer's buffers and workspace; call
        again after changing the layer's weights' storage."""
        self._stream_buffers()
        self._graphs = None
        comp = torch.cuda.current_stream(self.device)
        for b in range(2):
            self.forward(self._xbuf[b], y=self._ybuf[b])
        torch.cuda.synchronize(self.device)
        graphs = []
        for b in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.forward(self._xbuf[b], y=self._ybuf[b])
            graphs.append(g)
        comp.synchronize()
        self._graphs = graphs
        return graphs

    def _stream_buffers(self):
        if getattr(self, "_xbuf", None) is None:
            T, d = self.cfg.T, self.cfg.d
            self._xbuf = [torch.empty(T, d, dtype=torch.bfloat16, device=self.device)
                          for _ in range(2)]
            self._ybuf = [torch.empty(T, d, dtype=torch.bfloat16, device=self.device)
                          for _ in range(2)]

    def _copy_streams(self):
        if getattr(self, "_streams", None) is None:
            self._streams = (torch.cuda.Stream(self.device), torch.cuda.Stream(self.device))
        return self._streams

    def forward_host(self, x_host, y_host, x_dev=None):
        """End-to-end call with host buffers: copies pinned host x to the
        device, runs the layer, copies y back into pinned host y_host."""
        x_dev = x_dev if x_dev is not None else torch.empty_like(x_host, device=self.device)
        x_dev.copy_(x_host, non_blocking=True)
        y = self.forward(x_dev)
        y_host.copy_(y, non_blocking=True)
        return y_host
