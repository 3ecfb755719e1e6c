"""One MoE layer forward through the C ABI: the six steps of "LLM Internals §14.2.1"
as five library calls (router, dispatch, grouped SwiGLU, combine, balance stats).

`MoELayer` owns the device buffers of one batch shape; `forward` enqueues the calls on
the current stream and returns device tensors; `forward_host` is the end-to-end call a
host program makes (pinned host X in, host Y out).
"""

from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import binding as B
from .configs import MoEConfig


class MoELayer:
    def __init__(self, cfg: MoEConfig, weights: Dict[str, torch.Tensor],
                 ctx: Optional[B.Context] = None, device: int = 0,
                 capacity_factor: Optional[float] = None,
                 bias_gamma: Optional[float] = None):
        self.cfg = cfg
        # not None: every forward ends with the bias update step (update_bias)
        self.bias_gamma = bias_gamma
        self.w = weights
        self.dev = torch.device("cuda", device)
        self.ctx = ctx if ctx is not None else B.Context(device)
        self.score = B.MOE_SCORE_SIGMOID if cfg.score == "sigmoid" else B.MOE_SCORE_SOFTMAX
        self.capacity = (-1 if capacity_factor is None
                         else B.moe_capacity(capacity_factor, cfg.T, cfg.k, cfg.E))
        self.dtype_code = B.MOE_DTYPE_BF16 if cfg.dtype == "bf16" else B.MOE_DTYPE_F32
        self._alloc(cfg.T)
        self.fp8 = self._quantize_fp8() if cfg.fp8_experts else None

    def _quantize_fp8(self) -> Dict[str, torch.Tensor]:
        """FP8 E4M3 codes and per-output-channel scales of every expert weight (once)."""
        q = {}
        for name in ("gate", "up", "down", "s_gate", "s_up", "s_down"):
            shared = name.startswith("s_")
            src = ("Ws_" + name[2:]) if shared else ("W_" + name)
            if src not in self.w:
                continue
            W = self.w[src]
            codes = torch.empty(W.shape, dtype=torch.uint8, device=self.dev)
            scale = torch.empty(W.shape[:-1], dtype=torch.float32, device=self.dev)
            B.moe_quantize_fp8(self.ctx, W, codes, scale)
            tag = name[2:] if shared else name
            q[("Qs_" if shared else "Q_") + tag] = codes
            q[("Ss_" if shared else "S_") + tag] = scale
        torch.cuda.synchronize(self.dev)
        return q

    def _alloc(self, T: int) -> None:
        c, dev = self.cfg, self.dev
        i32, f32 = torch.int32, torch.float32
        xdt = torch.bfloat16 if c.dtype == "bf16" else torch.float32
        nbytes = B.moe_workspace_bytes(T, c.H, c.E, c.I, c.k, self.dtype_code, c.shared)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        B.moe_workspace_init(self.ws)
        self.idx = torch.empty(T, c.k, dtype=i32, device=dev)
        # expert-choice routing: E slots (token, expert) per token
        ks = c.E if c.expert_choice else c.k
        self.gate = torch.empty(T, ks, dtype=f32, device=dev)
        self.col_gap = torch.empty(c.E, dtype=f32, device=dev) if c.expert_choice else None
        self.gap = torch.empty(T, dtype=f32, device=dev)
        self.colsum = torch.empty(c.E, dtype=torch.float64, device=dev)
        self.counts = torch.empty(c.E, dtype=i32, device=dev)
        self.offsets = torch.empty(c.E + 1, dtype=i32, device=dev)
        self.row_of_slot = torch.empty(T * ks, dtype=i32, device=dev)
        self.slot_of_row = torch.empty(T * c.k, dtype=i32, device=dev)
        self.Xperm = torch.empty(T * c.k, c.H, dtype=xdt, device=dev)
        self.O = torch.empty(T * c.k, c.H, dtype=f32, device=dev)
        self.O_shared = torch.empty(T, c.H, dtype=f32, device=dev) if c.shared else None
        self.Y = torch.empty(T, c.H, dtype=f32, device=dev)
        self.f = torch.empty(c.E, dtype=torch.float64, device=dev)
        self.p = torch.empty(c.E, dtype=torch.float64, device=dev)
        self.stats = torch.empty(4, dtype=torch.float64, device=dev)
        # the balance statistics need only the routing and the counts, so they run on a
        # side stream beside the expert GEMMs and combine
        self._side = torch.cuda.Stream(device=dev)
        self._routed = torch.cuda.Event()
        self._stats_done = torch.cuda.Event()
        self.T = T

    def forward(self, X: torch.Tensor, stats: bool = True, stream=None,
                Y: Optional[torch.Tensor] = None,
                Y_bf16: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Enqueue the forward of X on `stream` (default: the current stream).  The fp32
        output goes to Y (default: the layer's own buffer), an optional bf16 copy to
        Y_bf16."""
        c, w = self.cfg, self.w
        if tuple(X.shape) != (self.T, c.H):
            raise ValueError(f"X has shape {tuple(X.shape)}, the layer takes {(self.T, c.H)}")
        if X.dtype != self.Xperm.dtype:
            raise TypeError(f"X is {X.dtype}, the layer computes in {self.Xperm.dtype}")
        Y = self.Y if Y is None else Y
        stream = torch.cuda.current_stream(self.dev) if stream is None else stream
        if c.expert_choice:
            return self._forward_expert_choice(X, Y, Y_bf16, stream)
        B.moe_router_topk(self.ctx, X, w["Wg"], c.k, self.score, c.renorm, self.idx,
                          self.gate, self.ws, bias=w.get("bias"),
                          logit_bias=w.get("logit_bias"), key_gap=self.gap,
                          prob_colsum=self.colsum, stream=stream,
                          n_groups=c.n_groups, topk_groups=c.topk_groups)
        B.moe_dispatch(self.ctx, self.idx, c.E, self.capacity, self.counts, self.offsets,
                       self.row_of_slot, self.slot_of_row, self.ws, X=X, Xperm=self.Xperm,
                       stream=stream)
        if stats:
            self._routed.record(stream)
            self._side.wait_event(self._routed)
            B.moe_balance_stats(self.ctx, self.T, c.k, self.counts, self.colsum, c.alpha,
                                self.f, self.p, self.stats, offsets=self.offsets,
                                stream=self._side)
            self._stats_done.record(self._side)
        self._experts(X, stream)
        B.moe_combine(self.ctx, self.O, self.row_of_slot, self.gate, Y,
                      O_shared=self.O_shared, Y_bf16=Y_bf16, stream=stream)
        if self.bias_gamma is not None:
            self.update_bias(self.bias_gamma, stream=stream)
        if stats:
            stream.wait_event(self._stats_done)   # the forward ends when both streams do
        return Y

    def _forward_expert_choice(self, X, Y, Y_bf16, stream) -> torch.Tensor:
        """Expert-choice routing: every expert takes its C = T*k/E best tokens; the expert
        stage is unchanged, the combine sums over the E (token, expert) slots."""
        c, w = self.cfg, self.w
        B.moe_expert_choice(self.ctx, X, w["Wg"], c.k, self.score, self.offsets,
                            self.row_of_slot, self.slot_of_row, self.gate, self.ws,
                            logit_bias=w.get("logit_bias"), col_gap=self.col_gap,
                            stream=stream)
        B.moe_gather_rows(self.ctx, self.slot_of_row, c.E, X, self.Xperm, self.ws,
                          stream=stream)
        self._experts(X, stream)
        B.moe_combine(self.ctx, self.O, self.row_of_slot, self.gate, Y,
                      O_shared=self.O_shared, Y_bf16=Y_bf16, stream=stream)
        return Y

    def _experts(self, X, stream) -> None:
        """Step 5: the grouped SwiGLU experts, from bf16/fp32 or FP8 weights."""
        c, w = self.cfg, self.w
        if self.fp8 is not None:
            B.moe_grouped_swiglu_fp8(self.ctx, X, self.Xperm, self.offsets, self.fp8, self.O,
                                     self.ws, c.k, O_shared=self.O_shared, stream=stream)
            return
        B.moe_grouped_swiglu(self.ctx, X, self.Xperm, self.offsets, w["W_gate"], w["W_up"],
                             w["W_down"], self.O, self.ws, c.k, Ws_gate=w.get("Ws_gate"),
                             Ws_up=w.get("Ws_up"), Ws_down=w.get("Ws_down"),
                             O_shared=self.O_shared, stream=stream)

    def update_bias(self, gamma: float, stream=None) -> None:
        """The balancing step after a forward: the selection bias moves by -gamma for
        every overloaded expert and +gamma for every underloaded one, from this forward's
        counts (in place on the layer's "bias" weight; enqueued on `stream`)."""
        stream = torch.cuda.current_stream(self.dev) if stream is None else stream
        B.moe_bias_update(self.ctx, self.T, self.cfg.k, self.counts, gamma, self.w["bias"],
                          stream=stream)

    def forward_host(self, X_host: torch.Tensor, Y_host: torch.Tensor,
                     X_dev: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """Host X (pinned) -> device, forward, device Y -> host Y (pinned), all three on
        `stream` (default: the current stream).  Returns once they are enqueued:
        synchronise the stream before reading Y_host."""
        s = torch.cuda.current_stream(self.dev) if stream is None else stream
        if X_dev is None:
            X_dev = torch.empty_like(X_host, device=self.dev)
        with torch.cuda.stream(s):
            X_dev.copy_(X_host, non_blocking=True)
            Y = self.forward(X_dev, stream=s)
            Y_host.copy_(Y, non_blocking=True)
        return Y_host

    def host_pipeline(self, X_host: torch.Tensor, Y_host: List[torch.Tensor], steps: int,
                      compute: torch.cuda.Stream) -> None:
        """`steps` end-to-end forwards from pinned host memory to pinned host memory, the
        copies overlapped with compute: step i's input copy (H2D stream) runs during
        step i-1's forward (compute stream), and step i's bf16 output copy (D2H stream)
        during step i+1's forward.  Device X and Y are double-buffered; events order the
        reuse of each buffer.  Y_host holds two pinned bf16 [T, H] buffers, used in turn."""
        dev = self.dev
        if not hasattr(self, "_pipe"):
            self._pipe = dict(
                h2d=torch.cuda.Stream(device=dev), d2h=torch.cuda.Stream(device=dev),
                X=[torch.empty_like(X_host, device=dev) for _ in range(2)],
                Y=[torch.empty(self.T, self.cfg.H, dtype=torch.float32, device=dev)
                   for _ in range(2)],
                Yb=[torch.empty(self.T, self.cfg.H, dtype=torch.bfloat16, device=dev)
                    for _ in range(2)])
        P = self._pipe
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [None, None]
        d2h_done = [None, None]
        for i in range(steps):
            b = i & 1
            with torch.cuda.stream(P["h2d"]):
                if comp_done[b] is not None:
                    P["h2d"].wait_event(comp_done[b])      # X[b] no longer read
                P["X"][b].copy_(X_host, non_blocking=True)
                h2d_done[b].record(P["h2d"])
            compute.wait_event(h2d_done[b])
            if d2h_done[b] is not None:
                compute.wait_event(d2h_done[b])             # Yb[b] already copied out
            self.forward(P["X"][b], stream=compute, Y=P["Y"][b], Y_bf16=P["Yb"][b])
            ev = torch.cuda.Event()
            ev.record(compute)
            comp_done[b] = ev
            with torch.cuda.stream(P["d2h"]):
                P["d2h"].wait_event(ev)
                Y_host[b].copy_(P["Yb"][b], non_blocking=True)
                ev2 = torch.cuda.Event()
                ev2.record(P["d2h"])
                d2h_done[b] = ev2
        for e in d2h_done:
            if e is not None:
                compute.wait_event(e)

    def capture(self, X: torch.Tensor, stats: bool = True,
                Y_bf16: Optional[torch.Tensor] = None) -> torch.cuda.CUDAGraph:
        """Record one forward of the device buffer X into a CUDA graph and return it;
        `graph.replay()` then reruns the whole forward on whatever X holds, with one
        launch from the host instead of one per kernel (small batches are host-bound).
        The forward allocates nothing and never synchronises, so it captures as is.  One
        eager forward first loads the module and fills the per-process caches; tracing
        must be off."""
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        self.forward(X, stats=stats, stream=s, Y_bf16=Y_bf16)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.forward(X, stats=stats, stream=s, Y_bf16=Y_bf16)
        return g

    def device_status(self) -> int:
        return B.moe_get_device_status(self.ctx, self.ws, reset=True)
