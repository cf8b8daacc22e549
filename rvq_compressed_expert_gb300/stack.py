"""Decode through a stack of MoE layers with the pages' router lookahead.

Per layer L, for one batch of tokens with residual h_L (page "Exécuter Kimi K3
avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée et prédiction du
routeur"):
  - x_L = rmsnorm(h_L)  (stand-in for the trunk's normalisation of the MoE
    input; without it the chain h <- h + MoE(h) diverges at these scales),
  - on the main stream layer L routes x_L (waste_moe_route),
  - on a side stream, once that route is done, layer L+1's router runs on x_L and
    its top-P experts are prefetched into L2 (waste_moe_prefetch),
  - on the main stream layer L applies its experts:
    h_{L+1} = h_L + combine (waste_moe_forward, mode 1, in place).
For one token the lookahead instead runs inside each layer's step, with no side
stream (waste_moe_set_lookahead).  The real router of each layer decides its
experts, so the lookahead changes neither the outputs nor the demand bytes.  The side stream starts behind layer
L's route, not beside it: the expert kernel is one cooperative launch that
needs every SM at once, and side-stream kernels still running when it is due
would hold it back; behind the route they fill the SMs that the expert kernel's
tail and the combine leave free.  x alternates between two buffers so the side
stream can still read x_L while x_{L+1} is written; layer L+1 routes only after
its prefetch has finished (an event), which also keeps the next write of x_L's
buffer behind the read.
"""
from __future__ import annotations

import torch

from . import binding as B


class DecodeStack:
    def __init__(self, layers, tokens: int, device="cuda", banked: bool = False):
        """banked: the layers' records live in a tiered bank (TieredStack); each layer's
        forward is then issued before the lookahead into the next layer, whose copies into
        the HBM cache run beside the forward's expert kernels."""
        self.banked = banked
        self.layers = layers
        self.T = tokens
        w = layers[0].w
        self.d = w.d
        self.h = torch.empty(tokens, w.d, dtype=torch.float32, device=device)
        self.x = [torch.empty(tokens, w.d, dtype=torch.float32, device=device) for _ in range(2)]
        self.idx = torch.empty(tokens, w.top_k, dtype=torch.int32, device=device)
        self.gate = torch.empty(tokens, w.top_k, dtype=torch.float32, device=device)

    def run(self, h0: torch.Tensor, lookahead: int, main: torch.cuda.Stream,
            side: torch.cuda.Stream | None = None, on_layer=None) -> torch.Tensor:
        """Enqueue one pass of h0 [T, d] fp32 through every layer on `main` (and `side` for
        the lookahead); returns the buffer that holds the output once `main` is done."""
        n = len(self.layers)
        T = self.T
        with torch.cuda.stream(main):
            self.h.copy_(h0)
        pending = None
        if self.banked:
            return self._run_banked(lookahead, main, side, on_layer)
        if T == 1:
            return self._run_one_token(lookahead, main, on_layer)
        for L in range(n):
            x = self.x[L & 1]
            B.waste_moe_rmsnorm(self.h, x, T, self.d, main)
            if pending is not None:
                main.wait_event(pending)  # layer L's prediction is in place before it routes
            self.layers[L].route(x, T, self.idx, self.gate, stream=main)
            ev = None
            if lookahead and L + 1 < n:
                side.wait_stream(main)  # x_L is ready and layer L has routed
                self.layers[L + 1].prefetch(x, T, lookahead, stream=side)
                ev = torch.cuda.Event()
                ev.record(side)
            # experts + combine (h += combine)
            self.layers[L].forward(x, T, self.idx, self.gate, self.h, 1, stream=main)
            if on_layer is not None:
                on_layer(L, self.idx, self.gate, main)
            pending = ev
        if pending is not None:
            main.wait_event(pending)
        return self.h

    def _run_one_token(self, lookahead, main, on_layer):
        """One token: the lookahead runs inside each layer's step (waste_moe_set_lookahead): layer
        L's router launch also runs layer L+1's router rows on x_L, and layer L's expert kernel
        predicts L+1's top-P experts and asks L2 for them with the SMs it leaves idle at its end.
        No side stream."""
        n = len(self.layers)
        for L in range(n):
            nxt = self.layers[L + 1].handle if lookahead and L + 1 < n else None
            B.waste_moe_set_lookahead(self.layers[L].handle, nxt, lookahead if nxt is not None else 0)
        for L in range(n):
            x = self.x[L & 1]
            B.waste_moe_rmsnorm(self.h, x, 1, self.d, main)
            self.layers[L].step(x, 1, self.idx, self.gate, self.h, 1, stream=main)
            if on_layer is not None:
                on_layer(L, self.idx, self.gate, main)
        return self.h

    def _run_banked(self, lookahead, main, side, on_layer):
        n = len(self.layers)
        T = self.T
        pending = None
        for L in range(n):
            x = self.x[L & 1]
            B.waste_moe_rmsnorm(self.h, x, T, self.d, main)
            x_ready = torch.cuda.Event()
            x_ready.record(main)
            if pending is not None:
                main.wait_event(pending)  # layer L's prediction is in place before it routes
            self.layers[L].step(x, T, self.idx, self.gate, self.h, 1, stream=main)
            if on_layer is not None:
                on_layer(L, self.idx, self.gate, main)
            pending = None
            if lookahead and L + 1 < n:
                side.wait_event(x_ready)
                self.layers[L + 1].prefetch(x, T, lookahead, stream=side)
                pending = torch.cuda.Event()
                pending.record(side)
        if pending is not None:
            main.wait_event(pending)
        return self.h
