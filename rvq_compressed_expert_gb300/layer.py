"""One MoE layer held on the GPU: weights, record bank and library handle.

Convenience wrapper over the C ABI for tests and the benchmark: it draws a
layer's synthetic weights (``synth``) on the device, writes the record bank
with ``waste_moe_pack_records`` and creates the handle.  All computation is
in the library's kernels.
"""
from __future__ import annotations

import torch

from . import binding as B
from . import synth


class MoELayer:
    def __init__(self, w: synth.Workload, seed: int, layer: int = 0, device="cuda",
                 max_tokens: int | None = None, flags: int = 0, lookahead: int | None = None,
                 keep_codes: bool = False, pack_batch: int = 32, inputs: synth.LayerInputs | None = None,
                 gen_device: str | None = None, crc: bool = False):
        self.w = w
        self.seed = seed
        self.layer = layer
        self.device = device
        gen_device = gen_device or device
        T = max_tokens if max_tokens is not None else w.tokens
        self.cfg = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, T,
                                 w.lookahead if lookahead is None else lookahead, flags, layer)
        self.stride, self.sec_off, self.sec_bytes = B.waste_moe_record_layout(self.cfg)
        li = inputs or synth.layer_inputs(w, seed, layer, gen_device, with_codes=False)
        self.router_w = li.router_w.to(device).contiguous()
        self.router_b = None if li.router_b is None else li.router_b.to(device).contiguous()
        self.codebooks = li.codebooks.to(device).contiguous()
        self.records = B.aligned_bytes(w.n_experts * self.stride, device)
        self.codes = None
        if inputs is not None and inputs.codes is not None:
            self.codes = tuple(c.to(device).contiguous() for c in inputs.codes)
            B.waste_moe_pack_records(self.cfg, layer, 0, w.n_experts, *self.codes, self.records,
                                     self.stride, int(crc))
            if not keep_codes:
                self.codes = None
        else:
            kept = [] if keep_codes else None
            for e0 in range(0, w.n_experts, pack_batch):
                n = min(pack_batch, w.n_experts - e0)
                parts = [synth.expert_codes(seed, layer, e, w.d, w.f, gen_device)
                         for e in range(e0, e0 + n)]
                gc, uc, dc = (torch.stack([p[i] for p in parts]).to(device).contiguous()
                              for i in range(3))
                B.waste_moe_pack_records(self.cfg, layer, e0, n, gc, uc, dc, self.records,
                                         self.stride, int(crc))
                if kept is not None:
                    kept.append((gc, uc, dc))
                else:
                    torch.cuda.current_stream().synchronize()
                    del gc, uc, dc
            if kept is not None:
                self.codes = tuple(torch.cat([k[i] for k in kept]) for i in range(3))
        self.handle = B.waste_moe_create(self.cfg, self.router_w, self.router_b, self.records,
                                         self.stride, self.codebooks)

    # ---- per-call wrappers
    def route(self, h, T, idx, gate, logits=None, stream=None):
        B.waste_moe_route(self.handle, h, T, idx, gate, logits, stream)

    def forward(self, h, T, idx, gate, out, mode=0, stream=None):
        B.waste_moe_forward(self.handle, h, T, idx, gate, out, mode, stream)

    def step(self, h, T, idx, gate, out, mode=0, logits=None, stream=None):
        B.waste_moe_step(self.handle, h, T, idx, gate, logits, out, mode, stream)

    def prefetch(self, h, T, n=-1, stream=None):
        B.waste_moe_prefetch(self.handle, h, T, n, stream)

    def stats(self):
        return B.waste_moe_stats(self.handle)

    def reset_stats(self):
        B.waste_moe_reset_stats(self.handle)

    def expert_codes_host(self, e: int, gen_device: str | None = None):
        """Logical codes of expert e, regenerated from the seed (for the oracle)."""
        if self.codes is not None:
            return tuple(c[e].cpu() for c in self.codes)
        return tuple(c.cpu() for c in synth.expert_codes(self.seed, self.layer, e, self.w.d,
                                                         self.w.f, gen_device or self.device))

    def close(self):
        if self.handle:
            B.waste_moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc_outputs(self, T: int):
        dev = self.device
        return (torch.empty(T, self.w.top_k, dtype=torch.int32, device=dev),
                torch.empty(T, self.w.top_k, dtype=torch.float32, device=dev),
                torch.empty(T, self.w.n_experts, dtype=torch.float32, device=dev),
                torch.empty(T, self.w.d, dtype=torch.float32, device=dev))
