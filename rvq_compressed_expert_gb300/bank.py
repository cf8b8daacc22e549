"""A tiered expert bank: the records of several layers in pinned host memory, read by the GPU,
with an HBM cache of a fixed number of records (waste_bank_create / waste_moe_create_banked).

Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", sections "Budget RAM et zone de
performance étroite" and "Lecture anticipée et prédiction du routeur": experts live in a
large slow tier, a bounded cache holds some, misses read the record from the slow tier, and
the next layer's router fills the cache ahead of demand.
"""
from __future__ import annotations

import torch

from . import binding as B
from . import synth
from .layer import MoELayer


class TieredStack:
    """n_layers layers of workload w whose records sit in one pinned host buffer behind one
    HBM cache of n_slots records.  `layers` are MoELayer objects holding banked handles, so
    DecodeStack runs them as it runs resident layers (banked=True)."""

    def __init__(self, w: synth.Workload, seed: int, n_layers: int, n_slots: int, device="cuda",
                 max_tokens: int | None = None, flags: int = 0, lookahead: int | None = None,
                 crc: bool = False):
        self.w = w
        T = max_tokens if max_tokens is not None else w.tokens
        cfg0 = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, T,
                             w.lookahead if lookahead is None else lookahead, flags, -1)
        self.stride, _, _ = B.waste_moe_record_layout(cfg0)
        per_layer = w.n_experts * self.stride
        self.host = B.pinned_bytes(n_layers * per_layer)
        self.layers = []
        for L in range(n_layers):
            ml = MoELayer(w, seed, L, device, max_tokens=T, flags=flags, lookahead=lookahead, crc=crc)
            self.host[L * per_layer:(L + 1) * per_layer].copy_(ml.records)
            torch.cuda.synchronize()
            B.waste_moe_destroy(ml.handle)
            ml.handle = None
            ml.records = None
            self.layers.append(ml)
        torch.cuda.empty_cache()
        self.cfg0 = cfg0
        self.bank = None
        self.rebank(n_slots)

    def rebank(self, n_slots: int, flags: int | None = None):
        """Replace the HBM cache by an empty one of n_slots records (same host records); with
        flags, the layer handles are made again with those configuration flags."""
        for ml in self.layers:
            if ml.handle:
                B.waste_moe_destroy(ml.handle)
                ml.handle = None
            if flags is not None:
                ml.cfg.flags = flags
        if self.bank:
            B.waste_bank_destroy(self.bank)
            self.bank = None
        self.n_slots = n_slots
        self.bank = B.waste_bank_create(self.cfg0, len(self.layers), self.host, self.stride, n_slots)
        for L, ml in enumerate(self.layers):
            ml.handle = B.waste_moe_create_banked(ml.cfg, ml.router_w, ml.router_b, self.bank, L,
                                                  ml.codebooks)

    def stats(self) -> dict:
        return B.waste_bank_stats(self.bank)

    def reset(self):
        B.waste_bank_reset(self.bank)

    def close(self):
        for ml in self.layers:
            ml.close()
        self.layers = []
        if self.bank:
            B.waste_bank_destroy(self.bank)
            self.bank = None
