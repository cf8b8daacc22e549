"""Routing trace of a decode run: which experts every layer picked for every token, with their
gates, written as JSON lines for offline study of expert popularity and reuse.

Recording is a copy of each layer's top-k on the stream that produced it (no host sync while
the stack runs); ``write`` waits for the device once and writes one line per (token, layer):
{"token": t, "layer": L, "experts": [...], "gates": [...]} (one list per token of the batch).
Hook it into ``DecodeStack.run(..., on_layer=trace.on_layer)`` and call ``next_token()``
between runs.
"""
from __future__ import annotations

import json

import torch


class RouteTrace:
    def __init__(self):
        self.token = 0
        self._rows = []  # (token, layer, idx copy, gate copy)

    def on_layer(self, layer: int, idx: torch.Tensor, gate: torch.Tensor, stream: torch.cuda.Stream):
        with torch.cuda.stream(stream):
            self._rows.append((self.token, layer, idx.clone(), gate.clone()))

    def next_token(self):
        self.token += 1

    def rows(self):
        """The trace as dictionaries (waits for the device)."""
        torch.cuda.synchronize()
        return [{"token": t, "layer": L, "experts": i.cpu().tolist(), "gates": g.cpu().tolist()}
                for t, L, i, g in self._rows]

    def write(self, path: str) -> int:
        rows = self.rows()
        with open(path, "w") as fh:
            for r in rows:
                fh.write(json.dumps(r) + "\n")
        return len(rows)
