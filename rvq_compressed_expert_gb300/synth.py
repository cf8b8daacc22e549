"""Seeded synthetic inputs for the routed-expert RVQ MoE step.

This module only draws random numbers with the shapes, dtypes and
distributions of the workloads; it holds none of the method's arithmetic
(no routing, no decoding, no matrix products).  Both the CUDA path and the
CPU oracle consume what it returns, so parity tests compare the two on the
very same arrays.

Every array is drawn from its own ``torch.Generator`` whose seed is a
counter-style mix of (seed, layer, expert, purpose), so any single expert of
any layer can be regenerated on its own (the full-size parity tests use this
to hand the oracle only the experts a token selected).  A generator on
``cuda`` and one on ``cpu`` give different streams: a test uses one device
for all of its draws.

Workload shapes follow the pages' model (16 experts per token over 92 layers,
3-stage RVQ with 256-entry codebooks over 8-weight vectors; page "Exécuter
Kimi K3 avec 29 Go de RAM à 0,50 tok/s", sections "Quantification et
exactitude" and "Budget RAM et zone de performance étroite").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

N_STAGES = 3
CODEBOOK_SIZE = 256
VEC = 8

# purposes mixed into every generator seed
_P_ROUTER, _P_BIAS, _P_CODEBOOK, _P_GATE, _P_UP, _P_DOWN, _P_HIDDEN, _P_DENSE, _P_INIT = range(1, 10)
_MASK64 = (1 << 64) - 1


def _mix(*key: int) -> int:
    """Fold integers into one 63-bit seed (splitmix64 finaliser per step)."""
    z = 0x9E3779B97F4A7C15
    for k in key:
        z = (z + (int(k) & _MASK64) + 0x9E3779B97F4A7C15) & _MASK64
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        z ^= z >> 31
    return z & ((1 << 63) - 1)


def _gen(device, *key: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*key))
    return g


@dataclass(frozen=True)
class Workload:
    """One synthetic configuration of the routed-expert step."""
    name: str
    d: int                 # hidden size
    f: int                 # expert FFN width
    n_experts: int         # experts per layer (E)
    top_k: int             # experts per token (k)
    tokens: int            # tokens per step (T)
    act_dtype: str = "f32"  # "f32" or "bf16" hidden states
    bias: str = "none"     # "none" | "offsets" | "zipf"
    n_layers: int = 1
    lookahead: int = 0
    seeds: tuple = (0,)
    bias_spacing: float = 1.0
    zipf_s: float = 1.1
    note: str = field(default="", compare=False)


WORKLOADS = {
    # d=256, f=128, E=8, top-2, 4 tokens, fp32, seed 0
    "tiny": Workload("tiny", 256, 128, 8, 2, 4, "f32", "none", seeds=(0,)),
    # one decode layer with the pages' expert shape: d=7168, f=1536, E=384, top-16, one token
    "decode": Workload("decode", 7168, 1536, 384, 16, 1, "f32", "offsets",
                       seeds=tuple(range(10))),
    # 92 MoE layers x 64 resident experts, one token, residual h += combine, lookahead 6
    "stack": Workload("stack", 7168, 1536, 64, 16, 1, "f32", "offsets", n_layers=92,
                      lookahead=6, seeds=tuple(range(10))),
    # 16 MoE layers x 64 experts behind a tiered bank (records in host memory, an HBM cache),
    # one token, Zipf(1.1) expert popularity, lookahead 6
    "tiered": Workload("tiered", 7168, 1536, 64, 16, 1, "f32", "zipf", n_layers=16,
                       lookahead=6, seeds=tuple(range(10))),
    # batched decode: 128 tokens, bf16 h, Zipf(1.1) expert popularity via router bias
    "batched": Workload("batched", 7168, 1536, 384, 16, 128, "bf16", "zipf",
                        seeds=tuple(range(10))),
    # prefill chunk: 512 tokens, bf16 h, no bias
    "prefill": Workload("prefill", 7168, 1536, 384, 16, 512, "bf16", "none",
                        seeds=tuple(range(10))),
}


def router_weight(seed: int, layer: int, n_experts: int, d: int, device="cpu") -> torch.Tensor:
    """W_r [E, d] fp32 with entries ~ N(0, 1/d) (variance 1/d)."""
    g = _gen(device, seed, layer, 0, _P_ROUTER)
    return torch.randn(n_experts, d, generator=g, device=device, dtype=torch.float32) / math.sqrt(d)


def router_bias(seed: int, layer: int, n_experts: int, kind: str, device="cpu",
                spacing: float = 1.0, zipf_s: float = 1.1) -> torch.Tensor | None:
    """Router bias [E] fp32, or None.

    ``offsets``: a seeded permutation of 0..E-1 times ``spacing`` -- distinct
    offsets that keep the top-k logits apart.
    ``zipf``: b_e = -s * ln(rank_e) over a seeded rank permutation (rank 1 is
    the most popular expert), which makes selection frequency fall off
    roughly like a Zipf(s) law.
    """
    if kind == "none":
        return None
    g = _gen("cpu", seed, layer, 0, _P_BIAS)
    perm = torch.randperm(n_experts, generator=g)
    if kind == "offsets":
        b = perm.to(torch.float32) * float(spacing)
    elif kind == "zipf":
        rank = perm.to(torch.float64) + 1.0
        b = (-float(zipf_s) * torch.log(rank)).to(torch.float32)
    else:
        raise ValueError(f"unknown bias kind {kind!r}")
    return b.to(device)


def codebooks(seed: int, layer: int, n_experts: int, device="cpu") -> torch.Tensor:
    """Codebooks [E, 3 matrices (gate, up, down), 3 stages, 256, 8] fp32.

    Stage s entries ~ N(0, std = 0.02 * 0.5**s).
    """
    g = _gen(device, seed, layer, 0, _P_CODEBOOK)
    cb = torch.randn(n_experts, 3, N_STAGES, CODEBOOK_SIZE, VEC, generator=g,
                     device=device, dtype=torch.float32)
    std = torch.tensor([0.02 * 0.5 ** s for s in range(N_STAGES)], dtype=torch.float32,
                       device=device).view(1, 1, N_STAGES, 1, 1)
    return cb * std


def expert_codes(seed: int, layer: int, expert: int, d: int, f: int, device="cpu"):
    """Codes of one expert in the logical layout, uint8 uniform on 0..255.

    Returns (gate [f, 3, d/8], up [f, 3, d/8], down [d, 3, f/8]):
    [output row][stage][vector along the input dimension].
    """
    out = []
    for purpose, (rows, n_in) in ((_P_GATE, (f, d)), (_P_UP, (f, d)), (_P_DOWN, (d, f))):
        g = _gen(device, seed, layer, expert, purpose)
        out.append(torch.randint(0, 256, (rows, N_STAGES, n_in // VEC), generator=g,
                                 device=device, dtype=torch.uint8))
    return tuple(out)


def layer_codes(seed: int, layer: int, n_experts: int, d: int, f: int, device="cpu"):
    """Codes of all experts of a layer: (gate [E,f,3,d/8], up [E,f,3,d/8], down [E,d,3,f/8])."""
    parts = [expert_codes(seed, layer, e, d, f, device) for e in range(n_experts)]
    return tuple(torch.stack([p[i] for p in parts]) for i in range(3))


def hidden(seed: int, tokens: int, d: int, act_dtype: str = "f32", device="cpu",
           stream: int = 0) -> torch.Tensor:
    """Hidden states h [T, d] ~ N(0, 1); fp32 or rounded to bf16."""
    g = _gen(device, seed, stream, 0, _P_HIDDEN)
    h = torch.randn(tokens, d, generator=g, device=device, dtype=torch.float32)
    if act_dtype == "bf16":
        return h.to(torch.bfloat16)
    if act_dtype != "f32":
        raise ValueError(act_dtype)
    return h


@dataclass
class LayerInputs:
    router_w: torch.Tensor
    router_b: torch.Tensor | None
    codebooks: torch.Tensor
    codes: tuple | None   # (gate, up, down) logical codes for all experts, or None


def layer_inputs(w: Workload, seed: int, layer: int = 0, device="cpu",
                 with_codes: bool = True) -> LayerInputs:
    """Router, bias, codebooks and (optionally) codes of one layer of a workload."""
    return LayerInputs(
        router_weight(seed, layer, w.n_experts, w.d, device),
        router_bias(seed, layer, w.n_experts, w.bias, device, w.bias_spacing, w.zipf_s),
        codebooks(seed, layer, w.n_experts, device),
        layer_codes(seed, layer, w.n_experts, w.d, w.f, device) if with_codes else None,
    )


def dense_matrix(seed: int, layer: int, expert: int, which: int, rows: int, cols: int, device="cpu",
                 std: float = 0.02) -> torch.Tensor:
    """A dense expert matrix [rows, cols] fp32 ~ N(0, std) (which: 0 gate, 1 up, 2 down), the
    input of the RVQ encoder."""
    g = _gen(device, seed, layer, expert, _P_DENSE, which)
    return torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * std


def rvq_init(seed: int, n_vectors: int, device="cpu") -> torch.Tensor:
    """[3, 256] int32 vector indices, uniform over [0, n_vectors): where each stage's centroids
    start (the encoder's only random draw)."""
    g = _gen("cpu", seed, n_vectors, 0, _P_INIT)
    return torch.randint(0, n_vectors, (3, CODEBOOK_SIZE), generator=g, dtype=torch.int32).to(device)
