"""Batched calls through the grouped tensor-core path, against the CPU oracle, through the C ABI.

Experts chosen by enough tokens of a call are applied on the tensor cores from fp16 weights
decoded out of their codes and fp16 activations, with fp32 accumulation; the others take the
fp32 lookup path.  The bar for this path is the one for bf16-activation variants: relative
L2 <= 2e-3 per token, plus a per-element bound of 4e-3 * max|y| (fp16 operands carry a
relative error of at most 2^-11 each; summed over thousands of products of random sign it
stays near 1e-3 of the output's scale).  Indices stay bit-exact: routing does not touch
this path.
"""
import numpy as np
import pytest
import torch

import oracle
from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth
from rvq_compressed_expert_gb300.layer import MoELayer

pytestmark = pytest.mark.gpu

REL_L2 = 2e-3
ELEM = 4e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rvq_compressed_expert_gb300 import _build
    _build.build()
    B.load()
    oracle.build()


def check_tokens(g_out, ref_out, tokens):
    for t in tokens:
        g = np.asarray(g_out[t], np.float64)
        r = np.asarray(ref_out[t], np.float64)
        rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
        assert rel <= REL_L2, f"token {t}: relative L2 {rel:.3e}"
        m = np.abs(g - r).max()
        assert m <= ELEM * np.abs(r).max(), f"token {t}: max |err| {m:.3e}"


def run_small(d, f, E, k, T, act, flags, bias="none", seed=0):
    w = synth.Workload("g", d, f, E, k, T, act, bias)
    li = synth.layer_inputs(w, seed, 0, "cpu", with_codes=True)
    h = synth.hidden(seed, T, d, act, "cpu")
    layer = MoELayer(w, seed, 0, "cuda", inputs=li, flags=flags)
    try:
        idx, gate, logits, out = layer.alloc_outputs(T)
        hd = h.cuda()
        layer.route(hd, T, idx, gate, logits)
        layer.forward(hd, T, idx, gate, out, 0)
        torch.cuda.synchronize()
        st = layer.stats()  # raises on a device-side error (bad index, timeout)
        ref = oracle.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, k)
        g_idx = idx.cpu().numpy()
        ok = [t for t in range(T) if oracle.topk_margin(ref["logits"][t], k) > 1e-4]
        assert ok, "no well-separated token"
        for t in ok:
            np.testing.assert_array_equal(g_idx[t], oracle.topk_softmax(ref["logits"][t], k)[0])
        check_tokens(out.cpu().numpy(), ref["out"], ok)
        return g_idx, out.cpu().numpy(), st
    finally:
        layer.close()


@pytest.mark.parametrize("act", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [
    (256, 128, 8, 2, 4),     # the tiny workload, every expert on the tensor cores
    (1032, 136, 12, 3, 5),   # ragged: K tail inside a chunk, 136 rows (M tail), 17 down vectors
    (512, 264, 20, 5, 3),    # 3 gate/up row blocks, 4 down row blocks, K tail on down
    (8, 8, 2, 1, 2),         # one vector per row, one K chunk, 8 of 128 rows
])
def test_forced_tensor_core_path_matches_oracle(shape, act):
    d, f, E, k, T = shape
    _, _, st = run_small(d, f, E, k, T, act, B.FLAG_FORCE_MMA)
    assert st["forward_slots"] == T * k


@pytest.mark.parametrize("shape,npads", [
    ((64, 64, 2, 1, 48), {32}),         # one K chunk: each issuer takes 16 of the 32 token columns
    ((64, 64, 2, 1, 80), {48}),         # one K chunk, 48 columns: 32 + 16
    ((128, 128, 4, 2, 60), {32}),       # two K chunks: each issuer one chunk per pass
    ((256, 136, 2, 1, 128), {64, 80}),  # 64 tokens: alternate K chunks; 80: 48 + 32 token columns;
                                        # down has 3 K chunks (the last one ragged)
])
def test_two_issuer_splits(shape, npads):
    """The MMAs of a chunk shared by two issuing threads: by alternate K chunks into two
    accumulators (<= 64 tokens, >= 2 K chunks) or by halves of the tokens."""
    d, f, E, k, T = shape
    g_idx, _, st = run_small(d, f, E, k, T, "bf16", B.FLAG_FORCE_MMA)
    counts = np.bincount(g_idx.ravel(), minlength=E)
    assert {(int(c) + 15) // 16 * 16 for c in counts if c > 0} == npads, counts
    assert st["forward_slots"] == T * k


def test_batched_bf16_mixed_paths():
    """bf16, 48 tokens, Zipf router bias: popular experts on the tensor cores, rare ones on
    the lookup path, combined per token in rank order."""
    d, f, E, k, T = 512, 256, 32, 4, 48
    g_idx, _, st = run_small(d, f, E, k, T, "bf16", 0, bias="zipf")
    counts = np.bincount(g_idx.ravel(), minlength=E)
    assert (counts >= 4).any() and ((counts > 0) & (counts < 4)).any(), counts
    # demand bytes: one read of the codes per tensor-core expert, one per lookup slot
    per_expert = oracle.expert_code_bytes(d, f)
    n_tc = int((counts >= 4).sum())
    n_lut = int(counts[counts < 4].sum())
    assert st["demand_code_bytes"] == (n_tc + n_lut) * per_expert


def test_more_tokens_than_one_chunk():
    """An expert chosen by more than 128 tokens is split into several token chunks."""
    d, f, E, k, T = 256, 128, 4, 2, 300
    g_idx, _, _ = run_small(d, f, E, k, T, "bf16", 0)
    assert np.bincount(g_idx.ravel(), minlength=E).max() > 128


def test_grouped_deterministic_and_gemv_flag():
    """Two runs are bit-identical; FORCE_GEMV keeps the batched bf16 call on the fp32 lookup
    path (then the fp32 bar holds)."""
    d, f, E, k, T = 512, 256, 16, 4, 32
    w = synth.Workload("g", d, f, E, k, T, "bf16", "none")
    li = synth.layer_inputs(w, 1, 0, "cpu", with_codes=True)
    h = synth.hidden(1, T, d, "bf16", "cuda")
    outs = {}
    for name, flags in (("tc", 0), ("gemv", B.FLAG_FORCE_GEMV)):
        layer = MoELayer(w, 1, 0, "cuda", inputs=li, flags=flags)
        try:
            idx, gate, logits, out = layer.alloc_outputs(T)
            layer.route(h, T, idx, gate, logits)
            res = []
            for _ in range(2):
                out.fill_(float("nan"))
                layer.forward(h, T, idx, gate, out, 0)
                torch.cuda.synchronize()
                res.append(out.clone())
            assert torch.equal(res[0], res[1]), name
            outs[name] = res[0].cpu().numpy()
        finally:
            layer.close()
    ref = oracle.moe_layer(h.cpu(), li.router_w, li.router_b, li.codebooks, li.codes, k)
    ok = [t for t in range(T) if oracle.topk_margin(ref["logits"][t], k) > 1e-4]
    check_tokens(outs["tc"], ref["out"], ok)
    for t in ok:
        g = outs["gemv"][t].astype(np.float64)
        r = ref["out"][t]
        assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 1e-5


def test_residual_mode_grouped():
    d, f, E, k, T = 512, 256, 8, 2, 16
    w = synth.Workload("g", d, f, E, k, T, "bf16", "none")
    li = synth.layer_inputs(w, 2, 0, "cpu", with_codes=True)
    h = synth.hidden(2, T, d, "bf16", "cuda")
    layer = MoELayer(w, 2, 0, "cuda", inputs=li)
    try:
        idx, gate, logits, out = layer.alloc_outputs(T)
        layer.route(h, T, idx, gate, logits)
        layer.forward(h, T, idx, gate, out, 0)
        base = torch.randn(T, d, generator=torch.Generator().manual_seed(5)).cuda()
        acc = base.clone()
        layer.forward(h, T, idx, gate, acc, 1)
        torch.cuda.synchronize()
        assert torch.equal(acc, base + out)
    finally:
        layer.close()


# ---------------------------------------------------------------- full batched shapes

def full_size(name, seed, n_check):
    w = synth.WORKLOADS[name]
    layer = MoELayer(w, seed, 0, "cuda")
    try:
        T = w.tokens
        h = synth.hidden(seed, T, w.d, w.act_dtype, "cuda")
        idx, gate, logits, out = layer.alloc_outputs(T)
        layer.route(h, T, idx, gate, logits)
        layer.forward(h, T, idx, gate, out, 0)
        torch.cuda.synchronize()
        layer.stats()
        g_idx = idx.cpu().numpy()
        counts = np.bincount(g_idx.ravel(), minlength=w.n_experts)
        # sampled tokens, spread over the batch; the oracle recomputes each from the router
        # and its 16 experts' codes
        rng = np.random.default_rng(seed)
        cand = rng.permutation(T)
        hc = h.cpu()
        g_out = out.cpu().numpy()
        checked = 0
        worst = 0.0
        for t in cand:
            ref = oracle.moe_token(hc[t], layer.router_w.cpu(),
                                   None if layer.router_b is None else layer.router_b.cpu(),
                                   layer.codebooks.cpu().numpy(),
                                   lambda e: layer.expert_codes_host(e), w.top_k)
            if oracle.topk_margin(ref["logits"], w.top_k) <= 1e-3:
                continue
            np.testing.assert_array_equal(g_idx[t], ref["idx"])
            check_tokens({t: g_out[t]}, {t: ref["out"]}, [t])
            r = ref["out"]
            worst = max(worst, float(np.linalg.norm(g_out[t].astype(np.float64) - r) / np.linalg.norm(r)))
            checked += 1
            if checked == n_check:
                break
        assert checked == n_check
        print(f"{name}: worst relative L2 over {n_check} sampled tokens {worst:.3e} (bar {REL_L2:.0e})")
        return counts
    finally:
        layer.close()


def test_batched_decode_full_size():
    """128 tokens, bf16, Zipf popularity, d=7168 f=1536 E=384 top-16 (sampled tokens)."""
    counts = full_size("batched", 0, 3)
    assert (counts >= 4).sum() > 0 and ((counts > 0) & (counts < 4)).sum() > 0


def test_prefill_full_size():
    """512 tokens, bf16, no bias, d=7168 f=1536 E=384 top-16 (32 sampled tokens, every one
    within the bf16 bar; the worst relative L2 is printed)."""
    counts = full_size("prefill", 0, 32)
    assert counts.sum() == 512 * 16
