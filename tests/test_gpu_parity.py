"""GPU path against the CPU oracle, element by element, through the C ABI.

Bar: expert indices bit-exact wherever the oracle's logits are separated by
more than the routing margin; fp32 outputs within relative L2 1e-5 and
per-element |err| <= 1e-4 * max|y| (bf16-activation variants: relative L2
2e-3 -- the activations are the same bf16 values on both sides, so the fp32
bound applies there too and is what is asserted).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth
from rvq_compressed_expert_gb300.layer import MoELayer
from tests import oracle_pins

pytestmark = pytest.mark.gpu

REL_L2 = 1e-5
ELEM = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rvq_compressed_expert_gb300 import _build
    _build.build()
    B.load()
    oracle.build()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_close(gpu, ref, rel=REL_L2, elem=ELEM):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    r = rel_l2(gpu, ref)
    assert r <= rel, f"relative L2 {r:.3e} > {rel:.1e}"
    m = float(np.abs(gpu - ref).max())
    assert m <= elem * float(np.abs(ref).max()) + 1e-30, f"max |err| {m:.3e}"


def margin_tau(logits):
    return 1e-4 * max(1.0, float(np.abs(logits).max()))


def check_routing(g_idx, g_gate, ref_logits, k):
    """Per token: bit-exact idx where the oracle's top-(k+1) margin exceeds tau, else the GPU's
    choice must be a valid top-k within tau.  Returns the tokens that are well separated."""
    ok_tokens = []
    for t in range(ref_logits.shape[0]):
        l = ref_logits[t]
        tau = margin_tau(l)
        ridx, rg = oracle.topk_softmax(l, k)
        if oracle.topk_margin(l, k) > tau:
            np.testing.assert_array_equal(g_idx[t], ridx, err_msg=f"token {t}")
            # the gates are an fp32 output of the path: held to the fp32 bar (relative 1e-5)
            np.testing.assert_allclose(g_gate[t], rg, rtol=1e-5, atol=1e-7)
            ok_tokens.append(t)
        else:
            kth = np.sort(l)[::-1][k - 1]
            assert all(l[e] >= kth - tau for e in g_idx[t])
            assert len(set(g_idx[t].tolist())) == k
    return ok_tokens


def run(layer, h, T, mode=0, out=None):
    idx, gate, logits, out0 = layer.alloc_outputs(T)
    out = out0 if out is None else out
    layer.route(h, T, idx, gate, logits)
    layer.forward(h, T, idx, gate, out, mode)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), gate.cpu().numpy(), logits.cpu().numpy(), out.cpu().numpy()


def small_layer(d, f, E, k, T, act="f32", seed=0, flags=0, bias="none"):
    w = synth.Workload("t", d, f, E, k, T, act, bias)
    li = synth.layer_inputs(w, seed, 0, "cpu", with_codes=True)
    h = synth.hidden(seed, T, d, act, "cpu")
    layer = MoELayer(w, seed, 0, "cuda", inputs=li, flags=flags)
    return w, li, h, layer


# ---------------------------------------------------------------- small shapes

@pytest.mark.parametrize("flags", [0, B.FLAG_K2_RECONSTRUCT], ids=["lut", "reconstruct"])
@pytest.mark.parametrize("act", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [
    (256, 128, 8, 2, 4),     # the tiny workload
    (1032, 136, 12, 3, 5),   # ragged: 129 input vectors (5 segments), 17 down vectors, 136 rows
    (512, 264, 20, 5, 3),    # several segments and row groups, odd down segment count
    (8, 8, 2, 1, 2),         # one vector per row
    (64, 16, 4, 4, 1),       # k = E
])
def test_layer_matches_oracle(shape, act, flags):
    d, f, E, k, T = shape
    # the lookup paths alone (batched bf16 calls would send popular experts to the
    # tensor cores, which tests/test_gpu_grouped.py covers at their own bar)
    w, li, h, layer = small_layer(d, f, E, k, T, act, flags=flags | B.FLAG_FORCE_GEMV)
    try:
        g_idx, g_gate, g_logits, g_out = run(layer, h.cuda(), T)
        ref = oracle.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, k)
        np.testing.assert_allclose(g_logits, ref["logits"], rtol=1e-5, atol=1e-5)
        ok = check_routing(g_idx, g_gate, ref["logits"], k)
        assert ok, "no well-separated token"
        assert_close(g_out[ok], ref["out"][ok])
    finally:
        layer.close()


def test_tiny_workload_exact_routing():
    w = synth.WORKLOADS["tiny"]
    li = synth.layer_inputs(w, 0, 0, "cpu", with_codes=True)
    h = synth.hidden(0, w.tokens, w.d, w.act_dtype, "cpu")
    layer = MoELayer(w, 0, 0, "cuda", inputs=li)
    try:
        g_idx, g_gate, _, g_out = run(layer, h.cuda(), w.tokens)
        ref = oracle.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, w.top_k)
        for t in range(w.tokens):
            assert oracle.topk_margin(ref["logits"][t], w.top_k) > 1e-3
        np.testing.assert_array_equal(g_idx, ref["idx"])
        np.testing.assert_allclose(g_gate.sum(1), 1.0, rtol=0, atol=4 * w.top_k * 2 ** -24)
        assert_close(g_out, ref["out"])
    finally:
        layer.close()


def test_hand_example_on_gpu():
    ex = oracle_pins.load_hand_example()
    for k in (2, 1):
        w = synth.Workload("hand", 8, 8, 2, k, 1)
        li = synth.LayerInputs(torch.tensor(ex["Wr"]), None, torch.tensor(ex["cbs"]),
                               tuple(torch.tensor(c) for c in ex["codes"]))
        layer = MoELayer(w, 0, 0, "cuda", inputs=li)
        try:
            h = torch.tensor(ex["h"], dtype=torch.float32)[None].cuda()
            g_idx, g_gate, g_logits, g_out = run(layer, h, 1)
            np.testing.assert_array_equal(g_logits[0], ex["expect"]["logits"])
            np.testing.assert_array_equal(g_idx[0], ex["expect"][f"idx_k{k}"].astype(np.int32))
            np.testing.assert_array_equal(g_gate[0], ex["expect"][f"gate_k{k}"])
            np.testing.assert_allclose(g_out[0], ex["expect"][f"out_k{k}"], rtol=2e-7, atol=1e-6)
        finally:
            layer.close()


@pytest.mark.parametrize("mode", [1, 2])
def test_residual_modes(mode):
    d, f, E, k, T = 256, 128, 8, 2, 4
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        base = torch.randn(T, d, generator=torch.Generator().manual_seed(5))
        out = (base if mode == 1 else torch.zeros(T, d)).cuda().contiguous()
        _, _, _, g_out = run(layer, h.cuda(), T, mode=mode, out=out)
        ref = oracle.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, k)
        expect = ref["out"] + (base.double().numpy() if mode == 1 else h.double().numpy())
        assert_close(g_out, expect)
    finally:
        layer.close()


def test_mode2_in_place():
    """out may alias h in mode 2 (residual update in place)."""
    d, f, E, k, T = 256, 128, 8, 2, 4
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        hd = h.cuda().contiguous()
        idx, gate, logits, _ = layer.alloc_outputs(T)
        layer.route(hd, T, idx, gate, logits)
        layer.forward(hd, T, idx, gate, hd, 2)
        torch.cuda.synchronize()
        ref = oracle.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, k, residual=True)
        assert_close(hd.cpu().numpy(), ref["out"])
    finally:
        layer.close()


def test_topk_ties_and_signed_zero():
    cases = [
        np.array([[1, 1, 1, 1, 0, 0, 0, 0]], np.float32),
        np.array([[0.0, -0.0, 0.0, -0.0, -1, 2, 2, -0.0]], np.float32),
        np.array([[3, 3, 3, 3, 3, 3, 3, 3]], np.float32),
        np.random.default_rng(0).integers(-3, 4, (7, 40)).astype(np.float32),
        np.array([[-np.inf, -np.inf, 5.0, -np.inf]], np.float32),
    ]
    for L in cases:
        T, E = L.shape
        for k in sorted({1, 2, min(E, 5), E if E <= 32 else 32}):
            dl = torch.tensor(L).cuda()
            idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
            gate = torch.empty(T, k, dtype=torch.float32, device="cuda")
            B.waste_moe_topk_from_logits(dl, T, E, k, idx, gate)
            torch.cuda.synchronize()
            for t in range(T):
                ridx, rg = oracle.topk_softmax(L[t].astype(np.float64), k)
                np.testing.assert_array_equal(idx[t].cpu().numpy(), ridx, err_msg=f"{L[t]} k={k}")
                np.testing.assert_allclose(gate[t].cpu().numpy(), rg, rtol=1e-6, atol=1e-7)


def test_empty_batch_is_noop():
    d, f, E, k, T = 256, 128, 8, 2, 4
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        out = torch.full((T, d), 7.0, device="cuda")
        idx, gate, logits, _ = layer.alloc_outputs(T)
        layer.route(h.cuda(), 0, idx, gate, logits)
        layer.forward(h.cuda(), 0, idx, gate, out, 0)
        torch.cuda.synchronize()
        assert bool((out == 7.0).all())
    finally:
        layer.close()


def test_tokens_above_max_rejected():
    d, f, E, k, T = 256, 128, 8, 2, 4
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        idx, gate, logits, out = layer.alloc_outputs(T)
        with pytest.raises(B.WasteError):
            layer.route(h.cuda(), T + 1, idx, gate, logits)
    finally:
        layer.close()


def test_bad_expert_index_flagged():
    """An index outside [0, E) contributes nothing and is reported by stats."""
    d, f, E, k, T = 256, 128, 8, 2, 1
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        hd = h.cuda()
        idx = torch.tensor([[3, E]], dtype=torch.int32, device="cuda")
        gate = torch.tensor([[0.5, 0.5]], device="cuda")
        out = torch.empty(T, d, device="cuda")
        layer.forward(hd, T, idx, gate, out, 0)
        torch.cuda.synchronize()
        e3 = oracle.expert_ffn(li.codebooks[3], li.codes[0][3], li.codes[1][3], li.codes[2][3], h[0])
        assert_close(out[0].cpu().numpy(), 0.5 * e3)
        with pytest.raises(B.WasteError):
            layer.stats()
        layer.reset_stats()
        layer.stats()
        # the launch's completion counters came back to zero around the invalid slot: the
        # next calls wait for their own gate/up units again
        for e in (5, 1):
            idx = torch.tensor([[e, 3]], dtype=torch.int32, device="cuda")
            layer.forward(hd, T, idx, gate, out, 0)
            torch.cuda.synchronize()
            ee = oracle.expert_ffn(li.codebooks[e], li.codes[0][e], li.codes[1][e], li.codes[2][e], h[0])
            assert_close(out[0].cpu().numpy(), 0.5 * ee + 0.5 * e3)
        layer.stats()
    finally:
        layer.close()


@pytest.mark.parametrize("shape", [(1032, 136, 12, 3, 5), (256, 128, 8, 2, 4), (8, 8, 2, 1, 2)])
def test_fused_step_equals_phases(shape):
    """The one-kernel step (route + forward) and forward through the fused kernel equal the
    per-phase kernels bit for bit, over several launches in a row (the device queue and
    counters must come back to zero after every launch)."""
    d, f, E, k, T = shape
    w, li, h, fused = small_layer(d, f, E, k, T, flags=B.FLAG_STEP_KERNEL)
    _, _, _, phases = small_layer(d, f, E, k, T)
    try:
        hd = h.cuda()
        ref = run(phases, hd, T)
        for _ in range(3):
            idx, gate, logits, out = fused.alloc_outputs(T)
            fused.step(hd, T, idx, gate, out, 0, logits)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(idx.cpu().numpy(), ref[0])
            assert np.array_equal(gate.cpu().numpy().view(np.uint32), ref[1].view(np.uint32))
            assert np.array_equal(out.cpu().numpy().view(np.uint32), ref[3].view(np.uint32))
            got = run(fused, hd, T)  # route, then forward through the fused kernel
            assert np.array_equal(got[3].view(np.uint32), ref[3].view(np.uint32))
        fused.stats()  # no timeout or bad index recorded
    finally:
        fused.close()
        phases.close()


def test_deterministic():
    d, f, E, k, T = 1032, 136, 12, 3, 5
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        a = run(layer, h.cuda(), T)[3]
        b = run(layer, h.cuda(), T)[3]
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    finally:
        layer.close()


@pytest.mark.parametrize("d, E, k, act", [(512, 384, 16, "f32"), (512, 12, 3, "f32"), (512, 4, 4, "f32"),
                                          (7168, 384, 16, "f32"), (7168, 384, 16, "bf16"), (8, 4, 2, "bf16")])
def test_one_token_routing_in_one_launch(d, E, k, act):
    """One token is routed in a single launch (one CTA per expert row, the row and the token
    moved into shared memory by bulk copies; the last CTA takes the top-k); the same token
    inside a batch of three goes through the staged router and the top-k kernel: indices,
    gates and logits agree bit for bit, and the counter is back at rest for the next call."""
    w = synth.Workload("r1", d, 64, E, k, 3, act, "offsets")
    li = synth.layer_inputs(w, 4, 0, "cpu", with_codes=True)
    h = synth.hidden(9, 3, d, act, "cpu").cuda()
    layer = MoELayer(w, 4, 0, "cuda", inputs=li)
    try:
        for rep in range(3):
            i3, g3, l3 = layer.alloc_outputs(3)[:3]
            layer.route(h, 3, i3, g3, l3)
            for t in range(3):
                i1, g1, l1 = layer.alloc_outputs(1)[:3]
                layer.route(h[t:t + 1].contiguous(), 1, i1, g1, l1)
                torch.cuda.synchronize()
                assert torch.equal(i1[0], i3[t]) and torch.equal(g1[0], g3[t]) and torch.equal(l1[0], l3[t])
    finally:
        layer.close()


@pytest.mark.parametrize("mode", [0, 1])
def test_output_in_pinned_host_memory(mode):
    """The step's output written straight into pinned host memory equals the device-memory
    output bit for bit (mode 0 =, mode 1 +=, the residual already in the host buffer)."""
    d, f, E, k, T = 512, 264, 20, 5, 3
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        hd = h.cuda()
        base = torch.randn(T, d, generator=torch.Generator().manual_seed(11))
        out_dev = base.cuda()
        out_host = base.clone().pin_memory()
        for out in (out_dev, out_host):
            idx, gate, logits, _ = layer.alloc_outputs(T)
            layer.step(hd, T, idx, gate, out, mode, logits=logits)
        torch.cuda.synchronize()
        assert torch.equal(out_dev.cpu(), out_host)
    finally:
        layer.close()


@pytest.mark.parametrize("T", [1, 3])
def test_largest_expert_count_and_top_k(T):
    """The configuration's limits: E = 4096 experts, top-32 (1,024 router CTAs; for one token the
    last of them takes the top-k, for three the top-k kernel does): logits, routing, gates and
    outputs against the oracle; plus the top-k alone on tied integer logits over 4096 experts."""
    d, f, E, k = 64, 16, 4096, 32
    w = synth.Workload("maxE", d, f, E, k, T, "f32", "offsets", bias_spacing=40.0)
    li = synth.layer_inputs(w, 5, 0, "cpu", with_codes=True)
    h = synth.hidden(6, T, d, "f32", "cpu")
    layer = MoELayer(w, 5, 0, "cuda", inputs=li)
    try:
        g_idx, g_gate, g_logits, g_out = run(layer, h.cuda(), T)
        ref = oracle.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, k)
        np.testing.assert_allclose(g_logits, ref["logits"], rtol=1e-5, atol=1e-5)
        ok = check_routing(g_idx, g_gate, ref["logits"], k)
        assert ok, "no well-separated token"
        assert_close(g_out[ok], ref["out"][ok])
    finally:
        layer.close()
    L = np.random.default_rng(1).integers(-4, 5, (2, E)).astype(np.float32)
    dl = torch.tensor(L).cuda()
    idx = torch.empty(2, k, dtype=torch.int32, device="cuda")
    gate = torch.empty(2, k, dtype=torch.float32, device="cuda")
    B.waste_moe_topk_from_logits(dl, 2, E, k, idx, gate)
    torch.cuda.synchronize()
    for t in range(2):
        ridx, rg = oracle.topk_softmax(L[t].astype(np.float64), k)
        np.testing.assert_array_equal(idx[t].cpu().numpy(), ridx)
        np.testing.assert_allclose(gate[t].cpu().numpy(), rg, rtol=1e-6, atol=1e-7)


def test_bad_record_header_refused():
    """create refuses a bank whose header has a wrong magic, expert id, layer or offset."""
    d, f, E, k, T = 256, 128, 8, 2, 1
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        rec = layer.records
        stride = layer.stride
        hdr_bytes = rec[: 128].clone()

        def expect_refusal(offset, value_bytes, cfg=None):
            saved = rec[offset: offset + len(value_bytes)].clone()
            rec[offset: offset + len(value_bytes)] = torch.tensor(list(value_bytes), dtype=torch.uint8,
                                                                 device="cuda")
            try:
                with pytest.raises(B.WasteError) as ei:
                    B.waste_moe_create(cfg or layer.cfg, layer.router_w, layer.router_b, rec, stride,
                                       layer.codebooks)
                assert ei.value.status == -4
            finally:
                rec[offset: offset + len(value_bytes)] = saved

        expect_refusal(0, b"XMOE")                                  # magic of record 0
        expect_refusal(3 * stride + 12, (7).to_bytes(4, "little"))  # expert id of record 3
        expect_refusal(5 * stride + 8, (9).to_bytes(4, "little"))   # layer of record 5
        expect_refusal(2 * stride + 40, (100).to_bytes(8, "little"))  # section offset not aligned
        expect_refusal(2 * stride + 56, (1 << 40).to_bytes(8, "little"))  # section past the record
        assert torch.equal(rec[:128], hdr_bytes)
    finally:
        layer.close()


def test_stats_count_algorithmic_bytes():
    d, f, E, k, T = 1032, 136, 12, 3, 5
    w, li, h, layer = small_layer(d, f, E, k, T)
    try:
        layer.reset_stats()
        run(layer, h.cuda(), T)
        st = layer.stats()
        assert st["demand_code_bytes"] == T * k * oracle.expert_code_bytes(d, f)
        assert st["codebook_bytes"] == T * k * 3 * 3 * 256 * 8 * 4
        assert st["router_bytes"] == E * d * 4
        assert st["routed_slots"] == T * k
        assert st["forward_slots"] == T * k
    finally:
        layer.close()


# ---------------------------------------------------------------- full decode shape

@pytest.mark.parametrize("seed", [0, 3])
def test_decode_layer_full_size(seed):
    """The decode workload (d=7168, f=1536, E=384, top-16, one token) at full size, in the
    launch configuration the benchmark times; the oracle recomputes the token from the
    router and the 16 selected experts' codes."""
    w = synth.WORKLOADS["decode"]
    layer = MoELayer(w, seed, 0, "cuda")
    try:
        h = synth.hidden(seed, 1, w.d, "f32", "cuda")
        g_idx, g_gate, g_logits, g_out = run(layer, h, 1)
        ref = oracle.moe_token(h[0].cpu(), layer.router_w.cpu(), layer.router_b.cpu(),
                               layer.codebooks.cpu().numpy(),
                               lambda e: layer.expert_codes_host(e), w.top_k)
        assert oracle.topk_margin(ref["logits"], w.top_k) > 1e-3
        np.testing.assert_allclose(g_logits[0], ref["logits"], rtol=1e-5, atol=1e-4)
        np.testing.assert_array_equal(g_idx[0], ref["idx"])
        np.testing.assert_allclose(g_gate[0], ref["gate"], rtol=1e-5, atol=1e-7)
        assert_close(g_out[0], ref["out"])
        st = layer.stats()
        assert st["demand_code_bytes"] == w.top_k * oracle.expert_code_bytes(w.d, w.f)
        # the register-reconstruct form of the expert kernels on the same records: the same
        # experts and the same output within the fp32 bar
        rcfg = B.make_config(w.d, w.f, w.n_experts, w.top_k, "f32", 1, 0, B.FLAG_K2_RECONSTRUCT, 0)
        rh = B.waste_moe_create(rcfg, layer.router_w, layer.router_b, layer.records, layer.stride,
                                layer.codebooks)
        try:
            idx = torch.empty(1, w.top_k, dtype=torch.int32, device="cuda")
            gate = torch.empty(1, w.top_k, dtype=torch.float32, device="cuda")
            out = torch.empty(1, w.d, dtype=torch.float32, device="cuda")
            B.waste_moe_route(rh, h, 1, idx, gate)
            B.waste_moe_forward(rh, h, 1, idx, gate, out, 0)
            torch.cuda.synchronize()
            B.waste_moe_stats(rh)
            np.testing.assert_array_equal(idx[0].cpu().numpy(), ref["idx"])
            assert_close(out[0].cpu().numpy(), ref["out"])
        finally:
            B.waste_moe_destroy(rh)
    finally:
        layer.close()
