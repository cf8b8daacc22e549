"""The decode stack with router lookahead: outputs and demand bytes do not depend on
the lookahead, graph replay equals eager launches, and the chain matches the oracle.

The pages state that the lookahead leaves the output exact (the real router still
decides) and leaves the total bytes read unchanged (page "Exécuter Kimi K3 avec 29
Go de RAM à 0,50 tok/s", section "Lecture anticipée et prédiction du routeur").
"""
import numpy as np
import pytest
import torch

import oracle
from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth
from rvq_compressed_expert_gb300.layer import MoELayer
from rvq_compressed_expert_gb300.stack import DecodeStack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rvq_compressed_expert_gb300 import _build
    _build.build()
    B.load()
    oracle.build()


SMALL = synth.Workload("small-stack", 512, 256, 16, 4, 2, "f32", "offsets", n_layers=6, lookahead=3)
# one token: the lookahead runs inside each layer's step (no side stream)
SMALL_ONE = synth.Workload("small-stack-1", 512, 256, 16, 4, 1, "f32", "offsets", n_layers=6, lookahead=3)


def make_layers(w, seed=0, device="cuda"):
    layers = []
    for L in range(w.n_layers):
        li = synth.layer_inputs(w, seed, L, "cpu", with_codes=True)
        layers.append((MoELayer(w, seed, L, device, inputs=li), li))
    return layers


def run_eager(stack, h0, P, record=None):
    main = torch.cuda.Stream()
    side = torch.cuda.Stream()
    main.wait_stream(torch.cuda.current_stream())
    out = stack.run(h0, P, main, side, on_layer=record)
    torch.cuda.current_stream().wait_stream(main)
    torch.cuda.synchronize()
    return out.clone()


@pytest.mark.parametrize("w", [SMALL, SMALL_ONE], ids=["two-tokens", "one-token"])
def test_stack_lookahead_invariant_and_matches_oracle(w):
    pairs = make_layers(w)
    layers = [p[0] for p in pairs]
    try:
        h0 = synth.hidden(3, w.tokens, w.d, "f32", "cpu")
        hd = h0.cuda()
        stack = DecodeStack(layers, w.tokens)
        routed = {}

        def record(L, idx, gate, main):
            with torch.cuda.stream(main):
                routed[L] = idx.clone()

        outs = {}
        for P in (0, w.lookahead):
            for l in layers:
                l.reset_stats()
            outs[P] = run_eager(stack, hd, P, record if P == 0 else None)
            sts = [l.stats() for l in layers]
            outs[(P, "bytes")] = sum(s["demand_code_bytes"] for s in sts)
            outs[(P, "hits")] = sum(s["prediction_hits"] for s in sts)
            outs[(P, "prefetch")] = sum(s["prefetch_experts"] for s in sts)
        assert torch.equal(outs[0], outs[w.lookahead]), "lookahead changed the output"
        assert outs[(0, "bytes")] == outs[(w.lookahead, "bytes")]
        assert outs[(0, "bytes")] == w.n_layers * w.tokens * w.top_k * oracle.expert_code_bytes(w.d, w.f)
        assert outs[(w.lookahead, "prefetch")] == (w.n_layers - 1) * w.tokens * w.lookahead
        assert outs[(0, "prefetch")] == 0 and outs[(0, "hits")] == 0
        # the oracle runs the same chain from h0 on its own
        ref_h, ref_idx, ref_logits = oracle.stack_chain(
            h0, [(li.router_w, li.router_b, li.codebooks, li.codes) for _, li in pairs], w.top_k)
        for L in range(w.n_layers):
            for t in range(w.tokens):
                assert oracle.topk_margin(ref_logits[L][t], w.top_k) > 1e-3
            np.testing.assert_array_equal(routed[L].cpu().numpy(), ref_idx[L], err_msg=f"layer {L}")
        got = outs[0].cpu().double().numpy()
        rel = np.linalg.norm(got - ref_h) / np.linalg.norm(ref_h)
        assert rel < 1e-5, rel
    finally:
        for l in layers:
            l.close()


def test_topk_survives_nonfinite_logits():
    """NaN and infinite logits (outside the contract) still give k distinct valid indices."""
    L = np.array([[np.nan, 1.0, np.inf, -np.inf, np.nan, 0.5, np.nan, -1.0] * 8], np.float32)
    for k in (1, 4, 16, 32):
        dl = torch.tensor(L).cuda()
        idx = torch.empty(1, k, dtype=torch.int32, device="cuda")
        gate = torch.empty(1, k, dtype=torch.float32, device="cuda")
        B.waste_moe_topk_from_logits(dl, 1, L.shape[1], k, idx, gate)
        torch.cuda.synchronize()
        got = idx[0].cpu().numpy()
        assert len(set(got.tolist())) == k
        assert got.min() >= 0 and got.max() < L.shape[1]


def test_rmsnorm_matches_oracle():
    x = torch.randn(5, 1032, generator=torch.Generator().manual_seed(0)) * 7
    y = torch.empty_like(x).cuda()
    B.waste_moe_rmsnorm(x.cuda(), y, 5, 1032)
    torch.cuda.synchronize()
    for t in range(5):
        ref = oracle.rmsnorm(x[t])
        np.testing.assert_allclose(y[t].cpu().numpy(), ref, rtol=2e-6, atol=1e-7)


def test_stack_graph_replay_equals_eager():
    w = SMALL
    pairs = make_layers(w, seed=1)
    layers = [p[0] for p in pairs]
    try:
        hd = synth.hidden(4, w.tokens, w.d, "f32", "cpu").cuda()
        stack = DecodeStack(layers, w.tokens)
        ref = run_eager(stack, hd, w.lookahead)
        for P in (0, w.lookahead):
            main = torch.cuda.Stream()
            side = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=main):
                out = stack.run(hd, P, main, side)
            for l in layers:
                l.reset_stats()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, ref), f"graph replay differs (lookahead {P})"
            sts = [l.stats() for l in layers]  # raises if a kernel saw a bad expert index
            assert sum(s["forward_slots"] for s in sts) == 3 * w.n_layers * w.tokens * w.top_k
            if P:
                assert sum(s["prefetch_experts"] for s in sts) == 3 * (w.n_layers - 1) * w.tokens * P
            del g
    finally:
        for l in layers:
            l.close()


def test_route_trace_jsonl(tmp_path):
    """The routing trace of two tokens through the stack: one JSON line per (token, layer) with
    the experts the oracle's chain picks and gates summing to one."""
    import json
    from rvq_compressed_expert_gb300.trace import RouteTrace
    w = SMALL
    pairs = make_layers(w)
    layers = [p[0] for p in pairs]
    try:
        stack = DecodeStack(layers, w.tokens)
        tr = RouteTrace()
        h0s = [synth.hidden(3 + i, w.tokens, w.d, "f32", "cpu") for i in range(2)]
        for h0 in h0s:
            run_eager(stack, h0.cuda(), 0, tr.on_layer)
            tr.next_token()
        path = tmp_path / "route.jsonl"
        assert tr.write(str(path)) == 2 * w.n_layers
        rows = [json.loads(l) for l in open(path)]
        assert [(r["token"], r["layer"]) for r in rows] == [(t, L) for t in range(2) for L in range(w.n_layers)]
        for t, h0 in enumerate(h0s):
            _, ref_idx, _ = oracle.stack_chain(
                h0, [(li.router_w, li.router_b, li.codebooks, li.codes) for _, li in pairs], w.top_k)
            for L in range(w.n_layers):
                r = rows[t * w.n_layers + L]
                assert r["experts"] == np.asarray(ref_idx[L]).tolist()
                assert all(abs(sum(g) - 1.0) < 1e-6 for g in r["gates"])
    finally:
        for l in layers:
            l.close()


def test_full_depth_token_matches_oracle():
    """One token through the full-depth stack -- 92 layers x 64 resident experts at d=7168,
    f=1536, top-16, lookahead 6 -- against the oracle's decode chain run on its own (only the 16
    selected experts' codes of each layer handed to it): every layer's experts bit-exact, the
    final h within the fp32 bar (relative L2 <= 1e-5, |err| <= 1e-4 max|h|).  Page "Exécuter
    Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Budget RAM et zone de performance
    étroite": 16 experts x 92 layers per token."""
    w = synth.WORKLOADS["stack"]
    free, _ = torch.cuda.mem_get_info()
    need = w.n_layers * w.n_experts * 12_390_400 * 1.05 + (4 << 30)
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free")
    layers = [MoELayer(w, 0, L, "cuda", max_tokens=1) for L in range(w.n_layers)]
    try:
        h0 = synth.hidden(7, 1, w.d, "f32", "cuda")
        stack = DecodeStack(layers, 1)
        routed = {}

        def record(L, idx, gate, main):
            with torch.cuda.stream(main):
                routed[L] = idx.clone()

        out = run_eager(stack, h0, w.lookahead, record)
        for l in layers:
            l.stats()  # raises on a latched device error
        ref_layers = []
        for L, ml in enumerate(layers):
            get = (lambda ml: lambda e: ml.expert_codes_host(e))(ml)
            ref_layers.append((ml.router_w.cpu(), ml.router_b.cpu(), ml.codebooks.cpu(), get))
        h, ref_idx, _, ref_logits = oracle.stack_token(h0[0].cpu(), ref_layers, w.top_k)
        for L in range(w.n_layers):
            assert oracle.topk_margin(ref_logits[L], w.top_k) > 1e-4, f"layer {L}: near-tie in the oracle"
            np.testing.assert_array_equal(routed[L][0].cpu().numpy(), ref_idx[L], err_msg=f"layer {L}")
        got = out[0].cpu().double().numpy()
        rel = np.linalg.norm(got - h) / np.linalg.norm(h)
        assert rel <= 1e-5, rel
        assert np.abs(got - h).max() <= 1e-4 * np.abs(h).max()
    finally:
        for l in layers:
            l.close()
        torch.cuda.empty_cache()


def test_lookahead_with_mispredictions():
    """A stack whose router bias gives Zipf-like expert popularity: the lookahead's predictions
    (layer L+1's router on layer L's input) miss some experts.  Outputs are still bit-identical
    with the lookahead on and off, demand bytes equal, and each prediction names the first row
    groups of gate and up plus their codebooks, whatever it hits."""
    # a weak Zipf law (s = 0.2): the bias orders the experts but the token still moves them
    w = synth.Workload("zipf-stack", 512, 256, 32, 4, 4, "f32", "zipf", n_layers=6, lookahead=3, zipf_s=0.2)
    pairs = make_layers(w)
    layers = [p[0] for p in pairs]
    try:
        hd = synth.hidden(5, w.tokens, w.d, "f32", "cuda")
        stack = DecodeStack(layers, w.tokens)
        res = {}
        for P in (0, w.lookahead):
            for l in layers:
                l.reset_stats()
            out = run_eager(stack, hd, P)
            sts = [l.stats() for l in layers]
            res[P] = (out, {k: sum(s[k] for s in sts) for k in sts[0]})
        (out0, s0), (out1, s1) = res[0], res[w.lookahead]
        assert torch.equal(out0, out1)
        assert s0["demand_code_bytes"] == s1["demand_code_bytes"]
        n_pred = (w.n_layers - 1) * w.tokens * w.lookahead
        assert s1["prefetch_experts"] == n_pred
        nseg = -(-w.d // 256)
        groups = -(-w.f // 16)
        per_expert = 2 * nseg * min(groups, 16) * 3 * 512 + 2 * 3 * 256 * 8 * 4
        assert s1["prefetch_issued_bytes"] == n_pred * per_expert
        assert 0 < s1["prediction_hits"] < n_pred, s1["prediction_hits"]
    finally:
        for l in layers:
            l.close()


def test_lookahead_inside_the_step_predicts_its_own_route():
    """waste_moe_set_lookahead with the layer as its own next layer: the step's router launch runs
    the layer's rows twice on the same input, its expert kernel predicts the top-P from the second
    set and prefetches them; the next step on the same input scores that prediction: every one of
    the P experts is among its top-k.  Outputs equal those without the lookahead, bit for bit."""
    w = synth.Workload("la-self", 1032, 136, 40, 6, 1, "f32", "none")
    layer = MoELayer(w, 0, 0, "cuda")
    plain = MoELayer(w, 0, 0, "cuda")
    try:
        idx, gate, logits, out = layer.alloc_outputs(1)
        idx2, gate2, logits2, out2 = plain.alloc_outputs(1)
        nseg = -(-w.d // 256)
        groups = -(-w.f // 16)
        per_expert = 2 * nseg * min(groups, 16) * 3 * 512 + 2 * 3 * 256 * 8 * 4
        for seed, P in ((1, 4), (2, 1), (3, 6)):
            x = synth.hidden(seed, 1, w.d, "f32", "cuda")
            B.waste_moe_set_lookahead(layer.handle, layer.handle, P)
            layer.route(x, 1, idx, gate, logits)  # scores (and so clears) a pending prediction
            layer.reset_stats()
            layer.step(x, 1, idx, gate, out, 0, logits)
            layer.step(x, 1, idx, gate, out, 0, logits)
            plain.step(x, 1, idx2, gate2, out2, 0, logits2)
            torch.cuda.synchronize()
            st = layer.stats()
            assert st["prefetch_experts"] == 2 * P
            assert st["prefetch_issued_bytes"] == 2 * P * per_expert
            assert st["prediction_hits"] == P
            assert torch.equal(idx, idx2)
            assert torch.equal(out.view(torch.int32), out2.view(torch.int32))
        B.waste_moe_set_lookahead(layer.handle, None, 0)
        layer.route(x, 1, idx, gate, logits)
        layer.reset_stats()
        layer.step(x, 1, idx, gate, out, 0, logits)
        torch.cuda.synchronize()
        st = layer.stats()
        assert st["prefetch_experts"] == 0 and st["prediction_hits"] == 0
    finally:
        layer.close()
        plain.close()


def test_set_lookahead_rejects_bad_arguments():
    w = synth.Workload("la-bad", 512, 256, 16, 4, 1, "f32", "none")
    a = MoELayer(w, 0, 0, "cuda")
    b = MoELayer(synth.Workload("la-bad2", 1024, 256, 16, 4, 1, "f32", "none"), 0, 1, "cuda")
    try:
        with pytest.raises(B.WasteError):
            B.waste_moe_set_lookahead(a.handle, a.handle, 17)  # more than the next layer's experts
        with pytest.raises(B.WasteError):
            B.waste_moe_set_lookahead(a.handle, b.handle, 2)  # another hidden size
        with pytest.raises(B.WasteError):
            B.waste_moe_set_lookahead(None, a.handle, 2)
        B.waste_moe_set_lookahead(a.handle, None, 0)
    finally:
        a.close()
        b.close()


def test_lookahead_inside_the_step_into_a_wider_layer():
    """The next layer may have more experts than the current one: its router rows ride on the
    current router launch all the same; its own route on the same input scores every one of the P
    predicted experts as a hit, and the current layer's outputs are unchanged."""
    wa = synth.Workload("la-a", 512, 256, 16, 4, 1, "f32", "none")
    wb = synth.Workload("la-b", 512, 256, 40, 6, 1, "f32", "none")
    a = MoELayer(wa, 0, 0, "cuda")
    b = MoELayer(wb, 0, 1, "cuda")
    try:
        ia, ga, la, oa = a.alloc_outputs(1)
        ib, gb, lb, ob = b.alloc_outputs(1)
        x = synth.hidden(9, 1, wa.d, "f32", "cuda")
        a.step(x, 1, ia, ga, oa, 0, la)
        torch.cuda.synchronize()
        ref = oa.clone()
        b.route(x, 1, ib, gb, lb)  # no prediction pending
        B.waste_moe_set_lookahead(a.handle, b.handle, 3)
        b.reset_stats()
        a.step(x, 1, ia, ga, oa, 0, la)
        b.route(x, 1, ib, gb, lb)
        torch.cuda.synchronize()
        st = b.stats()
        assert st["prefetch_experts"] == 3 and st["prediction_hits"] == 3
        assert torch.equal(oa.view(torch.int32), ref.view(torch.int32))
        B.waste_moe_set_lookahead(a.handle, None, 0)
    finally:
        a.close()
        b.close()
