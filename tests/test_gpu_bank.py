"""Tiered expert bank: records in pinned host memory, an HBM cache, device-side fetches.

Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", sections "Budget RAM et zone de
performance étroite" and "Lecture anticipée et prédiction du routeur": a bounded cache of
experts over a slow tier, misses read from the slow tier, the lookahead fills the cache ahead
of demand -- the outputs never change (the real router decides), only what is resident.
"""
import numpy as np
import pytest
import torch

import oracle
from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth
from rvq_compressed_expert_gb300.bank import TieredStack
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


def assert_oracle_chain(outs, w, hidden_seed0, n_layers, gen_device="cuda", seed=0):
    """Each token's output (the banked stack's) against the oracle's decode chain run on its own
    from the same token and weights: h <- h + MoE_L(rmsnorm(h)) over the layers, only the
    selected experts' codes fetched.  The bounded cache and the lookahead never change what a
    layer computes (page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", sections "Budget RAM
    et zone de performance étroite" and "Lecture anticipée et prédiction du routeur"), so the
    fp32 bar holds: relative L2 <= 1e-5 and |err| <= 1e-4 max|y|."""
    lis = [synth.layer_inputs(w, seed, L, gen_device, with_codes=False) for L in range(n_layers)]
    layers = []
    for L, li in enumerate(lis):
        get = (lambda L: lambda e: tuple(c.cpu() for c in synth.expert_codes(seed, L, e, w.d, w.f, gen_device)))(L)
        layers.append((li.router_w.cpu(), None if li.router_b is None else li.router_b.cpu(),
                       li.codebooks.cpu(), get))
    for i, got in enumerate(outs):
        h0 = synth.hidden(hidden_seed0 + i, w.tokens, w.d, "f32", "cuda")[0].cpu()
        ref, _, _, _ = oracle.stack_token(h0, layers, w.top_k)
        g = got[0].cpu().double().numpy()
        rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        assert rel <= 1e-5, f"token {i}: relative L2 {rel:.3e}"
        assert np.abs(g - ref).max() <= 1e-4 * np.abs(ref).max(), f"token {i}"


W = synth.Workload("bank", 512, 256, 16, 4, 1, "f32", "offsets", n_layers=4, lookahead=3)


def run_tokens(stack, tokens, lookahead):
    main = torch.cuda.Stream()
    side = torch.cuda.Stream()
    main.wait_stream(torch.cuda.current_stream())
    outs = []
    for i in range(tokens):
        with torch.cuda.stream(main):  # the token is drawn and the output read on `main`
            h0 = synth.hidden(50 + i, W.tokens, W.d, "f32", "cuda")
        out = stack.run(h0, lookahead, main, side)
        with torch.cuda.stream(main):
            outs.append(out.clone())
    torch.cuda.current_stream().wait_stream(main)
    torch.cuda.synchronize()
    return outs


def resident_outputs(tokens, lookahead):
    layers = [MoELayer(W, 0, L, "cuda") for L in range(W.n_layers)]
    try:
        return run_tokens(DecodeStack(layers, W.tokens), tokens, lookahead)
    finally:
        for l in layers:
            l.close()


@pytest.mark.parametrize("flags", [0, B.FLAG_BANK_SERIAL], ids=["overlap", "serial"])
@pytest.mark.parametrize("lookahead", [0, 3])
def test_banked_equals_resident(lookahead, flags):
    """6 slots for 4 layers x top-4: every layer evicts; outputs equal the resident stack's bit
    for bit, whether each expert is consumed as its copy lands (the step kernel's copy lanes)
    or after the whole copy; hits + misses count every routed expert; bytes copied = copies x
    record stride."""
    ref = resident_outputs(5, lookahead)
    ts = TieredStack(W, 0, W.n_layers, 6, flags=flags)
    try:
        got = run_tokens(DecodeStack(ts.layers, W.tokens, banked=True), 5, lookahead)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert_oracle_chain(got, W, 50, W.n_layers)
        st = ts.stats()
        assert st["demand_hits"] + st["demand_misses"] == 5 * W.n_layers * W.top_k
        assert st["copied_bytes"] == (st["demand_misses"] + st["prefetch_copies"]) * ts.stride
        for ml in ts.layers:
            ml.stats()  # raises if an expert had no slot
        if lookahead == 0:
            assert st["prefetch_copies"] == 0 and st["prefetch_present"] == 0
    finally:
        ts.close()


def test_lookahead_raises_demand_hits():
    """With the router's offsets making the prediction reliable, the lookahead turns demand
    misses into hits (16 slots: the cache holds about one layer's experts beside the next)."""
    res = {}
    for P in (0, 3):
        ts = TieredStack(W, 0, W.n_layers, 8)
        try:
            run_tokens(DecodeStack(ts.layers, W.tokens, banked=True), 4, P)
            res[P] = ts.stats()
        finally:
            ts.close()
    assert res[3]["demand_misses"] < res[0]["demand_misses"], res
    assert res[3]["prefetch_copies"] > 0


def test_bank_refusals():
    ts = TieredStack(W, 0, 1, 4)
    try:
        ml = ts.layers[0]
        cfg = B.make_config(W.d, W.f, W.n_experts, W.top_k, "f32", 2, 0, 0, 0)  # min(2 x 4, 16) > 4 slots
        with pytest.raises(B.WasteError) as ei:
            B.waste_moe_create_banked(cfg, ml.router_w, ml.router_b, ts.bank, 0, ml.codebooks)
        assert ei.value.status == -1
        with pytest.raises(B.WasteError):
            B.waste_moe_create_banked(ml.cfg, ml.router_w, ml.router_b, ts.bank, 1, ml.codebooks)  # no layer 1
    finally:
        ts.close()
    cfg = B.make_config(W.d, W.f, W.n_experts, W.top_k, "f32", 1, 0, 0, 0)
    stride, _, _ = B.waste_moe_record_layout(cfg)
    host = B.pinned_bytes(W.n_experts * stride + 8192)
    with pytest.raises(B.WasteError) as ei:  # not 4096-aligned
        B.waste_bank_create(cfg, 1, host[16:], stride, 4)
    assert ei.value.status == -4


@pytest.mark.parametrize("flags", [0, B.FLAG_BANK_SERIAL], ids=["overlap", "serial"])
def test_repeated_expert_across_tokens(flags):
    """Two tokens share experts that are not resident: each is copied once, the second token's
    units wait for the same copy (overlap) -- outputs equal the resident layer's."""
    w2 = synth.Workload("bank2", 512, 256, 12, 4, 2, "f32", "none")
    res = MoELayer(w2, 1, 0, "cuda")
    ts = TieredStack(w2, 1, 1, 8, flags=flags)
    try:
        h = synth.hidden(4, 2, w2.d, "f32", "cuda")
        gate = torch.rand(2, 4, device="cuda")
        for ids, misses in (([[5, 1, 2, 3], [5, 6, 1, 0]], 6), ([[7, 6, 9, 5], [9, 11, 7, 2]], 9)):
            idx = torch.tensor(ids, dtype=torch.int32, device="cuda")
            a = torch.empty(2, w2.d, device="cuda")
            b = torch.empty(2, w2.d, device="cuda")
            ts.layers[0].forward(h, 2, idx, gate, a)
            res.forward(h, 2, idx, gate, b)
            torch.cuda.synchronize()
            assert torch.equal(a, b)
            assert ts.stats()["demand_misses"] == misses, (ids, ts.stats())
        ts.layers[0].stats()
    finally:
        ts.close()
        res.close()


@pytest.mark.parametrize("flags", [0, B.FLAG_BANK_SERIAL], ids=["overlap", "serial"])
def test_many_ids_across_plan_chunks(flags):
    """16 tokens x top-4 = 64 ids, planned 32 at a time: experts repeated inside and across the
    two halves are copied once each, the repeats wait for those copies (overlap), and outputs
    equal the resident layer's; a second call with the same routing copies nothing."""
    w3 = synth.Workload("bank3", 512, 256, 20, 4, 16, "f32", "none")
    res = MoELayer(w3, 3, 0, "cuda")
    ts = TieredStack(w3, 3, 1, 20, flags=flags)
    try:
        h = synth.hidden(8, 16, w3.d, "f32", "cuda")
        g = torch.Generator().manual_seed(5)
        ids = torch.stack([torch.randperm(20, generator=g)[:4] for _ in range(16)]).to(torch.int32).cuda()
        gate = torch.rand(16, 4, generator=g).cuda()
        for rep in range(2):
            a = torch.empty(16, w3.d, device="cuda")
            b = torch.empty(16, w3.d, device="cuda")
            ts.layers[0].forward(h, 16, ids, gate, a)
            res.forward(h, 16, ids, gate, b)
            torch.cuda.synchronize()
            assert torch.equal(a, b)
            st = ts.stats()
            assert st["demand_misses"] == len(torch.unique(ids)), st
            assert st["demand_hits"] == (rep + 1) * 64 - st["demand_misses"]
        ts.layers[0].stats()
    finally:
        ts.close()
        res.close()


def test_large_cache_plan_from_global_memory():
    """7,000 slots (their ticks and keys do not fit the plan's shared memory, so it reads them
    from global memory): outputs equal the resident stack's, every expert is copied once, and a
    second token through the same layers only hits or copies the experts it has not seen."""
    ts = TieredStack(W, 0, W.n_layers, 7000)
    try:
        ref = resident_outputs(3, 0)
        got = run_tokens(DecodeStack(ts.layers, W.tokens, banked=True), 3, 0)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        st = ts.stats()
        assert st["demand_hits"] + st["demand_misses"] == 3 * W.n_layers * W.top_k
        assert st["demand_misses"] <= W.n_layers * W.n_experts  # nothing is ever evicted
        assert st["copied_bytes"] == st["demand_misses"] * ts.stride
    finally:
        ts.close()


@pytest.mark.parametrize("flags", [0, B.FLAG_BANK_SERIAL], ids=["overlap", "serial"])
def test_full_size_records(flags):
    """The decode shape (d=7168, f=1536, 12.4 MB records, 190 copy chunks each): 2 layers x 20
    experts, top-16, behind 24 slots (each layer's 16 experts evict the other's); four tokens
    through the banked stack equal the resident stack bit for bit."""
    wf = synth.Workload("bankf", 7168, 1536, 20, 16, 1, "f32", "offsets", n_layers=2, lookahead=4)
    layers = [MoELayer(wf, 0, L, "cuda") for L in range(2)]
    try:
        ref = run_tokens_w(DecodeStack(layers, 1), wf, 4, 0)
    finally:
        for l in layers:
            l.close()
    ts = TieredStack(wf, 0, 2, 24, flags=flags)
    try:
        got = run_tokens_w(DecodeStack(ts.layers, 1, banked=True), wf, 4, 0)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert_oracle_chain(got, wf, 70, 2)
        st = ts.stats()
        assert st["demand_hits"] + st["demand_misses"] == 4 * 2 * 16
        assert st["demand_misses"] >= 16 + 16
        for ml in ts.layers:
            ml.stats()
    finally:
        ts.close()


def run_tokens_w(stack, w, tokens, lookahead):
    main = torch.cuda.Stream()
    side = torch.cuda.Stream()
    main.wait_stream(torch.cuda.current_stream())
    outs = []
    for i in range(tokens):
        with torch.cuda.stream(main):
            h0 = synth.hidden(70 + i, w.tokens, w.d, "f32", "cuda")
        out = stack.run(h0, lookahead, main, side)
        with torch.cuda.stream(main):
            outs.append(out.clone())
    torch.cuda.current_stream().wait_stream(main)
    torch.cuda.synchronize()
    return outs


class LruModel:
    """The bank's replacement policy as documented: a demand call advances the clock; every
    requested expert already cached takes the call's stamp; then, in order, each miss takes the
    least (tick, slot) among slots stamped before the call (none left: not placed)."""

    def __init__(self, n_slots):
        self.tick = [0] * n_slots
        self.key_of = [-1] * n_slots
        self.slot_of = {}
        self.clock = 0
        self.hits = self.misses = 0
        self.present = self.copies = 0

    def demand(self, keys):
        self.clock += 1
        h, m = self._plan(keys)
        self.hits += h
        self.misses += m

    def lookahead(self, keys):
        """A lookahead fetch plans at the current clock (it does not advance it)."""
        h, m = self._plan(keys)
        self.present += h
        self.copies += m

    def _plan(self, keys):
        c = self.clock
        hits = misses = 0
        for k in keys:
            if k in self.slot_of:
                self.tick[self.slot_of[k]] = c
        for k in keys:
            if k in self.slot_of:
                hits += 1
                continue
            free = [(t, v) for v, t in enumerate(self.tick) if t < c]
            if not free:
                continue
            _, v = min(free)
            if self.key_of[v] >= 0:
                del self.slot_of[self.key_of[v]]
            self.slot_of[k] = v
            self.key_of[v] = k
            self.tick[v] = c
            misses += 1
        return hits, misses


@pytest.mark.parametrize("flags", [0, B.FLAG_BANK_SERIAL], ids=["overlap", "serial"])
def test_replacement_follows_the_lru_model(flags):
    """40 random calls (1-2 tokens, top-4 of 12 experts, repeats within and across tokens) on
    2 layers sharing 8 slots, most followed by a lookahead of 1-3 experts into the other layer:
    after every call the device's hit / miss and present / copied counts equal the model's, and
    the outputs equal the resident layers'."""
    w4 = synth.Workload("bank4", 512, 256, 12, 4, 2, "f32", "none", n_layers=2)
    res = [MoELayer(w4, 4, L, "cuda") for L in range(2)]
    ts = TieredStack(w4, 4, 2, 8, flags=flags)
    model = LruModel(8)
    g = torch.Generator().manual_seed(9)
    try:
        for call in range(40):
            L = int(torch.randint(0, 2, (1,), generator=g))
            T = int(torch.randint(1, 3, (1,), generator=g))
            ids = torch.stack([torch.randperm(12, generator=g)[:4] for _ in range(T)]).to(torch.int32)
            gate = torch.rand(T, 4, generator=g).cuda()
            h = synth.hidden(100 + call, T, w4.d, "f32", "cuda")
            a = torch.empty(T, w4.d, device="cuda")
            b = torch.empty(T, w4.d, device="cuda")
            ts.layers[L].forward(h, T, ids.cuda(), gate, a)
            res[L].forward(h, T, ids.cuda(), gate, b)
            torch.cuda.synchronize()
            assert torch.equal(a, b), call
            model.demand([L * 12 + int(e) for e in ids.reshape(-1)])
            # now and then a lookahead into the other layer: its top-P of the same token
            P = int(torch.randint(0, 4, (1,), generator=g))
            if P:
                o = 1 - L
                pidx = torch.empty(T, 4, dtype=torch.int32, device="cuda")
                pgate = torch.empty(T, 4, device="cuda")
                ts.layers[o].route(h, T, pidx, pgate)
                ts.layers[o].prefetch(h, T, P)
                torch.cuda.synchronize()
                model.lookahead([o * 12 + int(e) for e in pidx[:, :P].reshape(-1).cpu()])
            st = ts.stats()
            assert (st["demand_hits"], st["demand_misses"]) == (model.hits, model.misses), (call, st)
            assert (st["prefetch_present"], st["prefetch_copies"]) == (model.present, model.copies), (call, st)
    finally:
        ts.close()
        for l in res:
            l.close()


def test_plan_keeps_resident_experts_of_the_call():
    """4 slots, experts given to forward: {0,1,2,3} fills the cache; [4,0,1,2] then copies
    expert 4 alone, into the slot of 3 -- a miss listed before resident experts of the same
    call must not evict them.  Outputs equal the resident layer's."""
    w1 = synth.Workload("bank1", 512, 256, 8, 4, 1, "f32", "none")
    res = MoELayer(w1, 0, 0, "cuda")
    ts = TieredStack(w1, 0, 1, 4)
    try:
        h = synth.hidden(3, 1, w1.d, "f32", "cuda")
        gate = torch.full((1, 4), 0.25, device="cuda")
        for ids, misses in (([0, 1, 2, 3], 4), ([4, 0, 1, 2], 5), ([2, 3, 4, 1], 6)):
            idx = torch.tensor([ids], dtype=torch.int32, device="cuda")
            a = torch.empty(1, w1.d, device="cuda")
            b = torch.empty(1, w1.d, device="cuda")
            ts.layers[0].forward(h, 1, idx, gate, a)
            res.forward(h, 1, idx, gate, b)
            torch.cuda.synchronize()
            assert torch.equal(a, b)
            st = ts.stats()
            assert st["demand_misses"] == misses, (ids, st)
        # after [4,0,1,2] the cache held {4,0,1,2}: [2,3,4,1] misses only expert 3, evicting 0
        assert st["demand_hits"] == 12 - 6
    finally:
        ts.close()
        res.close()


def test_banked_grouped_bf16():
    """Batched bf16 calls on a bank take the grouped tensor-core path for experts with >= 4
    tokens (its producer reads the records through the slot map) and the lookup path for the
    rest: routing and outputs equal the resident layers' bit for bit.  16 slots hold one layer's
    16 experts (a call touches at most min(T * k, E) of them), so two layers evict each other."""
    wb = synth.Workload("bankb", 512, 256, 16, 4, 32, "bf16", "zipf")
    res = [MoELayer(wb, 2, L, "cuda") for L in range(2)]
    ts = TieredStack(wb, 2, 2, 16)
    try:
        h = synth.hidden(6, wb.tokens, wb.d, "bf16", "cuda")
        T, k = wb.tokens, wb.top_k
        first_seen = 0
        for rep in range(2):
            for L in range(2):
                outs = []
                for ml in (res[L], ts.layers[L]):
                    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
                    gate = torch.empty(T, k, device="cuda")
                    out = torch.empty(T, wb.d, device="cuda")
                    ml.step(h, T, idx, gate, out, 0)
                    outs.append((idx, gate, out))
                torch.cuda.synchronize()
                for a, b in zip(*outs):
                    assert torch.equal(a, b)
                if rep == 0:
                    first_seen += len(torch.unique(outs[1][0]))
        st = ts.stats()
        assert st["demand_hits"] + st["demand_misses"] == 2 * 2 * T * k
        assert st["demand_misses"] >= first_seen  # every expert came in when first routed
        for ml in ts.layers:
            ml.stats()
    finally:
        ts.close()
        for l in res:
            l.close()
