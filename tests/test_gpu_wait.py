"""Bounded device waits: a wait whose counter is withheld gives up, the handle reports it,
and the GPU stays usable.

Work items of the persistent step kernel wait on one another through device counters; each
wait is bounded and a wait that gives up is latched and reported as WASTE_ETIMEOUT -- the
pages' rule of refusing rather than degrading (page "Exécuter Kimi K3 avec 29 Go de RAM à
0,50 tok/s", section "Budget RAM et zone de performance étroite").  Here the counter is one
the test owns and never sets, with a 1 ms limit: nothing faults or hangs.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth
from rvq_compressed_expert_gb300.layer import MoELayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rvq_compressed_expert_gb300 import _build
    _build.build()
    B.load()
    oracle.build()


def tiny_step_matches_oracle(layer, w):
    h = synth.hidden(0, w.tokens, w.d, w.act_dtype, "cuda")
    idx, gate, logits, out = layer.alloc_outputs(w.tokens)
    layer.step(h, w.tokens, idx, gate, out, 0, logits)
    torch.cuda.synchronize()
    li = synth.layer_inputs(w, 0, 0, "cuda")
    ref = oracle.moe_layer(h.cpu(), li.router_w.cpu(), li.router_b, li.codebooks.cpu(),
                           tuple(c.cpu() for c in li.codes), w.top_k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
    got = out.cpu().double().numpy()
    assert np.linalg.norm(got - ref["out"]) <= 1e-5 * np.linalg.norm(ref["out"])


def test_withheld_counter_times_out_and_is_reported():
    w = synth.WORKLOADS["tiny"]
    layer = MoELayer(w, 0, 0, "cuda")
    try:
        counter = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        B.waste_moe_debug_wait(layer.handle, counter, 1, 1_000_000)  # 1 ms, never satisfied
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
        assert waited < 0.5, f"the 1 ms wait took {waited:.3f} s"
        with pytest.raises(B.WasteError) as ei:
            layer.stats()
        assert ei.value.status == -6  # WASTE_ETIMEOUT
        # the latched error stays until reset; afterwards the handle works again
        with pytest.raises(B.WasteError):
            layer.stats()
        layer.reset_stats()
        layer.stats()
        tiny_step_matches_oracle(layer, w)
        layer.stats()
        # a counter that is given: the wait returns at once and latches nothing
        counter.fill_(3)
        B.waste_moe_debug_wait(layer.handle, counter, 2, 1_000_000_000)
        torch.cuda.synchronize()
        layer.stats()
    finally:
        layer.close()
    # a fresh handle on the same context computes as before
    fresh = MoELayer(w, 0, 0, "cuda")
    try:
        tiny_step_matches_oracle(fresh, w)
        fresh.stats()
    finally:
        fresh.close()


def test_wait_limit_is_honoured():
    """The wait gives up after its limit, not before: 20 ms withheld takes at least 20 ms."""
    w = synth.WORKLOADS["tiny"]
    layer = MoELayer(w, 0, 0, "cuda")
    try:
        counter = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        B.waste_moe_debug_wait(layer.handle, counter, 1, 20_000_000)
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
        assert 0.02 <= waited < 1.0, waited
        with pytest.raises(B.WasteError) as ei:
            layer.stats()
        assert ei.value.status == -6
    finally:
        layer.close()
