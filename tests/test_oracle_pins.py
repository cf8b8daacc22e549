"""The CPU oracle against its pins (no GPU needed)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_mod):
    pin()


def test_tiny_layer_forms_agree(oracle_mod):
    """On the tiny workload the table form and the dense form give the same layer output."""
    from rvq_compressed_expert_gb300 import synth
    w = synth.WORKLOADS["tiny"]
    li = synth.layer_inputs(w, seed=0)
    h = synth.hidden(0, w.tokens, w.d, w.act_dtype)
    a = oracle_mod.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, w.top_k,
                             use_lut=True)
    b = oracle_mod.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, w.top_k,
                             use_lut=False)
    assert (a["idx"] == b["idx"]).all()
    num = ((a["out"] - b["out"]) ** 2).sum() ** 0.5
    den = (b["out"] ** 2).sum() ** 0.5
    assert num / den < 1e-12


def test_per_token_composition_matches_layer(oracle_mod):
    """moe_token (fetching only the selected experts) equals moe_layer on every token."""
    from rvq_compressed_expert_gb300 import synth
    w = synth.WORKLOADS["tiny"]
    li = synth.layer_inputs(w, seed=0)
    h = synth.hidden(0, w.tokens, w.d, w.act_dtype)
    full = oracle_mod.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, w.top_k,
                                residual=True)
    for t in range(w.tokens):
        r = oracle_mod.moe_token(h[t], li.router_w, li.router_b, li.codebooks,
                                 lambda e: (li.codes[0][e], li.codes[1][e], li.codes[2][e]),
                                 w.top_k, residual=True)
        assert (r["idx"] == full["idx"][t]).all()
        assert abs(r["out"] - full["out"][t]).max() < 1e-12


def test_stack_token_matches_chain(oracle_mod):
    """stack_token (one token, fetching only the selected experts) equals stack_chain on every
    token of a three-layer chain of the tiny workload's shapes."""
    from rvq_compressed_expert_gb300 import synth
    w = synth.WORKLOADS["tiny"]
    layers = [synth.layer_inputs(w, seed=0, layer=L) for L in range(3)]
    h = synth.hidden(0, w.tokens, w.d, w.act_dtype)
    full = [(li.router_w, li.router_b, li.codebooks, li.codes) for li in layers]
    h_all, idx_all, _ = oracle_mod.stack_chain(h, full, w.top_k)
    lazy = [(li.router_w, li.router_b, li.codebooks,
             (lambda li: lambda e: (li.codes[0][e], li.codes[1][e], li.codes[2][e]))(li)) for li in layers]
    for t in range(w.tokens):
        h_t, idxs, gates, _ = oracle_mod.stack_token(h[t], lazy, w.top_k)
        for L in range(3):
            assert (idxs[L] == idx_all[L][t]).all()
            assert abs(gates[L].sum() - 1.0) < 1e-12
        assert abs(h_t - h_all[t]).max() < 1e-12 * max(1.0, abs(h_all[t]).max())
