"""Seeded fuzz of tiny shapes: random (d, f, E, k, T), activation type, path flags and router
bias, each run through the C ABI and compared with the oracle on the same arrays.

Bars as in the parity tests: routing bit-exact where the oracle's top-k margin is clear;
outputs within relative L2 1e-5 on the fp32 lookup paths and 2e-3 where batched bf16 calls
send experts to the fp16 tensor-core path.
"""
import numpy as np
import pytest
import torch

import oracle
from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth
from rvq_compressed_expert_gb300.layer import MoELayer
from tests.test_gpu_parity import assert_close, check_routing

pytestmark = pytest.mark.gpu

FLAGS = [0, B.FLAG_FORCE_GEMV, B.FLAG_K2_RECONSTRUCT, B.FLAG_STEP_KERNEL, B.FLAG_FORCE_MMA]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rvq_compressed_expert_gb300 import _build
    _build.build()
    B.load()
    oracle.build()


def case(i):
    rng = np.random.default_rng(1000 + i)
    d = 8 * int(rng.integers(1, 161))
    f = 8 * int(rng.integers(1, 41))
    E = int(rng.integers(1, 41))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 7))
    act = ["f32", "bf16"][int(rng.integers(0, 2))]
    flags = FLAGS[int(rng.integers(0, len(FLAGS)))]
    bias = ["none", "offsets"][int(rng.integers(0, 2))]
    return d, f, E, k, T, act, flags, bias


@pytest.mark.parametrize("i", range(32))
def test_fuzz_case(i):
    d, f, E, k, T, act, flags, bias = case(i)
    w = synth.Workload("fuzz", d, f, E, k, T, act, bias)
    li = synth.layer_inputs(w, 50 + i, 0, "cpu", with_codes=True)
    h = synth.hidden(60 + i, T, d, act, "cpu")
    layer = MoELayer(w, 50 + i, 0, "cuda", inputs=li, flags=flags)
    try:
        idx, gate, logits, out = layer.alloc_outputs(T)
        layer.step(h.cuda(), T, idx, gate, out, 0, logits=logits)
        torch.cuda.synchronize()
        layer.stats()  # no device error
        ref = oracle.moe_layer(h, li.router_w, li.router_b, li.codebooks, li.codes, k)
        np.testing.assert_allclose(logits.cpu().numpy(), ref["logits"], rtol=1e-5, atol=1e-5)
        ok = check_routing(idx.cpu().numpy(), gate.cpu().numpy(), ref["logits"], k)
        if not ok:
            return  # every token's top-k within the rounding of its margin: routing checked above
        tc = act == "bf16" and (flags & B.FLAG_FORCE_MMA or (T > 1 and not flags & B.FLAG_FORCE_GEMV))
        tc = tc or bool(flags & B.FLAG_FORCE_MMA)
        got = out.cpu().numpy()[ok]
        if tc:
            assert_close(got, ref["out"][ok], rel=2e-3, elem=4e-3)
        else:
            assert_close(got, ref["out"][ok])
    finally:
        layer.close()
