"""waste_moe_forward_noalloc against waste_moe_forward, through the C ABI.

Some callers cannot allocate device memory: their serving engine owns all of
the GPU's memory and only hands out pointers, or they run where cudaMalloc is
not allowed.  The no-allocation entry point needs no handle and keeps its
partial sums in a fixed array inside the library's device image.  Each of two
calls in a row (the array keeps the previous call's contents) must match the
handle-based forward on the same inputs, within the tolerance the parity tests
use; for fp32 lookups, where the handle runs the gate/up and down units in one launch and
the no-allocation entry point runs them as two kernels, bit for bit.  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth
from rvq_compressed_expert_gb300.layer import MoELayer

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


def assert_close(got, ref):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= REL_L2, rel
    assert np.abs(got - ref).max() <= ELEM * np.abs(ref).max()


def two_calls(w, seeds, layer_seed=0, act="f32", exact=False):
    layer = MoELayer(w, layer_seed, 0, "cuda")
    try:
        idx, gate, logits, out_ref = layer.alloc_outputs(w.tokens)
        out_na = torch.empty_like(out_ref)
        for s in seeds:
            h = synth.hidden(s, w.tokens, w.d, act, "cuda")
            layer.route(h, w.tokens, idx, gate, logits)
            layer.forward(h, w.tokens, idx, gate, out_ref, 0)
            out_na.fill_(float("nan"))
            B.waste_moe_forward_noalloc(layer.cfg, layer.records, layer.stride, layer.codebooks,
                                        h, w.tokens, idx, gate, out_na, 0)
            torch.cuda.synchronize()
            assert_close(out_na, out_ref)
            if exact:
                # the handle runs the gate/up and down units in one launch, the no-allocation
                # entry point as two: the same units in the same order, so the same bits
                assert torch.equal(out_na.view(torch.int32), out_ref.view(torch.int32))
    finally:
        layer.close()


def test_noalloc_matches_forward_ragged_shapes():
    w = synth.Workload("ragged", 1032, 136, 12, 3, 5, "f32", "none")
    two_calls(w, seeds=(1, 2, 3), exact=True)


def test_noalloc_matches_forward_bf16():
    w = synth.Workload("ragged-bf16", 512, 264, 20, 5, 3, "bf16", "none")
    two_calls(w, seeds=(3, 4), act="bf16")


def test_noalloc_matches_forward_decode_shape():
    """The decode expert shape (d=7168, f=1536, top-16, one token): 16 slots fit the array."""
    w = synth.Workload("decode-e32", 7168, 1536, 32, 16, 1, "f32", "offsets")
    two_calls(w, seeds=(5, 6, 7), exact=True)


def test_noalloc_rejects_what_does_not_fit():
    """64 tokens x top-16 at the decode shape need about 264 MB of partial-sum scratch, far past
    the fixed array: refused on the host before anything is launched (the dummy buffers are
    never read)."""
    w = synth.Workload("decode-e32", 7168, 1536, 32, 16, 1, "f32", "offsets")
    T = 64
    cfg = B.make_config(w.d, w.f, w.n_experts, w.top_k, "f32", T)
    stride, _, _ = B.waste_moe_record_layout(cfg)
    dummy = B.aligned_bytes(4096, "cuda")
    with pytest.raises(B.WasteError) as ei:
        B.waste_moe_forward_noalloc(cfg, dummy, stride, dummy, dummy, T, dummy, dummy, dummy, 0)
    assert ei.value.status == -1
    assert "scratch" in ei.value.message
