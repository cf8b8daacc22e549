"""RVQ encoder on the device against the oracle's greedy residual k-means.

Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Quantification et
exactitude": 3 residual stages of 256 eight-dimensional vectors.  Codes and codebooks are
integers / values fixed by the encoder's rules (fp32 fused-multiply-add distances with
lower-index ties, exact fixed-point means), so they must match the oracle bit for bit; the
squared errors are sums in double taken in another order (relative 1e-9).
"""
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


def train_gpu(W, init, iters):
    rows, cols = W.shape
    cb = torch.empty(3, 256, 8, device="cuda")
    codes = torch.empty(rows, 3, cols // 8, dtype=torch.uint8, device="cuda")
    err = torch.empty(3, dtype=torch.float64, device="cuda")
    B.waste_rvq_train(W, init, iters, cb, codes, err)
    return cb.cpu().numpy(), codes.cpu().numpy(), err.cpu().numpy()


@pytest.mark.parametrize("iters", [0, 3])
@pytest.mark.parametrize("shape", [(64, 256), (37, 136), (5, 8), (300, 64)])
def test_train_matches_oracle(shape, iters):
    """Several CTAs and a ragged last one (2048, 629, 5 and 2400 vectors); 5 vectors for 256
    centroids makes every stage full of duplicate centroids (ties)."""
    rows, cols = shape
    W = synth.dense_matrix(1, 0, 0, 0, rows, cols, "cuda")
    init = synth.rvq_init(2, rows * cols // 8, "cuda")
    cb, codes, err = train_gpu(W, init, iters)
    ocb, ocodes, oerr = oracle.rvq_train(W.cpu().numpy(), init.cpu().numpy(), iters)
    assert np.array_equal(codes, ocodes)
    assert np.array_equal(cb, ocb)
    np.testing.assert_allclose(err, oerr, rtol=1e-9, atol=1e-30)


def test_encode_matches_oracle():
    W = synth.dense_matrix(3, 0, 0, 1, 96, 512, "cuda")
    cb = torch.randn(3, 256, 8, generator=torch.Generator("cuda").manual_seed(4), device="cuda") * 0.02
    codes = torch.empty(96, 3, 64, dtype=torch.uint8, device="cuda")
    err = torch.empty(3, dtype=torch.float64, device="cuda")
    B.waste_rvq_encode(W, cb, codes, err)
    ocodes, oerr = oracle.rvq_encode(W.cpu().numpy(), cb.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), ocodes)
    np.testing.assert_allclose(err.cpu().numpy(), oerr, rtol=1e-9)


def test_refusals():
    init = torch.zeros(3, 256, dtype=torch.int32, device="cuda")
    out = (torch.empty(3, 256, 8, device="cuda"), torch.empty(8, 3, 2, dtype=torch.uint8, device="cuda"),
           torch.empty(3, dtype=torch.float64, device="cuda"))
    W = torch.zeros(8, 16, device="cuda")
    W[3, 5] = float("nan")
    with pytest.raises(B.WasteError) as ei:
        B.waste_rvq_train(W, init, 1, *out)
    assert ei.value.status == -1
    W[3, 5] = 2.0 ** 22
    with pytest.raises(B.WasteError):
        B.waste_rvq_train(W, init, 1, *out)
    bad = init.clone()
    bad[1, 7] = 16
    with pytest.raises(B.WasteError):
        B.waste_rvq_train(torch.zeros(8, 16, device="cuda"), bad, 1, *out)
    with pytest.raises(B.WasteError):
        B.waste_rvq_train(torch.zeros(8, 12, device="cuda"), init, 1, *out)
    # after the refusals the device is fine and a valid call works
    B.waste_rvq_train(torch.zeros(8, 16, device="cuda") + 0.5, init, 1, *out)
    assert float(out[2].sum()) == 0.0


def test_mid_size_matches_oracle():
    """256 x 1024 (32,768 vectors, 64 CTAs x 2 rounds), 2 Lloyd rounds: bit-exact."""
    W = synth.dense_matrix(5, 0, 0, 2, 256, 1024, "cuda")
    init = synth.rvq_init(6, 256 * 128, "cuda")
    cb, codes, err = train_gpu(W, init, 2)
    ocb, ocodes, oerr = oracle.rvq_train(W.cpu().numpy(), init.cpu().numpy(), 2)
    assert np.array_equal(codes, ocodes) and np.array_equal(cb, ocb)
    np.testing.assert_allclose(err, oerr, rtol=1e-9)


def test_full_size_gate_matrix():
    """f x d = 1536 x 7168 (1.38M vectors), 4 Lloyd rounds: each stage's residual rebuilt in fp32
    from the codes; sampled vectors' codes are the oracle's nearest rows of the device's
    codebooks; the stage errors equal the rebuilt residuals' and fall stage by stage."""
    f, d = 1536, 7168
    W = synth.dense_matrix(7, 0, 0, 0, f, d, "cuda")
    init = synth.rvq_init(8, f * d // 8, "cuda")
    cb, codes, err = train_gpu(W, init, 4)
    R = W.cpu().numpy().reshape(-1, 8)
    rng = np.random.default_rng(9)
    sample = rng.choice(R.shape[0], 1500, replace=False)
    for s in range(3):
        c = codes[:, s, :].reshape(-1)
        for i in sample:
            assert oracle.rvq_nearest(R[i], cb[s]) == c[i]
        R = R - cb[s][c]
        e = float((R.astype(np.float64) ** 2).sum())
        assert abs(e - err[s]) <= 1e-9 * e
    total = float((W.double() ** 2).sum())
    assert total > err[0] > err[1] > err[2] > 0
    # 3 x 8 bits per 8 weights reconstruct N(0, 0.02^2) weights to a few percent
    assert err[2] / total < 0.05


def test_encoded_expert_through_the_path():
    """Dense gate/up/down encoded, packed and run through the expert kernels: the output equals
    the oracle's expert on the same codes, and is close to the dense expert."""
    d, f = 512, 256
    Ws = [synth.dense_matrix(10, 0, 0, k, *shape, "cuda") for k, shape in enumerate([(f, d), (f, d), (d, f)])]
    codes, cbs, rmse = [], [], []
    for k, W in enumerate(Ws):
        init = synth.rvq_init(11 + k, W.numel() // 8, "cuda")
        cb = torch.empty(3, 256, 8, device="cuda")
        c = torch.empty(W.shape[0], 3, W.shape[1] // 8, dtype=torch.uint8, device="cuda")
        err = torch.empty(3, dtype=torch.float64, device="cuda")
        B.waste_rvq_train(W, init, 3, cb, c, err)
        codes.append(c)
        cbs.append(cb)
        rmse.append((float(err[2]) / float((W.double() ** 2).sum())) ** 0.5)
    # Gaussian weights at 3 bits per weight: no code does better than the rate-distortion bound
    # D = sigma^2 2^(-2R), a relative rmse of 2^-3 (the codebooks' 6,144 values per matrix are
    # small next to the 131,072 weights); greedy k-means lands within 2x of it
    for r in rmse:
        assert 0.9 * 2.0 ** -3 < r < 2 * 2.0 ** -3, rmse
    w = synth.Workload("enc", d, f, 1, 1, 1, "f32", "none")
    li = synth.layer_inputs(w, 0, 0, "cuda", with_codes=False)
    li = synth.LayerInputs(li.router_w, li.router_b, torch.stack(cbs).unsqueeze(0).contiguous(), tuple(codes))
    layer = MoELayer(w, 0, 0, "cuda", inputs=li)
    try:
        x = synth.hidden(12, 1, d, "f32", "cuda")
        idx = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
        gate = torch.ones(1, 1, device="cuda")
        y = torch.empty(1, d, device="cuda")
        layer.forward(x, 1, idx, gate, y)
        torch.cuda.synchronize()
        yo = oracle.expert_ffn(li.codebooks[0].cpu(), *[c.cpu() for c in codes], x[0].cpu().double())
        got = y[0].cpu().double().numpy()
        assert np.linalg.norm(got - yo) <= 1e-5 * np.linalg.norm(yo)
        Wd = [W.cpu().double() for W in Ws]
        xd = x[0].cpu().double()
        zg, zu = Wd[0] @ xd, Wd[1] @ xd
        ydense = (Wd[2] @ (zg / (1 + torch.exp(-zg)) * zu)).numpy()
        rel = np.linalg.norm(got - ydense) / np.linalg.norm(ydense)
        # gate and up errors enter the SwiGLU product, the down error adds on top: about the sum
        # of the three relative errors
        assert rel < 1.5 * sum(rmse), (rel, rmse)
    finally:
        layer.close()
