"""Pins of the CPU oracle to facts other than the oracle itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
a value fixed by the pages or by mathematics: the hand-worked example in
``golden/hand_2expert.txt``, closed forms, invariants, library routines
(numpy matmul, Python's stable sort) and brute force on tiny inputs.  The
set is chosen so that a plausible slip anywhere in the oracle (a dropped
stage or term, a wrong sign, index or tie order, a transposed operand)
fails at least one of them; ``test_oracle_mutants.py`` plants such slips in
a copy of the oracle and checks that they are caught.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- fixtures

def load_hand_example():
    """Parse golden/hand_2expert.txt into arrays (d = f = 8, E = 2)."""
    d = f = 8
    E = 2
    cb_one = np.zeros((3, 256, 8), np.float32)
    codes = {m: np.zeros((E, 8, 3, 1), np.uint8) for m in range(3)}
    Wr = np.zeros((E, d), np.float32)
    h = None
    expect = {}
    with open(os.path.join(GOLDEN, "hand_2expert.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "codebook":
                s, c = int(tok[1]), int(tok[2])
                cb_one[s, c] = [float(v) for v in tok[3:11]]
            elif tok[0] == "code":
                e, m, r = int(tok[1]), int(tok[2]), int(tok[3])
                codes[m][e, r, :, 0] = [int(v) for v in tok[4:7]]
            elif tok[0] == "router":
                Wr[int(tok[1])] = [float(v) for v in tok[2:10]]
            elif tok[0] == "hidden":
                h = np.array([float(v) for v in tok[1:9]], np.float64)
            elif tok[0] == "expect":
                expect[tok[1]] = np.array([float(v) for v in tok[2:]], np.float64)
    cbs = np.broadcast_to(cb_one, (E, 3, 3, 256, 8)).copy()
    return dict(d=d, f=f, E=E, cbs=cbs, codes=(codes[0], codes[1], codes[2]), Wr=Wr, h=h,
                expect=expect)


def _rand_matrix(rng, n_out, n_in):
    cb = (rng.standard_normal((3, 256, 8)) * np.array([0.02, 0.01, 0.005])[:, None, None]
          ).astype(np.float32)
    codes = rng.integers(0, 256, (n_out, 3, n_in // 8), dtype=np.uint8)
    return cb, codes


def _rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- pins

def pin_hand_example_layer():
    """Hand-worked 2-expert example: exact tie, k = 2 and k = 1, both product forms."""
    ex = load_hand_example()
    for use_lut in (True, False):
        for k in (2, 1):
            r = oracle.moe_layer(ex["h"][None], ex["Wr"], None, ex["cbs"], ex["codes"], k,
                                 use_lut=use_lut)
            np.testing.assert_allclose(r["logits"][0], ex["expect"]["logits"], rtol=0, atol=0)
            np.testing.assert_array_equal(r["idx"][0], ex["expect"][f"idx_k{k}"].astype(np.int32))
            np.testing.assert_allclose(r["gate"][0], ex["expect"][f"gate_k{k}"], rtol=0, atol=1e-15)
            np.testing.assert_allclose(r["out"][0], ex["expect"][f"out_k{k}"], rtol=1e-14, atol=1e-14)


def pin_hand_example_experts():
    """Each expert of the hand example on its own matches the worked values."""
    ex = load_hand_example()
    for e in range(2):
        for use_lut in (True, False):
            y = oracle.expert_ffn(ex["cbs"][e], ex["codes"][0][e], ex["codes"][1][e],
                                  ex["codes"][2][e], ex["h"], use_lut)
            np.testing.assert_allclose(y, ex["expect"][f"y_expert{e}"], rtol=1e-14, atol=1e-14)


def pin_chain_hand_example():
    """Two chained copies of the hand example (h <- h + MoE(rmsnorm(h))), worked by hand in
    the golden file: layer-by-layer h, layer 2's logits, gates and routing, k = 2 and k = 1."""
    ex = load_hand_example()
    X = ex["expect"]
    layer = (ex["Wr"], None, ex["cbs"], ex["codes"])
    for k in (2, 1):
        r1 = oracle.residual_layer(ex["h"][None], *layer, k)
        np.testing.assert_array_equal(r1["idx"][0], np.arange(k, dtype=np.int32))
        np.testing.assert_allclose(r1["h"][0], X[f"chain_h1_k{k}"], rtol=1e-14, atol=1e-14)
        r2 = oracle.residual_layer(r1["h"], *layer, k)
        np.testing.assert_array_equal(r2["idx"][0], np.arange(k, dtype=np.int32))
        np.testing.assert_allclose(r2["logits"][0], X[f"chain_logits2_k{k}"], rtol=1e-14, atol=1e-14)
        if k == 2:
            np.testing.assert_allclose(r2["gate"][0], X["chain_gate2_k2"], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(r2["h"][0], X[f"chain_h2_k{k}"], rtol=1e-14, atol=1e-14)
        h2, idxs, logits = oracle.stack_chain(ex["h"][None], [layer, layer], k)
        np.testing.assert_allclose(h2[0], X[f"chain_h2_k{k}"], rtol=1e-14, atol=1e-14)
        assert len(idxs) == 2 and len(logits) == 2


def pin_chain_zero_codebooks():
    """Layers whose codebooks are all zero give zero expert outputs, so the chain leaves h
    exactly as it was (whatever the routing)."""
    rng = np.random.default_rng(11)
    T, d, f, E, k = 3, 64, 32, 6, 2
    layers = []
    for _ in range(3):
        Wr = rng.standard_normal((E, d)).astype(np.float32)
        b = rng.standard_normal(E).astype(np.float32)
        cbs = np.zeros((E, 3, 3, 256, 8), np.float32)
        codes = (rng.integers(0, 256, (E, f, 3, d // 8), dtype=np.uint8),
                 rng.integers(0, 256, (E, f, 3, d // 8), dtype=np.uint8),
                 rng.integers(0, 256, (E, d, 3, f // 8), dtype=np.uint8))
        layers.append((Wr, b, cbs, codes))
    h0 = rng.standard_normal((T, d))
    h, idxs, _ = oracle.stack_chain(h0, layers, k)
    np.testing.assert_array_equal(h, h0)
    assert len(idxs) == 3


def pin_dequant_stage_placement():
    """Closed form: with stage-s codebook entry c equal to c * 256**s on component s
    (zero elsewhere), W[r][8j+s] is code_s(r, j) * 256**s and every other weight is 0."""
    rng = np.random.default_rng(1)
    n_out, n_in = 24, 40
    cb = np.zeros((3, 256, 8), np.float32)
    for s in range(3):
        cb[s, :, s] = np.arange(256, dtype=np.float32) * float(256 ** s)
    codes = rng.integers(0, 256, (n_out, 3, n_in // 8), dtype=np.uint8)
    W = oracle.dequant(cb, codes)
    expect = np.zeros((n_out, n_in))
    for r in range(n_out):
        for j in range(n_in // 8):
            for s in range(3):
                expect[r, 8 * j + s] = float(codes[r, s, j]) * 256.0 ** s
    np.testing.assert_array_equal(W, expect)


def pin_dequant_residual_sum():
    """Residual stages add: W from all three stages equals the sum of W from each stage alone."""
    rng = np.random.default_rng(2)
    cb, codes = _rand_matrix(rng, 16, 32)
    parts = []
    for s in range(3):
        cb_s = np.zeros_like(cb)
        cb_s[s] = cb[s]
        parts.append(oracle.dequant(cb_s, codes))
    np.testing.assert_allclose(oracle.dequant(cb, codes), parts[0] + parts[1] + parts[2],
                               rtol=1e-15, atol=1e-18)


def pin_matvec_dense_library():
    """Dense product against numpy's matmul."""
    rng = np.random.default_rng(3)
    W = rng.standard_normal((37, 53))
    x = rng.standard_normal(53)
    np.testing.assert_allclose(oracle.matvec_dense(W, x), W @ x, rtol=1e-12, atol=1e-12)


def pin_lut_equals_dequant():
    """The pages' table form equals dequantise-then-multiply (numpy matmul) on tiny shapes."""
    rng = np.random.default_rng(4)
    for n_out, n_in in ((8, 8), (16, 16), (5, 64), (33, 256), (64, 8)):
        cb, codes = _rand_matrix(rng, n_out, n_in)
        x = rng.standard_normal(n_in)
        W = oracle.dequant(cb, codes)
        assert _rel(oracle.matvec_lut(cb, codes, x), W @ x) < 1e-12


def pin_lut_unit_vectors():
    """Brute force: the table form applied to unit vector e_i returns column i of W."""
    rng = np.random.default_rng(5)
    cb, codes = _rand_matrix(rng, 7, 24)
    W = oracle.dequant(cb, codes)
    for i in range(24):
        x = np.zeros(24)
        x[i] = 1.0
        np.testing.assert_allclose(oracle.matvec_lut(cb, codes, x), W[:, i], rtol=1e-13, atol=1e-16)


def pin_router_library():
    """Router logits against numpy: W_r h + b, with and without bias."""
    rng = np.random.default_rng(6)
    Wr = rng.standard_normal((11, 40)).astype(np.float32)
    b = rng.standard_normal(11).astype(np.float32)
    h = rng.standard_normal(40)
    np.testing.assert_allclose(oracle.router(Wr, None, h), Wr.astype(np.float64) @ h, rtol=1e-12)
    np.testing.assert_allclose(oracle.router(Wr, b, h), Wr.astype(np.float64) @ h + b, rtol=1e-12)


def pin_topk_against_sort():
    """Top-k against Python's stable sort on key (-logit, index), ties and +-0 included."""
    rng = np.random.default_rng(7)
    cases = [rng.standard_normal(8), rng.integers(-2, 3, 16).astype(np.float64),
             np.array([0.0, -0.0, 0.0, -0.0, 1.0, 1.0, -1.0]), np.ones(5),
             rng.standard_normal(64)]
    for l in cases:
        order = sorted(range(len(l)), key=lambda e: (-l[e], e))
        for k in range(1, len(l) + 1):
            idx, _ = oracle.topk_softmax(l, k)
            assert idx.tolist() == order[:k], (l, k)


def pin_topk_exhaustive_small():
    """Brute force over all 2-subsets of 8 experts: the chosen pair is the one whose
    smaller logit beats every logit outside it."""
    rng = np.random.default_rng(8)
    for _ in range(20):
        l = rng.standard_normal(8)
        best = [S for S in itertools.combinations(range(8), 2)
                if min(l[list(S)]) > max(l[[e for e in range(8) if e not in S]])]
        assert len(best) == 1
        idx, _ = oracle.topk_softmax(l, 2)
        assert sorted(idx.tolist()) == list(best[0])
        assert l[idx[0]] >= l[idx[1]]


def pin_gate_invariants():
    """Gates sum to 1; k = 1 gives exactly 1; equal logits give 1/k; ratios are exp of gaps."""
    rng = np.random.default_rng(9)
    l = rng.standard_normal(32) * 3
    idx, g = oracle.topk_softmax(l, 6)
    assert abs(g.sum() - 1.0) < 1e-15
    for a in range(6):
        for b in range(6):
            assert abs(g[a] / g[b] - math.exp(l[idx[a]] - l[idx[b]])) < 1e-12 * max(1, g[a] / g[b])
    _, g1 = oracle.topk_softmax(l, 1)
    assert g1[0] == 1.0
    _, geq = oracle.topk_softmax(np.full(9, 0.25), 4)
    np.testing.assert_allclose(geq, np.full(4, 0.25), rtol=0, atol=1e-16)
    assert np.all(np.diff(g) <= 0)


def pin_silu_closed_forms():
    """silu(0) = 0; silu(x) - silu(-x) = x; silu(ln 3) = 0.75 ln 3; silu(x) -> x for large x."""
    assert oracle.silu(0.0) == 0.0
    for x in (0.1, 0.7, 2.5, 9.0):
        assert abs(oracle.silu(x) - oracle.silu(-x) - x) < 1e-14 * max(1, x)
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12


def pin_swiglu_roles():
    """Gate and up play different roles: with U = 0 the output is 0 whatever G is, and
    with the gate matrix zero the output is 0 too (silu(0) = 0)."""
    rng = np.random.default_rng(10)
    d, f = 16, 8
    cb = np.stack([_rand_matrix(rng, 1, 8)[0] for _ in range(3)])
    gc = rng.integers(0, 256, (f, 3, d // 8), dtype=np.uint8)
    uc = rng.integers(0, 256, (f, 3, d // 8), dtype=np.uint8)
    dc = rng.integers(0, 256, (d, 3, f // 8), dtype=np.uint8)
    x = rng.standard_normal(d)
    for zero_mat in (0, 1):
        cbz = cb.copy()
        cbz[zero_mat] = 0
        assert np.all(oracle.expert_ffn(cbz, gc, uc, dc, x) == 0.0)
    # and the full product against a numpy composition of the dequantised matrices
    G = oracle.dequant(cb[0], gc)
    U = oracle.dequant(cb[1], uc)
    D = oracle.dequant(cb[2], dc)
    zg = G @ x
    a = zg / (1 + np.exp(-zg)) * (U @ x)
    assert _rel(oracle.expert_ffn(cb, gc, uc, dc, x), D @ a) < 1e-12


def pin_down_linearity():
    """Doubling the down codebooks doubles the expert output exactly."""
    rng = np.random.default_rng(11)
    d, f = 24, 16
    cb = np.stack([_rand_matrix(rng, 1, 8)[0] for _ in range(3)])
    gc = rng.integers(0, 256, (f, 3, d // 8), dtype=np.uint8)
    uc = rng.integers(0, 256, (f, 3, d // 8), dtype=np.uint8)
    dc = rng.integers(0, 256, (d, 3, f // 8), dtype=np.uint8)
    x = rng.standard_normal(d)
    cb2 = cb.copy()
    cb2[2] *= 2
    np.testing.assert_array_equal(oracle.expert_ffn(cb2, gc, uc, dc, x),
                                  2 * oracle.expert_ffn(cb, gc, uc, dc, x))


def pin_combine():
    """Combine: k = 1 with gate 1 returns y; the base is added; gates weight the outputs."""
    rng = np.random.default_rng(12)
    ys = rng.standard_normal((3, 10))
    base = rng.standard_normal(10)
    np.testing.assert_array_equal(oracle.combine([1.0], ys[:1]), ys[0])
    np.testing.assert_allclose(oracle.combine([0.2, 0.3, 0.5], ys, base),
                               base + 0.2 * ys[0] + 0.3 * ys[1] + 0.5 * ys[2], rtol=1e-14)


def pin_code_bytes_match_pages():
    """Per-token expert bytes: 16 experts x 92 layers of 3-bit codes at K3's shapes
    (d = 7168, f = 1536) come to 16.98 GiB, the pages' "17.0 GB" per token; one expert's
    codes fill exactly 3024 pages of 4 KiB."""
    b = oracle.expert_code_bytes(7168, 1536)
    assert b == 12_386_304
    assert b % 4096 == 0 and b // 4096 == 3024
    assert abs(16 * 92 * b / 2 ** 30 - 17.0) < 0.05


def pin_rmsnorm():
    """RMS normalisation: a constant vector c maps to sign(c) (up to the 1e-6 floor), the
    output's mean square is 1 up to the floor, and scaling the input does not change it."""
    for c in (3.0, -0.5):
        out = oracle.rmsnorm(np.full(16, c))
        np.testing.assert_allclose(out, np.sign(c) * abs(c) / math.sqrt(c * c + 1e-6), rtol=1e-14)
    rng = np.random.default_rng(13)
    x = rng.standard_normal(100) * 5
    out = oracle.rmsnorm(x)
    ms = float(np.mean(x * x))
    assert abs(float(np.mean(out * out)) - ms / (ms + 1e-6)) < 1e-13
    np.testing.assert_allclose(oracle.rmsnorm(4 * x), out, rtol=1e-7)


def pin_crc32():
    """crc32: the standard check value of "123456789" (0xCBF43926), the empty string, and
    zlib's crc32 on random byte strings of several lengths."""
    import zlib
    assert oracle.crc32(b"123456789") == 0xCBF43926
    assert oracle.crc32(b"") == 0
    rng = np.random.default_rng(14)
    for n in (1, 7, 4096, 10000):
        a = rng.integers(0, 256, n, dtype=np.uint8)
        assert oracle.crc32(a) == zlib.crc32(a.tobytes())


def _rvq_data(rng, rows, cols, scale=0.02):
    return (rng.standard_normal((rows, cols)) * scale).astype(np.float32)


def pin_rvq_nearest():
    """Nearest codebook row: equals the float64 argmin wherever the best two distances are
    apart by more than fp32 rounding; a row equal to x wins with distance 0; among equal rows
    the lower index wins."""
    rng = np.random.default_rng(21)
    checked = 0
    for _ in range(300):
        C = rng.standard_normal((256, 8)).astype(np.float32)
        x = rng.standard_normal(8).astype(np.float32)
        d = ((x.astype(np.float64) - C.astype(np.float64)) ** 2).sum(1)
        o = np.argsort(d)
        if d[o[1]] - d[o[0]] > 1e-5 * d[o[1]]:
            assert oracle.rvq_nearest(x, C) == o[0]
            checked += 1
    assert checked > 250
    C = rng.standard_normal((256, 8)).astype(np.float32)
    assert oracle.rvq_nearest(C[77], C) == 77
    C[200] = C[31]
    assert oracle.rvq_nearest(C[31] + np.float32(1e-3), C) == 31
    C[:] = C[5]
    assert oracle.rvq_nearest(rng.standard_normal(8).astype(np.float32), C) == 0


def pin_rvq_exact_for_few_distinct_vectors():
    """A matrix built from 200 distinct vectors, each stage-0 centroid started on one of them:
    stage 0 reproduces every vector exactly (residual 0, later stages add zeros), so the codes
    dequantise to W exactly and each code names a row equal to its vector."""
    rng = np.random.default_rng(22)
    base = (rng.standard_normal((200, 8)) * 0.05).astype(np.float32)
    pick = rng.integers(0, 200, 24 * 40)
    pick[:200] = rng.permutation(200)
    W = base[pick].reshape(24, 320)
    first = {int(b): i for i, b in reversed(list(enumerate(pick)))}
    init = np.zeros((3, 256), np.int32)
    init[0, :200] = [first[b] for b in range(200)]
    init[0, 200:] = rng.integers(0, len(pick), 56)
    init[1:] = rng.integers(0, len(pick), (2, 256))
    cb, codes, err = oracle.rvq_train(W, init, 3)
    assert err[0] == 0.0 and err[1] == 0.0 and err[2] == 0.0
    assert np.array_equal(oracle.dequant(cb, codes), W.astype(np.float64))
    for r, j in [(0, 0), (5, 17), (23, 39)]:
        assert np.array_equal(cb[0, codes[r, 0, j]], W[r, 8 * j:8 * j + 8])


def pin_rvq_residual_bookkeeping():
    """err[2] equals the squared difference between W and the codes dequantised stage by stage
    in fp32 (((w - c0) - c1) - c2), and the stage errors fall; encoding with the trained
    codebooks gives the same codes and errors (the final assignments)."""
    rng = np.random.default_rng(23)
    W = _rvq_data(rng, 40, 96)
    init = rng.integers(0, 40 * 12, (3, 256)).astype(np.int32)
    cb, codes, err = oracle.rvq_train(W, init, 4)
    nv = 12
    R = W.reshape(40, nv, 8).copy()
    for s_ in range(3):
        R = R - cb[s_][codes[:, s_, :]]
        e = float((R.astype(np.float64) ** 2).sum())
        assert abs(e - err[s_]) <= 1e-12 * max(e, 1e-30)
    assert err[0] > err[1] > err[2] >= 0
    assert err[0] < float((W.astype(np.float64) ** 2).sum())
    c2, e2 = oracle.rvq_encode(W, cb)
    assert np.array_equal(c2, codes) and np.array_equal(e2, err)
    # with no Lloyd round each stage's codebook is its residual at the init indices
    cb0, codes0, _ = oracle.rvq_train(W, init, 0)
    R = W.reshape(-1, 8).copy()
    for s_ in range(3):
        assert np.array_equal(cb0[s_], R[init[s_]])
        R = R - cb0[s_][codes0[:, s_, :].reshape(-1)]


def pin_rvq_lloyd_monotone_and_means():
    """Lloyd rounds never raise the stage-0 error (beyond the 2^-40 rounding of the means);
    after enough rounds the assignment is stable, and then every used centroid is the mean of
    its members (float64 mean, to the fixed-point rounding)."""
    rng = np.random.default_rng(24)
    W = _rvq_data(rng, 64, 64)
    init = rng.integers(0, 512, (3, 256)).astype(np.int32)
    errs = [oracle.rvq_train(W, init, it)[2][0] for it in range(6)]
    for a, b in zip(errs, errs[1:]):
        assert b <= a * (1 + 1e-12)
    assert errs[-1] < errs[0]
    cb, codes, _ = oracle.rvq_train(W, init, 60)
    V = W.reshape(-1, 8).astype(np.float64)
    c0 = codes[:, 0, :].reshape(-1)
    used = np.unique(c0)
    assert len(used) > 100
    for c in used[:64]:
        m = V[c0 == c].mean(0)
        assert np.all(np.abs(cb[0, c] - m) <= 2.0 ** -40 + 2.0 ** -24 * np.abs(m) + 1e-30)


def pin_rvq_refusals():
    """cols not a multiple of 8, a non-finite or too large weight, an init index outside the
    vectors: refused."""
    rng = np.random.default_rng(25)
    init = np.zeros((3, 256), np.int32)
    for W in (_rvq_data(rng, 4, 12), np.full((2, 8), np.nan, np.float32),
              np.full((2, 8), 2.0 ** 22, np.float32)):
        try:
            oracle.rvq_train(W, init, 1)
        except ValueError:
            pass
        else:
            raise AssertionError("accepted")
    bad = init.copy()
    bad[2, 3] = 2
    try:
        oracle.rvq_train(_rvq_data(rng, 1, 16), bad, 1)
    except ValueError:
        pass
    else:
        raise AssertionError("accepted")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
