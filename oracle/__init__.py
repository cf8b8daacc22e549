"""CPU oracle for the routed-expert RVQ MoE step -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline
leg may import this package.  It wraps ``oracle.c`` (plain single-threaded C,
double accumulation) with ctypes and composes its functions per token.  It
shares no code with the CUDA library and never calls it.

The pages describe the engine this step comes from:
"Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s" (sections "Quantification
et exactitude", "Lecture anticipée et prédiction du routeur", "Architecture
de streaming depuis le disque").  ``oracle.c`` cites the passage each
function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_lib/liboracle.so (gcc, -O2, no fast-math)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    """Declare the argument types of every exported oracle function on a loaded library."""
    lib.oracle_dequant.argtypes = [_i, _i, _fp, _u8p, _dp]
    lib.oracle_matvec_dense.argtypes = [_i, _i, _dp, _dp, _dp]
    lib.oracle_matvec_lut.argtypes = [_i, _i, _fp, _u8p, _dp, _dp]
    lib.oracle_router.argtypes = [_i, _i, _fp, _fp, _dp, _dp]
    lib.oracle_topk_softmax.argtypes = [_i, _i, _dp, _i32p, _dp]
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_expert_ffn.argtypes = [_i, _i, _fp, _u8p, _u8p, _u8p, _dp, _dp, _i]
    lib.oracle_combine.argtypes = [_i, _i, _dp, _dp, _dp, _dp]
    lib.oracle_moe_layer.argtypes = [_i, _i, _i, _i, _i, _fp, _fp, _fp, _u8p, _u8p, _u8p,
                                     _dp, _i, _i, _dp, _dp, _i32p, _dp]
    lib.oracle_rmsnorm.argtypes = [_i, _dp, _dp]
    lib.oracle_residual_layer.argtypes = [_i, _i, _i, _i, _i, _fp, _fp, _fp, _u8p, _u8p, _u8p,
                                          _dp, _i, _dp, _i32p, _dp]
    lib.oracle_expert_code_bytes.argtypes = [_i, _i]
    lib.oracle_expert_code_bytes.restype = ctypes.c_uint64
    lib.oracle_crc32.argtypes = [_u8p, ctypes.c_size_t]
    lib.oracle_rvq_nearest.argtypes = [_fp, _fp]
    lib.oracle_rvq_nearest.restype = ctypes.c_int
    lib.oracle_rvq_train.argtypes = [_i, _i, _fp, _i32p, _i, _fp, _u8p, _dp]
    lib.oracle_rvq_train.restype = ctypes.c_int
    lib.oracle_rvq_encode.argtypes = [_i, _i, _fp, _fp, _u8p, _dp]
    lib.oracle_rvq_encode.restype = ctypes.c_int
    lib.oracle_crc32.restype = ctypes.c_uint32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _np(a, dtype):
    """Contiguous numpy array of dtype from a numpy array or a CPU/GPU torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach()
        if a.dtype.is_floating_point and dtype in (np.float64, np.float32):
            a = a.to("cpu").double() if dtype == np.float64 else a.to("cpu").float()
        else:
            a = a.to("cpu")
        a = a.numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def dequant(cb, codes):
    """W [n_out, n_in] (float64) of one matrix: cb [3,256,8] fp32, codes [n_out,3,nv] u8."""
    cb = _np(cb, np.float32)
    codes = _np(codes, np.uint8)
    n_out, _, nv = codes.shape
    W = np.empty((n_out, nv * 8), np.float64)
    _load().oracle_dequant(n_out, nv * 8, _ptr(cb, ctypes.c_float), _ptr(codes, ctypes.c_uint8),
                           _ptr(W, ctypes.c_double))
    return W


def matvec_dense(W, x):
    W = _np(W, np.float64)
    x = _np(x, np.float64)
    y = np.empty(W.shape[0], np.float64)
    _load().oracle_matvec_dense(W.shape[0], W.shape[1], _ptr(W, ctypes.c_double),
                                _ptr(x, ctypes.c_double), _ptr(y, ctypes.c_double))
    return y


def matvec_lut(cb, codes, x):
    cb = _np(cb, np.float32)
    codes = _np(codes, np.uint8)
    x = _np(x, np.float64)
    n_out, _, nv = codes.shape
    y = np.empty(n_out, np.float64)
    _load().oracle_matvec_lut(n_out, nv * 8, _ptr(cb, ctypes.c_float), _ptr(codes, ctypes.c_uint8),
                              _ptr(x, ctypes.c_double), _ptr(y, ctypes.c_double))
    return y


def router(Wr, bias, h):
    """Logits [E] (float64) of one token."""
    Wr = _np(Wr, np.float32)
    h = _np(h, np.float64)
    E, d = Wr.shape
    b = None if bias is None else _np(bias, np.float32)
    out = np.empty(E, np.float64)
    _load().oracle_router(E, d, _ptr(Wr, ctypes.c_float),
                          None if b is None else _ptr(b, ctypes.c_float),
                          _ptr(h, ctypes.c_double), _ptr(out, ctypes.c_double))
    return out


def topk_softmax(logits, k):
    """(idx [k] int32 in rank order, gate [k] float64) of one token."""
    l = _np(logits, np.float64)
    idx = np.empty(k, np.int32)
    g = np.empty(k, np.float64)
    _load().oracle_topk_softmax(l.shape[0], k, _ptr(l, ctypes.c_double), _ptr(idx, ctypes.c_int32),
                                _ptr(g, ctypes.c_double))
    return idx, g


def silu(z: float) -> float:
    return _load().oracle_silu(float(z))


def expert_ffn(cb_e, gate_codes, up_codes, down_codes, x, use_lut=True):
    """y [d] (float64) of one expert on one token; cb_e [3,3,256,8]."""
    cb_e = _np(cb_e, np.float32)
    gc = _np(gate_codes, np.uint8)
    uc = _np(up_codes, np.uint8)
    dc = _np(down_codes, np.uint8)
    x = _np(x, np.float64)
    f = gc.shape[0]
    d = dc.shape[0]
    y = np.empty(d, np.float64)
    _load().oracle_expert_ffn(d, f, _ptr(cb_e, ctypes.c_float), _ptr(gc, ctypes.c_uint8),
                              _ptr(uc, ctypes.c_uint8), _ptr(dc, ctypes.c_uint8),
                              _ptr(x, ctypes.c_double), _ptr(y, ctypes.c_double), int(use_lut))
    return y


def combine(gate, ys, base=None):
    g = _np(gate, np.float64)
    ys = _np(ys, np.float64)
    k, d = ys.shape
    b = None if base is None else _np(base, np.float64)
    out = np.empty(d, np.float64)
    _load().oracle_combine(d, k, _ptr(g, ctypes.c_double), _ptr(ys, ctypes.c_double),
                           None if b is None else _ptr(b, ctypes.c_double),
                           _ptr(out, ctypes.c_double))
    return out


def crc32(data) -> int:
    """crc32 (IEEE 802.3 / zlib) of a byte string, numpy uint8 array or uint8 tensor."""
    if isinstance(data, (bytes, bytearray)):
        a = np.frombuffer(bytes(data), np.uint8)
    else:
        a = _np(data, np.uint8).reshape(-1)
    a = np.ascontiguousarray(a)
    return int(_load().oracle_crc32(_ptr(a, ctypes.c_uint8), a.size))


def rmsnorm(x):
    """x / sqrt(mean(x^2) + 1e-6) of one row (float64)."""
    x = _np(x, np.float64)
    out = np.empty_like(x)
    _load().oracle_rmsnorm(x.shape[0], _ptr(x, ctypes.c_double), _ptr(out, ctypes.c_double))
    return out


def residual_layer(h, Wr, bias, cbs, codes, k, use_lut=True):
    """One layer of the decode chain on all tokens: h_t <- h_t + MoE(rmsnorm(h_t)).

    h [T,d] (not modified); codes = (gate [E,f,3,d/8], up [E,f,3,d/8], down [E,d,3,f/8]).
    Returns dict(h [T,d] after the layer, logits [T,E], idx [T,k], gate [T,k]).
    """
    h = _np(h, np.float64).copy()
    Wr = _np(Wr, np.float32)
    cbs = _np(cbs, np.float32)
    gc, uc, dc = (_np(c, np.uint8) for c in codes)
    b = None if bias is None else _np(bias, np.float32)
    T, d = h.shape
    E = Wr.shape[0]
    f = gc.shape[1]
    logits = np.empty((T, E), np.float64)
    idx = np.empty((T, k), np.int32)
    gate = np.empty((T, k), np.float64)
    _load().oracle_residual_layer(T, d, f, E, k, _ptr(Wr, ctypes.c_float),
                                  None if b is None else _ptr(b, ctypes.c_float),
                                  _ptr(cbs, ctypes.c_float), _ptr(gc, ctypes.c_uint8),
                                  _ptr(uc, ctypes.c_uint8), _ptr(dc, ctypes.c_uint8),
                                  _ptr(h, ctypes.c_double), int(bool(use_lut)),
                                  _ptr(logits, ctypes.c_double), _ptr(idx, ctypes.c_int32),
                                  _ptr(gate, ctypes.c_double))
    return dict(h=h, logits=logits, idx=idx, gate=gate)


def stack_chain(h0, layers, k, n_layers=None):
    """Decode chain h <- h + MoE_L(rmsnorm(h)) over the given layers, in order.

    layers: list of (Wr, bias, cbs, codes) with codes = (gate, up, down) for all experts.
    Returns (final h [T,d], list of idx [T,k] per layer, list of logits [T,E] per layer).
    """
    h = _np(h0, np.float64).copy()
    idxs, logits = [], []
    for Wr, bias, cbs, codes in layers[:n_layers]:
        r = residual_layer(h, Wr, bias, cbs, codes, k)
        h = r["h"]
        idxs.append(r["idx"])
        logits.append(r["logits"])
    return h, idxs, logits


def stack_token(h_t, layers, k):
    """The same chain for one token, fetching only the selected experts' codes.

    layers: iterable of (Wr, bias, cbs, get_expert_codes) per layer, where cbs is
    [E,3,3,256,8] or a callable e -> [3,3,256,8] and get_expert_codes(e) returns
    (gate [f,3,d/8], up [f,3,d/8], down [d,3,f/8]).  Returns (final h [d], and per layer the
    lists of idx [k], gate [k] and logits [E]).
    """
    h = _np(h_t, np.float64).copy()
    idxs, gates, logits = [], [], []
    for Wr, bias, cbs, get_codes in layers:
        r = moe_token(rmsnorm(h), Wr, bias, cbs, get_codes, k)
        h = h + r["out"]
        idxs.append(r["idx"])
        gates.append(r["gate"])
        logits.append(r["logits"])
    return h, idxs, gates, logits


def expert_code_bytes(d: int, f: int) -> int:
    return int(_load().oracle_expert_code_bytes(d, f))


def moe_layer(h, Wr, bias, cbs, codes, k, residual=False, use_lut=True):
    """One layer over all tokens with every expert's arrays given.

    h [T,d]; codes = (gate [E,f,3,d/8], up [E,f,3,d/8], down [E,d,3,f/8]).
    Returns dict(out [T,d], logits [T,E], idx [T,k], gate [T,k]).
    """
    h = _np(h, np.float64)
    Wr = _np(Wr, np.float32)
    cbs = _np(cbs, np.float32)
    gc, uc, dc = (_np(c, np.uint8) for c in codes)
    b = None if bias is None else _np(bias, np.float32)
    T, d = h.shape
    E = Wr.shape[0]
    f = gc.shape[1]
    out = np.empty((T, d), np.float64)
    logits = np.empty((T, E), np.float64)
    idx = np.empty((T, k), np.int32)
    gate = np.empty((T, k), np.float64)
    _load().oracle_moe_layer(T, d, f, E, k, _ptr(Wr, ctypes.c_float),
                             None if b is None else _ptr(b, ctypes.c_float),
                             _ptr(cbs, ctypes.c_float), _ptr(gc, ctypes.c_uint8),
                             _ptr(uc, ctypes.c_uint8), _ptr(dc, ctypes.c_uint8),
                             _ptr(h, ctypes.c_double), int(bool(residual)), int(bool(use_lut)),
                             _ptr(out, ctypes.c_double), _ptr(logits, ctypes.c_double),
                             _ptr(idx, ctypes.c_int32), _ptr(gate, ctypes.c_double))
    return dict(out=out, logits=logits, idx=idx, gate=gate)


def moe_token(h_t, Wr, bias, cbs, get_expert_codes, k, residual=False, use_lut=True):
    """One layer for one token, fetching only the selected experts' codes.

    get_expert_codes(e) -> (gate [f,3,d/8], up [f,3,d/8], down [d,3,f/8]);
    cbs is [E,3,3,256,8] or a callable e -> [3,3,256,8].
    Returns dict(out [d], logits [E], idx [k], gate [k]).
    """
    h_t = _np(h_t, np.float64)
    logits = router(Wr, bias, h_t)
    idx, g = topk_softmax(logits, k)
    ys = np.empty((k, h_t.shape[0]), np.float64)
    for i, e in enumerate(idx.tolist()):
        cb_e = cbs(e) if callable(cbs) else cbs[e]
        gc, uc, dc = get_expert_codes(e)
        ys[i] = expert_ffn(cb_e, gc, uc, dc, h_t, use_lut)
    out = combine(g, ys, h_t if residual else None)
    return dict(out=out, logits=logits, idx=idx, gate=g)


def topk_margin(logits, k):
    """Smallest gap between adjacent ranks 1..k+1 of one token's logits (inf if k == E)."""
    l = np.sort(np.asarray(logits, np.float64))[::-1]
    m = min(k + 1, l.shape[0])
    if m < 2:
        return float("inf")
    return float(np.min(l[: m - 1] - l[1:m]))


def rvq_nearest(x, C) -> int:
    """Index of the codebook row of C [256, 8] nearest to x [8] (fp32 distance, lower index on
    ties)."""
    x = _np(x, np.float32)
    C = _np(C, np.float32)
    return int(_load().oracle_rvq_nearest(_ptr(x, ctypes.c_float), _ptr(C, ctypes.c_float)))


def rvq_train(W, init, iters: int):
    """Greedy residual k-means of W [rows, cols] fp32: returns (codebooks [3,256,8] fp32, codes
    [rows,3,cols/8] u8, err [3] float64 = sum of squared residuals after each stage).  init
    [3,256] int32: the vector index each stage's centroids start from.  Raises ValueError on
    refused inputs."""
    W = _np(W, np.float32)
    init = _np(init, np.int32)
    rows, cols = W.shape
    cb = np.zeros((3, 256, 8), np.float32)
    codes = np.zeros((rows, 3, max(cols // 8, 0)), np.uint8)
    err = np.zeros(3, np.float64)
    rc = _load().oracle_rvq_train(rows, cols, _ptr(W, ctypes.c_float), _ptr(init, ctypes.c_int32), int(iters),
                                  _ptr(cb, ctypes.c_float), _ptr(codes, ctypes.c_uint8), _ptr(err, ctypes.c_double))
    if rc:
        raise ValueError("rvq_train refused its inputs")
    return cb, codes, err


def rvq_encode(W, cb):
    """The three nearest-codebook assignments of W with given codebooks: (codes, err)."""
    W = _np(W, np.float32)
    cb = _np(cb, np.float32)
    rows, cols = W.shape
    codes = np.zeros((rows, 3, max(cols // 8, 0)), np.uint8)
    err = np.zeros(3, np.float64)
    rc = _load().oracle_rvq_encode(rows, cols, _ptr(W, ctypes.c_float), _ptr(cb, ctypes.c_float),
                                   _ptr(codes, ctypes.c_uint8), _ptr(err, ctypes.c_double))
    if rc:
        raise ValueError("rvq_encode refused its inputs")
    return codes, err
