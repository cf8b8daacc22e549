"""ctypes binding of libwaste_moe (include/waste_moe.h): same names, argument marshalling only.

Tensors are passed as torch tensors (their data pointers are handed to the
library) or as raw integer addresses; streams as ``torch.cuda.Stream``, an
integer handle, or None for torch's current stream.  Every compute step runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback: if the
library has not been built, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libwaste_moe.so")

ABI_VERSION = 1
ACT_F32, ACT_BF16 = 0, 1
FLAG_VERIFY_CRC = 1 << 0
FLAG_FORCE_GEMV = 1 << 2
FLAG_FORCE_MMA = 1 << 3
FLAG_K2_RECONSTRUCT = 1 << 4
FLAG_STEP_KERNEL = 1 << 5
FLAG_BANK_SERIAL = 1 << 6
RECORD_ALIGN = 4096
RECORD_MAGIC = 0x454F4D57

STATUS = {0: "WASTE_OK", -1: "WASTE_EINVAL", -2: "WASTE_ENOMEM", -3: "WASTE_ECUDA",
          -4: "WASTE_ELAYOUT", -5: "WASTE_ECRC", -6: "WASTE_ETIMEOUT", -7: "WASTE_ENOTIMPL"}

EXPORTED = ["waste_moe_record_layout", "waste_moe_pack_records", "waste_moe_create",
            "waste_moe_route", "waste_moe_forward", "waste_moe_prefetch", "waste_moe_destroy",
            "waste_moe_stats", "waste_moe_reset_stats", "waste_moe_last_error",
            "waste_moe_topk_from_logits", "waste_moe_set_profiling", "waste_moe_read_profile",
            "waste_moe_rmsnorm", "waste_moe_forward_noalloc", "waste_moe_step", "waste_moe_set_trace",
            "waste_bank_create", "waste_bank_destroy", "waste_bank_reset", "waste_bank_stats",
            "waste_moe_set_lookahead",
            "waste_moe_create_banked", "waste_rvq_train", "waste_rvq_encode", "waste_moe_debug_wait"]


class waste_moe_config(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_uint32), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("lookahead", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("layer", ctypes.c_int32)]


class waste_record_header(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32),
                ("layer", ctypes.c_int32), ("expert_id", ctypes.c_int32),
                ("d", ctypes.c_int32), ("f", ctypes.c_int32), ("n_stages", ctypes.c_int32),
                ("codebook_size", ctypes.c_int32), ("vec", ctypes.c_int32),
                ("layout_id", ctypes.c_uint32), ("section_offset", ctypes.c_uint64 * 3),
                ("section_bytes", ctypes.c_uint64 * 3), ("record_bytes", ctypes.c_uint64),
                ("payload_crc32", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class waste_moe_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "demand_code_bytes", "codebook_bytes", "router_bytes", "prefetch_issued_bytes",
        "prefetch_experts", "prediction_hits", "routed_slots", "forward_slots")]


class waste_bank_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "demand_hits", "demand_misses", "prefetch_copies", "prefetch_present", "copied_bytes")]


class WasteError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (no build step here: a missing library is an error)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libwaste_moe.so not found at {path}; build it first "
                           "(rvq_compressed_expert_gb300._build.build())")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    cfgp = ctypes.POINTER(waste_moe_config)
    lib.waste_moe_record_layout.argtypes = [cfgp, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                            ctypes.POINTER(sz)]
    lib.waste_moe_pack_records.argtypes = [cfgp, i32, i32, i32, vp, vp, vp, vp, sz, i32, vp]
    lib.waste_moe_create.argtypes = [cfgp, vp, vp, vp, sz, vp, ctypes.POINTER(vp)]
    lib.waste_moe_route.argtypes = [vp, vp, i32, vp, vp, vp, vp]
    lib.waste_moe_forward.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp]
    lib.waste_moe_prefetch.argtypes = [vp, vp, i32, i32, vp]
    lib.waste_moe_destroy.argtypes = [vp]
    lib.waste_moe_destroy.restype = None
    lib.waste_moe_stats.argtypes = [vp, ctypes.POINTER(waste_moe_stats_t)]
    lib.waste_moe_reset_stats.argtypes = [vp]
    lib.waste_moe_last_error.argtypes = []
    lib.waste_moe_last_error.restype = ctypes.c_char_p
    lib.waste_moe_topk_from_logits.argtypes = [vp, i32, i32, i32, vp, vp, vp]
    lib.waste_moe_set_profiling.argtypes = [vp, i32]
    lib.waste_moe_read_profile.argtypes = [vp, ctypes.POINTER(ctypes.c_float)]
    lib.waste_moe_rmsnorm.argtypes = [vp, vp, i32, i32, vp]
    lib.waste_moe_step.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, vp]
    lib.waste_moe_set_trace.argtypes = [vp, vp, i32]
    lib.waste_moe_set_lookahead.argtypes = [vp, vp, i32]
    lib.waste_moe_forward_noalloc.argtypes = [cfgp, vp, sz, vp, vp, i32, vp, vp, vp, i32, vp]
    lib.waste_bank_create.argtypes = [cfgp, i32, vp, sz, i32, ctypes.POINTER(vp)]
    lib.waste_bank_destroy.argtypes = [vp]
    lib.waste_bank_destroy.restype = None
    lib.waste_bank_reset.argtypes = [vp]
    lib.waste_bank_stats.argtypes = [vp, ctypes.POINTER(waste_bank_stats_t)]
    lib.waste_moe_create_banked.argtypes = [cfgp, vp, vp, vp, i32, vp, ctypes.POINTER(vp)]
    lib.waste_rvq_train.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp]
    lib.waste_rvq_encode.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    lib.waste_moe_debug_wait.argtypes = [vp, vp, ctypes.c_uint32, ctypes.c_uint64, vp]
    for name in EXPORTED:
        if name not in ("waste_moe_destroy", "waste_moe_last_error", "waste_bank_destroy"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int):
    if rc != 0:
        raise WasteError(rc, load().waste_moe_last_error().decode())
    return rc


def make_config(d, f, n_experts, top_k, act_dtype="f32", max_tokens=1, lookahead=6, flags=0,
                layer=-1) -> waste_moe_config:
    return waste_moe_config(ABI_VERSION, d, f, n_experts, top_k,
                            ACT_BF16 if act_dtype == "bf16" else ACT_F32, max_tokens, lookahead,
                            flags, layer)


def waste_moe_last_error() -> str:
    return load().waste_moe_last_error().decode()


def waste_moe_record_layout(cfg: waste_moe_config):
    """(stride, [section offsets], [section bytes])."""
    st = ctypes.c_size_t()
    off = (ctypes.c_size_t * 3)()
    by = (ctypes.c_size_t * 3)()
    _check(load().waste_moe_record_layout(ctypes.byref(cfg), ctypes.byref(st), off, by))
    return st.value, list(off), list(by)


def waste_moe_pack_records(cfg, layer, expert_begin, n_experts, gate_codes, up_codes, down_codes,
                           records, record_stride, compute_crc=0, stream=None):
    return _check(load().waste_moe_pack_records(
        ctypes.byref(cfg), layer, expert_begin, n_experts, _ptr(gate_codes), _ptr(up_codes),
        _ptr(down_codes), _ptr(records), record_stride, compute_crc, _stream(stream)))


def waste_moe_create(cfg, router_w, router_bias, records, record_stride, codebooks) -> int:
    out = ctypes.c_void_p()
    _check(load().waste_moe_create(ctypes.byref(cfg), _ptr(router_w), _ptr(router_bias),
                                   _ptr(records), record_stride, _ptr(codebooks),
                                   ctypes.byref(out)))
    return out.value


def waste_moe_route(h, d_h, T, d_idx, d_gate, d_logits=None, stream=None):
    return _check(load().waste_moe_route(h, _ptr(d_h), T, _ptr(d_idx), _ptr(d_gate),
                                         _ptr(d_logits), _stream(stream)))


def waste_moe_forward(h, d_h, T, d_idx, d_gate, d_out, mode=0, stream=None):
    return _check(load().waste_moe_forward(h, _ptr(d_h), T, _ptr(d_idx), _ptr(d_gate),
                                           _ptr(d_out), mode, _stream(stream)))


def waste_moe_step(h, d_h, T, d_idx, d_gate, d_logits, d_out, mode=0, stream=None):
    return _check(load().waste_moe_step(h, _ptr(d_h), T, _ptr(d_idx), _ptr(d_gate), _ptr(d_logits),
                                        _ptr(d_out), mode, _stream(stream)))


def waste_moe_set_trace(h, d_trace, n_items):
    """Record {start ns, end ns, SM, CTA} per work item of the step kernel into d_trace."""
    return _check(load().waste_moe_set_trace(h, _ptr(d_trace), n_items))


def waste_moe_prefetch(next_layer, d_h, T, n_prefetch=-1, side=None):
    return _check(load().waste_moe_prefetch(next_layer, _ptr(d_h), T, n_prefetch, _stream(side)))


def waste_moe_destroy(h):
    if h:
        load().waste_moe_destroy(h)


def waste_moe_stats(h) -> dict:
    st = waste_moe_stats_t()
    _check(load().waste_moe_stats(h, ctypes.byref(st)))
    return {n: getattr(st, n) for n, _ in waste_moe_stats_t._fields_}


def waste_moe_reset_stats(h):
    return _check(load().waste_moe_reset_stats(h))


def waste_moe_topk_from_logits(d_logits, T, E, k, d_idx, d_gate, stream=None):
    return _check(load().waste_moe_topk_from_logits(_ptr(d_logits), T, E, k, _ptr(d_idx),
                                                    _ptr(d_gate), _stream(stream)))


def waste_moe_set_profiling(h, enable=True):
    return _check(load().waste_moe_set_profiling(h, int(bool(enable))))


def waste_moe_set_lookahead(h, next_layer, n_prefetch):
    """The lookahead inside h's one-token steps into next_layer (None or 0: off)."""
    return _check(load().waste_moe_set_lookahead(h, next_layer, n_prefetch))


def waste_moe_read_profile(h) -> dict:
    """Milliseconds per kernel of the last profiled route and forward."""
    ms = (ctypes.c_float * 6)()
    _check(load().waste_moe_read_profile(h, ms))
    out = dict(zip(("router", "topk", "gate_up", "down", "combine", "step"), list(ms)))
    if out["down"] < 0 <= out["gate_up"]:  # gate/up and down units in one launch
        out["experts"] = out.pop("gate_up")
    return out


def waste_moe_debug_wait(h, d_counter, target, limit_ns, stream=None):
    """The library's bounded device wait on a caller-owned uint32 counter (test aid)."""
    return _check(load().waste_moe_debug_wait(h, _ptr(d_counter), target, limit_ns, _stream(stream)))


def waste_moe_rmsnorm(d_in, d_out, T, d, stream=None):
    return _check(load().waste_moe_rmsnorm(_ptr(d_in), _ptr(d_out), T, d, _stream(stream)))


def waste_moe_forward_noalloc(cfg, records, record_stride, codebooks, d_h, T, d_idx, d_gate, d_out,
                              mode=0, stream=None):
    """waste_moe_forward without a handle; its scratch is a fixed 8 MiB device array."""
    return _check(load().waste_moe_forward_noalloc(
        ctypes.byref(cfg), _ptr(records), record_stride, _ptr(codebooks), _ptr(d_h), T,
        _ptr(d_idx), _ptr(d_gate), _ptr(d_out), mode, _stream(stream)))


def waste_bank_create(cfg, n_layers, host_records, record_stride, n_slots) -> int:
    out = ctypes.c_void_p()
    _check(load().waste_bank_create(ctypes.byref(cfg), n_layers, _ptr(host_records), record_stride, n_slots,
                                    ctypes.byref(out)))
    return out.value


def waste_bank_destroy(bank):
    if bank:
        load().waste_bank_destroy(bank)


def waste_bank_reset(bank):
    return _check(load().waste_bank_reset(bank))


def waste_bank_stats(bank) -> dict:
    st = waste_bank_stats_t()
    _check(load().waste_bank_stats(bank, ctypes.byref(st)))
    return {n: getattr(st, n) for n, _ in waste_bank_stats_t._fields_}


def waste_moe_create_banked(cfg, router_w, router_bias, bank, layer, codebooks) -> int:
    out = ctypes.c_void_p()
    _check(load().waste_moe_create_banked(ctypes.byref(cfg), _ptr(router_w), _ptr(router_bias), bank, layer,
                                          _ptr(codebooks), ctypes.byref(out)))
    return out.value


def pinned_bytes(nbytes: int, align: int = RECORD_ALIGN) -> torch.Tensor:
    """A uint8 pinned host buffer of nbytes whose start is align-aligned."""
    raw = torch.empty(nbytes + align, dtype=torch.uint8, pin_memory=True)
    off = (-raw.data_ptr()) % align
    return raw[off:off + nbytes]


def aligned_bytes(nbytes: int, device="cuda", align: int = RECORD_ALIGN) -> torch.Tensor:
    """A uint8 device buffer of nbytes whose start is align-aligned (view into a larger one)."""
    raw = torch.empty(nbytes + align, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % align
    return raw[off:off + nbytes]


def waste_rvq_train(w, init, iters: int, codebooks, codes, err, stream=None):
    """Greedy residual k-means of w [rows, cols] fp32 (device): codebooks [3,256,8] fp32, codes
    [rows,3,cols/8] u8, err [3] float64 (device, written).  init [3,256] int32 (device)."""
    rows, cols = w.shape
    return _check(load().waste_rvq_train(_ptr(w), rows, cols, _ptr(init), int(iters), _ptr(codebooks),
                                         _ptr(codes), _ptr(err), _stream(stream)))


def waste_rvq_encode(w, codebooks, codes, err, stream=None):
    rows, cols = w.shape
    return _check(load().waste_rvq_encode(_ptr(w), rows, cols, _ptr(codebooks), _ptr(codes), _ptr(err),
                                          _stream(stream)))
