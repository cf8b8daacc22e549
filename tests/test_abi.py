"""The C ABI library: builds, loads, exports what include/waste_moe.h declares,
and rejects bad arguments on the host (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

from rvq_compressed_expert_gb300 import _build
from rvq_compressed_expert_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "waste_moe.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(waste_(?:moe|bank|rvq)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("waste_moe_create", "waste_moe_route", "waste_moe_forward",
                     "waste_moe_prefetch", "waste_moe_destroy"):
        assert required in names
    assert sorted(B.EXPORTED) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and they are plain C symbols (not C++-mangled)
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, re.M), name


def test_record_layout_matches_format(lib):
    cfg = B.make_config(7168, 1536, 384, 16)
    stride, off, by = B.waste_moe_record_layout(cfg)
    # 3 sections of 4,128,768 B (1008 pages each) behind a 4 KiB header
    assert by == [4_128_768] * 3
    assert off == [4096, 4096 + 4_128_768, 4096 + 2 * 4_128_768]
    assert stride == 12_390_400
    # tiny shapes: down matrix (256 rows x 16 vectors) pads its 16 vectors to one 32-vector segment
    # gate/up: 1 segment x 8 row groups x 1536 B = 3 pages; down: 1 x 16 x 1536 B = 6 pages
    stride, off, by = B.waste_moe_record_layout(B.make_config(256, 128, 8, 2))
    assert by == [12288, 12288, 24576]
    assert off == [4096, 16384, 28672]
    assert stride == 53248


def test_header_struct_size():
    assert ctypes.sizeof(B.waste_record_header) == 4 * 10 + 8 * 7 + 8


@pytest.mark.parametrize("field,value", [("abi_version", 99), ("d", 12), ("f", 0),
                                         ("n_experts", 0), ("top_k", 0), ("top_k", 9),
                                         ("act_dtype", 3), ("max_tokens", 0), ("lookahead", -1),
                                         ("flags", 1 << 30)])
def test_bad_config_rejected(lib, field, value):
    cfg = B.make_config(256, 128, 8, 2)
    setattr(cfg, field, value)
    with pytest.raises(B.WasteError) as ei:
        B.waste_moe_record_layout(cfg)
    assert ei.value.status == -1
    assert B.waste_moe_last_error()


def test_create_rejects_null_and_misaligned(lib):
    cfg = B.make_config(256, 128, 8, 2)
    with pytest.raises(B.WasteError) as ei:
        B.waste_moe_create(cfg, None, None, None, 0, None)
    assert ei.value.status == -1
    with pytest.raises(B.WasteError) as ei:
        B.waste_moe_create(cfg, 4096, None, 4096 + 16, 1 << 20, 4096)
    assert ei.value.status == -4  # record base not 4 KiB aligned
    with pytest.raises(B.WasteError) as ei:
        B.waste_moe_create(cfg, 4096, None, 8192, 4096, 4096)
    assert ei.value.status == -4  # stride too small for the sections


def test_topk_rejects_bad_sizes(lib):
    for T, E, k in ((-1, 8, 2), (1, 8, 0), (1, 8, 9), (1, 0, 1), (1, 5000, 2), (1, 64, 33)):
        with pytest.raises(B.WasteError):
            B.waste_moe_topk_from_logits(None, T, E, k, None, None, stream=0)
    B.waste_moe_topk_from_logits(None, 0, 8, 2, None, None, stream=0)  # T = 0: nothing to do


def test_null_handle_rejected(lib):
    with pytest.raises(B.WasteError):
        B.waste_moe_route(None, None, 1, None, None, stream=0)
    with pytest.raises(B.WasteError):
        B.waste_moe_forward(None, None, 1, None, None, None, stream=0)
    with pytest.raises(B.WasteError):
        B.waste_moe_prefetch(None, None, 1, side=0)
    with pytest.raises(B.WasteError):
        B.waste_moe_stats(None)
    with pytest.raises(B.WasteError):
        B.waste_moe_debug_wait(None, 4096, 1, 1_000_000, stream=0)
    B.waste_moe_destroy(None)
