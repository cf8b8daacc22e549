"""Record payload crc32 on the device: written by pack, checked by create.

Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Architecture de
streaming depuis le disque": records carry a crc32 checked behind --verify.  The device
crc (4 KiB chunks folded with the GF(2) "advance" matrix) must equal the oracle's
bit-at-a-time crc32 and zlib's of the same payload bytes; a flipped byte must make create
refuse the layer.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from rvq_compressed_expert_gb300 import binding as B
from rvq_compressed_expert_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rvq_compressed_expert_gb300 import _build
    _build.build()
    B.load()
    oracle.build()


def packed(w, seed, compute_crc, flags=0):
    cfg = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, 1, 0, flags, 0)
    stride, off, by = B.waste_moe_record_layout(cfg)
    li = synth.layer_inputs(w, seed, 0, "cuda", with_codes=True)
    records = B.aligned_bytes(w.n_experts * stride, "cuda")
    B.waste_moe_pack_records(cfg, 0, 0, w.n_experts, *[c.contiguous() for c in li.codes], records, stride,
                             compute_crc)
    torch.cuda.synchronize()
    return cfg, stride, off, by, li, records


def header_crc(records, stride, e):
    hdr = records[e * stride:e * stride + 4096].cpu().numpy()
    off = B.waste_record_header.payload_crc32.offset
    return int(hdr[off:off + 4].view(np.uint32)[0])


def payload(records, stride, off, by, e):
    lo = e * stride + off[0]
    return records[lo:lo + by[0] + by[1] + by[2]].cpu().numpy()


@pytest.mark.parametrize("shape", [(256, 128, 4), (1032, 136, 3)])
def test_pack_writes_payload_crc(shape):
    d, f, E = shape
    w = synth.Workload("crc", d, f, E, 1, 1, "f32", "none")
    cfg, stride, off, by, li, records = packed(w, 0, 1)
    for e in range(E):
        p = payload(records, stride, off, by, e)
        want = oracle.crc32(p)
        assert want == zlib.crc32(p.tobytes())
        assert header_crc(records, stride, e) == want


def test_verify_accepts_and_refuses():
    w = synth.Workload("crc", 512, 264, 6, 2, 1, "f32", "none")
    cfg, stride, off, by, li, records = packed(w, 1, 1, B.FLAG_VERIFY_CRC)
    h = B.waste_moe_create(cfg, li.router_w, li.router_b, records, stride, li.codebooks)
    B.waste_moe_destroy(h)
    # one flipped payload byte of record 4: refused with the flag, accepted without it
    pos = 4 * stride + off[1] + 12345
    records[pos] ^= 0x10
    with pytest.raises(B.WasteError) as ei:
        B.waste_moe_create(cfg, li.router_w, li.router_b, records, stride, li.codebooks)
    assert ei.value.status == -5 and "record 4" in ei.value.message
    cfg0 = B.make_config(w.d, w.f, w.n_experts, w.top_k, w.act_dtype, 1, 0, 0, 0)
    B.waste_moe_destroy(B.waste_moe_create(cfg0, li.router_w, li.router_b, records, stride, li.codebooks))
    # packed without a crc: the header holds 0, which the check refuses
    cfg2, stride2, _, _, li2, records2 = packed(w, 2, 0, B.FLAG_VERIFY_CRC)
    with pytest.raises(B.WasteError) as ei:
        B.waste_moe_create(cfg2, li2.router_w, li2.router_b, records2, stride2, li2.codebooks)
    assert ei.value.status == -5


def test_crc_full_decode_shape():
    """Records of the decode shape (d=7168, f=1536: 3024 pages of payload each)."""
    w = synth.Workload("crc-decode", 7168, 1536, 4, 2, 1, "f32", "none")
    cfg, stride, off, by, li, records = packed(w, 3, 1, B.FLAG_VERIFY_CRC)
    for e in range(w.n_experts):
        assert header_crc(records, stride, e) == zlib.crc32(payload(records, stride, off, by, e).tobytes())
    B.waste_moe_destroy(B.waste_moe_create(cfg, li.router_w, li.router_b, records, stride, li.codebooks))
