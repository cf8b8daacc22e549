"""Planted slips in a copy of the oracle must each fail at least one pin.

Each mutant replaces one snippet of oracle.c (a dropped term, a flipped sign,
a transposed index, a reversed tie order ...), compiles the copy on the CPU
and runs every pin against it.  A mutant that passes all pins would mean the
pins cannot see that kind of mistake.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "dequant_drops_stage": ("for (int s = 0; s < OR_STAGES; ++s)\n                    w += ",
                            "for (int s = 0; s < 2; ++s)\n                    w += "),
    "dequant_transposed_vector": ("W[(size_t)r * n_in + (size_t)j * OR_V + v] = w;",
                                  "W[(size_t)r * n_in + (size_t)v * nv + j] = w;"),
    "lut_wrong_stage_table": ("double t2 = T[((size_t)2 * nv + j)", "double t2 = T[((size_t)1 * nv + j)"),
    "lut_drops_stage": ("acc += t0 + t1 + t2;", "acc += t0 + t1;"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "swiglu_swapped": ("a[r] = oracle_silu(zg[r]) * zu[r];", "a[r] = oracle_silu(zu[r]) * zg[r];"),
    "tie_break_reversed": ("return a < b;", "return a > b;"),
    "topk_ascending": ("if (l[a] > l[b]) return 1;\n    if (l[a] < l[b]) return 0;",
                       "if (l[a] < l[b]) return 1;\n    if (l[a] > l[b]) return 0;"),
    "gates_unnormalised": ("gate[i] = exp(logits[idx[i]] - lmax) / z;", "gate[i] = exp(logits[idx[i]] - lmax);"),
    "combine_drops_gate": ("acc += gate[t] * ys[(size_t)t * d + i];", "acc += ys[(size_t)t * d + i];"),
    "router_drops_bias": ("logits[e] = acc + (bias ? (double)bias[e] : 0.0);", "logits[e] = acc;"),
    "router_transposed": ("acc += (double)Wr[(size_t)e * d + i] * h[i];",
                          "acc += (double)Wr[(size_t)(i % n_experts) * d + (e % d)] * h[i];"),
    "dense_transposed": ("acc += W[(size_t)r * n_in + i] * x[i];",
                         "acc += W[(size_t)(i % n_out) * n_in + (r % n_in)] * x[i];"),
    "rmsnorm_no_mean": ("double scale = 1.0 / sqrt(ss / (double)d + 1e-6);",
                        "double scale = 1.0 / sqrt(ss + 1e-6);"),
    "code_bytes_wrong": ("return (uint64_t)3 * (uint64_t)OR_STAGES", "return (uint64_t)2 * (uint64_t)OR_STAGES"),
    "crc_not_complemented": ("    return ~c;\n}", "    return c;\n}"),
    "crc_wrong_polynomial": ("(0xEDB88320u & (0u - (c & 1u)))", "(0x04C11DB7u & (0u - (c & 1u)))"),
    "rvq_ties_to_higher": ("        if (d < bd) {\n            bd = d;", "        if (d <= bd) {\n            bd = d;"),
    "rvq_residual_not_updated": ("R[i * OR_V + v] = R[i * OR_V + v] - C[(size_t)c * OR_V + v];",
                                 "R[i * OR_V + v] = R[i * OR_V + v];"),
    "rvq_mean_not_divided": ("(double)sum[c][v] / (double)cnt[c]", "(double)sum[c][v]"),
    "rvq_init_from_weights": ("C[(size_t)c * OR_V + v] = R[(size_t)init[s * OR_K + c] * OR_V + v];",
                              "C[(size_t)c * OR_V + v] = W[(size_t)init[s * OR_K + c] * OR_V + v];"),
    "rvq_codes_transposed": ("codes[code_index(nv, r, s, j)] = code[(size_t)r * nv + j];",
                             "codes[code_index(nv, r, s, j)] = code[(size_t)j * rows + r];"),
    "rvq_distance_abs": ("d = fmaf(t, t, d);", "d = d + fabsf(t);"),
    "chain_router_on_h": ("oracle_router(n_experts, d, Wr, bias, x, lt);",
                          "oracle_router(n_experts, d, Wr, bias, ht, lt);"),
    "chain_experts_on_h": ("down_codes + (size_t)e * dn_exp, x,", "down_codes + (size_t)e * dn_exp, ht,"),
    "chain_drops_residual": ("ht[i] = ht[i] + y[i];", "ht[i] = y[i];"),
    "chain_norm_written_back": ("oracle_rmsnorm(d, ht, x);", "oracle_rmsnorm(d, ht, x);\n        memcpy(ht, x, sizeof(double) * (size_t)d);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, oracle_mod):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"snippet for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"])
    saved = oracle._lib
    oracle._lib = oracle._bind(ctypes.CDLL(str(so)))
    failed = []
    try:
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    finally:
        oracle._lib = saved
    assert failed, f"mutant {name} passed every pin"
