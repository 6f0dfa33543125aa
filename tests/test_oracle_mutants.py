"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies ``oracle/moe_oracle.c``, replaces one snippet with a
plausible mistake (a wrong index, a dropped term, a swapped operand, a
wrong order), builds the copy into a temporary library and runs every pin
on it. At least one pin must fail. The planted mistakes live only in the
temporary copies; the oracle itself is untouched.
"""
import os

import pytest

from oracle import oracle as oracle_mod
from oracle_pins import ALL_PINS

MUTANTS = {
    "lane_of_chunk": ("int L = c % 32;", "int L = c % 16;"),
    "butterfly_order": ("for (int s = 16; s >= 1; s /= 2)", "for (int s = 1; s <= 16; s *= 2)"),
    "gate_transposed": ("Wg[(int64_t)h * E + e]", "Wg[(int64_t)e * H + h]"),
    "bias_dropped": ("if (bias) l = l + bias[e];", "if (bias) l = l;"),
    "tie_to_higher": ("l[e] > l[best]", "l[e] >= l[best]"),
    "weights_unnormalised": ("- m) / den);", "- m));"),
    "w1_w3_swapped": ("g[f] = a[f] / (1.0 + exp(-a[f])) * b[f];",
                      "g[f] = b[f] / (1.0 + exp(-b[f])) * a[f];"),
    "silu_sign": ("(1.0 + exp(-a[f]))", "(1.0 + exp(a[f]))"),
    "permute_unstable": ("for (int64_t f = 0; f < R; ++f) {\n        int32_t p",
                         "for (int64_t f = R - 1; f >= 0; --f) {\n        int32_t p"),
    "offsets_wrong_count": ("offsets[e + 1] = offsets[e] + counts[e];",
                            "offsets[e + 1] = offsets[e] + counts[(e + 1) % E];"),
    "shared_scaled": ("for (int32_t n = 0; n < H; ++n) o[n] += y[n];",
                      "for (int32_t n = 0; n < H; ++n) o[n] += 0.5 * y[n];"),
    "combine_rank0_weight": ("double w = (double)topk_w[t * k + j];",
                             "double w = (double)topk_w[t * k];"),
    "w2_transposed": ("y[n] += gv * (double)bf16_to_float(w2[n]);",
                      "y[n] += gv * (double)bf16_to_float(W2[(int64_t)n * F + f]);"),
    "expert_stride": ("W1 + e * H * (int64_t)F, W3 + e * H * (int64_t)F",
                      "W1 + e * (int64_t)F, W3 + e * H * (int64_t)F"),
    "full_softmax_over_k_only": ("for (int32_t e = 0; e < E; ++e) den_all += exp((double)l[e] - m);",
                                 "for (int32_t e = 0; e < k; ++e) den_all += exp((double)l[topk_idx[t * k + e]] - m);"),
    "shared_gate_sign": ("scale[t] = 1.0 / (1.0 + exp(-d));", "scale[t] = 1.0 / (1.0 + exp(d));"),
    "shared_gate_dropped": ("for (int32_t n = 0; n < H; ++n) o[n] += sc * y[n];",
                            "for (int32_t n = 0; n < H; ++n) o[n] += y[n];"),
    "x_row_stride": ("const uint16_t* xrow = x + t * (int64_t)H;\n                double* y",
                     "const uint16_t* xrow = x + (t / k) * (int64_t)H;\n                double* y"),
    # the canonical order: elements of a chunk taken from the top down
    "chunk_order_reversed": ("for (int32_t h = 8 * c; h < 8 * c + 8 && h < H; ++h) {",
                             "for (int32_t h = (8 * c + 7 < H ? 8 * c + 7 : H - 1); h >= 8 * c; --h) {"),
    # the canonical order: 16-element chunks
    "chunk_of_16": ("int32_t n_chunks = (H + 7) / 8;\n    for (int32_t c = 0; c < n_chunks; ++c) {\n"
                    "        int L = c % 32;\n        for (int32_t h = 8 * c; h < 8 * c + 8 && h < H; ++h) {",
                    "int32_t n_chunks = (H + 15) / 16;\n    for (int32_t c = 0; c < n_chunks; ++c) {\n"
                    "        int L = c % 32;\n        for (int32_t h = 16 * c; h < 16 * c + 16 && h < H; ++h) {"),
    # the butterfly updated in place, from the top lane down: lane 0 reads a
    # partner it already overwrote (upwards in place happens to leave lane 0 right)
    "butterfly_in_place": ("for (int i = 0; i < 32; ++i) next[i] = lane[i] + lane[i ^ s];\n"
                           "        for (int i = 0; i < 32; ++i) lane[i] = next[i];",
                           "for (int i = 31; i >= 0; --i) lane[i] = lane[i] + lane[i ^ s];\n"
                           "        for (int i = 0; i < 32; ++i) next[i] = lane[i];"),
    # top-k that does not exclude the experts already chosen
    "topk_no_exclusion": ("                if (taken[e]) continue;\n", "                if (0) continue;\n"),
    # h rounded to bf16 in the reference (the definition keeps g in full precision)
    "g_rounded_bf16": ("for (int32_t f = 0; f < F; ++f) g[f] = a[f] / (1.0 + exp(-a[f])) * b[f];",
                       "for (int32_t f = 0; f < F; ++f) g[f] = (double)(float)(a[f] / (1.0 + exp(-a[f])) * b[f]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle_mod.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle_mod.build(str(mutant_src), str(tmp_path / f"libmutant_{name}.so"))
    O = oracle_mod.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(O)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"
