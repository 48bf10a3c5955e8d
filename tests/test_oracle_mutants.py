"""The pins catch plausible oracle mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source (a
dropped term, a wrong sign or index, a transposed operand, a misplaced scale),
compiles it on the CPU, and checks that the golden fixtures and the library
cross-check reject it.  The committed oracle is never modified.
"""
import os

import numpy as np
import pytest

import oracle
import workloads
from test_oracle_pins import _golden_cases, _sdpa_reference, quantize_pins, run_golden

SRC = os.path.join(os.path.dirname(oracle.__file__), "verify_oracle.c")

MUTANTS = {
    "drop_own_draft_key": ("if (!p->custom_mask) return t <= i;", "if (!p->custom_mask) return t < i;"),
    "k_scale_on_drafts": ("? p->sm_scale * dot : -INFINITY", "? p->sm_scale * p->k_scale * dot : -INFINITY"),
    "tree_mask_transposed": ("p->mask_indptr[b] + i * (P_b + L_b) + P_b + t]", "p->mask_indptr[b] + t * (P_b + L_b) + P_b + i]"),
    "tree_mask_prefix_offset": ("i * (P_b + L_b) + P_b + t]", "i * (P_b + L_b) + t]"),
    "v_scale_dropped": ("acc[c] += w * p->v_scale * pool_elem(p, p->v_pool", "acc[c] += w * pool_elem(p, p->v_pool"),
    "gqa_modulo": ("const int64_t kvh = h / group;", "const int64_t kvh = h % p->h_kv;"),
    "no_indirection": ("return p->paged ? paged_row(p, b, j) : kv_index(p, p_b + j);",
                       "return p->paged ? paged_row(p, b, j) : p_b + j;"),
    "paged_page_offset": ("* p->page_size + j % p->page_size;", "* p->page_size + j / p->page_size;"),
    "paged_draft_unscaled": ("return p->v_scale * pool_elem(p, p->v_pool, paged_row", "return pool_elem(p, p->v_pool, paged_row"),
    "softmax_sign": ("exp(score[j] - mx)", "exp(mx - score[j])"),
    "pool_strides_transposed": ("loc * p->kp_s0 + kvh * p->kp_s1", "loc * p->kp_s1 + kvh * p->kp_s0"),
    "draft_value_row": ("p->v_ext[(s_b + t) * p->ve_s0", "p->v_ext[(s_b + 0) * p->ve_s0"),
    "store_multiplies_scale": ("const float y = x / scale;", "const float y = x * scale;"),
    "e4m3_ties_away": ("(dh == dl && (c & 1) == 0)", "(dh == dl)"),
    "e4m3_sign_dropped": ("const uint8_t sign = signbit(y) ? 0x80 : 0x00;", "const uint8_t sign = 0x00;"),
    "bf16_truncates": ("if (dh < dl || (dh == dl && ((hi >> 16) & 1u) == 0)) return (uint16_t)(hi >> 16);", ""),
}


def _build_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert old in src, f"mutation site for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.build(str(path), str(tmp_path / f"lib{name}.so"), force=True)
    return oracle.load(so)


def _detected(lib):
    try:
        quantize_pins(lib)
    except AssertionError:
        return True
    for case in _golden_cases():
        fn, pd = case.values
        try:
            run_golden(fn, pd, lib=lib)
        except AssertionError:
            return True
    prob = workloads.make_problem(workloads.TINY, "cpu")
    got = oracle.verify_forward(workloads.to_oracle_arrays(prob), lib=lib)["o"]
    return not np.allclose(got, _sdpa_reference(prob), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    lib = _build_mutant(name, tmp_path)
    assert _detected(lib), f"planted mistake {name} passed every pin"
