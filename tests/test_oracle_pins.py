"""Pins for the fp64 CPU oracle: checks against things other than itself.

- exhaustive format decoders against torch's own conversions;
- hand-derived closed-form fixtures under ``tests/golden/`` (each cites the
  passage of the "verify_splitkv.py" page it follows);
- a library cross-check: the whole operation is one masked softmax attention
  over the concatenated key set, which torch's scaled_dot_product_attention
  computes in fp64;
- invariants the definition fixes: single key, identical keys, scale
  equivalences, slot-permutation invariance, key-order invariance, causal and
  GQA dependency structure, the log-sum-exp merge identity of the debug outputs.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decoders
def test_bf16_decoder_exhaustive():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_bf16(codes)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decoder_exhaustive():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 for both signs
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0 and got[1] == 2.0 ** -9


# ---------------------------------------------------------------- golden fixtures
def _parse_value(s):
    if isinstance(s, (int, float)):
        return float(s)
    s = s.strip()
    if s == "-inf":
        return -math.inf
    if s == "nan":
        return math.nan
    if s.startswith("ln(") and s.endswith(")"):
        return math.log(float(Fraction(s[3:-1])))
    return float(Fraction(s))


def _parse_array(a):
    if isinstance(a, list):
        return [_parse_array(x) for x in a]
    return _parse_value(a)


def _golden_arrays(fx, pool_dtype):
    def bits16(a):
        t = torch.tensor(_parse_array(a), dtype=torch.float64)
        b = t.to(torch.bfloat16)
        assert torch.equal(b.to(torch.float64).nan_to_num(7.5), t.nan_to_num(7.5)), "fixture value not exact in bf16"
        return b.view(torch.int16).numpy().view(np.uint16)

    def pool(a):
        if pool_dtype == "bf16":
            return bits16(a)
        t = torch.tensor(_parse_array(a), dtype=torch.float64)
        f8 = t.to(torch.float8_e4m3fn)
        assert torch.equal(f8.to(torch.float64).nan_to_num(7.5), t.nan_to_num(7.5)), "fixture value not exact in e4m3"
        return f8.view(torch.uint8).numpy()

    if fx.get("paged"):
        n, hq = len(fx["q"]), len(fx["q"][0])
        hkv, d = len(fx["k_pool"][0]), len(fx["k_pool"][0][0])
        dv = len(fx["v_pool"][0][0])
        fx = dict(fx, k_ext=[[[0] * d] * hkv] * n, v_ext=[[[0] * dv] * hkv] * n)
    return {
        **({"block_table": np.array(fx["block_table"], dtype=np.int32), "page_size": fx["page_size"],
            "seq_lens": np.array(fx["seq_lens"], dtype=np.int32)} if fx.get("paged") else
           {"kv_indptr": np.array(fx["kv_indptr"], dtype=np.int32),
            "kv_indices": np.array(fx["kv_indices"], dtype=np.int64)}),
        "q": bits16(fx["q"]), "k_ext": bits16(fx["k_ext"]), "v_ext": bits16(fx["v_ext"]),
        "k_pool": pool(fx["k_pool"]), "v_pool": pool(fx["v_pool"]), "pool_dtype": pool_dtype,
        "qo_indptr": np.array(fx["qo_indptr"], dtype=np.int32),
        "sm_scale": _parse_value(fx["sm_scale"]), "k_scale": fx["k_scale"], "v_scale": fx["v_scale"],
        **({"custom_mask": np.array(fx["custom_mask"], dtype=np.uint8),
            "mask_indptr": np.array(fx["mask_indptr"], dtype=np.int64)} if "custom_mask" in fx else {}),
    }


def _golden_cases():
    cases = []
    for fn in sorted(os.listdir(GOLDEN)):
        if fn.endswith(".json"):
            with open(os.path.join(GOLDEN, fn)) as f:
                fx = json.load(f)
            for pd in fx["pool_dtypes"]:
                cases.append(pytest.param(fn, pd, id=f"{fn[:-5]}-{pd}"))
    return cases


def run_golden(fn, pool_dtype, lib=None):
    with open(os.path.join(GOLDEN, fn)) as f:
        fx = json.load(f)
    arrays = _golden_arrays(fx, pool_dtype)
    res = oracle.verify_forward(arrays, debug=True, lib=lib)
    for key, exp in fx["expected"].items():
        want = np.array(_parse_array(exp), dtype=np.float64)
        got = res[key]
        assert got.shape == want.shape, (key, got.shape, want.shape)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12, err_msg=f"{fn}:{key}")


@pytest.mark.parametrize("fn,pool_dtype", _golden_cases())
def test_golden(fn, pool_dtype):
    run_golden(fn, pool_dtype)


def test_golden_fixtures_present():
    names = {f for f in os.listdir(GOLDEN) if f.endswith(".json")}
    assert {"scales_causal.json", "gqa_mapping.json", "indptr_empty_prefix.json", "tree_mask.json",
            "paged_drafts_in_cache.json"} <= names


# ---------------------------------------------------------------- library cross-check
def _sdpa_reference(prob):
    """fp64 torch scaled_dot_product_attention over [scaled prefix keys ; drafts]
    with a boolean mask (prefix always visible, draft t visible to row i iff t <= i)."""
    d64 = torch.float64
    q, ke, ve = prob["q"].to(d64), prob["k_ext"].to(d64), prob["v_ext"].to(d64)
    kb, vb = prob["k_buffer"].to(d64), prob["v_buffer"].to(d64)
    qo, kvp, kvi = prob["qo_indptr"], prob["kv_indptr"], prob["kv_indices"].long()
    h_q, h_kv = q.shape[1], ke.shape[1]
    g = h_q // h_kv
    out = torch.empty(q.shape[0], h_q, ve.shape[2], dtype=d64)
    for b in range(qo.numel() - 1):
        s, e = int(qo[b]), int(qo[b + 1])
        ps, pe = int(kvp[b]), int(kvp[b + 1])
        loc = kvi[ps:pe]
        L, P = e - s, pe - ps
        kcat = torch.cat([prob["k_scale"] * kb[loc], ke[s:e]], 0)       # [P+L, h_kv, d]
        vcat = torch.cat([prob["v_scale"] * vb[loc], ve[s:e]], 0)
        mask = torch.ones(L, P + L, dtype=torch.bool)
        if prob.get("custom_mask") is not None:
            mi = prob["mask_indptr"]
            m = prob["custom_mask"][int(mi[b]):int(mi[b + 1])].view(L, P + L).bool()
            mask[:, P:] = m[:, P:]  # prefix columns are not applied
        else:
            mask[:, P:] = torch.tril(torch.ones(L, L, dtype=torch.bool))
        qh = q[s:e].transpose(0, 1)                                     # [h_q, L, d]
        kh = kcat.transpose(0, 1).repeat_interleave(g, 0)               # [h_q, P+L, d]
        vh = vcat.transpose(0, 1).repeat_interleave(g, 0)
        o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask, scale=prob["sm_scale"])
        out[s:e] = o.transpose(0, 1)
    return out.numpy()


SDPA_CASES = [
    workloads.TINY,
    workloads.Spec("mixed_empty", (0, 37, 5, 130), 3, 6, 2, 64, 64, perm=True, pool_extra=11, seed=7),
    workloads.Spec("fp8_scales", (40, 75), 4, 8, 2, 64, 64, pool="e4m3", perm=True, k_scale=0.5,
                   v_scale=0.25, seed=8),
    workloads.Spec("l1_decode", (50, 17), 1, 8, 8, 64, 64, seed=9, idx_dtype="int32"),
    workloads.Spec("d_ne_dv", (33, 20), 2, 4, 2, 64, 128, seed=10),
    workloads.Spec("long_chain", (16,), 8, 4, 1, 64, 64, seed=11),
    workloads.Spec("tree_random", (0, 23, 40), 6, 8, 2, 64, 64, perm=True, tree="random", seed=12),
    workloads.Spec("tree_star_fp8", (30, 9), 5, 4, 2, 64, 64, pool="e4m3", tree="star", k_scale=0.5, v_scale=2.0,
                   seed=13),
]


@pytest.mark.parametrize("spec", SDPA_CASES, ids=lambda s: s.name)
def test_sdpa_library_crosscheck(spec):
    prob = workloads.make_problem(spec, "cpu")
    got = oracle.verify_forward(workloads.to_oracle_arrays(prob))["o"]
    ref = _sdpa_reference(prob)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- invariants
def _run(prob, **kw):
    return oracle.verify_forward(workloads.to_oracle_arrays(prob), **kw)


def test_single_key_returns_its_value():
    prob = workloads.make_problem(workloads.Spec("single", (0, 0, 0), 3, 4, 2, 64, 64, seed=21), "cpu")
    o = _run(prob)["o"]
    ve = prob["v_ext"].to(torch.float64).numpy()
    for b in range(3):
        row = 3 * b  # draft row 0 sees only its own draft key
        for h in range(4):
            assert np.array_equal(o[row, h], ve[row, h // 2])


def test_identical_keys_give_mean_of_values():
    spec = workloads.Spec("ident", (20, 9), 3, 4, 2, 64, 64, v_scale=0.5, seed=22)
    prob = workloads.make_problem(spec, "cpu")
    k = prob["k_buffer"][0:1, :, :].clone()
    prob["k_buffer"][:] = k
    prob["k_ext"][:] = k[0]
    o = _run(prob)["o"]
    vb = prob["v_buffer"].to(torch.float64) * 0.5
    ve = prob["v_ext"].to(torch.float64)
    for b, (ps, pe) in enumerate([(0, 20), (20, 29)]):
        for i in range(3):
            row = 3 * b + i
            vis = torch.cat([vb[ps:pe], ve[3 * b: 3 * b + i + 1]], 0)  # [n, h_kv, dv]
            mean = vis.mean(0).numpy()
            for h in range(4):
                np.testing.assert_allclose(o[row, h], mean[h // 2], rtol=1e-13, atol=1e-14)


def test_k_scale_equals_prescaled_keys_and_v_scale_equals_prescaled_values():
    base = workloads.Spec("sc", (30, 45), 4, 8, 2, 64, 64, perm=True, seed=23)
    a = workloads.make_problem(base, "cpu", k_scale=2.0, v_scale=0.5)
    b = workloads.make_problem(base, "cpu")
    b["k_buffer"] = (b["k_buffer"].to(torch.float64) * 2.0).to(torch.bfloat16)
    b["v_buffer"] = (b["v_buffer"].to(torch.float64) * 0.5).to(torch.bfloat16)
    oa, ob = _run(a)["o"], _run(b)["o"]
    np.testing.assert_allclose(oa, ob, rtol=1e-14, atol=1e-15)


def test_scales_do_not_touch_drafts():
    base = workloads.Spec("nodraftscale", (0, 0), 4, 4, 1, 64, 64, seed=24)
    a = _run(workloads.make_problem(base, "cpu"))["o"]
    b = _run(workloads.make_problem(base, "cpu", k_scale=0.25, v_scale=3.0))["o"]
    assert np.array_equal(a, b)


def test_scales_do_touch_the_prefix():
    base = workloads.Spec("prefscale", (12, 5), 2, 4, 1, 64, 64, seed=25)
    a = _run(workloads.make_problem(base, "cpu"))["o"]
    b = _run(workloads.make_problem(base, "cpu", k_scale=0.5))["o"]
    c = _run(workloads.make_problem(base, "cpu", v_scale=0.5))["o"]
    assert np.abs(a - b).max() > 1e-3 and np.abs(a - c).max() > 1e-3


def test_pool_slot_permutation_is_invisible():
    spec = workloads.Spec("slotperm", (25, 60, 3), 3, 4, 2, 64, 64, perm=True, pool_extra=9, seed=26)
    prob = workloads.make_problem(spec, "cpu")
    o1 = _run(prob)["o"]
    n = prob["k_buffer"].shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n)
    prob2 = dict(prob)
    prob2["k_buffer"] = prob["k_buffer"][perm]           # new slot s holds old slot perm[s]
    prob2["v_buffer"] = prob["v_buffer"][perm]
    prob2["kv_indices"] = inv[prob["kv_indices"]]
    o2 = _run(prob2)["o"]
    assert np.array_equal(o1, o2)


def test_prefix_key_order_changes_only_rounding():
    spec = workloads.Spec("keyorder", (80, 33), 4, 4, 1, 64, 64, perm=True, seed=27)
    prob = workloads.make_problem(spec, "cpu")
    o1 = _run(prob)["o"]
    kvi = prob["kv_indices"].clone()
    kvi[0:80] = kvi[0:80].flip(0)
    kvi[80:113] = kvi[80:113][torch.randperm(33, generator=torch.Generator().manual_seed(3))]
    prob2 = dict(prob, kv_indices=kvi)
    o2 = _run(prob2)["o"]
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)


def test_causal_dependency_structure():
    spec = workloads.Spec("causal", (10, 7), 4, 2, 1, 64, 64, seed=28)
    prob = workloads.make_problem(spec, "cpu")
    o1 = _run(prob)["o"]
    t = 2  # perturb draft key/value row t of sequence 1
    row = 4 + t
    prob["k_ext"][row] = prob["k_ext"][row] * -2
    prob["v_ext"][row] = prob["v_ext"][row] + 1
    o2 = _run(prob)["o"]
    changed = np.abs(o1 - o2).max(axis=(1, 2)) > 0
    assert changed.tolist() == [False] * 4 + [False, False, True, True]


def test_gqa_dependency_structure():
    spec = workloads.Spec("gqa", (20, 11), 2, 8, 4, 64, 64, seed=29)
    prob = workloads.make_problem(spec, "cpu")
    o1 = _run(prob)["o"]
    kvh = 2
    prob["v_buffer"][:, kvh] = prob["v_buffer"][:, kvh] + 1
    o2 = _run(prob)["o"]
    changed = np.abs(o1 - o2).max(axis=(0, 2)) > 0
    assert changed.tolist() == [h // 2 == kvh for h in range(8)]


def test_every_row_sees_the_whole_prefix():
    spec = workloads.Spec("fullprefix", (40,), 4, 2, 1, 64, 64, seed=30)
    prob = workloads.make_problem(spec, "cpu")
    o1 = _run(prob)["o"]
    last = int(prob["kv_indices"][39])
    prob["v_buffer"][last] = prob["v_buffer"][last] + 4
    o2 = _run(prob)["o"]
    assert (np.abs(o1 - o2).max(axis=2) > 0).all()


def test_lse_merge_identity_of_debug_parts():
    spec = workloads.Spec("merge", (0, 50, 9), 3, 4, 2, 64, 64, perm=True, k_scale=0.5, v_scale=2.0, seed=31)
    prob = workloads.make_problem(spec, "cpu")
    r = _run(prob, debug=True)
    lp, ld = r["lse_prefix"][..., None], r["lse_draft"][..., None]
    m = np.maximum(lp, ld)
    wp, wd = np.exp(lp - m), np.exp(ld - m)
    merged = (r["o_prefix"] * wp + r["o_draft"] * wd) / (wp + wd)
    np.testing.assert_allclose(r["o"], merged, rtol=1e-12, atol=1e-13)
    assert np.isneginf(r["lse_prefix"][0:3]).all()  # sequence 0 has no prefix


def test_large_scores_stay_finite_and_convex():
    spec = workloads.Spec("large", (64, 31), 2, 4, 2, 64, 64, seed=32)
    prob = workloads.make_problem(spec, "cpu")
    prob["q"] = (prob["q"].to(torch.float64) * 64).to(torch.bfloat16)  # scores in the hundreds
    o = _run(prob)["o"]
    assert np.isfinite(o).all()
    vmax = max(prob["v_buffer"].abs().max().item(), prob["v_ext"].abs().max().item())
    assert np.abs(o).max() <= vmax + 1e-12


def test_ranges_compute_only_what_is_asked():
    prob = workloads.make_problem(workloads.TINY, "cpu")
    full = _run(prob)["o"]
    part = oracle.verify_forward(workloads.to_oracle_arrays(prob), b_range=(1, 2), h_range=(2, 4))["o"]
    assert np.isnan(part[0:4]).all() and np.isnan(part[4:8, 0:2]).all()
    assert np.array_equal(part[4:8, 2:4], full[4:8, 2:4])


def test_thread_count_does_not_change_results():
    prob = workloads.make_problem(workloads.Spec("threads", (100, 64, 3), 4, 8, 2, 64, 64, seed=33), "cpu")
    a = oracle.verify_forward(workloads.to_oracle_arrays(prob), nthreads=1)["o"]
    b = oracle.verify_forward(workloads.to_oracle_arrays(prob), nthreads=4)["o"]
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- tree verify (custom mask)
def test_chain_tree_mask_equals_causal():
    spec = workloads.Spec("chain", (0, 31, 64), 6, 8, 2, 64, 64, perm=True, seed=41)
    causal = _run(workloads.make_problem(spec, "cpu"))["o"]
    chain = _run(workloads.make_problem(spec, "cpu", tree="chain"))["o"]
    assert np.array_equal(causal, chain)


def test_tree_mask_prefix_columns_are_not_applied():
    spec = workloads.Spec("prefcols", (17, 40), 5, 4, 1, 64, 64, perm=True, tree="random", seed=42)
    prob = workloads.make_problem(spec, "cpu")
    a = _run(prob)["o"]
    cm = prob["custom_mask"].clone()
    mi = prob["mask_indptr"]
    for b, P in enumerate(prob["prefix_lens"]):
        m = cm[int(mi[b]):int(mi[b + 1])].view(5, P + 5)
        m[:, :P] = 0
    b_ = _run(dict(prob, custom_mask=cm))["o"]
    assert np.array_equal(a, b_)


def test_tree_mask_row_with_nothing_visible_is_zero():
    spec = workloads.Spec("empty_row", (0,), 3, 2, 1, 64, 64, tree="chain", seed=43)
    prob = workloads.make_problem(spec, "cpu")
    cm = prob["custom_mask"].clone()
    cm[3:6] = 0  # row 1 sees nothing (no prefix, no draft)
    r = _run(dict(prob, custom_mask=cm), debug=True)
    assert np.array_equal(r["o"][1], np.zeros_like(r["o"][1]))
    assert np.isfinite(r["o"]).all() and np.isneginf(r["lse_draft"][1]).all()


# ---------------------------------------------------------------- drafts in a paged cache
def _sdpa_paged(prob):
    """fp64 SDPA over each sequence's cache positions 0 .. P+L-1 (scaled keys
    and values), prefix visible, drafts causal."""
    d64 = torch.float64
    q = prob["q"].to(d64)
    kc, vc = prob["k_buffer"].to(d64), prob["v_buffer"].to(d64)
    bt, ps = prob["block_table"].long(), prob["page_size"]
    h_q, h_kv = q.shape[1], kc.shape[1]
    g = h_q // h_kv
    L = prob["max_len_extend"]
    out = torch.empty(q.shape[0], h_q, vc.shape[2], dtype=d64)
    for b, P in enumerate(prob["seq_lens"].tolist()):
        j = torch.arange(P + L)
        rows = bt[b, j // ps] * ps + j % ps
        k = prob["k_scale"] * kc[rows]
        v = prob["v_scale"] * vc[rows]
        mask = torch.ones(L, P + L, dtype=torch.bool)
        mask[:, P:] = torch.tril(torch.ones(L, L, dtype=torch.bool))
        qh = q[b * L:(b + 1) * L].transpose(0, 1)
        o = torch.nn.functional.scaled_dot_product_attention(
            qh, k.transpose(0, 1).repeat_interleave(g, 0), v.transpose(0, 1).repeat_interleave(g, 0),
            attn_mask=mask, scale=prob["sm_scale"])
        out[b * L:(b + 1) * L] = o.transpose(0, 1)
    return out.numpy()


PAGED_CASES = [
    workloads.Spec("paged_ps16", (100, 0, 37), 4, 8, 2, 64, 64, perm=True, page_size=16, pool_extra=40, seed=51),
    workloads.Spec("paged_ps1_fp8", (30, 61), 3, 4, 2, 64, 64, pool="e4m3", perm=True, page_size=1, k_scale=0.5,
                   v_scale=2.0, seed=52),
    workloads.Spec("paged_decode_ps64", (200, 129, 5), 1, 8, 8, 64, 64, perm=True, page_size=64, seed=53),
]


@pytest.mark.parametrize("spec", PAGED_CASES, ids=lambda s: s.name)
def test_paged_sdpa_crosscheck(spec):
    prob = workloads.make_problem(spec, "cpu")
    got = _run(prob)["o"]
    np.testing.assert_allclose(got, _sdpa_paged(prob), rtol=1e-11, atol=1e-12)


def test_paged_equals_flat_when_scales_are_one():
    spec = workloads.Spec("paged_eq", (70, 3, 0), 4, 8, 4, 64, 64, perm=True, page_size=8, pool_extra=24, seed=54)
    prob = workloads.make_problem(spec, "cpu")
    paged = _run(prob)["o"]
    flat = {k: v for k, v in prob.items() if k not in ("block_table", "page_size", "seq_lens")}
    assert np.array_equal(paged, _run(flat)["o"])


def test_paged_poisoned_pages_are_never_read():
    spec = workloads.Spec("paged_poison", (50, 9), 4, 4, 1, 64, 64, perm=True, page_size=4, pool_extra=64,
                          poison=True, seed=55)
    assert np.isfinite(_run(workloads.make_problem(spec, "cpu"))["o"]).all()


# ---------------------------------------------------------------- quantised store of new K/V rows
def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _e4m3_midpoints():
    """Every value halfway between two adjacent non-negative finite e4m3 codes."""
    vals = np.array([oracle.decode_e4m3(np.array([c], dtype=np.uint8))[0] for c in range(0x7F)])
    return (vals[:-1] + vals[1:]) / 2


def quantize_pins(lib=None):
    """Every check of the quantised store; raises AssertionError on a miss.
    Pinned to: the e4m3 and bf16 format definitions (round trip of every
    code, the tie rule, saturation) and torch's own round-to-nearest-even
    float8 / bfloat16 casts (a library routine the oracle does not use)."""
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_e4m3(codes, lib=lib)
    finite = ~np.isnan(vals)
    # 1. decode -> store at scale 1 returns every finite code (both zeros included)
    rt = oracle.quantize(_bf16_bits(torch.tensor(vals[finite])), 1.0, "e4m3", lib=lib)
    np.testing.assert_array_equal(rt, codes[finite])
    # 2. torch's cast on in-range binary32 values: random magnitudes and every midpoint, both signs
    g = torch.Generator().manual_seed(71)
    mag = torch.exp2(torch.empty(20000).uniform_(-12, 8.85, generator=g))
    mid = torch.tensor(_e4m3_midpoints(), dtype=torch.float32)
    v = torch.cat([mag, -mag, mid, -mid, torch.tensor([0.0, -0.0, 448.0, -448.0, 463.0])])
    want = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.encode_e4m3(v.numpy(), lib=lib), want)
    # 3. ties go to the even code; beyond 448 (and infinity) saturates; NaN stays NaN
    got = oracle.encode_e4m3(np.array([1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10, 464.0, 465.0, 1e30,
                                       -1e30, np.inf, np.nan], dtype=np.float32), lib=lib)
    assert got.tolist() == [0x38, 0x3A, 0x02, 0x00, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0x7F]
    # 4. bf16 store: torch's cast on random binary32 values and exact ties
    f = torch.randn(20000, generator=g) * torch.exp2(torch.empty(20000).uniform_(-30, 30, generator=g))
    w = torch.randint(0, 2 ** 16, (4000,), generator=g, dtype=torch.int32) << 16 | 0x8000
    ties = w.view(torch.float32)
    ties = ties[torch.isfinite(ties)]
    for x in (f, ties):
        want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(oracle.encode_bf16(x.numpy(), lib=lib), want)
    # 5. the scale divides, in binary32, before the cast (both cache dtypes)
    x = torch.randn(4096, generator=g).to(torch.bfloat16)
    for s in (0.5, 0.75, 2.0, 1.3):
        q = (x.float() / s)
        keep = q.abs() < 464
        want8 = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got8 = oracle.quantize(_bf16_bits(x), s, "e4m3", lib=lib)
        np.testing.assert_array_equal(got8[keep.numpy()], want8[keep.numpy()])
        want16 = q.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(oracle.quantize(_bf16_bits(x), s, "bf16", lib=lib), want16)


def test_quantised_store_pins():
    quantize_pins()


def test_store_then_read_is_within_half_a_step():
    """decode(store(x, s)) * s is the nearest representable value: relative
    error at most 2^-4 for normal e4m3 values, 2^-8 for bf16."""
    g = torch.Generator().manual_seed(72)
    x = (torch.randn(8192, generator=g) * 4).to(torch.bfloat16)
    xd = x.double().numpy()
    for s in (0.25, 1.0, 3.0):
        back = oracle.decode_e4m3(oracle.quantize(_bf16_bits(x), s, "e4m3")) * s
        normal = np.abs(xd / s) >= 2.0 ** -6
        assert np.all(np.abs(back - xd)[normal] <= 2.0 ** -4 * np.abs(xd)[normal] + 1e-300)
        back16 = oracle.decode_bf16(oracle.quantize(_bf16_bits(x), s, "bf16")) * s
        assert np.all(np.abs(back16 - xd) <= 2.0 ** -8 * np.abs(xd))


def test_write_rows_replaces_only_the_named_rows():
    g = torch.Generator().manual_seed(73)
    pool = _bf16_bits(torch.randn(10, 2, 8, generator=g))
    new = _bf16_bits(torch.randn(3, 2, 8, generator=g))
    out = oracle.write_rows(pool, [7, 1, 4], new, 1.0, "bf16")
    np.testing.assert_array_equal(out[[7, 1, 4]], new)
    keep = [0, 2, 3, 5, 6, 8, 9]
    np.testing.assert_array_equal(out[keep], pool[keep])
    pool8 = np.zeros((10, 2, 8), dtype=np.uint8)
    out8 = oracle.write_rows(pool8, [2, 9, 0], new, 0.5, "e4m3")
    np.testing.assert_array_equal(out8[[2, 9, 0]], oracle.quantize(new, 0.5, "e4m3"))
