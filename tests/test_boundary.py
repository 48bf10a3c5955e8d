"""Host-side boundary tests (no GPU needed).

The gate follows ``can_handle`` on the "verify_splitkv.py" page and the
fallback tests of the "test_verify_splitkv.py" page (non-causal, sinks,
sliding window, logit cap, ragged extend); the build's own limits are checked
too.  ``vsk_can_handle`` never dereferences tensor data, so CPU tensors stand
in for device tensors here.
"""
import ctypes
import re

import pytest
import torch

import workloads
import speculative_decode_verify_prefix_gb300 as vsk
from speculative_decode_verify_prefix_gb300 import _native


@pytest.fixture(scope="module", autouse=True)
def built():
    vsk.build()


def _inputs(**over):
    spec = workloads.Spec("gate", (512, 512), 4, 16, 2, 256, 256, seed=3)
    p = workloads.make_problem(spec, "cpu", **over)
    return [p["q"], p["k_ext"], p["v_ext"], p["k_buffer"], p["v_buffer"], p["qo_indptr"], p["kv_indptr"],
            p["kv_indices"], None, True, None, p["max_len_extend"]]


def test_accepts_the_verify_shape():
    assert vsk.can_handle(*_inputs())


def test_fallback_non_causal():
    a = _inputs()
    a[9] = False
    assert not vsk.can_handle(*a)
    assert "causal" in vsk.last_error()


def test_fallback_exotic_features():
    a = _inputs()
    assert not vsk.can_handle(*a, sinks=torch.zeros(16))
    assert not vsk.can_handle(*a, sliding_window_size=128)
    assert not vsk.can_handle(*a, logit_cap=30.0)
    assert not vsk.can_handle(*a, xai_temperature_len=4)
    assert vsk.can_handle(*a, sliding_window_size=-1, logit_cap=0.0, xai_temperature_len=-1)


def test_fallback_ragged_extend():
    a = _inputs()
    a[11] = a[11] + 1
    assert not vsk.can_handle(*a)
    assert "ragged" in vsk.last_error()
    a[11] = "four"
    assert not vsk.can_handle(*a)
    a[11] = 0
    assert not vsk.can_handle(*a)


def test_rejects_shape_mismatches():
    q, ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle = _inputs()
    assert not vsk.can_handle(q[:, :15], ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle)  # 15 % 2
    assert not vsk.can_handle(q, ke, ve, kb[:, :1], vb, qo, kvp, kvi, cm, causal, mi, mle)
    assert not vsk.can_handle(q, ke, ve, kb, vb[:, :, :128], qo, kvp, kvi, cm, causal, mi, mle)
    assert not vsk.can_handle(q, ke[:, :, :128], ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle)
    assert not vsk.can_handle(q, ke, ve, kb, vb, qo[:1], kvp, kvi, cm, causal, mi, mle)  # bs < 1
    assert not vsk.can_handle(q, ke, ve, kb, vb, qo, kvp[:2], kvi, cm, causal, mi, mle)
    assert not vsk.can_handle(q[0], ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle)  # not 3-d


def test_rejects_unbuilt_dtypes_and_sizes():
    q, ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle = _inputs()
    assert not vsk.can_handle(q.half(), ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle)
    assert not vsk.can_handle(q, ke, ve, kb, vb.to(torch.float8_e4m3fn), qo, kvp, kvi, cm, causal, mi, mle)
    assert not vsk.can_handle(q, ke, ve, kb, vb, qo.long(), kvp, kvi, cm, causal, mi, mle)
    assert not vsk.can_handle(q, ke, ve, kb, vb, qo, kvp, kvi.float(), cm, causal, mi, mle)
    # head_dim not built
    spec = workloads.Spec("d96", (20,), 4, 4, 1, 96, 96, seed=4)
    p = workloads.make_problem(spec, "cpu")
    assert not vsk.can_handle(p["q"], p["k_ext"], p["v_ext"], p["k_buffer"], p["v_buffer"], p["qo_indptr"],
                              p["kv_indptr"], p["kv_indices"], None, True, None, 4)
    # D != Dv: built for D, Dv in {64, 128, 256}; any other v_head_dim is not
    spec = workloads.Spec("dne", (20,), 4, 4, 1, 64, 128, seed=4)
    p = workloads.make_problem(spec, "cpu")
    assert vsk.can_handle(p["q"], p["k_ext"], p["v_ext"], p["k_buffer"], p["v_buffer"], p["qo_indptr"],
                          p["kv_indptr"], p["kv_indices"], None, True, None, 4)
    spec = workloads.Spec("dv96", (20,), 4, 4, 1, 64, 96, seed=4)
    p = workloads.make_problem(spec, "cpu")
    assert not vsk.can_handle(p["q"], p["k_ext"], p["v_ext"], p["k_buffer"], p["v_buffer"], p["qo_indptr"],
                              p["kv_indptr"], p["kv_indices"], None, True, None, 4)
    assert "v_head_dim" in vsk.last_error()


def test_packed_row_limit():
    ok = workloads.Spec("r128", (20,), 8, 16, 1, 128, 128, seed=5)        # 16 * 8 = 128 rows
    too = workloads.Spec("r256", (20,), 8, 32, 1, 128, 128, seed=5)       # 256 rows
    d256 = workloads.Spec("r128d256", (20,), 8, 16, 1, 256, 256, seed=5)  # 128 rows at D=256
    for spec, want in ((ok, True), (too, False), (d256, False)):
        p = workloads.make_problem(spec, "cpu")
        got = vsk.can_handle(p["q"], p["k_ext"], p["v_ext"], p["k_buffer"], p["v_buffer"], p["qo_indptr"],
                             p["kv_indptr"], p["kv_indices"], None, True, None, 8)
        assert got == want, spec.name


def test_rejects_misaligned_pool():
    q, ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle = _inputs()
    flat = torch.zeros(kb.numel() + 8, dtype=torch.bfloat16)
    shifted = flat[1:1 + kb.numel()].view(kb.shape)  # 2-byte offset
    assert not vsk.can_handle(q, ke, ve, shifted, vb, qo, kvp, kvi, cm, causal, mi, mle)
    assert "16-byte" in vsk.last_error()


def test_fwd_returns_false_without_launch_when_gate_fails():
    a = _inputs()
    o = torch.empty(a[0].shape[0], 16, 256, dtype=torch.bfloat16)
    a[9] = False
    assert vsk.verify_splitkv_fwd(a[0], a[1], a[2], o, a[3], a[4], a[5], a[6], a[7], None, False, None, a[11],
                                  1.0, 1.0) is False


def test_c_fwd_rejects_bad_output_before_any_cuda_call():
    lib = _native.lib()
    q, ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle = _inputs()
    o_bad = torch.empty(q.shape[0], 16, 128, dtype=torch.bfloat16)  # wrong Dv
    r = vsk.api._ref
    ok = lib.verify_splitkv_fwd(r(q), r(ke), r(ve), r(o_bad), r(kb), r(vb), r(qo), r(kvp), r(kvi), 1, mle,
                                1.0, 1.0, 0.0, None, 0, None)
    assert ok == 0 and "o_extend" in vsk.last_error()


def test_workspace_bound_for_sms():
    lib = _native.lib()
    a = lib.vsk_workspace_size_for_sms(152, 64, 32, 8, 128, 128, 4)
    b = lib.vsk_workspace_size_for_sms(152, 128, 32, 8, 128, 128, 4)
    assert 0 < a < b
    # head_dim != v_head_dim: the partials hold v_head_dim columns
    c = lib.vsk_workspace_size_for_sms(152, 64, 32, 8, 128, 64, 4)
    d = lib.vsk_workspace_size_for_sms(152, 64, 32, 8, 128, 256, 4)
    assert 0 < c < a < d
    assert lib.vsk_workspace_size_for_sms(152, 64, 32, 8, 128, 96, 4) == 0
    # serving shape: partial slots (4 CTAs/SM bound + one per segment) x 8 heads x 16 rows x (128 + 1) fp32
    slots = 4 * 152 + 64
    assert a >= slots * 8 * 16 * 129 * 4
    assert a < 64 * 2 ** 20
    assert lib.vsk_workspace_size_for_sms(152, 64, 32, 8, 96, 96, 4) == 0
    assert lib.vsk_workspace_size_for_sms(0, 64, 32, 8, 128, 128, 4) == 0


def _header_functions():
    with open(_native.HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|void|char)\s*\*?\s*(\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    names = _header_functions()
    assert {"verify_splitkv_fwd", "vsk_can_handle", "vsk_workspace_size"} <= set(names)
    lib = ctypes.CDLL(_native.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/verify_splitkv.h but not exported"


def test_version_string():
    assert vsk.version().startswith("verify_splitkv-gb300")


def test_tree_entry_rejects_bad_mask_arguments():
    lib = _native.lib()
    q, ke, ve, kb, vb, qo, kvp, kvi, cm, causal, mi, mle = _inputs()
    o = torch.empty(q.shape[0], 16, 256, dtype=torch.bfloat16)
    r = vsk.api._ref
    good_mask = torch.ones(2 * 4 * (512 + 4), dtype=torch.uint8)
    good_ind = torch.tensor([0, 4 * 516, 8 * 516], dtype=torch.int64)
    for mask, ind, msg in ((good_mask.float(), good_ind, "uint8"), (good_mask, good_ind.float(), "int32 or int64"),
                           (good_mask, good_ind[:2], "B+1")):
        ok = lib.verify_splitkv_tree_fwd(r(q), r(ke), r(ve), r(o), r(kb), r(vb), r(qo), r(kvp), r(kvi), r(mask),
                                         r(ind), mle, 1.0, 1.0, 0.0, None, 0, None)
        assert ok == 0 and msg in vsk.last_error()


def test_python_tree_path_needs_skip_prefix():
    a = _inputs()
    o = torch.empty(a[0].shape[0], 16, 256, dtype=torch.bfloat16)
    mask = torch.ones(2 * 4 * 516, dtype=torch.uint8)
    ind = torch.tensor([0, 4 * 516, 8 * 516], dtype=torch.int64)
    assert vsk.verify_splitkv_fwd(a[0], a[1], a[2], o, a[3], a[4], a[5], a[6], a[7], mask, True, ind, a[11], 1.0, 1.0,
                                  skip_prefix_custom_mask=False) is False


def _paged_inputs(**over):
    spec = workloads.Spec("gate_paged", (100, 37), 4, 16, 2, 128, 128, page_size=16, seed=6)
    p = workloads.make_problem(spec, "cpu", **over)
    o = torch.empty(p["q"].shape, dtype=torch.bfloat16)
    return dict(q=p["q"], o=o, kc=p["k_buffer"], vc=p["v_buffer"], bt=p["block_table"], sl=p["seq_lens"],
                ps=16, mle=4)


def _paged_call(a):
    r = vsk.api._ref
    return _native.lib().verify_splitkv_paged_fwd(r(a["q"]), r(a["o"]), r(a["kc"]), r(a["vc"]), r(a["bt"]),
                                                  r(a["sl"]), a["ps"], a["mle"], 1.0, 1.0, 0.0, None, 0, None)


@pytest.mark.parametrize("change,msg", [
    (dict(ps=0), "page_size"),
    (dict(mle=3), "ragged"),
    (dict(bt="long"), "int32"),
    (dict(sl="long"), "int32"),
    (dict(bt="drop_row"), "one row per sequence"),
    (dict(kc="drop_rows"), "k_cache and v_cache"),
    (dict(kc="odd_pages", vc="odd_pages"), "whole number of pages"),
    (dict(o="short"), "o must be"),
    (dict(vc="fp8"), "both be bf16 or both fp8"),
    (dict(bt="one_col", ps=2), "fewer than max_len_extend"),
])
def test_paged_entry_rejects_bad_arguments(change, msg):
    a = _paged_inputs()
    for k, v in change.items():
        if v == "long":
            a[k] = a[k].long()
        elif v == "drop_row":
            a[k] = a[k][:1]
        elif v == "drop_rows":
            a[k] = a[k][:-16]
        elif v == "odd_pages":
            a[k] = a[k][:-1]
        elif v == "short":
            a[k] = a[k][:, :, :64]
        elif v == "fp8":
            a[k] = a[k].to(torch.float8_e4m3fn)
        elif v == "one_col":
            a[k] = a[k][:, :1].contiguous()
        else:
            a[k] = v
    assert _paged_call(a) == 0
    assert msg in vsk.last_error(), vsk.last_error()


def test_call_form_names_the_form_of_each_shape():
    """vsk_call_form: the form the planner takes for static shapes and the
    pool dtype (default switches), consistent with vsk_launches_per_call; then
    the head_dim 256 forms with the tensor-memory streams switched off, and
    with each of them forced."""
    f = vsk.call_form

    def check(cases):
        for args, want in cases:
            assert f(*args) == want, (args, f(*args))
            b, hq, hkv, d, dv, l, t, _ = args
            if want and d == dv:
                assert vsk.launches_per_call(b, hq, hkv, d, l, t) == (1 if want in ("cluster", "one_launch") else 2)

    rows = "tensor_memory_rows"
    check([
        ((2, 4, 1, 64, 64, 4, 160, False), "stream_only"),              # the tiny case
        ((4, 16, 2, 128, 128, 4, 1028, False), "stream_only"),          # 2,056 token-heads
        ((64, 32, 8, 128, 128, 4, 64 * 20000, False), "one_launch"),    # the serving batch
        ((3, 16, 2, 256, 256, 4, 1536, False), rows),                   # 3,072 token-heads
        ((2, 16, 2, 256, 256, 4, 72000, True), rows),                   # e4m3, R = 32: any size up to 2^23
        ((64, 16, 2, 256, 256, 4, 64 * 20000, True), rows),             # the long e4m3 batch
        ((1, 16, 2, 256, 256, 4, 393215, False), rows),                 # bf16, R = 32: below 786,432 token-heads
        ((1, 16, 2, 256, 256, 4, 393216, False), "stream_only"),        # ... from there
        ((64, 16, 2, 256, 256, 4, 64 * 20000, False), "stream_only"),   # the long bf16 batch
        ((8, 8, 2, 256, 256, 4, 8 * 20000, False), rows),               # bf16, R = 16: any size up to 2^23
        ((1, 8, 2, 256, 256, 4, 524287, True), rows),                   # e4m3, R = 16: below 2^20
        ((1, 8, 2, 256, 256, 4, 524288, True), "stream_only"),          # ... from there
        ((64, 16, 2, 256, 256, 4, 64 * 65536, True), rows),             # exactly 2^23 token-heads
        ((64, 16, 2, 256, 256, 4, 64 * 65537, True), "one_launch"),     # past 2^23 token-heads
        ((64, 16, 2, 256, 256, 4, 64 * 65537, False), "one_launch"),
        ((2, 64, 2, 256, 256, 4, 100, False), "one_launch"),            # R = 128
        ((2, 16, 2, 128, 256, 4, 1000, False), "one_launch"),           # head_dim != v_head_dim
        ((2, 16, 2, 96, 96, 4, 1000, False), ""),                       # not built
    ])
    try:
        vsk.set_tuning_tc(0)  # the mma.sync forms only
        check([
            ((3, 16, 2, 256, 256, 4, 1536, False), "column_split"),     # 3,072 token-heads
            ((2, 16, 2, 256, 256, 4, 72000, False), "column_split"),    # 144,000: below 2^18 (bf16)
            ((2, 16, 2, 256, 256, 4, 72000, True), "stream_only"),      # ... from 2^17 (e4m3)
            ((8, 8, 2, 256, 256, 4, 8 * 20000, False), "stream_only"),
            ((64, 16, 2, 256, 256, 4, 64 * 20000, True), "stream_only"),
            ((64, 16, 2, 256, 256, 4, 64 * 65537, False), "one_launch"),
        ])
        # a forced tensor-memory stream takes every head_dim 256 call of <= 32 packed rows
        for mode, want in ((1, "tensor_memory"), (2, rows)):
            vsk.set_tuning_tc(mode)
            assert f(64, 16, 2, 256, 256, 4, 64 * 20000, False) == want
            assert f(64, 16, 2, 256, 256, 4, 64 * 65537, True) == want
            assert f(3, 16, 2, 256, 256, 4, 1536, False) == want
            assert f(2, 64, 2, 256, 256, 4, 100, False) == "one_launch"   # R = 128
            assert f(64, 32, 8, 128, 128, 4, 64 * 20000, False) == "one_launch"
    finally:
        vsk.set_tuning_tc()


def test_launches_per_call_follows_the_form_switches():
    """Head_dim 256 with at most 32 packed rows per KV head takes two launches
    up to 2^23 prefix tokens x KV heads, whichever stream serves it: with the
    tensor-memory streams off (as here), the column-split stream below 2^18
    (bf16; 2^17 for e4m3 pools, which the host-only query does not know), the
    stream-only kernel from there, each followed by the combine launch; with
    the column split off, the stream-only form from 2,048.  The tensor-memory
    switch takes precedence (by default within the same 2^23 window).  Head_dim 64 / 128 with at most 32 drafts takes the
    stream-only kernel plus the combine launch inside its own size window.
    The cluster form (one launch; off by default) takes small calls first when
    it is on.  Everything else is one launch."""
    f = vsk.launches_per_call
    try:
        vsk.set_tuning_tc(0)
        vsk.set_tuning_cluster(1)
        # the cluster form (one launch): fewer than 2,048 token-heads, at most 512 segments
        assert f(2, 4, 1, 64, 4, 160) == 1                          # the tiny case
        assert f(4, 16, 2, 128, 4, 1020) == 1                       # 2,040 token-heads
        assert f(4, 16, 2, 128, 4, 1028) == 2                       # 2,056: stream + combine
        assert f(3, 16, 2, 256, 4, 1536) == 2                       # 3,072: column split + combine
        assert f(2, 64, 2, 256, 4, 100) == 1                        # R = 128 at head_dim 256: one-launch kernel
        assert f(300, 16, 2, 128, 4, 3000) == 2                     # 600 segments: past 512
        vsk.set_tuning_cluster(2)
        assert f(3, 16, 2, 256, 4, 1536) == 1                       # mode 2: wherever it applies
        assert f(64, 32, 8, 128, 4, 64 * 20000) == 1
        assert f(2, 64, 2, 256, 4, 100) == 1                        # (one-launch kernel: R = 128 at 256)
        vsk.set_tuning_cluster(0)
        vsk.set_tuning_colsplit(1)
        assert f(64, 32, 8, 128, 4, 64 * 20000) == 1                 # head_dim 128
        assert f(3, 16, 2, 256, 4, 1536) == 2                       # R = 32, 3,072 token-heads: column split
        assert f(8, 8, 2, 256, 4, 8 * 20000) == 2                   # R = 16, 320,000: stream only
        assert f(16, 16, 2, 256, 4, 524288) == 2                    # 1,048,576: stream only
        assert f(64, 16, 2, 256, 4, 64 * 20000) == 2                # the long batch: stream only
        assert f(64, 16, 2, 256, 4, 64 * 65536) == 2                # exactly 2^23 token-heads
        assert f(64, 16, 2, 256, 4, 64 * 65537) == 1                # one token past it per sequence
        assert f(2, 64, 2, 256, 4, 100) == 1                        # R = 128: one-launch kernel
        # head_dim 64 / 128: stream + combine up to 2^22 (R > 16) or 2^23 (R <= 16) token-heads
        assert f(2, 4, 1, 64, 4, 160) == 2                          # the tiny case
        assert f(2, 16, 2, 128, 4, 1024) == 2                       # 2,048 token-heads
        assert f(16, 16, 2, 128, 4, 2097152) == 2                   # R = 32, 2^22
        assert f(16, 16, 2, 128, 4, 2097168) == 1
        assert f(16, 32, 8, 128, 4, 1048576) == 2                   # R = 16, 2^23
        assert f(16, 32, 8, 128, 4, 1048592) == 1
        assert f(64, 32, 8, 128, 4, 64 * 20480) == 1                # the serving batch: one launch
        assert f(2, 64, 2, 128, 33, 4000) == 1                      # 33 drafts: beyond the combine kernel
        vsk.set_tuning_split_launch(0)
        assert f(16, 32, 8, 128, 4, 524288) == 1
        vsk.set_tuning_split_launch(2)
        assert f(64, 32, 8, 128, 4, 64 * 20000) == 2
        vsk.set_tuning_split_launch(1)
        vsk.set_tuning_colsplit(2)
        assert f(64, 16, 2, 256, 4, 64 * 20000) == 2
        assert f(64, 32, 8, 128, 4, 64 * 20000) == 1
        vsk.set_tuning_colsplit(0)
        assert f(3, 16, 2, 256, 4, 1536) == 2                       # stream only at any size
        assert f(2, 16, 2, 256, 4, 1000) == 2
        vsk.set_tuning_split_launch(0)
        assert f(3, 16, 2, 256, 4, 1536) == 1                       # both off: one launch
        vsk.set_tuning_split_launch(1)
        vsk.set_tuning_tc(True)
        assert f(64, 16, 2, 256, 4, 64 * 20000) == 2
        assert f(3, 16, 2, 256, 4, 1536) == 2                       # over the one-launch switches
        vsk.set_tuning_tc(2)
        assert f(64, 16, 2, 256, 4, 64 * 65537) == 2
        vsk.set_tuning_tc()                                          # the default: the 2^23 window
        assert f(3, 16, 2, 256, 4, 1536) == 2
        assert f(64, 16, 2, 256, 4, 64 * 65536) == 2
        assert f(64, 16, 2, 256, 4, 64 * 65537) == 1
    finally:
        vsk.set_tuning_tc()
        vsk.set_tuning_colsplit(1)
        vsk.set_tuning_split_launch(1)
        vsk.set_tuning_cluster(0)
    assert f(0, 16, 2, 256, 4, 10) == 0                             # no sequences
    assert f(2, 15, 2, 256, 4, 10) == 0                             # h_q not a multiple of h_kv
    assert f(2, 16, 2, 96, 4, 10) == 0                              # head_dim not built
