"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance: atol 2e-2, rtol 1e-2 on the bf16 output against the oracle's fp64
value (the parity tolerance of the "test_verify_splitkv.py" page); integer
index handling is checked bit-exactly (int32 vs int64 indices, pool-slot
permutations, repeated calls).

At long prefixes the outputs are small (a softmax-weighted mean of thousands
of N(0, 1) rows: |o| of order 1/sqrt(n)), so the page's absolute tolerance
alone would pass an output that is off by tens of percent.  The long-context
cases therefore also bound the error by a fraction of the output's magnitude:
max |err| <= SCALED * max |ref|.  The kernels' own error is bf16 rounding of
the output (at most 2^-9 of |o|) and of the softmax weights, about 0.3 % of
max |ref| at most, so SCALED = 1e-2 leaves room for rounding and none for a
wrong result (a dropped piece, a wrong scale).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2
SCALED = 1e-2  # max |err| <= SCALED * max |ref| on the long-context cases


@pytest.fixture(scope="module")
def vsk():
    import speculative_decode_verify_prefix_gb300 as m

    m.build()
    yield m
    m.set_tuning(0, 0)


def run_gpu(vsk, prob, o=None, **kw):
    q = prob["q"]
    if o is None:
        o = torch.full((q.shape[0], q.shape[1], prob["v_ext"].shape[2]), float("nan"), dtype=torch.bfloat16,
                       device=q.device)
    cm = kw.pop("custom_mask", None)
    mi = kw.pop("mask_indptr", None)
    ran = vsk.verify_splitkv_fwd(q, prob["k_ext"], prob["v_ext"], o, prob["k_buffer"], prob["v_buffer"],
                                 prob["qo_indptr"], prob["kv_indptr"], prob["kv_indices"], cm, True, mi,
                                 prob["max_len_extend"], prob["k_scale"], prob["v_scale"],
                                 sm_scale=prob["sm_scale"], **kw)
    assert ran, vsk.last_error()
    torch.cuda.synchronize()
    return o


def oracle_o(prob, **kw):
    return oracle.verify_forward(workloads.to_oracle_arrays(prob), **kw)["o"]


def check(got, ref, atol=ATOL, rtol=RTOL, rows=None, scaled=None):
    """The page's tolerance element by element and, with ``scaled``, also
    max |err| <= scaled * max |ref| (the bound scaled to the output's
    magnitude).  Returns the largest absolute error."""
    g = got.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} elements out of tolerance; max abs err {err.max():.3e}"
    if scaled is not None:
        bound = scaled * float(np.abs(ref).max())
        assert err.max() <= bound, f"max abs err {err.max():.3e} above {scaled:g} x max|ref| = {bound:.3e}"
    return float(err.max())


def check_every_sequence(p, o, scaled=SCALED, planted_seq=None):
    """Every sequence of a large batch (all heads, all draft rows) against the
    oracle, one sequence at a time (its referenced pool rows gathered to the
    host), each with the magnitude-scaled bound.  With ``planted_seq``, that
    sequence's oracle output is also scaled by 1.1 (a mistake planted in the
    oracle's result, on the CPU) and the check must reject it, which shows the
    scaled bound sees a 10 % error the page's absolute tolerance lets through.
    Returns the largest error relative to max |ref| over the batch."""
    worst = 0.0
    for b in range(len(p["prefix_lens"])):
        sub, (s, e) = _subproblem(p, b)
        ref = oracle_o(sub, nthreads=0)
        err = check(o[s:e], ref, scaled=scaled)
        worst = max(worst, err / float(np.abs(ref).max()))
        if b == planted_seq:
            planted = ref * 1.1
            check(o[s:e], planted)  # the page's tolerance alone: passes
            with pytest.raises(AssertionError):
                check(o[s:e], planted, scaled=scaled)
    return worst


def gpu_problem(spec, **over):
    return workloads.make_problem(spec, "cuda", **over)


# ----------------------------------------------------------------- the five workloads
def test_tiny(vsk):
    p = gpu_problem(workloads.TINY)
    o, ref = run_gpu(vsk, p), oracle_o(p)
    err = check(o, ref)
    assert err < 4e-3  # bf16 output rounding plus bf16 softmax weights, nothing more
    assert vsk.read_error_flags() == 0


def test_head_dim_256(vsk):
    p = gpu_problem(workloads.D256)
    check(run_gpu(vsk, p), oracle_o(p), scaled=SCALED)


@pytest.mark.parametrize("spec", workloads.gqa_sweep(), ids=lambda s: s.name)
def test_gqa_extend_sweep(vsk, spec):
    p = gpu_problem(spec)
    check(run_gpu(vsk, p), oracle_o(p), scaled=SCALED)


def test_fp8_pool_with_scales(vsk):
    p = gpu_problem(workloads.FP8)
    o, ref = run_gpu(vsk, p), oracle_o(p)
    err = check(o, ref, scaled=SCALED)
    assert err < 2e-3  # fp8 decode is exact on both sides; outputs are ~v_scale/sqrt(n)


DV_PAIRS = [(64, 128), (64, 256), (128, 64), (128, 256), (256, 64), (256, 128)]


@pytest.mark.parametrize("pool", ["bf16", "e4m3"])
@pytest.mark.parametrize("d,dv", DV_PAIRS, ids=lambda x: str(x))
def test_head_dim_differs_from_v_head_dim(vsk, d, dv, pool):
    """head_dim != v_head_dim (the value rows, the partials and the output
    have v_head_dim columns), one launch; empty, short and multi-piece
    prefixes, permuted pool slots, scales on the e4m3 pool."""
    fp8 = pool == "e4m3"
    spec = workloads.Spec(f"dv_{d}_{dv}_{pool}", (0, 17, 300, 2500), 4, 16, 2, d, dv, pool=pool, perm=True,
                          pool_extra=20, k_scale=0.5 if fp8 else 1.0, v_scale=0.75 if fp8 else 1.0,
                          seed=900 + d + dv + (7 if fp8 else 0))
    p = gpu_problem(spec)
    assert vsk.launches_per_call(4, 16, 2, d, 4, p["kv_indices"].shape[0]) >= 1
    vsk.read_error_flags()
    o = run_gpu(vsk, p)
    assert o.shape[2] == dv
    check(o, oracle_o(p), scaled=SCALED)
    assert vsk.read_error_flags() == 0
    # the split of the prefix across CTAs changes the rounding order only
    vsk.set_tuning(7, 16)
    try:
        o2 = run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
    check(o2, oracle_o(p), scaled=SCALED)


def _subproblem(prob, b):
    """Sequence b alone, with its referenced pool rows gathered to the host."""
    kvp, qo = prob["kv_indptr"].cpu(), prob["qo_indptr"].cpu()
    s, e = int(qo[b]), int(qo[b + 1])
    ps, pe = int(kvp[b]), int(kvp[b + 1])
    loc = prob["kv_indices"][ps:pe].long()
    uniq, inv = torch.unique(loc, return_inverse=True)
    sub = {
        "q": prob["q"][s:e].cpu(), "k_ext": prob["k_ext"][s:e].cpu(), "v_ext": prob["v_ext"][s:e].cpu(),
        "k_buffer": prob["k_buffer"][uniq].cpu(), "v_buffer": prob["v_buffer"][uniq].cpu(),
        "qo_indptr": torch.tensor([0, e - s], dtype=torch.int32),
        "kv_indptr": torch.tensor([0, pe - ps], dtype=torch.int32),
        "kv_indices": inv.cpu().to(torch.int64),
        "sm_scale": prob["sm_scale"], "k_scale": prob["k_scale"], "v_scale": prob["v_scale"],
    }
    return sub, (s, e)


def test_serving_scale_every_sequence(vsk):
    """Full serving-scale batch (64 sequences, prefixes U[8192, 32768]) in the
    benchmark's launch configuration; the oracle checks every sequence (all
    heads, all draft rows) with the page's tolerance and the magnitude-scaled
    bound, and a 10 % error planted in the oracle's result is rejected."""
    p = gpu_problem(workloads.SERVING)
    o = run_gpu(vsk, p)
    assert torch.isfinite(o.float()).all()
    assert vsk.read_error_flags() == 0
    worst = check_every_sequence(p, o, planted_seq=0)
    assert worst < 5e-3, worst  # bf16 rounding only
    del p
    torch.cuda.empty_cache()


def test_head_dim_256_long_every_sequence(vsk):
    """The bf16 head_dim 256 benchmark shape (64 sequences, prefixes
    U[8192, 32768], h_q/h_kv 16/2, 4 drafts) in its default form; the oracle
    checks every sequence with the page's tolerance and the magnitude-scaled
    bound, and a 10 % error planted in the oracle's result is rejected."""
    spec = workloads.Spec("d256_b64_p8k_32k", None, 4, 16, 2, 256, 256, perm=True, batch=64,
                          len_range=(8192, 32768), seed=1239)
    p = gpu_problem(spec)
    o = run_gpu(vsk, p)
    assert torch.isfinite(o.float()).all()
    assert vsk.read_error_flags() == 0
    worst = check_every_sequence(p, o, planted_seq=0)
    assert worst < 5e-3, worst  # bf16 rounding only
    del p
    torch.cuda.empty_cache()


# ----------------------------------------------------------------- edge cases
EDGE = [
    workloads.Spec("mixed_ragged_empty", (0, 1, 15, 16, 17, 300, 0, 1000), 3, 8, 2, 128, 128, perm=True,
                   pool_extra=50, seed=101),
    workloads.Spec("all_empty", (0, 0, 0), 4, 8, 4, 128, 128, seed=102),
    workloads.Spec("l1_decode", (700, 33), 1, 32, 8, 128, 128, perm=True, seed=103),
    workloads.Spec("rows128", (333, 1024), 8, 16, 1, 128, 128, perm=True, seed=104),
    workloads.Spec("d256_rows64", (250, 517), 8, 16, 2, 256, 256, perm=True, seed=105),
    workloads.Spec("d64_hkv8", (129, 77, 400), 4, 32, 8, 64, 64, perm=True, seed=106),
    workloads.Spec("bf16_scales", (1024, 2048), 4, 16, 2, 256, 256, k_scale=0.5, v_scale=0.25, seed=107),
    workloads.Spec("fp8_d64", (100, 257), 2, 8, 4, 64, 64, pool="e4m3", perm=True, k_scale=2.0, v_scale=0.5,
                   seed=108),
    workloads.Spec("fp8_d128_hkv8", (1000, 35, 513), 4, 32, 8, 128, 128, pool="e4m3", perm=True, k_scale=0.75,
                   v_scale=1.5, seed=109),
    workloads.Spec("hkv6", (200, 90), 3, 12, 6, 128, 128, perm=True, seed=110),
    workloads.Spec("single_seq_long", (20000,), 4, 8, 2, 128, 128, perm=True, seed=111),
    # 600 short sequences: the block scan gives each thread several sequences
    workloads.Spec("many_short_seqs", None, 2, 8, 2, 64, 64, perm=True, batch=600, len_range=(0, 40), seed=119),
    # one 200k-token prefix: a long segment merged in two levels
    workloads.Spec("one_200k_prefix", (200000,), 4, 16, 2, 128, 128, perm=True, seed=120),
]


LONG_EDGE = {"rows128", "bf16_scales", "single_seq_long", "one_200k_prefix"}


@pytest.mark.parametrize("spec", EDGE, ids=lambda s: s.name)
def test_edge_cases(vsk, spec):
    p = gpu_problem(spec)
    check(run_gpu(vsk, p), oracle_o(p), scaled=SCALED if spec.name in LONG_EDGE else None)
    assert vsk.read_error_flags() == 0


def test_poisoned_unreferenced_slots(vsk):
    spec = workloads.Spec("poison", (40, 0, 129), 4, 8, 2, 128, 128, perm=True, pool_extra=300, poison=True,
                          seed=112)
    p = gpu_problem(spec)
    check(run_gpu(vsk, p), oracle_o(p))


@pytest.mark.parametrize("num_ctas,min_tok", [(1, 0), (2, 16), (3, 16), (7, 16), (64, 16), (1000, 16), (0, 16)])
def test_split_count_independence(vsk, num_ctas, min_tok):
    spec = workloads.Spec("splits", (2000, 5, 0, 777, 64), 4, 16, 4, 128, 128, perm=True, seed=113)
    p = gpu_problem(spec)
    vsk.set_tuning_cluster(0)  # the forms whose split the CTA count sets
    try:
        vsk.set_tuning(0, 0)
        base = run_gpu(vsk, p).float()
        vsk.set_tuning(num_ctas, min_tok)
        o = run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
        vsk.set_tuning_cluster(0)
    check(o, oracle_o(p))
    assert (o.float() - base).abs().max().item() < 1e-3 * 8  # a few bf16 ulps at |o| < 1


def test_int32_indices_bitwise_equal(vsk):
    spec = workloads.Spec("idx", (500, 37, 1200), 4, 16, 2, 128, 128, perm=True, pool_extra=20, seed=114)
    a = run_gpu(vsk, gpu_problem(spec))
    b = run_gpu(vsk, gpu_problem(spec, idx_dtype="int32"))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_slot_permutation_bitwise_equal(vsk):
    spec = workloads.Spec("slots", (300, 1000), 4, 8, 2, 128, 128, perm=True, pool_extra=7, seed=115)
    p = gpu_problem(spec)
    a = run_gpu(vsk, p)
    n = p["k_buffer"].shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(9)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n, device="cuda")
    p2 = dict(p, k_buffer=p["k_buffer"][perm].contiguous(), v_buffer=p["v_buffer"][perm].contiguous(),
              kv_indices=inv[p["kv_indices"]])
    b = run_gpu(vsk, p2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_repeated_calls_identical(vsk):
    """Tickets are left at zero after each call and pieces merge in a fixed
    order: back-to-back calls agree bitwise."""
    spec = workloads.Spec("repeat", (3000, 4000, 10), 4, 32, 8, 128, 128, perm=True, seed=116)
    p = gpu_problem(spec)
    vsk.set_tuning(16, 64)  # force multi-CTA segments
    try:
        a = run_gpu(vsk, p)
        b = run_gpu(vsk, p)
        c = run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_strided_views(vsk):
    """Pool heads not contiguous within a token and q/o as strided views."""
    spec = workloads.Spec("strided", (300, 45), 4, 8, 2, 128, 128, perm=True, seed=117)
    p = gpu_problem(spec)
    ref = oracle_o(p)
    big_k = torch.zeros(p["k_buffer"].shape[0], 2, 2 * 128, dtype=torch.bfloat16, device="cuda")
    big_v = torch.zeros_like(big_k)
    big_k[:, :, 64:192] = p["k_buffer"]
    big_v[:, :, 128:256] = p["v_buffer"]
    big_q = torch.zeros(p["q"].shape[0], 8, 3 * 128, dtype=torch.bfloat16, device="cuda")
    big_q[:, :, 128:256] = p["q"]
    big_o = torch.full((p["q"].shape[0], 8, 2 * 128), 7.0, dtype=torch.bfloat16, device="cuda")
    p2 = dict(p, k_buffer=big_k[:, :, 64:192], v_buffer=big_v[:, :, 128:256], q=big_q[:, :, 128:256])
    run_gpu(vsk, p2, o=big_o[:, :, 0:128])
    check(big_o[:, :, 0:128], ref)
    assert (big_o[:, :, 128:] == 7.0).all()  # nothing written outside the view


def test_out_of_range_index_is_flagged_not_read(vsk):
    spec = workloads.Spec("badidx", (50, 60), 2, 4, 1, 64, 64, seed=118)
    p = gpu_problem(spec)
    ref_other = oracle_o(p)
    kvi = p["kv_indices"].clone()
    kvi[55] = p["k_buffer"].shape[0]      # one past the pool (sequence 1)
    kvi[70] = -3                          # negative (sequence 1)
    p2 = dict(p, kv_indices=kvi)
    vsk.read_error_flags()
    o = run_gpu(vsk, p2)
    assert vsk.read_error_flags() & 1
    assert torch.isfinite(o.float()).all()
    check(o, ref_other, rows=slice(0, 2))  # sequence 0 untouched
    # sequence 1 equals the definition with those two keys removed
    keep = torch.ones(60, dtype=torch.bool)
    keep[[5, 20]] = False
    p3 = dict(p, kv_indices=torch.cat([kvi[:50], kvi[50:][keep.cuda()]]),
              kv_indptr=torch.tensor([0, 50, 108], dtype=torch.int32, device="cuda"))
    check(o, oracle_o(p3), rows=slice(2, 4))


def test_cuda_graph_replay_matches_eager(vsk):
    spec = workloads.Spec("graph", (900, 50, 2048), 4, 32, 8, 128, 128, perm=True, seed=119)
    p = gpu_problem(spec)
    eager = run_gpu(vsk, p)
    ws = vsk.get_workspace("cuda", 3, 32, 8, 128, 128, 4)
    o = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_gpu(vsk, p, o=o, workspace=ws)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    o.fill_(0)
    with torch.cuda.graph(g):
        vsk.verify_splitkv_fwd(p["q"], p["k_ext"], p["v_ext"], o, p["k_buffer"], p["v_buffer"], p["qo_indptr"],
                               p["kv_indptr"], p["kv_indices"], None, True, None, 4, 1.0, 1.0,
                               sm_scale=p["sm_scale"], workspace=ws)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), eager.view(torch.int16))


# ----------------------------------------------------------------- tree verify (custom mask)
TREES = [
    workloads.Spec("tree_rand_l8", (0, 17, 300, 1024), 8, 16, 2, 128, 128, perm=True, tree="random", seed=201),
    workloads.Spec("tree_star_l4", (2000, 33), 4, 32, 8, 128, 128, perm=True, tree="star", seed=202),
    workloads.Spec("tree_rand_d256_fp8", (700, 90), 6, 16, 2, 256, 256, pool="e4m3", perm=True, tree="random",
                   k_scale=0.5, v_scale=0.25, seed=203),
    workloads.Spec("tree_rand_d64_l16", (129, 64), 16, 8, 1, 64, 64, perm=True, tree="random", seed=204),
    workloads.Spec("tree_rand_d256_dv128", (500, 33), 6, 8, 2, 256, 128, perm=True, tree="random", seed=205),
]


def run_tree(vsk, prob, o=None, **kw):
    return run_gpu(vsk, prob, o=o, custom_mask=prob["custom_mask"], mask_indptr=prob["mask_indptr"], **kw)


@pytest.mark.parametrize("spec", TREES, ids=lambda s: s.name)
def test_tree_verify_matches_oracle(vsk, spec):
    p = gpu_problem(spec)
    check(run_tree(vsk, p), oracle_o(p))
    assert vsk.read_error_flags() == 0


def test_chain_tree_is_bitwise_the_causal_path(vsk):
    spec = workloads.Spec("chain", (500, 0, 1200), 4, 32, 8, 128, 128, perm=True, tree="chain", seed=205)
    p = gpu_problem(spec)
    a = run_gpu(vsk, p)
    b = run_tree(vsk, p)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_tree_prefix_columns_and_indptr_dtype(vsk):
    spec = workloads.Spec("cols", (77, 300), 5, 8, 2, 128, 128, perm=True, tree="random", seed=206)
    p = gpu_problem(spec)
    a = run_tree(vsk, p)
    cm = p["custom_mask"].clone()
    mi = p["mask_indptr"].cpu()
    for b, P in enumerate(p["prefix_lens"]):
        cm[int(mi[b]):int(mi[b + 1])].view(5, P + 5)[:, :P] = 0
    b_ = run_gpu(vsk, p, custom_mask=cm.bool(), mask_indptr=p["mask_indptr"].to(torch.int32))
    assert torch.equal(a.view(torch.int16), b_.view(torch.int16))


def test_tree_row_with_nothing_visible_is_zero(vsk):
    spec = workloads.Spec("emptyrow", (0, 40), 3, 4, 1, 64, 64, tree="chain", seed=207)
    p = gpu_problem(spec)
    cm = p["custom_mask"].clone()
    cm[3:6] = 0  # sequence 0, draft row 1: no prefix and no visible draft
    p2 = dict(p, custom_mask=cm)
    o = run_tree(vsk, p2)
    ref = oracle_o(p2)
    check(o, ref)
    assert (o[1].float() == 0).all()


def test_tree_bad_mask_indptr_is_flagged_not_read(vsk):
    spec = workloads.Spec("badmask", (50, 60), 4, 8, 2, 128, 128, tree="random", seed=208)
    p = gpu_problem(spec)
    mi = p["mask_indptr"].clone()
    mi[1] = p["custom_mask"].numel()  # sequence 1's rows would start past the end
    vsk.read_error_flags()
    o = run_gpu(vsk, p, custom_mask=p["custom_mask"], mask_indptr=mi)
    assert vsk.read_error_flags() & 16
    causal = oracle_o({k: v for k, v in p.items() if k not in ("custom_mask", "mask_indptr")})
    check(o, causal, rows=slice(4, 8))              # sequence 1 fell back to causal drafts
    check(o, oracle_o(p), rows=slice(0, 4))         # sequence 0 kept its tree


# ----------------------------------------------------------------- drafts already in a paged cache
PAGED = [
    workloads.Spec("paged_ps1", (0, 17, 300, 1024), 4, 16, 2, 128, 128, perm=True, page_size=1, pool_extra=33,
                   seed=301),
    workloads.Spec("paged_ps16_fp8", (700, 5, 90), 4, 32, 8, 128, 128, pool="e4m3", perm=True, page_size=16,
                   k_scale=0.5, v_scale=0.25, seed=302),
    workloads.Spec("paged_ps64_d256", (1000, 63, 64, 0), 6, 16, 2, 256, 256, perm=True, page_size=64,
                   k_scale=1.5, v_scale=0.75, seed=303),
    workloads.Spec("paged_decode_ps16", (2000, 1, 0, 513, 16), 1, 32, 8, 128, 128, perm=True, page_size=16,
                   seed=304),
    workloads.Spec("paged_ps32_d64_l8", (129, 4000), 8, 8, 1, 64, 64, pool="e4m3", perm=True, page_size=32,
                   k_scale=2.0, v_scale=0.5, seed=305),
    # page sizes that are not powers of two (the page division is a multiply-high)
    workloads.Spec("paged_ps3", (1, 2, 3, 1000), 3, 16, 4, 128, 128, perm=True, page_size=3, seed=311),
    workloads.Spec("paged_ps24_fp8", (23, 24, 25, 3000), 4, 8, 2, 128, 128, pool="e4m3", perm=True, page_size=24,
                   k_scale=0.75, v_scale=1.25, seed=312),
    workloads.Spec("paged_ps100_d64", (99, 100, 101, 1234), 5, 16, 8, 64, 64, perm=True, page_size=100, seed=313),
    # head_dim != v_head_dim
    workloads.Spec("paged_ps16_d128_dv64", (300, 0, 1500), 4, 16, 2, 128, 64, perm=True, page_size=16, seed=314),
    workloads.Spec("paged_ps8_d64_dv256_fp8", (77, 900), 2, 16, 4, 64, 256, pool="e4m3", perm=True, page_size=8,
                   k_scale=0.5, v_scale=1.5, seed=315),
]


def run_paged(vsk, prob, o=None, **kw):
    q = prob["q"]
    if o is None:
        o = torch.full((q.shape[0], q.shape[1], prob["v_buffer"].shape[2]), float("nan"), dtype=torch.bfloat16,
                       device=q.device)
    vsk.verify_splitkv_paged_fwd(q, o, prob["k_buffer"], prob["v_buffer"], prob["block_table"], prob["seq_lens"],
                                 prob["page_size"], prob["max_len_extend"], prob["k_scale"], prob["v_scale"],
                                 sm_scale=prob["sm_scale"], **kw)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("spec", PAGED, ids=lambda s: s.name)
def test_paged_drafts_match_oracle(vsk, spec):
    p = gpu_problem(spec)
    vsk.read_error_flags()
    check(run_paged(vsk, p), oracle_o(p))
    assert vsk.read_error_flags() == 0


def test_paged_poisoned_pages(vsk):
    spec = workloads.Spec("paged_poison", (40, 0, 129), 4, 8, 2, 128, 128, perm=True, page_size=16, pool_extra=200,
                          poison=True, seed=306)
    p = gpu_problem(spec)
    check(run_paged(vsk, p), oracle_o(p))


def test_paged_bf16_unit_scales_is_bitwise_the_flat_path(vsk):
    """With a bf16 cache and unit scales the paged call and the flat call
    (prefix through kv_indices, drafts gathered into k_extend / v_extend) see
    the same keys in the same order and must agree bit for bit."""
    spec = workloads.Spec("paged_vs_flat", (900, 3, 0, 2500), 4, 32, 8, 128, 128, perm=True, page_size=16, seed=307)
    p = gpu_problem(spec)
    vsk.set_tuning(0, 256)  # the same split for both (their default floors come from different static shapes)
    vsk.set_tuning_cluster(0)  # (the cluster form sizes its clusters from the static shapes too)
    try:
        a = run_paged(vsk, p)
        b = run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
        vsk.set_tuning_cluster(0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_paged_split_count_independence(vsk):
    spec = workloads.Spec("paged_splits", (2000, 5, 777), 4, 16, 4, 128, 128, perm=True, page_size=8, seed=308)
    p = gpu_problem(spec)
    ref = oracle_o(p)
    for n in (1, 7, 1000):
        vsk.set_tuning(n, 16)
        vsk.set_tuning_cluster(0)  # the forms whose split the CTA count sets
        try:
            o = run_paged(vsk, p)
        finally:
            vsk.set_tuning(0, 0)
            vsk.set_tuning_cluster(0)
        check(o, ref)


def test_paged_bad_page_and_length_are_flagged_not_read(vsk):
    spec = workloads.Spec("paged_bad", (50, 60, 70), 2, 4, 1, 64, 64, page_size=16, seed=309)
    p = gpu_problem(spec)
    ref = oracle_o(p)
    n_pages = p["k_buffer"].shape[0] // 16
    bt = p["block_table"].clone()
    bt[1, 1] = n_pages          # one past the cache: positions 16..31 of sequence 1
    sl = p["seq_lens"].clone()
    sl[2] = -5                  # sequence 2: negative length
    vsk.read_error_flags()
    o = run_paged(vsk, dict(p, block_table=bt, seq_lens=sl))
    flags = vsk.read_error_flags()
    assert flags & 1 and flags & 2
    assert torch.isfinite(o.float()).all()
    check(o, ref, rows=slice(0, 2))  # sequence 0 untouched
    # sequence 1 equals the definition with positions 16..31 of its prefix removed
    keep = torch.ones(60, dtype=torch.bool)
    keep[16:32] = False
    kvi = p["kv_indices"].cpu()
    p3 = dict(p, kv_indices=torch.cat([kvi[:50], kvi[50:110][keep]]).cuda(),
              kv_indptr=torch.tensor([0, 50, 94, 94], dtype=torch.int32, device="cuda"))
    p3.pop("block_table")
    check(o, oracle_o(p3), rows=slice(2, 4))


def test_paged_cuda_graph_replay(vsk):
    spec = workloads.Spec("paged_graph", (900, 50, 2048), 4, 32, 8, 128, 128, perm=True, page_size=16, seed=310)
    p = gpu_problem(spec)
    eager = run_paged(vsk, p)
    ws = vsk.get_workspace("cuda", 3, 32, 8, 128, 128, 4)
    o = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_paged(vsk, p, o=o, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    o.fill_(0)
    with torch.cuda.graph(g):
        vsk.verify_splitkv_paged_fwd(p["q"], o, p["k_buffer"], p["v_buffer"], p["block_table"], p["seq_lens"], 16, 4,
                                     sm_scale=p["sm_scale"], workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), eager.view(torch.int16))


# ----------------------------------------------------------------- fused store of the new drafts
def _bits_np(t):
    return workloads._bits(t)


def _pool_np(t):
    a = t.cpu().contiguous()
    return a.view(torch.uint8).numpy() if a.dtype == torch.float8_e4m3fn else a.view(torch.int16).numpy().view(np.uint16)


WRITE_FLAT = [
    workloads.Spec("write_bf16", (300, 0, 1000), 4, 16, 2, 128, 128, perm=True, pool_extra=64, seed=401),
    workloads.Spec("write_fp8_d256", (700, 90), 4, 16, 2, 256, 256, pool="e4m3", perm=True, pool_extra=32,
                   k_scale=0.5, v_scale=0.25, seed=402),
    workloads.Spec("write_fp8_d64_l8", (129, 64, 5), 8, 8, 1, 64, 64, pool="e4m3", perm=True, pool_extra=48,
                   k_scale=2.0, v_scale=0.75, seed=403),
    workloads.Spec("write_bf16_scaled", (500,), 3, 32, 8, 128, 128, perm=True, pool_extra=8, k_scale=1.5,
                   v_scale=0.5, seed=404),
    workloads.Spec("write_fp8_d128_dv256", (400, 7), 4, 16, 2, 128, 256, pool="e4m3", perm=True, pool_extra=40,
                   k_scale=0.5, v_scale=0.25, seed=405),
]


def _free_rows(p, n, seed):
    """n distinct pool rows that no prefix references, in random order."""
    used = torch.zeros(p["k_buffer"].shape[0], dtype=torch.bool)
    used[p["kv_indices"].cpu()] = True
    free = torch.nonzero(~used).flatten()
    assert free.numel() >= n
    return free[torch.randperm(free.numel(), generator=torch.Generator().manual_seed(seed))[:n]]


@pytest.mark.parametrize("spec", WRITE_FLAT, ids=lambda s: s.name)
@pytest.mark.parametrize("loc_dtype", [torch.int64, torch.int32])
def test_fused_store_flat(vsk, spec, loc_dtype):
    p = gpu_problem(spec)
    plain = run_gpu(vsk, p)
    n = p["q"].shape[0]
    loc = _free_rows(p, n, spec.seed).to(loc_dtype)
    kb, vb = p["k_buffer"].clone(), p["v_buffer"].clone()
    o = torch.full_like(plain, float("nan"))
    vsk.read_error_flags()
    vsk.verify_splitkv_write_fwd(p["q"], p["k_ext"], p["v_ext"], o, kb, vb, p["qo_indptr"], p["kv_indptr"],
                                 p["kv_indices"], loc.cuda(), p["max_len_extend"], p["k_scale"], p["v_scale"],
                                 sm_scale=p["sm_scale"])
    torch.cuda.synchronize()
    assert vsk.read_error_flags() == 0
    assert torch.equal(o.view(torch.int16), plain.view(torch.int16))  # the attention is untouched
    dt = "e4m3" if spec.pool == "e4m3" else "bf16"
    rows = loc.long().numpy()
    for pool, new, sc in ((kb, p["k_ext"], p["k_scale"]), (vb, p["v_ext"], p["v_scale"])):
        old = p["k_buffer"] if pool is kb else p["v_buffer"]
        want = oracle.write_rows(_pool_np(old), rows, _bits_np(new), sc, dt)
        np.testing.assert_array_equal(_pool_np(pool), want)  # exactly those rows, exactly those codes


PAGED_WRITE = [
    workloads.Spec("pwrite_ps16_fp8", (700, 5, 90, 0), 4, 32, 8, 128, 128, pool="e4m3", perm=True, page_size=16,
                   k_scale=0.5, v_scale=0.25, seed=411),
    workloads.Spec("pwrite_ps1_bf16", (0, 17, 300), 4, 16, 2, 128, 128, perm=True, page_size=1, seed=412),
    workloads.Spec("pwrite_ps3_d256_fp8", (23, 1000), 6, 16, 2, 256, 256, pool="e4m3", perm=True, page_size=3,
                   k_scale=1.5, v_scale=0.75, seed=413),
    workloads.Spec("pwrite_decode_ps64_d64", (2000, 1, 63), 1, 8, 8, 64, 64, perm=True, page_size=64, k_scale=0.8,
                   v_scale=1.25, seed=414),
    workloads.Spec("pwrite_ps16_bf16_poison", (40, 0, 129), 4, 8, 2, 128, 128, perm=True, page_size=16,
                   pool_extra=200, poison=True, k_scale=1.25, v_scale=2.0, seed=415),
    workloads.Spec("pwrite_ps16_d256_dv64_fp8", (600, 3), 4, 16, 2, 256, 64, pool="e4m3", perm=True, page_size=16,
                   k_scale=0.5, v_scale=0.75, seed=416),
]


def _draft_rows(p):
    bt, ps, L = p["block_table"].cpu().numpy(), p["page_size"], p["max_len_extend"]
    rows = []
    for b, P in enumerate(p["prefix_lens"]):
        j = np.arange(P, P + L)
        rows.append(bt[b, j // ps].astype(np.int64) * ps + j % ps)
    return np.concatenate(rows)


@pytest.mark.parametrize("spec", PAGED_WRITE, ids=lambda s: s.name)
def test_fused_store_paged(vsk, spec):
    p = gpu_problem(spec)
    g = torch.Generator(device="cuda").manual_seed(spec.seed + 1000)
    k_new = torch.randn(p["k_ext"].shape, generator=g, device="cuda").to(torch.bfloat16)
    v_new = torch.randn(p["v_ext"].shape, generator=g, device="cuda").to(torch.bfloat16)
    kc, vc = p["k_buffer"].clone(), p["v_buffer"].clone()
    o = torch.full((p["q"].shape[0], p["q"].shape[1], vc.shape[2]), float("nan"), dtype=torch.bfloat16,
                   device="cuda")
    vsk.read_error_flags()
    vsk.verify_splitkv_paged_write_fwd(p["q"], k_new, v_new, o, kc, vc, p["block_table"], p["seq_lens"],
                                       p["page_size"], p["max_len_extend"], p["k_scale"], p["v_scale"],
                                       sm_scale=p["sm_scale"])
    torch.cuda.synchronize()
    assert vsk.read_error_flags() == 0
    dt = "e4m3" if spec.pool == "e4m3" else "bf16"
    rows = _draft_rows(p)
    want_k = oracle.write_rows(_pool_np(p["k_buffer"]), rows, _bits_np(k_new), p["k_scale"], dt)
    want_v = oracle.write_rows(_pool_np(p["v_buffer"]), rows, _bits_np(v_new), p["v_scale"], dt)
    np.testing.assert_array_equal(_pool_np(kc), want_k)
    np.testing.assert_array_equal(_pool_np(vc), want_v)
    # attention = the definition over the cache as stored
    arrays = workloads.to_oracle_arrays(p)
    arrays["k_pool"], arrays["v_pool"] = want_k, want_v
    check(o, oracle.verify_forward(arrays)["o"])
    # ... and bit for bit what the plain paged call computes on that cache
    again = run_paged(vsk, dict(p, k_buffer=kc, v_buffer=vc))
    assert torch.equal(o.view(torch.int16), again.view(torch.int16))


def test_one_workspace_serves_calls_of_any_shape(vsk):
    """Tickets sit at a fixed place at the end of the buffer: calls of
    different batch sizes, head counts and CTA counts sharing one caller
    workspace agree bitwise with calls on a fresh zeroed workspace."""
    specs = [
        workloads.Spec("ws_a", (3000, 200, 4000, 17, 900, 1200, 5, 2500), 4, 32, 8, 128, 128, perm=True, seed=501),
        workloads.Spec("ws_b", (5000, 64), 4, 16, 2, 256, 256, perm=True, seed=502),
        workloads.Spec("ws_c", (2000, 5, 0, 777, 64), 4, 16, 4, 128, 128, perm=True, seed=503),
    ]
    shared = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    plan = [(0, 0, 0), (1000, 16, 0), (64, 16, 0), (0, 0, 1), (7, 16, 0), (300, 16, 0)]
    for i, (nc, mt, cl) in enumerate(plan):
        for spec in specs:
            p = gpu_problem(spec)
            vsk.set_tuning(nc, mt)
            vsk.set_tuning_cluster(cl)  # mostly the forms with tickets or a second launch
            try:
                got = run_gpu(vsk, p, workspace=shared)
                fresh = run_gpu(vsk, p, workspace=torch.zeros_like(shared))
            finally:
                vsk.set_tuning(0, 0)
                vsk.set_tuning_cluster(0)
            assert torch.equal(got.view(torch.int16), fresh.view(torch.int16)), (i, spec.name)
    assert vsk.read_error_flags(shared) == 0


def test_large_ticket_region_on_a_reused_buffer(vsk):
    """A one-launch call with more than 16,384 tickets (decode, l_ext = 1,
    h_q / h_kv = 32 / 8, 9,000 short prefixes: two per segment plus one per
    CTA) on a buffer whose bytes before its last 64 KiB are not zero, as an
    earlier call's partials leave them: the part of the ticket region beyond
    the last 64 KiB is cleared by the call itself.  Checked against the
    oracle on two calls in a row, the first after a head_dim 256 call with a
    large partial region on the same buffer."""
    rng = np.random.default_rng(801)
    spec = workloads.Spec("tickets_9000", tuple(int(x) for x in rng.integers(0, 9, 9000)), 1, 32, 8, 128, 128,
                          perm=True, seed=801)
    big = workloads.Spec("tickets_first", None, 4, 16, 2, 256, 256, perm=True, batch=48, len_range=(2000, 6000),
                         seed=802)
    p = gpu_problem(spec)
    B = len(spec.prefix_lens)
    need = vsk.workspace_size(B, 32, 8, 128, 128, 1)
    assert need > 0
    shared = torch.full((need + (1 << 20),), 0x5A, dtype=torch.uint8, device="cuda")
    shared[:256] = 0        # the error word
    shared[-65536:] = 0     # the tail every call leaves at zero
    ref = oracle_o(p)
    vsk.set_tuning_split_launch(0)  # the one-launch kernel: the form that draws tickets
    vsk.set_tuning_colsplit(0)
    vsk.set_tuning_cluster(0)
    vsk.set_tuning_tc(0)
    try:
        assert vsk.launches_per_call(B, 32, 8, 128, 1, p["kv_indices"].shape[0]) == 1
        pb = gpu_problem(big)
        ob = run_gpu(vsk, pb, workspace=shared)
        for _ in range(2):
            o = run_gpu(vsk, p, workspace=shared)
            check(o, ref)
        assert vsk.read_error_flags(shared) == 0
    finally:
        vsk.set_tuning_split_launch(1)
        vsk.set_tuning_colsplit(1)
        vsk.set_tuning_cluster(0)
        vsk.set_tuning_tc()
    check(ob, oracle_o(pb), scaled=SCALED)


def test_head_dim_256_stream_only_with_64_packed_rows(vsk):
    """The stream-only head_dim 256 kernel with four 16-row tiles per KV head
    (h_q / h_kv = 16, 4 drafts), forced on, then the combine kernel."""
    spec = workloads.Spec("so256_r64", (3000, 0, 1700, 65), 4, 16, 1, 256, 256, perm=True, seed=851)
    p = gpu_problem(spec)
    vsk.set_tuning_colsplit(0)
    vsk.set_tuning_split_launch(2)
    vsk.set_tuning_cluster(0)
    try:
        assert vsk.launches_per_call(4, 16, 1, 256, 4, p["kv_indices"].shape[0]) == 2
        o = run_gpu(vsk, p)
    finally:
        vsk.set_tuning_colsplit(1)
        vsk.set_tuning_split_launch(1)
        vsk.set_tuning_cluster(0)
    check(o, oracle_o(p), scaled=SCALED)
    assert vsk.read_error_flags() == 0


def _combine_grid_specs():
    # The combine kernel stages 2 x nb pieces per CTA, nb chosen by its grid
    # (16 up to two CTAs per SM, 8 up to three, 4 beyond).  With 32 combine
    # CTAs per sequence at both shapes below, 8 / 12 / 20 sequences fall in the
    # three classes on a 152-SM GB300; lengths up to 3,000 tokens give
    # segments of tens of pieces, so several batches run per CTA.
    rng = np.random.default_rng(811)
    out = []
    for B in (8, 12, 20):
        lens = tuple(int(x) for x in rng.integers(100, 3000, B))
        out.append(workloads.Spec(f"combine_b{B}_d128", lens, 4, 32, 8, 128, 128, perm=True, seed=811 + B))
        out.append(workloads.Spec(f"combine_b{B}_d256_fp8", lens, 4, 16, 2, 256, 256, pool="e4m3", perm=True,
                                  k_scale=0.5, v_scale=0.25, seed=831 + B))
    return out


@pytest.mark.parametrize("spec", _combine_grid_specs(), ids=lambda s: s.name)
def test_combine_kernel_grid_sizes(vsk, spec):
    """Two-launch calls whose combine grids take each staging batch size."""
    p = gpu_problem(spec)
    B = len(spec.prefix_lens)
    assert vsk.launches_per_call(B, spec.h_q, spec.h_kv, spec.d, spec.l_ext, p["kv_indices"].shape[0]) == 2
    check(run_gpu(vsk, p), oracle_o(p), scaled=SCALED)
    assert vsk.read_error_flags() == 0


TILES = [
    workloads.Spec("tiles_r32", (700, 0, 2100), 4, 16, 2, 128, 128, perm=True, seed=601),
    workloads.Spec("tiles_r64_fp8", (333, 1500), 8, 8, 1, 128, 128, pool="e4m3", perm=True, k_scale=0.5,
                   v_scale=0.75, seed=602),
    workloads.Spec("tiles_r128_d64", (90, 1200), 8, 16, 1, 64, 64, perm=True, seed=603),
    workloads.Spec("tiles_r32_tree", (40, 900), 4, 8, 1, 128, 128, perm=True, tree="random", seed=604),
    workloads.Spec("tiles_r32_paged_fp8", (17, 1000), 4, 16, 2, 128, 128, pool="e4m3", perm=True, page_size=16,
                   k_scale=1.5, v_scale=0.5, seed=605),
]


@pytest.mark.parametrize("tiles", [1, 2])
@pytest.mark.parametrize("spec", TILES, ids=lambda s: s.name)
def test_one_or_two_tiles_per_warp(vsk, spec, tiles):
    """Packed rows > 16 at head_dim <= 128: each consumer warp serves one or
    two 16-row tiles; both CTA shapes match the oracle."""
    p = gpu_problem(spec)
    vsk.set_tuning_tiles(tiles)
    try:
        if spec.tree:
            o = run_tree(vsk, p)
        elif spec.page_size:
            o = run_paged(vsk, p)
        else:
            o = run_gpu(vsk, p)
    finally:
        vsk.set_tuning_tiles(0)
    check(o, oracle_o(p))
    assert vsk.read_error_flags() == 0
