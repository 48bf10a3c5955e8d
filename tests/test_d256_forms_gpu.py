"""GPU parity of the two-launch forms (a prefix stream, then the combine
kernel), against the fp64 oracle, with the one-launch mma.sync kernel checked
beside each:

- "tc": the tensor-memory stream (tcgen05.mma, accumulators in TMEM), head_dim 256,
  keys on the MMAs' M side;
- "tcr": the tensor-memory stream with the packed query rows on M (e4m3
  queries split into two exact e4m3 terms), head_dim 256;
- "colsplit": the column-split mma.sync stream (two warps per 16-row query
  tile, each holding half the head dimension), head_dim 256;
- "split": the stream-only mma.sync kernel at head_dim 64 and 128 (every case
  below rewritten to one of them, chosen by a hash of its name);
- "split256": the stream-only mma.sync kernel at head_dim 256 (one tile per
  warp; e4m3 pools with pipelined stages);
- "colsplit2": the column-split stream with both 16-row tiles in each warp
  of the pair (head_dim 256, 17 to 32 packed rows; cases with fewer rows take
  the one-tile split);
- "cluster": the cluster form (one launch: a thread-block cluster per
  (sequence, KV head) streams it and folds its own partials after a cluster
  barrier), at head_dim 64, 128 or 256 (chosen by a hash of the case's name).

All serve at most 32 packed query rows per KV head (head_dim 256) or 32 drafts
(64 / 128) and fold their partials after the stream: in a second launch, or
(the cluster form) in the same one.  Same tolerance as the other parity tests
(atol 2e-2, rtol 1e-2 on the bf16 output); stored cache codes and repeated /
graph-replayed calls are compared bit for bit.  Every call also checks the
device error word, whose timeout bit would report a pipeline wait that gave up.
"""
import numpy as np
import pytest
import torch

import zlib

import oracle
import workloads
from test_parity_gpu import gpu_problem as _gpu_problem
from test_parity_gpu import (_bits_np, _draft_rows, _free_rows, _pool_np, _subproblem, check,
                             check_every_sequence, oracle_o, run_gpu, run_paged, run_tree)

pytestmark = pytest.mark.gpu
S = workloads.Spec


FORM = {"name": "tc"}


def _adapt(spec):
    """The case as the form under test serves it: the "split" form runs it at
    head_dim 64 or 128, the "cluster" form at 64, 128 or 256."""
    h = zlib.crc32(spec.name.encode()) % 3
    if FORM["name"] == "split":
        d = 64 if h == 0 else 128
    elif FORM["name"] == "cluster":
        d = (64, 128, 256)[h]
    else:
        return spec
    return workloads.replace(spec, d=d, dv=d)


def gpu_problem(spec, **over):
    return _gpu_problem(_adapt(spec), **over)


def _select(m, form):
    m.set_tuning_tc(2 if form == "tcr" else 1 if form == "tc" else 0)
    m.set_tuning_colsplit(2 if form in ("colsplit", "colsplit2") else 0)
    m.set_tuning_colsplit2(2 if form == "colsplit2" else 0)
    m.set_tuning_split_launch(2 if form in ("split", "split256") else 0)
    m.set_tuning_cluster(2 if form == "cluster" else 0)


@pytest.fixture(scope="module", params=["tc", "tcr", "colsplit", "colsplit2", "split", "split256", "cluster"])
def vsk(request):
    import speculative_decode_verify_prefix_gb300 as m

    m.build()
    m.form = request.param
    FORM["name"] = m.form
    _select(m, m.form)
    yield m
    m.set_tuning(0, 0)
    m.set_tuning_tc()
    m.set_tuning_colsplit(1)
    m.set_tuning_colsplit2(1)
    m.set_tuning_split_launch(1)
    m.set_tuning_cluster(0)
    FORM["name"] = "tc"


def both(vsk, fn):
    """fn() on the form under test, then on the one-launch mma.sync kernel."""
    a = fn()
    _select(vsk, "one_launch")
    try:
        b = fn()
    finally:
        _select(vsk, vsk.form)
    return a, b


TC = [
    # prefixes around the 64-key tile: empty, one key, a tile minus / plus one, several tiles
    S("tc_ragged_bf16", (0, 1, 63, 64, 65, 127, 128, 129, 1000, 4097), 4, 16, 2, 256, 256, perm=True,
      pool_extra=40, seed=701),
    S("tc_ragged_fp8", (0, 1, 63, 64, 65, 191, 2000), 4, 16, 2, 256, 256, pool="e4m3", perm=True, k_scale=0.5,
      v_scale=0.25, seed=702),
    S("tc_rows16", (300, 1500, 7), 4, 8, 2, 256, 256, perm=True, seed=703),               # R = 16
    S("tc_rows8_fp8", (513, 2048), 2, 8, 2, 256, 256, pool="e4m3", perm=True, k_scale=1.5, v_scale=0.5,
      seed=704),                                                                          # R = 8 (16-row tile)
    S("tc_decode_l1", (4000, 31, 0, 65), 1, 32, 4, 256, 256, perm=True, seed=705),        # one draft, R = 8
    S("tc_hkv8_r32", (900, 2500), 4, 64, 8, 256, 256, perm=True, seed=706),               # 8 KV heads, R = 32
    S("tc_gq32_fp8", (3000, 100), 1, 32, 1, 256, 256, pool="e4m3", perm=True, k_scale=0.75, v_scale=1.25,
      seed=707),                                                                          # one KV head, R = 32
    S("tc_int32_idx", (700, 64, 1), 4, 16, 2, 256, 256, perm=True, idx_dtype="int32", seed=708),
    S("tc_bf16_scales", (1024, 2048), 3, 16, 2, 256, 256, k_scale=0.5, v_scale=0.25, seed=709),
    # 70,000 prefix tokens: at head_dim 64 / 128 warps take two 16-row tiles
    S("tc_two_tiles", (40000, 30000), 4, 16, 2, 256, 256, perm=True, seed=770),
    # more sequences than a block has threads (the combine kernel's length scan loops)
    S("tc_300_short", tuple(int(x) for x in np.random.default_rng(761).integers(0, 41, 300)), 4, 16, 2, 256, 256,
      perm=True, seed=761),
]


@pytest.mark.parametrize("spec", TC, ids=lambda s: s.name)
def test_form_matches_oracle(vsk, spec):
    p = gpu_problem(spec)
    ref = oracle_o(p)
    vsk.read_error_flags()
    a, b = both(vsk, lambda: run_gpu(vsk, p))
    assert vsk.read_error_flags() == 0
    check(a, ref)
    check(b, ref)


def _scale_k_rows(p, factor_of_position):
    """Multiply the K row of every referenced prefix token by a factor of its
    position in its sequence (the pool keeps its dtype)."""
    kb = p["k_buffer"]
    kf = kb.float()
    kvp = p["kv_indptr"].cpu().tolist()
    kvi = p["kv_indices"].long()
    for b in range(len(kvp) - 1):
        n = kvp[b + 1] - kvp[b]
        if n == 0:
            continue
        f = factor_of_position(torch.arange(n, device=kb.device, dtype=torch.float32), n)
        rows = kvi[kvp[b]:kvp[b + 1]]
        kf[rows] = kf[rows] * f[:, None, None]
    return dict(p, k_buffer=kf.to(kb.dtype))


@pytest.mark.parametrize("pool", ["bf16", "e4m3"])
def test_form_rising_scores_rescale_the_accumulator(vsk, pool):
    """K rows grow with their position, so scores keep rising along each
    prefix and the running maximum is raised (O rescaled in TMEM) many times
    inside a piece."""
    spec = S("tc_rising", (3000, 1777, 70), 4, 16, 2, 256, 256, pool=pool, perm=True, seed=711)
    p = _scale_k_rows(gpu_problem(spec), lambda t, n: 1.0 + 6.0 * t / n)
    vsk.read_error_flags()
    a, b = both(vsk, lambda: run_gpu(vsk, p))
    assert vsk.read_error_flags() == 0
    ref = oracle_o(p)
    check(a, ref)
    check(b, ref)


def test_form_single_dominant_key(vsk):
    """One key per sequence with a huge K row (scores of either sign, far
    beyond the others) late in the prefix: the maximum jumps once by a lot."""
    spec = S("tc_spike", (2000, 700), 4, 16, 2, 256, 256, perm=True, seed=712)
    p = _scale_k_rows(gpu_problem(spec), lambda t, n: torch.where(t == n - 37, 40.0, 1.0))
    a, b = both(vsk, lambda: run_gpu(vsk, p))
    ref = oracle_o(p)
    check(a, ref)
    check(b, ref)
    assert vsk.read_error_flags() == 0


TC_PAGED = [
    S("tcp_ps1", (0, 17, 300, 1024), 4, 16, 2, 256, 256, perm=True, page_size=1, pool_extra=33, seed=721),
    S("tcp_ps16_fp8", (700, 5, 90), 4, 16, 2, 256, 256, pool="e4m3", perm=True, page_size=16, k_scale=0.5,
      v_scale=0.25, seed=722),
    S("tcp_ps64", (1000, 63, 64, 0), 4, 16, 2, 256, 256, perm=True, page_size=64, k_scale=1.5, v_scale=0.75,
      seed=723),
    S("tcp_ps3_decode", (2000, 1, 0, 513), 1, 32, 8, 256, 256, perm=True, page_size=3, seed=724),
]


@pytest.mark.parametrize("spec", TC_PAGED, ids=lambda s: s.name)
def test_form_paged_matches_oracle(vsk, spec):
    p = gpu_problem(spec)
    ref = oracle_o(p)
    vsk.read_error_flags()
    a, b = both(vsk, lambda: run_paged(vsk, p))
    assert vsk.read_error_flags() == 0
    check(a, ref)
    check(b, ref)


TC_TREE = [
    S("tct_rand", (0, 17, 300, 1024), 4, 16, 2, 256, 256, perm=True, tree="random", seed=731),
    S("tct_star_fp8", (2000, 33), 4, 16, 2, 256, 256, pool="e4m3", perm=True, tree="star", k_scale=0.5,
      v_scale=2.0, seed=732),
]


@pytest.mark.parametrize("spec", TC_TREE, ids=lambda s: s.name)
def test_form_tree_matches_oracle(vsk, spec):
    p = gpu_problem(spec)
    ref = oracle_o(p)
    a, b = both(vsk, lambda: run_tree(vsk, p))
    check(a, ref)
    check(b, ref)
    assert vsk.read_error_flags() == 0


@pytest.mark.parametrize("pool", ["bf16", "e4m3"])
def test_form_fused_store_flat(vsk, pool):
    spec = S("tcw_flat", (700, 90, 0), 4, 16, 2, 256, 256, pool=pool, perm=True, pool_extra=32, k_scale=0.5,
             v_scale=0.25, seed=741)
    p = gpu_problem(spec)
    plain = run_gpu(vsk, p)
    loc = _free_rows(p, p["q"].shape[0], spec.seed)
    kb, vb = p["k_buffer"].clone(), p["v_buffer"].clone()
    o = torch.full_like(plain, float("nan"))
    vsk.read_error_flags()
    vsk.verify_splitkv_write_fwd(p["q"], p["k_ext"], p["v_ext"], o, kb, vb, p["qo_indptr"], p["kv_indptr"],
                                 p["kv_indices"], loc.cuda(), p["max_len_extend"], p["k_scale"], p["v_scale"],
                                 sm_scale=p["sm_scale"])
    torch.cuda.synchronize()
    assert vsk.read_error_flags() == 0
    assert torch.equal(o.view(torch.int16), plain.view(torch.int16))
    rows = loc.long().numpy()
    for pool_t, new, sc, old in ((kb, p["k_ext"], p["k_scale"], p["k_buffer"]),
                                 (vb, p["v_ext"], p["v_scale"], p["v_buffer"])):
        want = oracle.write_rows(_pool_np(old), rows, _bits_np(new), sc, pool)
        np.testing.assert_array_equal(_pool_np(pool_t), want)


@pytest.mark.parametrize("pool", ["bf16", "e4m3"])
def test_form_fused_store_paged(vsk, pool):
    spec = S("tcw_paged", (23, 1000, 0, 64), 4, 16, 2, 256, 256, pool=pool, perm=True, page_size=16,
             k_scale=1.5, v_scale=0.75, seed=742)
    p = gpu_problem(spec)
    g = torch.Generator(device="cuda").manual_seed(spec.seed + 1000)
    k_new = torch.randn(p["k_ext"].shape, generator=g, device="cuda").to(torch.bfloat16)
    v_new = torch.randn(p["v_ext"].shape, generator=g, device="cuda").to(torch.bfloat16)
    kc, vc = p["k_buffer"].clone(), p["v_buffer"].clone()
    o = torch.full(p["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vsk.read_error_flags()
    vsk.verify_splitkv_paged_write_fwd(p["q"], k_new, v_new, o, kc, vc, p["block_table"], p["seq_lens"],
                                       p["page_size"], p["max_len_extend"], p["k_scale"], p["v_scale"],
                                       sm_scale=p["sm_scale"])
    torch.cuda.synchronize()
    assert vsk.read_error_flags() == 0
    rows = _draft_rows(p)
    want_k = oracle.write_rows(_pool_np(p["k_buffer"]), rows, _bits_np(k_new), p["k_scale"], pool)
    want_v = oracle.write_rows(_pool_np(p["v_buffer"]), rows, _bits_np(v_new), p["v_scale"], pool)
    np.testing.assert_array_equal(_pool_np(kc), want_k)
    np.testing.assert_array_equal(_pool_np(vc), want_v)
    arrays = workloads.to_oracle_arrays(p)
    arrays["k_pool"], arrays["v_pool"] = want_k, want_v
    check(o, oracle.verify_forward(arrays)["o"])


@pytest.mark.parametrize("num_ctas,min_tok", [(1, 0), (3, 16), (150, 16), (1000, 16), (0, 64)])
def test_form_split_count_independence(vsk, num_ctas, min_tok):
    spec = S("tc_splits", (2000, 5, 0, 777, 64), 4, 16, 2, 256, 256, pool="e4m3", perm=True, k_scale=0.5,
             v_scale=1.5, seed=751)
    p = gpu_problem(spec)
    vsk.set_tuning(num_ctas, min_tok)
    try:
        o = run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
    check(o, oracle_o(p))
    assert vsk.read_error_flags() == 0


@pytest.mark.parametrize("pool", ["bf16", "e4m3"])
def test_form_two_tiles_per_warp(vsk, pool):
    """Warps with two 16-row tiles (forced; at head_dim 64 / 128 the stream-only
    kernel takes them from 2^18 prefix tokens): no effect on the head_dim 256
    forms."""
    spec = S(f"tc_two_tiles_forced_{pool}", (9000, 0, 4097, 700), 4, 16, 2, 256, 256, pool=pool, perm=True,
             k_scale=0.5 if pool == "e4m3" else 1.0, v_scale=0.75, seed=771)
    p = gpu_problem(spec)
    vsk.set_tuning_tiles(2)
    try:
        o = run_gpu(vsk, p)
    finally:
        vsk.set_tuning_tiles(0)
    check(o, oracle_o(p))
    assert vsk.read_error_flags() == 0


@pytest.mark.parametrize("pool", ["bf16", "e4m3"])
def test_form_one_segment_many_pieces(vsk, pool):
    """One sequence and one KV head cut into 1000 pieces (1000 stream CTAs of
    50 tokens): the combine step folds them all."""
    spec = S(f"tc_one_long_{pool}", (50000,), 4, 8, 1, 256, 256, pool=pool, perm=True,
             k_scale=0.5 if pool == "e4m3" else 1.0, seed=762)
    p = gpu_problem(spec)
    vsk.set_tuning(1000, 16)
    try:
        o = run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
    check(o, oracle_o(p))
    assert vsk.read_error_flags() == 0


def test_form_repeated_calls_and_graph_replay_identical(vsk):
    """Two launches per call (stream, then combine): no state is left behind,
    so repeated calls and CUDA-graph replays agree bit for bit."""
    spec = S("tc_repeat", (3000, 4000, 10), 4, 16, 2, 256, 256, perm=True, seed=752)
    p = gpu_problem(spec)
    vsk.set_tuning(16, 64)  # multi-CTA segments
    try:
        a = run_gpu(vsk, p)
        b = run_gpu(vsk, p)
        ws = vsk.get_workspace("cuda", 3, 16, 2, p["q"].shape[2], p["v_ext"].shape[2], 4)
        o = torch.empty_like(a)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run_gpu(vsk, p, o=o, workspace=ws)
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
    finally:
        vsk.set_tuning(0, 0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(o.view(torch.int16), a.view(torch.int16))
    check(a, oracle_o(p))


def test_form_poisoned_unreferenced_slots(vsk):
    spec = S("tc_poison", (40, 0, 129, 64), 4, 16, 2, 256, 256, perm=True, pool_extra=300, poison=True, seed=753)
    p = gpu_problem(spec)
    check(run_gpu(vsk, p), oracle_o(p))
    assert vsk.read_error_flags() == 0


@pytest.mark.parametrize("spec", TC[:4] + TC[9:10], ids=lambda s: s.name)
def test_form_with_programmatic_dependent_launch(vsk, spec):
    """The two-launch forms with the combine kernel launched as a
    programmatic dependent of the stream (it starts early and waits for the
    stream grid before reading partials), forced on: bitwise the result of
    plain stream order, forced off."""
    p = gpu_problem(spec)
    vsk.read_error_flags()
    vsk.set_tuning_pdl(0)
    try:
        a = run_gpu(vsk, p)
        vsk.set_tuning_pdl(2)
        b = run_gpu(vsk, p)
        c = run_gpu(vsk, p)
    finally:
        vsk.set_tuning_pdl(1)
    assert vsk.read_error_flags() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))
    check(b, oracle_o(p))


def test_form_out_of_range_index_is_flagged_not_read(vsk):
    spec = S("tc_badidx", (50, 130), 4, 16, 2, 256, 256, seed=754)
    p = gpu_problem(spec)
    ref_other = oracle_o(p)
    kvi = p["kv_indices"].clone()
    kvi[55] = p["k_buffer"].shape[0]      # one past the pool (sequence 1, key 5)
    kvi[150] = -3                         # negative (sequence 1, key 100)
    vsk.read_error_flags()
    o = run_gpu(vsk, dict(p, kv_indices=kvi))
    assert vsk.read_error_flags() & 1
    assert torch.isfinite(o.float()).all()
    check(o, ref_other, rows=slice(0, 4))  # sequence 0 untouched
    keep = torch.ones(130, dtype=torch.bool)
    keep[[5, 100]] = False
    p3 = dict(p, kv_indices=torch.cat([kvi[:50], kvi[50:][keep.cuda()]]),
              kv_indptr=torch.tensor([0, 50, 178], dtype=torch.int32, device="cuda"))
    check(o, oracle_o(p3), rows=slice(4, 8))  # sequence 1 without those two keys


def test_form_fp8_long_every_sequence(vsk):
    """The e4m3 head_dim 256 benchmark shape (64 sequences, prefixes
    U[8192, 32768]) in this form; the oracle checks every sequence with the
    page's tolerance and the magnitude-scaled bound."""
    spec = S("fp8_b64_p8k_32k", None, 4, 16, 2, 256, 256, pool="e4m3", perm=True, k_scale=0.5, v_scale=0.25,
             batch=64, len_range=(8192, 32768), seed=1240)
    p = gpu_problem(spec)
    o = run_gpu(vsk, p)
    assert torch.isfinite(o.float()).all()
    assert vsk.read_error_flags() == 0
    check_every_sequence(p, o, planted_seq=0)
    del p
    torch.cuda.empty_cache()


def _tc_cases(n=24, seed=2025):
    """Seeded random head_dim 256 problems the tensor-memory stream serves
    (at most 32 packed rows per KV head): lengths, head layouts, pools, scales,
    index dtypes, forms (causal, tree, paged) and CTA splits."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        h_kv = int(rng.choice([1, 2, 4, 8]))
        L = int(rng.integers(1, 9))
        gq = int(rng.choice([g for g in (1, 2, 4, 8) if g * L <= 32]))
        B = int(rng.integers(1, 6))
        kind = rng.choice(["empty", "short", "mid", "long"], size=B, p=[0.1, 0.3, 0.4, 0.2])
        lens = tuple(int({"empty": 0, "short": rng.integers(1, 70), "mid": rng.integers(70, 700),
                          "long": rng.integers(700, 3000)}[k]) for k in kind)
        form = str(rng.choice(["flat", "tree", "paged"], p=[0.5, 0.2, 0.3]))
        pool = str(rng.choice(["bf16", "e4m3"]))
        ks = float(rng.choice([1.0, 0.5, 1.5])) if pool == "e4m3" else float(rng.choice([1.0, 0.75]))
        vs = float(rng.choice([1.0, 0.5, 2.0])) if pool == "e4m3" else float(rng.choice([1.0, 1.25]))
        spec = S(f"tcfuzz{i}_{form}", lens, L, gq * h_kv, h_kv, 256, 256, pool=pool, perm=bool(rng.integers(0, 2)),
                 k_scale=ks, v_scale=vs, idx_dtype=str(rng.choice(["int32", "int64"])),
                 pool_extra=int(rng.integers(0, 64)), poison=bool(rng.integers(0, 2)),
                 tree="random" if form == "tree" else "",
                 page_size=int(rng.choice([1, 3, 16, 64])) if form == "paged" else 0, seed=4000 + i)
        tuning = (0, 0) if rng.random() < 0.6 else (int(rng.integers(1, 400)), 16)
        out.append((spec, form, tuning))
    return out


@pytest.mark.parametrize("case", _tc_cases(), ids=lambda c: c[0].name)
def test_form_random_problem_matches_oracle(vsk, case):
    spec, form, (nc, mt) = case
    p = workloads.make_problem(_adapt(spec), "cuda")
    vsk.read_error_flags()
    vsk.set_tuning(nc, mt)
    try:
        o = run_tree(vsk, p) if form == "tree" else run_paged(vsk, p) if form == "paged" else run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
    check(o, oracle_o(p))
    assert vsk.read_error_flags() == 0
