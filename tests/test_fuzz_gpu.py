"""Randomised GPU parity sweep: seeded random shapes, lengths, head layouts,
pool dtypes, index dtypes, scales, verify forms (causal, tree, paged) and CTA
splits, each compared element by element with the fp64 oracle.  The draws are
fixed (seed 2024), so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

import workloads
from test_parity_gpu import check, oracle_o, run_gpu, run_paged, run_tree

pytestmark = pytest.mark.gpu


def _cases(n=48, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(rng.choice([64, 128, 256]))
        h_kv = int(rng.choice([1, 2, 4, 8]))
        max_r = 64 if d == 256 else 128
        L = int(rng.integers(1, 9))
        gq = int(rng.choice([g for g in (1, 2, 4, 8) if g * L <= max_r]))
        B = int(rng.integers(1, 7))
        kind = rng.choice(["empty", "short", "mid", "long"], size=B, p=[0.1, 0.3, 0.4, 0.2])
        lens = tuple(int({"empty": 0, "short": rng.integers(1, 40), "mid": rng.integers(40, 700),
                          "long": rng.integers(700, 3000)}[k]) for k in kind)
        form = str(rng.choice(["flat", "tree", "paged"], p=[0.45, 0.25, 0.3]))
        pool = str(rng.choice(["bf16", "e4m3"]))
        ks = float(rng.choice([1.0, 0.5, 1.5, 0.25])) if pool == "e4m3" else float(rng.choice([1.0, 0.75]))
        vs = float(rng.choice([1.0, 0.5, 2.0, 0.25])) if pool == "e4m3" else float(rng.choice([1.0, 1.25]))
        spec = workloads.Spec(f"fuzz{i}_{form}", lens, L, gq * h_kv, h_kv, d, d, pool=pool,
                              perm=bool(rng.integers(0, 2)), k_scale=ks, v_scale=vs,
                              idx_dtype=str(rng.choice(["int32", "int64"])),
                              pool_extra=int(rng.integers(0, 64)), poison=bool(rng.integers(0, 2)),
                              tree="random" if form == "tree" else "",
                              page_size=int(rng.choice([1, 3, 16, 64])) if form == "paged" else 0,
                              seed=3000 + i)
        tuning = (0, 0) if rng.random() < 0.6 else (int(rng.integers(1, 400)), 16)
        out.append((spec, form, tuning))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def vsk():
    import speculative_decode_verify_prefix_gb300 as m

    m.build()
    yield m
    m.set_tuning(0, 0)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_random_problem_matches_oracle(vsk, case):
    spec, form, (nc, mt) = case
    p = workloads.make_problem(spec, "cuda")
    vsk.read_error_flags()
    vsk.set_tuning(nc, mt)
    try:
        if form == "tree":
            o = run_tree(vsk, p)
        elif form == "paged":
            o = run_paged(vsk, p)
        else:
            o = run_gpu(vsk, p)
    finally:
        vsk.set_tuning(0, 0)
    check(o, oracle_o(p))
    assert vsk.read_error_flags() == 0
