"""The launch count a call reports (vsk_launches_per_call, which bench.py's
gpu_launches uses) against the kernels the CUDA profiler sees for the call:
one launch for the one-launch kernel, two for the stream + combine forms."""
import pytest
import torch

import workloads
from test_parity_gpu import gpu_problem, run_gpu

pytestmark = pytest.mark.gpu
S = workloads.Spec


@pytest.fixture(scope="module")
def vsk():
    import speculative_decode_verify_prefix_gb300 as m
    from torch.profiler import ProfilerActivity, profile

    m.build()
    # the first profiling session of a process can come back empty while the
    # CUDA activity tracer starts: run one on a throwaway kernel
    with profile(activities=[ProfilerActivity.CUDA]):
        torch.ones(1024, device="cuda").sum()
        torch.cuda.synchronize()
    yield m
    m.set_tuning_tc()
    m.set_tuning_colsplit(1)
    m.set_tuning_split_launch(1)
    m.set_tuning_cluster(0)


def _kernels_of_one_call(vsk, p):
    from torch.profiler import ProfilerActivity, profile

    run_gpu(vsk, p)  # warm (library load, workspace)
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        run_gpu(vsk, p)
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    if not names:
        pytest.skip("the CUDA profiler recorded no kernels here")
    return [n for n in names if "vsk_" in n or "vtr_" in n or "vtc_" in n]


CASES = [
    # (spec, colsplit mode, split-launch mode, cluster mode, tensor-memory mode)
    (workloads.TINY, 1, 1, 1, 3),                                             # tiny: the cluster form (mode 1), one launch
    (workloads.TINY, 1, 1, 0, 3),                                             # tiny by default: stream only + combine
    (workloads.TINY, 1, 0, 0, 3),                                             # tiny, both off: one launch
    (workloads.D256, 1, 1, 0, 3),                                             # by default: rows-on-M stream + combine
    (workloads.FP8, 1, 1, 0, 3),                                              # (e4m3 too)
    (workloads.D256, 1, 1, 1, 0),                                             # past the cluster form's window
    (workloads.D256, 1, 1, 0, 0),                                             # column split + combine
    (workloads.D256, 0, 1, 0, 0),                                             # column split off: stream only + combine
    (workloads.D256, 0, 0, 0, 0),                                             # all off: one launch
    (workloads.D256, 0, 2, 0, 0),                                             # stream-only head_dim 256 + combine
    (S("lc_gqa", (3000, 2500), 4, 16, 2, 128, 128, perm=True, seed=790), 1, 1, 0, 3),  # stream + combine
    (S("lc_gqa_one", (3000, 2500), 4, 16, 2, 128, 128, perm=True, seed=790), 1, 0, 0, 3),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}_cs{c[1]}_sl{c[2]}_cl{c[3]}_tc{c[4]}")
def test_reported_launches_match_the_profiled_kernels(vsk, case):
    spec, cs, sl, cl, tc = case
    vsk.set_tuning_tc(tc)
    vsk.set_tuning_colsplit(cs)
    vsk.set_tuning_split_launch(sl)
    vsk.set_tuning_cluster(cl)
    p = gpu_problem(spec)
    B = len(p["prefix_lens"])
    want = vsk.launches_per_call(B, spec.h_q, spec.h_kv, spec.d, p["max_len_extend"], p["kv_indices"].shape[0])
    got = _kernels_of_one_call(vsk, p)
    assert want in (1, 2)
    assert len(got) == want, got
    if want == 2:
        assert any("vsk_combine_kernel" in n for n in got)
    if spec.d == 256 and cs == 0 and sl == 2:
        assert any("vsk_kernel<256, false, 1, 1, true" in n for n in got), got
    if spec.d == 256 and tc == 3 and cl == 0:
        assert any("vtr_kernel" in n for n in got), got
