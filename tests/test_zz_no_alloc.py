"""The allocation-free entry point against the oracle and the workspace entry point.

verify_splitkv_fwd_noalloc exists for callers that may not allocate device
memory: engines that hand all free HBM to their own pool allocator at start-up
(a stray cudaMalloc there can fail, fragment the pool or stall the device) and
plugin hosts whose interface passes only input and output pointers.  Its
scratch is an array built into the library's device image, shared by every
call and keeping whatever the previous call left.

These tests call it through the C ABI several times in a row, with problems
of different shapes and forms in turn (a head_dim 256 e4m3 call served by the
rows-on-M tensor-memory stream plus a combine launch, a head_dim 128 stream plus combine,
a cluster-form call and a one-launch call with tickets), so each call runs on
what a differently shaped call left in the array.  Each result is compared with the fp64 oracle (the page's
tolerance and the magnitude-scaled bound of the other parity tests) and with
verify_splitkv_fwd given a caller workspace.  The device's free memory must
not change across the calls.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2
SCALED = 1e-2
NOALLOC_SCRATCH = ctypes.c_void_p(1)  # VSK_NOALLOC_SCRATCH: selects the built-in scratch


@pytest.fixture(scope="module")
def lib():
    import speculative_decode_verify_prefix_gb300 as vsk
    from speculative_decode_verify_prefix_gb300 import _native

    vsk.build()
    vsk.set_tuning(0, 0)
    L = _native.lib()
    P = ctypes.POINTER(_native.VskTensor)
    L.verify_splitkv_fwd_noalloc.restype = ctypes.c_int
    L.verify_splitkv_fwd_noalloc.argtypes = [P] * 9 + [ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                                       ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
    return L


def _noalloc(lib, p, o, kv_indices=None):
    import speculative_decode_verify_prefix_gb300 as vsk

    r = vsk.api._ref
    stream = torch.cuda.current_stream()
    kvi = p["kv_indices"] if kv_indices is None else kv_indices
    return lib.verify_splitkv_fwd_noalloc(
        r(p["q"]), r(p["k_ext"]), r(p["v_ext"]), r(o), r(p["k_buffer"]), r(p["v_buffer"]), r(p["qo_indptr"]),
        r(p["kv_indptr"]), r(kvi), 1, p["max_len_extend"], p["k_scale"], p["v_scale"],
        p["sm_scale"], ctypes.c_void_p(stream.cuda_stream))


def _noalloc_flags(lib):
    flags = ctypes.c_uint32(0)
    stream = torch.cuda.current_stream()
    assert lib.vsk_read_error_flags(NOALLOC_SCRATCH, ctypes.c_void_p(stream.cuda_stream), ctypes.byref(flags)) == 1
    return int(flags.value)


def _with_workspace(p):
    import speculative_decode_verify_prefix_gb300 as vsk

    q = p["q"]
    o = torch.empty(q.shape[0], q.shape[1], p["v_ext"].shape[2], dtype=torch.bfloat16, device=q.device)
    ws = torch.zeros(vsk.workspace_size(len(p["prefix_lens"]), q.shape[1], p["k_ext"].shape[1], q.shape[2],
                                        p["v_ext"].shape[2], p["max_len_extend"]), dtype=torch.uint8,
                     device=q.device)
    assert vsk.verify_splitkv_fwd(q, p["k_ext"], p["v_ext"], o, p["k_buffer"], p["v_buffer"], p["qo_indptr"],
                                  p["kv_indptr"], p["kv_indices"], None, True, None, p["max_len_extend"],
                                  p["k_scale"], p["v_scale"], sm_scale=p["sm_scale"], workspace=ws)
    torch.cuda.synchronize()
    return o


def _check(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - ref)
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"max abs err {err.max():.3e}"
    assert err.max() <= SCALED * np.abs(ref).max(), f"max abs err {err.max():.3e} vs max|ref| {np.abs(ref).max():.3e}"


# four shapes and forms, called in turn: each call finds the array as a call
# of another shape (another workspace layout) left it.  Form switches:
# (cluster, column split, stream + combine) modes.
SPECS = [
    (workloads.Spec("noalloc_fp8_d256", (4096, 1500), 4, 16, 2, 256, 256, pool="e4m3", perm=True, k_scale=0.5,
                    v_scale=0.25, seed=202), (0, 1, 1), 2),    # rows-on-M tensor-memory stream + combine
    (workloads.Spec("noalloc_bf16_d128", (3000, 4000, 10, 0, 777), 4, 32, 8, 128, 128, perm=True, seed=201),
     (0, 1, 1), 2),                                            # stream + combine
    (workloads.Spec("noalloc_tiny", (64, 96), 4, 4, 1, 64, 64, seed=204), (1, 1, 1), 1),  # the cluster form
    (workloads.Spec("noalloc_one_launch", (2500, 33, 700), 4, 16, 2, 128, 128, perm=True, seed=206),
     (0, 1, 0), 1),                                            # one launch: tickets in the array
]


def _form(modes):
    import speculative_decode_verify_prefix_gb300 as vsk

    cl, cs, sl = modes
    vsk.set_tuning_cluster(cl)
    vsk.set_tuning_colsplit(cs)
    vsk.set_tuning_split_launch(sl)


def test_noalloc_matches_oracle_across_shapes(lib):
    import speculative_decode_verify_prefix_gb300 as vsk

    probs = [workloads.make_problem(spec, "cuda") for spec, _, _ in SPECS]
    try:
        for (spec, modes, launches), p in zip(SPECS, probs):
            _form(modes)
            assert vsk.launches_per_call(len(p["prefix_lens"]), spec.h_q, spec.h_kv, spec.d, spec.l_ext,
                                         p["kv_indices"].shape[0]) == launches, spec.name
        refs = [oracle.verify_forward(workloads.to_oracle_arrays(p))["o"] for p in probs]
        with_ws = []
        for (_, modes, _), p in zip(SPECS, probs):
            _form(modes)
            with_ws.append(_with_workspace(p).float().cpu().numpy())
        outs = [torch.empty(p["q"].shape[0], p["q"].shape[1], p["v_ext"].shape[2], dtype=torch.bfloat16,
                            device="cuda") for p in probs]
        # one round first: the library's module and kernels are loaded
        for (_, modes, _), p, o in zip(SPECS, probs, outs):
            _form(modes)
            assert _noalloc(lib, p, o) == 1, lib.vsk_last_error().decode()
        torch.cuda.synchronize()
        n = len(SPECS)
        for rnd in range(2):
            for i in range(n) if rnd == 0 else reversed(range(n)):
                _form(SPECS[i][1])
                outs[i].fill_(float("nan"))
                torch.cuda.synchronize()
                free0 = torch.cuda.mem_get_info()[0]
                assert _noalloc(lib, probs[i], outs[i]) == 1, lib.vsk_last_error().decode()
                torch.cuda.synchronize()
                assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated"
                _check(outs[i], refs[i])
                np.testing.assert_allclose(outs[i].float().cpu().numpy(), with_ws[i], atol=ATOL, rtol=RTOL)
                assert _noalloc_flags(lib) == 0
    finally:
        _form((0, 1, 1))


def test_noalloc_flags_an_out_of_range_index(lib):
    spec = workloads.Spec("noalloc_badidx", (50, 130), 4, 16, 2, 128, 128, seed=205)
    p = workloads.make_problem(spec, "cuda")
    ref = oracle.verify_forward(workloads.to_oracle_arrays(p))["o"]
    kvi = p["kv_indices"].clone()
    kvi[55] = p["k_buffer"].shape[0]  # one past the pool (sequence 1)
    o = torch.empty(p["q"].shape[0], 16, 128, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, p, o, kv_indices=kvi) == 1, lib.vsk_last_error().decode()
    torch.cuda.synchronize()
    assert _noalloc_flags(lib) & 1
    _check(o[:4], ref[:4])  # sequence 0 does not read the bad index
    # the next call starts from a clear error word
    assert _noalloc(lib, p, o) == 1
    torch.cuda.synchronize()
    assert _noalloc_flags(lib) == 0
    _check(o, ref)


def test_noalloc_rejects_problems_beyond_the_builtin_scratch(lib):
    spec = workloads.Spec("noalloc_big", tuple([4] * 2048), 4, 32, 8, 128, 128, seed=203)
    p = workloads.make_problem(spec, "cuda")
    o = torch.empty(p["q"].shape[0], 32, 128, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, p, o) == 0
    msg = lib.vsk_last_error().decode()
    assert "bytes of scratch" in msg and "built into the library" in msg
