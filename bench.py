"""Benchmark: split-KV verify attention on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one call of the whole hot path (one verify_splitkv_fwd launch) over
the serving-scale verify batch: B = 64 sequences, prefix lengths drawn
uniformly from [8192, 32768], l_ext = 4 draft rows, h_q = 32, h_kv = 8,
head_dim 128, bf16 K/V pool addressed through a random permutation
(page size 1).  Inputs are synthetic and seeded (workloads.py), resident in
HBM when the timed region starts, and larger than L2 (5.4 GB pool vs 129 MB).

value  = algorithmic bytes per call / mean device time per call (GB/s).
e2e    = the same metric through the public API with pinned host inputs:
         every step copies all inputs host->device and the output back.
roofline.achieved = algorithmic bytes per launch / mean launch duration,
         against the measured HBM copy peak.
cpu_baseline = the fp64 CPU oracle on a bounded sample of the same workload.

--impl reference times that oracle instead (the reference arm): each step is a
bounded sample of the workload on the host cores, reported in the same metric.
Under torchrun (N > 1) every rank runs an independent replica (the path
shards by sequence with no exchange), timings are maxed over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verify-attn KV GB/s (fraction of GB300 HBM peak) and µs/call, 1 GPU"
FALLBACK_HBM_GBS = 6800.0
KERNEL_DIR = os.path.join(ROOT, "speculative_decode_verify_prefix_gb300", "csrc")
KERNEL_SRCS = ("verify_kernel.cuh", "verify_combine.cuh", "verify_tc.cuh", "verify_tr.cuh")  # every kernel of a call
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (every file a call's kernels come
    from): comments and blank space are left out, so an edit of comments
    alone keeps the ncu figures valid."""
    import re

    src = ""
    for name in KERNEL_SRCS:
        with open(os.path.join(KERNEL_DIR, name)) as f:
            src += f.read() + "\n"
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    src = " ".join(src.split())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def traffic_per_launch(workload: str):
    """DRAM bytes per launch from the committed ncu summaries, or None when
    there is none for this workload or it was taken on another kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return t.get("workloads", {}).get(workload, {}).get("dram_bytes_per_launch")


WORKLOADS = {
    "serving": workloads.SERVING,
    # same length distribution, 8 sequences (~0.67 GB > L2): the case multi-pass
    # ncu captures run on
    "serving_b8": workloads.replace(workloads.SERVING, name="serving_b8_p8k_32k", batch=8),
    "tiny": workloads.TINY,
    "d256": workloads.D256,
    "fp8": workloads.FP8,
    # the same batch with the drafts already in a 16-token-page cache
    # (verify_splitkv_paged_fwd)
    "serving_paged": workloads.replace(workloads.SERVING, name="serving_paged16_b64_p8k_32k", page_size=16),
    # the head_dim 256 and fp8-pool shapes at the serving batch and length mix
    "d256_long": workloads.Spec("d256_b64_p8k_32k", None, 4, 16, 2, 256, 256, perm=True, batch=64,
                                len_range=(8192, 32768), seed=1239),
    "fp8_long": workloads.Spec("fp8_b64_p8k_32k", None, 4, 16, 2, 256, 256, pool="e4m3", perm=True, k_scale=0.5,
                               v_scale=0.25, batch=64, len_range=(8192, 32768), seed=1240),
    # head_dim 256 with 8 sequences (~0.33 GB > L2): multi-pass ncu captures
    "d256_b8": workloads.Spec("d256_b8_p8k_32k", None, 4, 16, 2, 256, 256, perm=True, batch=8,
                              len_range=(8192, 32768), seed=1239),
    # the e4m3 head_dim 256 shape with 8 sequences (~0.17 GB > L2): multi-pass ncu captures
    "fp8_b8": workloads.Spec("fp8_b8_p8k_32k", None, 4, 16, 2, 256, 256, pool="e4m3", perm=True, k_scale=0.5,
                             v_scale=0.25, batch=8, len_range=(8192, 32768), seed=1240),
    "fp8_cfg": workloads.FP8,
    # the serving batch over an e4m3 cache (k_scale 0.5, v_scale 0.25): half the bytes per token
    "serving_fp8": workloads.replace(workloads.SERVING, name="serving_fp8_b64_p8k_32k", pool="e4m3", k_scale=0.5,
                                     v_scale=0.25),
    "serving_fp8_b8": workloads.replace(workloads.SERVING, name="serving_fp8_b8_p8k_32k", batch=8, pool="e4m3",
                                        k_scale=0.5, v_scale=0.25),
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="serving")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU-baseline sample time")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--one-launch", action="store_true",
                    help="keep every call on the one-launch kernel (no column split, no stream + combine launches)")
    ap.add_argument("--tc", type=int, nargs="?", const=2, default=None, metavar="MODE",
                    help="head_dim 256 tensor-memory streams (tcgen05; two launches per call, then the "
                         "combine kernel): 2 (the bare flag) vtr_kernel, packed query rows on the MMAs' M side, "
                         "wherever it applies; 1 vtc_kernel, keys on M; 0 neither; unset: the library's "
                         "default (vtr_kernel where it measured faster)")
    ap.add_argument("--report-configs", action="store_true",
                    help="print a per-configuration table (tiny, d256, GQA sweep, fp8, serving) instead of the JSON line")
    ap.add_argument("--config-calls", type=int, default=0, metavar="N",
                    help="call every small parity configuration (tiny, d256, GQA sweep, fp8) N times in its default "
                         "form and print the kernel launches per call, nothing timed: the command an ncu launch list "
                         "of those configurations runs")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- ranks
class Dist:
    """Process layout: torchrun env vars when present, else a single process."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local_rank])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        return reduce_max(x, self.pg)

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def reduce_max(x: float, pg) -> float:
    """Max of a scalar over all ranks (identity on one process)."""
    if pg is None:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() and \
        pg.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, max_seconds: float, world: int) -> float:
    """Whole-job throughput: units every rank processed over the slowest rank's time."""
    return per_rank_units * world / max_seconds


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = str(index)
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        return parse_clock_rows(rows, self.REASONS)


def parse_clock_rows(rows, reason_names) -> dict:
    sm, smax, reasons = [], [], set()
    for r in rows:
        r = [x.strip() for x in r]
        if len(r) < 9:
            continue
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
        except ValueError:
            continue
        for name, val in zip(reason_names, r[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


# ----------------------------------------------------------------------------- accounting
def seq_bytes(prob, b: int) -> int:
    """Algorithmic bytes of sequence b: its prefix K/V rows once per KV head,
    its indices, queries, drafts and output."""
    q, ke, ve = prob["q"], prob["k_ext"], prob["v_ext"]
    P = prob["prefix_lens"][b]
    h_q, h_kv, d, dv = q.shape[1], ke.shape[1], ke.shape[2], ve.shape[2]
    L = prob["max_len_extend"]
    e = prob["k_buffer"].element_size()
    if prob.get("block_table") is not None:
        pages = -(-(P + L) // prob["page_size"])
        return int((P + L) * h_kv * (d + dv) * e + 4 * pages + 4 + L * (2 * h_q * d + 2 * h_q * dv))
    idx = prob["kv_indices"].element_size()
    return int(P * h_kv * (d + dv) * e + P * idx + L * (2 * h_q * d + 2 * h_kv * (d + dv) + 2 * h_q * dv))


def sample_arrays(prob, seqs):
    """Host arrays for the oracle holding only the listed sequences, with each
    sequence's referenced pool rows gathered (in first-use order) to the host."""
    kvp = prob["kv_indptr"].cpu().tolist()
    qo = prob["qo_indptr"].cpu().tolist()
    qs, ks, vs, locs, lens, rows = [], [], [], [], [], []
    for b in seqs:
        qs.append(prob["q"][qo[b]:qo[b + 1]])
        ks.append(prob["k_ext"][qo[b]:qo[b + 1]])
        vs.append(prob["v_ext"][qo[b]:qo[b + 1]])
        locs.append(prob["kv_indices"][kvp[b]:kvp[b + 1]].long())
        lens.append(kvp[b + 1] - kvp[b])
        rows.append(qo[b + 1] - qo[b])
    loc = torch.cat(locs)
    uniq, inv = torch.unique(loc, return_inverse=True)
    sub = {
        "q": torch.cat(qs), "k_ext": torch.cat(ks), "v_ext": torch.cat(vs),
        "k_buffer": prob["k_buffer"][uniq], "v_buffer": prob["v_buffer"][uniq],
        "kv_indptr": torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32),
        "qo_indptr": torch.tensor([0] + np.cumsum(rows).tolist(), dtype=torch.int32),
        "kv_indices": inv.to(torch.int64),
        "sm_scale": prob["sm_scale"], "k_scale": prob["k_scale"], "v_scale": prob["v_scale"],
    }
    return workloads.to_oracle_arrays(sub)


class OracleSampler:
    """Times the fp64 oracle on (sequence, query-head block) units of a workload."""

    def __init__(self, prob, seqs):
        import oracle

        self.oracle = oracle
        self.prob = prob
        self.cores = oracle.max_threads(0)
        self.seqs = list(seqs)
        self.arrays = sample_arrays(prob, self.seqs)
        self.h_q = prob["q"].shape[1]
        self.out = {}

    def run(self, units):
        """units: list of (local sequence index, h0, h1).  Returns (seconds, bytes)."""
        t0 = time.perf_counter()
        for (s, h0, h1) in units:
            self.oracle.verify_forward(self.arrays, b_range=(s, s + 1), h_range=(h0, h1), out=self.out)
        dt = time.perf_counter() - t0
        nbytes = sum(seq_bytes(self.prob, self.seqs[s]) * (h1 - h0) / self.h_q for (s, h0, h1) in units)
        return dt, nbytes


def cpu_baseline(prob, target_s: float) -> dict:
    """The oracle as it stands on the host cores, on whole sequences of the
    workload until about target_s seconds of CPU work."""
    B = len(prob["prefix_lens"])
    cal = OracleSampler(prob, [0])
    h_q = cal.h_q
    t1, _ = cal.run([(0, 0, h_q)])
    n = max(1, min(B - 1, 32, int(target_s / max(t1, 1e-6))))
    samp = OracleSampler(prob, range(1, 1 + n))
    dt, nbytes, passes = 0.0, 0.0, 0
    while dt < target_s and passes < 64:
        d, b = samp.run([(s, 0, h_q) for s in range(n)])
        dt, nbytes, passes = dt + d, nbytes + b, passes + 1
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": samp.cores, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"{passes} pass(es) over {n} whole sequences (all {h_q} query heads, all draft rows) of "
                      f"the same workload, fp64, OpenMP over (sequence, head); bytes counted as the "
                      f"sequences' algorithmic bytes"}


def oracle_config_times(min_seconds: float = 0.25) -> list:
    """The oracle as it stands on the four small configurations (tiny, head_dim
    256, the GQA / draft-length sweep, the e4m3 pool), whole problems on the
    host: one thread, and all cores.  Each figure is the mean over repeats
    filling at least min_seconds.  A reported baseline, not a target."""
    import oracle

    specs = [workloads.TINY, workloads.D256] + workloads.gqa_sweep() + [workloads.FP8]
    cores = oracle.max_threads(0)
    rows = []
    for spec in specs:
        prob = workloads.make_problem(spec, "cpu")
        arrays = workloads.to_oracle_arrays(prob)
        nbytes = workloads.algorithmic_bytes(prob)
        row = {"config": spec.name, "bytes_per_call": nbytes}
        for label, nt in (("1thread", 1), ("all_cores", 0)):
            oracle.verify_forward(arrays, nthreads=nt)
            n, t0 = 0, time.perf_counter()
            while True:
                oracle.verify_forward(arrays, nthreads=nt)
                n += 1
                dt = time.perf_counter() - t0
                if dt >= min_seconds:
                    break
            row[f"us_per_call_{label}"] = round(dt / n * 1e6, 1)
            row[f"gbs_{label}"] = round(nbytes / (dt / n) / 1e9, 4)
        rows.append(row)
    return [{"cores_all": cores}] + rows


# ----------------------------------------------------------------------------- our arm
def _call(vsk, prob, o, ws):
    if prob.get("block_table") is not None:
        vsk.verify_splitkv_paged_fwd(prob["q"], o, prob["k_buffer"], prob["v_buffer"], prob["block_table"],
                                     prob["seq_lens"], prob["page_size"], prob["max_len_extend"], prob["k_scale"],
                                     prob["v_scale"], sm_scale=prob["sm_scale"], workspace=ws)
        return True
    return vsk.verify_splitkv_fwd(prob["q"], prob["k_ext"], prob["v_ext"], o, prob["k_buffer"], prob["v_buffer"],
                                  prob["qo_indptr"], prob["kv_indptr"], prob["kv_indices"], None, True, None,
                                  prob["max_len_extend"], prob["k_scale"], prob["v_scale"],
                                  sm_scale=prob["sm_scale"], workspace=ws)


def time_kernel(vsk, prob, o, ws, steps: int, warmup: int, dist: Dist, gpu_index: int):
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        assert _call(vsk, prob, o, ws), vsk.last_error()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clk:
        t0.record(stream)
        for i in range(steps):
            starts[i].record(stream)
            _call(vsk, prob, o, ws)
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    region_ms = t0.elapsed_time(t1)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return region_ms, statistics.fmean(launch_ms), statistics.median(launch_ms), clk.summary()


def time_e2e(vsk, prob, steps: int, warmup: int):
    """Public API end to end: pinned host inputs copied in, result copied out.
    The first steps after pinning run slower (first touch of the pinned pages
    and device mappings); the median over the timed steps is reported."""
    if prob.get("block_table") is not None:
        names = ["q", "k_buffer", "v_buffer", "block_table", "seq_lens"]
    else:
        names = ["q", "k_ext", "v_ext", "k_buffer", "v_buffer", "qo_indptr", "kv_indptr", "kv_indices"]
    host = {k: prob[k].cpu().pin_memory() for k in names}
    dev = {k: torch.empty_like(prob[k]) for k in names}
    o = torch.empty(prob["q"].shape[0], prob["q"].shape[1], prob["v_ext"].shape[2], dtype=torch.bfloat16,
                    device=prob["q"].device)
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_host.numel() * o_host.element_size()
    d = dict(prob, **dev)
    ws = vsk.get_workspace(o.device, len(prob["prefix_lens"]), o.shape[1], prob["k_ext"].shape[1],
                           prob["q"].shape[2], prob["v_ext"].shape[2], prob["max_len_extend"])
    stream = torch.cuda.current_stream()
    times = []
    for i in range(warmup + steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in names:
            dev[k].copy_(host[k], non_blocking=True)
        assert _call(vsk, d, o, ws), vsk.last_error()
        o_host.copy_(o, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
    del host, dev
    return statistics.median(times), h2d, d2h


def run_ours(args, dist: Dist) -> dict:
    import speculative_decode_verify_prefix_gb300 as vsk

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    spec = WORKLOADS[args.workload]
    # the tensor-memory stream serves head_dim 256 with at most 32 packed rows per KV head
    vsk.set_tuning_tc(0 if args.one_launch else (3 if args.tc is None else int(args.tc)))
    vsk.set_tuning_colsplit(0 if args.one_launch else 1)
    vsk.set_tuning_split_launch(0 if args.one_launch else 1)
    vsk.set_tuning_cluster(0)
    prob = workloads.make_problem(spec, dev)
    B = len(prob["prefix_lens"])
    nbytes = workloads.algorithmic_bytes(prob)
    o = torch.empty(prob["q"].shape[0], prob["q"].shape[1], prob["v_ext"].shape[2], dtype=torch.bfloat16,
                    device=dev)
    ws = vsk.get_workspace(dev, B, prob["q"].shape[1], prob["k_ext"].shape[1], prob["q"].shape[2],
                           prob["v_ext"].shape[2], prob["max_len_extend"])
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    gpu_index = visible.split(",")[dist.local_rank].strip() if visible else str(dist.local_rank)
    region_ms, launch_ms, launch_med_ms, clocks = time_kernel(vsk, prob, o, ws, args.steps, args.warmup, dist,
                                                              gpu_index)
    flags = vsk.read_error_flags(ws)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} after the timed region")
    region_s = dist.max(region_ms / 1e3)
    launch_s = dist.max(launch_ms / 1e3)
    ms_per_step = region_s * 1e3 / args.steps
    value = aggregate(nbytes * args.steps, region_s, dist.world) / 1e9
    peak, peak_kind = hbm_peak()
    achieved = nbytes / launch_s / 1e9
    # the committed ncu figures are for the default forms only
    default_form = not args.one_launch and args.tc in (None, 3)
    traffic = traffic_per_launch(args.workload) if default_form else None
    if prob.get("block_table") is not None:
        tokens = B * prob["block_table"].shape[1] * prob["page_size"]
    else:
        tokens = prob["kv_indices"].shape[0]
    launches = vsk.launches_per_call(B, spec.h_q, spec.h_kv, spec.d, prob["max_len_extend"], tokens)
    form = vsk.call_form(B, spec.h_q, spec.h_kv, spec.d, spec.dv, prob["max_len_extend"], tokens,
                         spec.pool == "e4m3")
    kernel = {"tensor_memory": "vtc_kernel (+ vsk_combine_kernel)",
              "tensor_memory_rows": "vtr_kernel (+ vsk_combine_kernel)",
              "column_split": "vsk_kernel column-split stream (+ vsk_combine_kernel)",
              "column_split_two_tiles": "vsk_kernel two-tile column-split stream (+ vsk_combine_kernel)",
              "stream_only": "vsk_kernel stream only (+ vsk_combine_kernel)",
              "cluster": "vsk_kernel cluster form"}.get(form, f"vsk_kernel<{spec.d},{str(spec.pool == 'e4m3').lower()}>")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_call": round(ms_per_step * 1e3, 2), "frac_of_hbm_peak": round(value / peak, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; workloads.py)",
        "config": workload_config(spec, prob, nbytes),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": kernel,
                     "launch_us_mean": round(launch_s * 1e6, 2), "launch_us_median": round(launch_med_ms * 1e3, 2),
                     "bytes_per_launch": nbytes},
        "gpu_launches": args.steps * launches,
        "clocks": clocks,
    }
    line["config"]["kernel_launches_per_step"] = launches
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(vsk, prob, args.e2e_steps, 3)
        e2e_s = dist.max(e2e_ms / 1e3)
        line["e2e"] = {"value": round(aggregate(nbytes, e2e_s, dist.world) / 1e9, 3), "unit": "GB/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3),
                       "steps": args.e2e_steps, "statistic": "median of the timed steps after 3 warm-up steps"}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob, args.cpu_seconds)
        line["cpu_baseline"]["small_configs"] = oracle_config_times()
    return line


def workload_config(spec, prob, nbytes) -> dict:
    lens = prob["prefix_lens"]
    return {
        "workload": spec.name, "batch": len(lens), "prefix_tokens": int(sum(lens)),
        "prefix_len_min": int(min(lens)), "prefix_len_max": int(max(lens)),
        "prefix_lens": (f"uniform int [{spec.len_range[0]}, {spec.len_range[1]}], seed {spec.seed}"
                        if spec.prefix_lens is None else list(spec.prefix_lens)),
        "l_ext": spec.l_ext, "h_q": spec.h_q, "h_kv": spec.h_kv, "head_dim": spec.d, "v_head_dim": spec.dv,
        "kv_pool": spec.pool,
        "kv_indices": (("random page permutation, int32 block table" if spec.page_size > 0 else
                        ("random permutation" if spec.perm else "arange") + f", {spec.idx_dtype}")),
        "k_scale": spec.k_scale, "v_scale": spec.v_scale, "page_size": max(1, spec.page_size),
        "drafts": "in the paged cache (block table)" if spec.page_size > 0 else "k_extend / v_extend",
        "algorithmic_bytes_per_call": nbytes,
        "l2": "inputs larger than L2 (no flush)" if nbytes > 129e6 else "inputs fit in L2 (L2-resident figure)",
        "kernel_launches_per_step": 1,
    }


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, dist: Dist) -> dict | None:
    """The oracle, as it stands, on the host cores: each step computes a bounded
    sample (one sequence x a block of query heads) of the same workload."""
    if dist.rank != 0:
        return None
    dev = torch.device("cuda", dist.local_rank) if torch.cuda.is_available() else torch.device("cpu")
    spec = WORKLOADS[args.workload]
    prob = workloads.make_problem(spec, dev)
    B = len(prob["prefix_lens"])
    n_seq = min(B, 8)
    samp = OracleSampler(prob, range(n_seq))
    h_q = samp.h_q
    hb = max(1, min(h_q, samp.cores))  # one query head per core per step
    units = [(s, h0, min(h_q, h0 + hb)) for s in range(n_seq) for h0 in range(0, h_q, hb)]
    for i in range(args.warmup):
        samp.run([units[i % len(units)]])
    tot_s, tot_b = 0.0, 0.0
    for i in range(args.steps):
        dt, nb = samp.run([units[(args.warmup + i) % len(units)]])
        tot_s += dt
        tot_b += nb
    value = tot_b / tot_s / 1e9
    nbytes = workloads.algorithmic_bytes(prob)
    sample = (f"per step: 1 sequence x {hb} query heads (all draft rows) of the {spec.name} workload, "
              f"cycling over its first {n_seq} sequences; fp64 oracle, OpenMP over heads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; workloads.py)", "config": workload_config(spec, prob, nbytes),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": samp.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def report_configs(args) -> str:
    """Per-configuration timings: median of >= 100 launches after 10 warm-up
    launches, each launch timed alone with CUDA events; cold = the L2 flushed
    before every launch by reading a 512 MB buffer (clean lines, so no write
    back lands inside the timed launch), warm = back-to-back launches with the
    inputs L2-resident when they fit.  Eager launches and CUDA-graph replays."""
    import speculative_decode_verify_prefix_gb300 as vsk

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = hbm_peak()
    flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)  # 512 MB
    specs = [workloads.TINY, workloads.D256] + workloads.gqa_sweep() + [workloads.FP8, workloads.SERVING]
    rows = ["| config | B | R | D | pool | bytes / call | us / call cold (eager) | us / call cold (graph) | "
            "us / call warm (graph) | GB/s cold (graph) | K/V-only GB/s cold | of measured peak (cold) |",
            "|" + "---|" * 12]
    for spec in specs:
        prob = workloads.make_problem(spec, dev)
        B = len(prob["prefix_lens"])
        nbytes = workloads.algorithmic_bytes(prob)
        kv = int(sum(prob["prefix_lens"])) * spec.h_kv * (spec.d + spec.dv) * prob["k_buffer"].element_size()
        o = torch.empty(prob["q"].shape[0], spec.h_q, spec.dv, dtype=torch.bfloat16, device=dev)
        ws = vsk.get_workspace(dev, B, spec.h_q, spec.h_kv, spec.d, spec.dv, spec.l_ext)
        n = 100 if nbytes > 129e6 else 200

        def timed(run, cold=True):
            ts = []
            for i in range(10 + n):
                if cold:
                    flush.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                run()
                e1.record()
                ts.append((e0, e1))
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in ts[10:]) * 1e3

        eager = timed(lambda: _call(vsk, prob, o, ws))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            _call(vsk, prob, o, ws)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            _call(vsk, prob, o, ws)
        graph = timed(g.replay)
        warm = timed(g.replay, cold=False)
        if vsk.read_error_flags(ws):
            raise RuntimeError(f"device error flags after {spec.name}")
        rows.append(f"| {spec.name} | {B} | {(spec.h_q // spec.h_kv) * spec.l_ext} | {spec.d} | {spec.pool} | {nbytes:,} | "
                    f"{eager:.2f} | {graph:.2f} | {warm:.2f} | {nbytes / graph / 1e3:.0f} | {kv / graph / 1e3:.0f} | "
                    f"{nbytes / graph / 1e3 / peak:.3f} |")
        del prob, o, g
        torch.cuda.empty_cache()
    rows.append(f"\npeak: {peak} GB/s ({peak_kind}); cold: L2 flushed by reading 512 MB before every launch")
    return "\n".join(rows)


def config_calls(n: int) -> None:
    """Every small parity configuration, n calls each in its default form (in
    the order tiny, d256, GQA sweep, fp8), one line per configuration with the
    kernel launches each call makes: the launch list of an ncu run over this
    command maps back to the configurations by those counts."""
    import speculative_decode_verify_prefix_gb300 as vsk

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for spec in [workloads.TINY, workloads.D256] + workloads.gqa_sweep() + [workloads.FP8]:
        prob = workloads.make_problem(spec, dev)
        B = len(prob["prefix_lens"])
        o = torch.empty(prob["q"].shape[0], spec.h_q, spec.dv, dtype=torch.bfloat16, device=dev)
        ws = vsk.get_workspace(dev, B, spec.h_q, spec.h_kv, spec.d, spec.dv, spec.l_ext)
        for _ in range(n):
            assert _call(vsk, prob, o, ws), vsk.last_error()
        torch.cuda.synchronize()
        if vsk.read_error_flags(ws):
            raise RuntimeError(f"device error flags after {spec.name}")
        print(spec.name, vsk.launches_per_call(B, spec.h_q, spec.h_kv, spec.d, spec.l_ext,
                                               prob["kv_indices"].shape[0]), flush=True)
        del prob, o
        torch.cuda.empty_cache()


def main(argv=None):
    args = parse_args(argv)
    if args.report_configs:
        print(report_configs(args), flush=True)
        return
    if args.config_calls > 0:
        config_calls(args.config_calls)
        return
    dist = Dist()
    try:
        if args.impl == "reference":
            line = run_reference(args, dist)
        else:
            line = run_ours(args, dist)
        if dist.rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
