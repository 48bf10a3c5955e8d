"""Seeded synthetic verify-attention workloads.

The one module both the CUDA path's tests/benchmark and the CPU oracle take
their inputs from.  It holds no attention arithmetic: it only draws random
tensors, builds index arrays and marshals tensors into the plain arrays the
oracle reads.

Input layout follows the "test_verify_splitkv.py" page (``_build_verify_inputs``)
and the target-verify branch of the "aiter_backend.py" page
(``init_forward_metadata``, target-verify, non-MLA): a constant number of draft
rows ``l_ext`` per sequence with ``qo_indptr = arange(0, B*l_ext + 1, l_ext)``
(int32), ``kv_indptr = [0, cumsum(prefix_lens)]`` (int32, prefix tokens only),
``kv_indices`` int64 (int32 also accepted) addressing a token pool of shape
``[pool_tokens, h_kv, head_dim]``, and q / k_ext / v_ext drawn N(0, 1) in bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Spec:
    name: str
    prefix_lens: tuple | None  # explicit lengths, or None for drawn lengths
    l_ext: int
    h_q: int
    h_kv: int
    d: int
    dv: int
    pool: str = "bf16"          # "bf16" | "e4m3"
    perm: bool = False          # kv_indices a random permutation of pool slots
    k_scale: float = 1.0
    v_scale: float = 1.0
    batch: int = 0              # used when prefix_lens is None
    len_range: tuple = (0, 0)   # inclusive range of drawn prefix lengths
    idx_dtype: str = "int64"
    pool_extra: int = 0         # unreferenced pool slots beyond sum(prefix_lens)
    poison: bool = False        # fill unreferenced pool slots with NaN
    tree: str = ""              # "" causal drafts; "chain" | "star" | "random": tree-verify mask
    page_size: int = 0          # > 0: drafts already in a paged cache, addressed by a block table
    seed: int = 0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads: a tiny case, head_dim 256, a GQA / draft-length sweep,
# an fp8 e4m3 pool with dequant scales, and a serving-scale batch.
TINY = Spec("tiny", (64, 96), 4, 4, 1, 64, 64, seed=1234)
D256 = Spec("d256_b3_p512", (512, 512, 512), 4, 16, 2, 256, 256, seed=1235)
FP8 = Spec("fp8_pool_p4k_8k", (4096, 8192), 4, 16, 2, 256, 256, pool="e4m3", perm=True,
           k_scale=0.5, v_scale=0.25, seed=1237)
SERVING = Spec("serving_b64_p8k_32k", None, 4, 32, 8, 128, 128, perm=True, batch=64,
               len_range=(8192, 32768), seed=1238)


def gqa_sweep() -> list[Spec]:
    out = []
    for h_kv in (1, 2, 4, 8):
        for l_ext in (1, 2, 4, 8):
            out.append(Spec(f"gqa_hkv{h_kv}_l{l_ext}", (1024, 2048), l_ext, 8, h_kv, 128, 128,
                            seed=1236 + 100 * h_kv + l_ext))
    return out


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _make_paged(spec: Spec, device, g, lens) -> dict:
    """Drafts-in-cache problem: every sequence's prefix and drafts occupy
    ceil((P_b + l_ext) / page_size) pages of a shared cache, listed in a
    zero-padded int32 block table (the unified target-verify layout)."""
    ps, L, B = spec.page_size, spec.l_ext, int(lens.numel())
    npages = [-(-(int(P) + L) // ps) for P in lens.tolist()]
    used = sum(npages)
    num_pages = used + -(-int(spec.pool_extra) // ps)
    bf16 = torch.bfloat16
    k_cache = torch.randn(num_pages * ps, spec.h_kv, spec.d, generator=g, device=device, dtype=bf16)
    v_cache = torch.randn(num_pages * ps, spec.h_kv, spec.dv, generator=g, device=device, dtype=bf16)
    order = (torch.randperm(num_pages, generator=g, device=device) if spec.perm
             else torch.arange(num_pages, device=device)).to(torch.int32).cpu()
    max_pages = max(npages) if npages else 1
    bt = torch.zeros(B, max_pages, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(npages):
        bt[b, :n] = order[pos:pos + n]
        pos += n
    n_ext = B * L
    q = torch.randn(n_ext, spec.h_q, spec.d, generator=g, device=device, dtype=bf16)
    rows = []  # pool row of every cache position, per sequence
    for b, P in enumerate(lens.tolist()):
        j = torch.arange(int(P) + L)
        rows.append((bt[b, j // ps].long() * ps + j % ps))
    if spec.poison:
        unref = torch.ones(num_pages * ps, dtype=torch.bool)
        if rows:
            unref[torch.cat(rows)] = False
        k_cache[unref.to(device)] = float("nan")
        v_cache[unref.to(device)] = float("nan")
    if spec.pool == "e4m3":
        k_cache = k_cache.to(torch.float8_e4m3fn)
        v_cache = v_cache.to(torch.float8_e4m3fn)
    # flat equivalents (prefix through kv_indices, drafts as k_ext / v_ext), for comparisons
    pre = [r[:int(P)] for r, P in zip(rows, lens.tolist())]
    drf = torch.cat([r[int(P):] for r, P in zip(rows, lens.tolist())]) if rows else torch.zeros(0, dtype=torch.long)
    kv_indices = (torch.cat(pre) if pre else torch.zeros(0, dtype=torch.long)).to(torch.int64)
    kv_indptr = torch.zeros(B + 1, dtype=torch.int32)
    kv_indptr[1:] = torch.cumsum(lens, 0).to(torch.int32)
    d_dev = drf.to(device)
    k_ext = k_cache[d_dev].to(bf16) if n_ext else torch.zeros(0, spec.h_kv, spec.d, dtype=bf16, device=device)
    v_ext = v_cache[d_dev].to(bf16) if n_ext else torch.zeros(0, spec.h_kv, spec.dv, dtype=bf16, device=device)
    return {
        "spec": spec, "q": q, "k_ext": k_ext, "v_ext": v_ext, "k_buffer": k_cache, "v_buffer": v_cache,
        "block_table": bt.to(device), "page_size": ps, "seq_lens": lens.to(torch.int32).to(device),
        "qo_indptr": torch.arange(0, n_ext + 1, L, dtype=torch.int32).to(device),
        "kv_indptr": kv_indptr.to(device), "kv_indices": kv_indices.to(device),
        "max_len_extend": L, "sm_scale": spec.sm_scale, "k_scale": spec.k_scale, "v_scale": spec.v_scale,
        "prefix_lens": [int(x) for x in lens.tolist()], "pool_dtype": spec.pool,
    }


def make_problem(spec: Spec, device="cpu", **overrides) -> dict:
    """Draw one problem.  Every tensor lives on ``device``; draws are seeded by
    ``spec.seed`` in a fixed order, so a (spec, device) pair is reproducible."""
    if overrides:
        spec = replace(spec, **overrides)
    device = torch.device(device)
    g = _gen(device, spec.seed)
    if spec.prefix_lens is not None:
        lens = torch.tensor(list(spec.prefix_lens), dtype=torch.int64)
    else:
        lo, hi = spec.len_range
        lens = torch.randint(lo, hi + 1, (spec.batch,), generator=g, device=device).cpu()
    if spec.page_size > 0:
        return _make_paged(spec, device, g, lens)
    B = int(lens.numel())
    T = int(lens.sum())
    pool_tokens = T + int(spec.pool_extra)
    bf16 = torch.bfloat16

    k_buffer = torch.randn(pool_tokens, spec.h_kv, spec.d, generator=g, device=device, dtype=bf16)
    v_buffer = torch.randn(pool_tokens, spec.h_kv, spec.dv, generator=g, device=device, dtype=bf16)
    if spec.perm:
        kv_indices = torch.randperm(pool_tokens, generator=g, device=device)[:T].to(torch.int64)
    else:
        kv_indices = torch.arange(T, device=device, dtype=torch.int64)
    n_ext = B * spec.l_ext
    q = torch.randn(n_ext, spec.h_q, spec.d, generator=g, device=device, dtype=bf16)
    k_ext = torch.randn(n_ext, spec.h_kv, spec.d, generator=g, device=device, dtype=bf16)
    v_ext = torch.randn(n_ext, spec.h_kv, spec.dv, generator=g, device=device, dtype=bf16)

    if spec.poison and pool_tokens > 0:
        unref = torch.ones(pool_tokens, dtype=torch.bool, device=device)
        if T:
            unref[kv_indices] = False
        k_buffer[unref] = float("nan")
        v_buffer[unref] = float("nan")
    if spec.pool == "e4m3":
        k_buffer = k_buffer.to(torch.float8_e4m3fn)
        v_buffer = v_buffer.to(torch.float8_e4m3fn)

    kv_indptr = torch.zeros(B + 1, dtype=torch.int32)
    kv_indptr[1:] = torch.cumsum(lens, 0).to(torch.int32)
    qo_indptr = torch.arange(0, n_ext + 1, spec.l_ext, dtype=torch.int32)
    if spec.idx_dtype == "int32":
        kv_indices = kv_indices.to(torch.int32)
    extra = {}
    if spec.tree:
        cm, mi = tree_mask([int(x) for x in lens.tolist()], spec.l_ext, spec.tree, spec.seed + 7, device)
        extra = {"custom_mask": cm, "mask_indptr": mi}
    return {**extra,
        "spec": spec,
        "q": q, "k_ext": k_ext, "v_ext": v_ext,
        "k_buffer": k_buffer, "v_buffer": v_buffer,
        "qo_indptr": qo_indptr.to(device), "kv_indptr": kv_indptr.to(device),
        "kv_indices": kv_indices,
        "max_len_extend": spec.l_ext,
        "sm_scale": spec.sm_scale, "k_scale": spec.k_scale, "v_scale": spec.v_scale,
        "prefix_lens": [int(x) for x in lens.tolist()],
        "pool_dtype": spec.pool,
    }


def tree_parents(kind: str, L: int, gen: torch.Generator) -> list:
    """Parent of each draft node of a speculation tree (node 0 is the root):
    a chain (i -> i-1), a star (every node under the root) or a random tree."""
    if kind == "chain":
        return [-1] + list(range(L - 1))
    if kind == "star":
        return [-1] + [0] * (L - 1)
    return [-1] + [int(torch.randint(0, i, (1,), generator=gen)) for i in range(1, L)]


def tree_mask(prefix_lens, L: int, kind: str, seed: int, device="cpu"):
    """Target-verify mask of speculation trees, in the layout the
    "aiter_backend.py" page builds: per sequence an L x (P_b + L) uint8 matrix,
    row-major, prefix columns all visible, draft column t visible to row i iff
    t is i or an ancestor of i; ``mask_indptr`` (int64) holds the running
    offsets."""
    gen = torch.Generator().manual_seed(seed)
    parts, offs = [], [0]
    for P in prefix_lens:
        par = tree_parents(kind, L, gen)
        m = torch.zeros(L, P + L, dtype=torch.uint8)
        m[:, :P] = 1
        for i in range(L):
            a = i
            while a >= 0:
                m[i, P + a] = 1
                a = par[a]
        parts.append(m.flatten())
        offs.append(offs[-1] + m.numel())
    cm = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.uint8)
    return cm.to(device), torch.tensor(offs, dtype=torch.int64, device=device)


def _bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 (uint16) or e4m3 (uint8) tensor, on the host."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(f"unexpected dtype {t.dtype}")


def to_oracle_arrays(prob: dict) -> dict:
    """Host numpy views of a problem in the form the oracle reads."""
    return {
        "q": _bits(prob["q"]), "k_ext": _bits(prob["k_ext"]), "v_ext": _bits(prob["v_ext"]),
        "k_pool": _bits(prob["k_buffer"]), "v_pool": _bits(prob["v_buffer"]),
        "pool_dtype": "e4m3" if prob["k_buffer"].dtype == torch.float8_e4m3fn else "bf16",
        "qo_indptr": prob["qo_indptr"].cpu().numpy(),
        "kv_indptr": prob["kv_indptr"].cpu().numpy(),
        "kv_indices": prob["kv_indices"].cpu().numpy(),
        "sm_scale": prob["sm_scale"], "k_scale": prob["k_scale"], "v_scale": prob["v_scale"],
        **({"custom_mask": prob["custom_mask"].cpu().numpy(), "mask_indptr": prob["mask_indptr"].cpu().numpy()}
           if prob.get("custom_mask") is not None else {}),
        **({"block_table": prob["block_table"].cpu().numpy(), "page_size": prob["page_size"],
            "seq_lens": prob["seq_lens"].cpu().numpy()} if prob.get("block_table") is not None else {}),
    }


def algorithmic_bytes(prob: dict) -> int:
    """Bytes the method must move once: every referenced prefix K/V row once per
    KV head, the indices, the queries, the draft K/V and the output."""
    q, ke, ve = prob["q"], prob["k_ext"], prob["v_ext"]
    T = int(sum(prob["prefix_lens"]))
    h_kv, d = ke.shape[1], ke.shape[2]
    dv = ve.shape[2]
    e = prob["k_buffer"].element_size()
    idx = prob["kv_indices"].element_size()
    n_rows, h_q = q.shape[0], q.shape[1]
    if prob.get("block_table") is not None:
        # drafts come from the cache too; one page id per page and one length per sequence
        ps, L = prob["page_size"], prob["max_len_extend"]
        pages = sum(-(-(P + L) // ps) for P in prob["prefix_lens"])
        return int((T + n_rows) * h_kv * (d + dv) * e + 4 * pages + 4 * len(prob["prefix_lens"])
                   + 2 * n_rows * h_q * d + 2 * n_rows * h_q * dv)
    kv = T * h_kv * (d + dv) * e
    return int(kv + T * idx + 2 * n_rows * h_q * d + 2 * n_rows * h_kv * (d + dv) + 2 * n_rows * h_q * dv)
