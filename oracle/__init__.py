"""Python face of the fp64 CPU oracle for split-KV verify attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use it; the CUDA product path never does.
It imports nothing from the product package and the product imports nothing
from here.

The arithmetic lives in ``verify_oracle.c`` (plain loops, fp64, full score
rows); this module only compiles it with gcc, marshals numpy arrays into its
problem struct and returns numpy results.  What it computes and the readings
it takes are stated in the header comment of ``verify_oracle.c``; the sources
are the "verify_splitkv.py" page (module docstring, ``_verify_prefix_stage1``,
``_verify_combine_stage2``) and the "test_verify_splitkv.py" page
(``_build_verify_inputs``: the input layout).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, f"libverify_oracle_{platform.machine()}.so")

POOL_BF16 = 0
POOL_E4M3 = 1
IDX_I32 = 0
IDX_I64 = 1


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("h_q", ctypes.c_int64),
        ("h_kv", ctypes.c_int64),
        ("d", ctypes.c_int64),
        ("dv", ctypes.c_int64),
        ("n_rows", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("q_s0", ctypes.c_int64), ("q_s1", ctypes.c_int64),
        ("k_ext", ctypes.c_void_p), ("ke_s0", ctypes.c_int64), ("ke_s1", ctypes.c_int64),
        ("v_ext", ctypes.c_void_p), ("ve_s0", ctypes.c_int64), ("ve_s1", ctypes.c_int64),
        ("k_pool", ctypes.c_void_p), ("kp_s0", ctypes.c_int64), ("kp_s1", ctypes.c_int64),
        ("v_pool", ctypes.c_void_p), ("vp_s0", ctypes.c_int64), ("vp_s1", ctypes.c_int64),
        ("pool_dtype", ctypes.c_int32),
        ("idx_dtype", ctypes.c_int32),
        ("qo_indptr", ctypes.c_void_p),
        ("kv_indptr", ctypes.c_void_p),
        ("kv_indices", ctypes.c_void_p),
        ("sm_scale", ctypes.c_double),
        ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
        ("custom_mask", ctypes.c_void_p),
        ("mask_indptr", ctypes.c_void_p),
        ("paged", ctypes.c_int32),
        ("block_table", ctypes.c_void_p),
        ("bt_s0", ctypes.c_int64),
        ("page_size", ctypes.c_int64),
        ("seq_lens", ctypes.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def build(source: str = _SRC, out_path: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the oracle into a shared library with gcc (OpenMP over heads)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    if not force and os.path.exists(out_path) and os.path.getmtime(out_path) >= os.path.getmtime(source):
        return out_path
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _bind(lib):
    lib.orc_verify_forward.restype = ctypes.c_int
    lib.orc_verify_forward.argtypes = [ctypes.POINTER(_Problem)] + [ctypes.c_int64] * 4 + [ctypes.c_void_p] * 5 + [ctypes.c_int]
    lib.orc_max_threads.restype = ctypes.c_int
    lib.orc_max_threads.argtypes = [ctypes.c_int]
    lib.orc_decode_bf16.restype = None
    lib.orc_decode_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.orc_decode_e4m3.restype = None
    lib.orc_decode_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.orc_quantize.restype = None
    lib.orc_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_void_p]
    lib.orc_encode_e4m3.restype = None
    lib.orc_encode_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.orc_encode_bf16.restype = None
    lib.orc_encode_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; a path loads a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _strides(a: np.ndarray):
    it = a.itemsize
    assert a.ndim == 3, "expected a 3-d array"
    if a.size == 0:
        return a.shape[1] * a.shape[2], a.shape[2]
    assert a.strides[2] == it, "last dimension must be contiguous"
    return a.strides[0] // it, a.strides[1] // it


def decode_bf16(bits: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.orc_decode_bf16(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_e4m3(codes: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib.orc_decode_e4m3(_ptr(codes), _ptr(out), codes.size)
    return out


def encode_e4m3(values: np.ndarray, lib=None) -> np.ndarray:
    """e4m3 codes of binary32 values (nearest, ties to even, saturating)."""
    lib = lib or load()
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib.orc_encode_e4m3(_ptr(v), _ptr(out), v.size)
    return out


def encode_bf16(values: np.ndarray, lib=None) -> np.ndarray:
    """bf16 bit patterns of binary32 values (nearest, ties to even)."""
    lib = lib or load()
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib.orc_encode_bf16(_ptr(v), _ptr(out), v.size)
    return out


def quantize(bits: np.ndarray, scale: float, pool_dtype: str, lib=None) -> np.ndarray:
    """Cache codes of bf16 values (uint16 bit patterns) stored with a
    dequantisation scale: the cache dtype's nearest value to x / scale
    (binary32 quotient).  ``pool_dtype`` "e4m3" gives uint8 codes, "bf16"
    uint16 bit patterns."""
    lib = lib or load()
    src = np.ascontiguousarray(bits, dtype=np.uint16)
    e4m3 = pool_dtype == "e4m3"
    out = np.empty(src.shape, dtype=np.uint8 if e4m3 else np.uint16)
    lib.orc_quantize(_ptr(src), src.size, float(scale), POOL_E4M3 if e4m3 else POOL_BF16, _ptr(out))
    return out


def write_rows(pool: np.ndarray, rows: np.ndarray, new_bits: np.ndarray, scale: float, pool_dtype: str,
               lib=None) -> np.ndarray:
    """A copy of ``pool`` [n, h_kv, d] with rows ``rows`` replaced by the
    quantised ``new_bits`` [len(rows), h_kv, d] (the cache after a K or V
    store of new tokens)."""
    out = np.array(pool, copy=True)
    out[np.asarray(rows, dtype=np.int64)] = quantize(new_bits, scale, pool_dtype, lib=lib)
    return out


def max_threads(nthreads: int = 0, lib=None) -> int:
    lib = lib or load()
    return int(lib.orc_max_threads(int(nthreads)))


def verify_forward(prob: dict, b_range=None, h_range=None, debug: bool = False,
                   nthreads: int = 0, lib=None, out: dict | None = None) -> dict:
    """Run the oracle on a problem held as numpy arrays.

    ``prob`` keys: ``q``, ``k_ext``, ``v_ext`` (uint16 bf16 bit patterns,
    shapes [n_rows, h_q, d], [n_rows, h_kv, d], [n_rows, h_kv, dv]);
    ``k_pool``, ``v_pool`` (uint16 bf16 bits or uint8 e4m3 codes, [pool_tokens,
    h_kv, d|dv]); ``pool_dtype`` ("bf16" | "e4m3"); ``qo_indptr``,
    ``kv_indptr`` (int32 [B+1]); ``kv_indices`` (int32 or int64);
    ``sm_scale``, ``k_scale``, ``v_scale`` (floats); optionally
    ``custom_mask`` (uint8, flattened per-sequence [L, P+L] row-major draft
    visibility, nonzero = visible) with ``mask_indptr`` (int64 [B+1]) for tree
    verify; without them the drafts are causal.  A paged problem (drafts
    already in the cache) instead gives ``block_table`` (int32 [B, max_blocks]),
    ``page_size`` and ``seq_lens`` (int32 [B], cached tokens before the
    drafts); its ``kv_indptr`` / ``kv_indices`` / ``k_ext`` / ``v_ext`` are
    not read (``k_ext`` / ``v_ext`` may be empty [n_rows, h_kv, d] arrays).

    Returns ``{"o": float64 [n_rows, h_q, dv]}`` (NaN where not computed) and,
    with ``debug``, ``o_prefix``, ``lse_prefix``, ``o_draft``, ``lse_draft``.
    """
    lib = lib or load()
    q, ke, ve = prob["q"], prob["k_ext"], prob["v_ext"]
    kp, vp = prob["k_pool"], prob["v_pool"]
    qo = np.ascontiguousarray(prob["qo_indptr"], dtype=np.int32)
    kvp = np.ascontiguousarray(prob.get("kv_indptr", np.zeros(1, dtype=np.int32)), dtype=np.int32)
    kvi = np.ascontiguousarray(prob.get("kv_indices", np.zeros(0, dtype=np.int64)))
    if kvi.dtype not in (np.int32, np.int64):
        raise TypeError("kv_indices must be int32 or int64")
    for name, a in (("q", q), ("k_ext", ke), ("v_ext", ve)):
        if a.dtype != np.uint16:
            raise TypeError(f"{name} must hold bf16 bit patterns (uint16)")
    pool_dtype = POOL_E4M3 if prob["pool_dtype"] == "e4m3" else POOL_BF16
    want = np.uint8 if pool_dtype == POOL_E4M3 else np.uint16
    if kp.dtype != want or vp.dtype != want:
        raise TypeError("pool arrays do not match pool_dtype")
    n_rows, h_q, d = q.shape
    h_kv, dv = ke.shape[1], ve.shape[2]
    B = qo.shape[0] - 1

    P = _Problem()
    P.batch, P.h_q, P.h_kv, P.d, P.dv, P.n_rows = B, h_q, h_kv, d, dv, n_rows
    P.q, (P.q_s0, P.q_s1) = _ptr(q), _strides(q)
    P.k_ext, (P.ke_s0, P.ke_s1) = _ptr(ke), _strides(ke)
    P.v_ext, (P.ve_s0, P.ve_s1) = _ptr(ve), _strides(ve)
    P.k_pool, (P.kp_s0, P.kp_s1) = _ptr(kp), _strides(kp)
    P.v_pool, (P.vp_s0, P.vp_s1) = _ptr(vp), _strides(vp)
    P.pool_dtype = pool_dtype
    P.idx_dtype = IDX_I64 if kvi.dtype == np.int64 else IDX_I32
    P.qo_indptr, P.kv_indptr, P.kv_indices = _ptr(qo), _ptr(kvp), _ptr(kvi) if kvi.size else 0
    P.sm_scale = float(prob["sm_scale"])
    P.k_scale = float(prob.get("k_scale", 1.0))
    P.v_scale = float(prob.get("v_scale", 1.0))
    cm = prob.get("custom_mask")
    mi = None
    if cm is not None:
        cm = np.ascontiguousarray(cm).view(np.uint8) if cm.dtype == np.bool_ else np.ascontiguousarray(cm, dtype=np.uint8)
        mi = np.ascontiguousarray(prob["mask_indptr"], dtype=np.int64)
        P.custom_mask, P.mask_indptr = (_ptr(cm) if cm.size else 0), _ptr(mi)

    b0, b1 = b_range if b_range is not None else (0, B)
    h0, h1 = h_range if h_range is not None else (0, h_q)
    res = out if out is not None else {}
    if "o" not in res:
        res["o"] = np.full((n_rows, h_q, dv), np.nan, dtype=np.float64)
    dbg = [0, 0, 0, 0]
    if debug:
        for k, shp in (("o_prefix", (n_rows, h_q, dv)), ("lse_prefix", (n_rows, h_q)),
                       ("o_draft", (n_rows, h_q, dv)), ("lse_draft", (n_rows, h_q))):
            if k not in res:
                res[k] = np.full(shp, np.nan, dtype=np.float64)
        dbg = [_ptr(res["o_prefix"]), _ptr(res["lse_prefix"]), _ptr(res["o_draft"]), _ptr(res["lse_draft"])]
    bt = sl = None
    if prob.get("block_table") is not None:
        bt = np.ascontiguousarray(prob["block_table"], dtype=np.int32)
        sl = np.ascontiguousarray(prob["seq_lens"], dtype=np.int32)
        P.paged, P.block_table, P.bt_s0, P.page_size, P.seq_lens = 1, _ptr(bt), bt.shape[1], int(prob["page_size"]), _ptr(sl)
    keep = (q, ke, ve, kp, vp, qo, kvp, kvi, cm, mi, bt, sl)  # noqa: F841  (alive across the call)
    rc = lib.orc_verify_forward(ctypes.byref(P), b0, b1, h0, h1, _ptr(res["o"]), *dbg, int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the requested ranges or head counts")
    return res
