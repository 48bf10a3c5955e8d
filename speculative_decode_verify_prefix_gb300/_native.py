"""Build and load the in-tree CUDA library (libverify_splitkv.so, sm_103a).

The library is compiled from ``csrc/*.cu`` with nvcc into ``_build/`` next to
this file: every translation unit (the host side, and the kernels of each
head_dim) in parallel, then linked into one shared library.  Loading never
falls back to anything: if the library is missing or fails to load, callers
get an exception.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(_HERE, "csrc")
SRCS = sorted(os.path.join(CSRC, n) for n in os.listdir(CSRC) if n.endswith(".cu"))
HEADER = os.path.join(os.path.dirname(_HERE), "include", "verify_splitkv.h")
BUILD_DIR = os.path.join(_HERE, "_build")
OBJ_DIR = os.path.join(BUILD_DIR, f"obj_{platform.machine()}")
LIB_PATH = os.path.join(BUILD_DIR, f"libverify_splitkv_{platform.machine()}.so")
NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [*NVCC_ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC"]


def nvcc_path() -> str:
    for cand in (os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"), "nvcc"):
        if os.path.sep not in cand or os.path.exists(cand):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library for sm_103a (no-op when up to date): each
    translation unit in parallel, then one link.  ``verbose`` passes
    ``-Xptxas=-v`` (registers, spills, shared memory per kernel)."""
    from concurrent.futures import ThreadPoolExecutor

    os.makedirs(OBJ_DIR, exist_ok=True)
    headers = [HEADER] + [os.path.join(CSRC, n) for n in os.listdir(CSRC) if n.endswith(".cuh")]
    newest_header = max(os.path.getmtime(h) for h in headers)
    if not force and os.path.exists(LIB_PATH):
        if os.path.getmtime(LIB_PATH) >= max(newest_header, *(os.path.getmtime(s) for s in SRCS)):
            return LIB_PATH
    nvcc = nvcc_path()

    def compile_one(src):
        obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(newest_header, os.path.getmtime(src)):
            return obj, ""
        tmp = obj + f".tmp{os.getpid()}"
        cmd = [nvcc, *NVCC_FLAGS, *(["-Xptxas=-v"] if verbose else []), "-c", src, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        os.replace(tmp, obj)
        return obj, r.stderr

    with ThreadPoolExecutor(len(SRCS)) as ex:
        results = list(ex.map(compile_one, SRCS))
    if verbose:
        for _, log in results:
            print(log, end="")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *NVCC_ARCH, "-shared", *[o for o, _ in results], "-o", tmp], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class VskTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 3),
        ("stride", ctypes.c_int64 * 3),
    ]


DTYPE_BF16, DTYPE_FP8E4M3, DTYPE_I32, DTYPE_I64, DTYPE_U8 = 0, 1, 2, 3, 4

_lib = None
_lock = threading.Lock()

_P = ctypes.POINTER(VskTensor)


def _bind(lib):
    lib.vsk_can_handle.restype = ctypes.c_int
    lib.vsk_can_handle.argtypes = [_P] * 8 + [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                              ctypes.c_float, ctypes.c_int64]
    lib.verify_splitkv_fwd.restype = ctypes.c_int
    lib.verify_splitkv_fwd.argtypes = [_P] * 9 + [ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                                                  ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.verify_splitkv_tree_fwd.restype = ctypes.c_int
    lib.verify_splitkv_tree_fwd.argtypes = [_P] * 11 + [ctypes.c_int64, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.verify_splitkv_paged_fwd.restype = ctypes.c_int
    lib.verify_splitkv_paged_fwd.argtypes = [_P] * 6 + [ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                                                        ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                                                        ctypes.c_void_p]
    lib.verify_splitkv_write_fwd.restype = ctypes.c_int
    lib.verify_splitkv_write_fwd.argtypes = [_P] * 10 + [ctypes.c_int64, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.verify_splitkv_paged_write_fwd.restype = ctypes.c_int
    lib.verify_splitkv_paged_write_fwd.argtypes = [_P] * 8 + [ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                                              ctypes.c_float, ctypes.c_float, ctypes.c_void_p,
                                                              ctypes.c_size_t, ctypes.c_void_p]
    lib.vsk_workspace_size.restype = ctypes.c_size_t
    lib.vsk_workspace_size.argtypes = [ctypes.c_int64] * 6
    lib.vsk_workspace_size_for_sms.restype = ctypes.c_size_t
    lib.vsk_workspace_size_for_sms.argtypes = [ctypes.c_int] + [ctypes.c_int64] * 6
    lib.vsk_workspace_init.restype = ctypes.c_int
    lib.vsk_workspace_init.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.vsk_read_error_flags.restype = ctypes.c_int
    lib.vsk_read_error_flags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    lib.vsk_set_tuning.restype = None
    lib.vsk_set_tuning.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.vsk_set_tuning_tiles.restype = None
    lib.vsk_set_tuning_tiles.argtypes = [ctypes.c_int]
    lib.vsk_set_tuning_tc.restype = None
    lib.vsk_set_tuning_tc.argtypes = [ctypes.c_int]
    lib.vsk_set_tuning_colsplit.restype = None
    lib.vsk_set_tuning_colsplit.argtypes = [ctypes.c_int]
    lib.vsk_set_tuning_split_launch.restype = None
    lib.vsk_set_tuning_split_launch.argtypes = [ctypes.c_int]
    lib.vsk_set_tuning_cluster.restype = None
    lib.vsk_set_tuning_cluster.argtypes = [ctypes.c_int]
    lib.vsk_set_tuning_pdl.restype = None
    lib.vsk_set_tuning_pdl.argtypes = [ctypes.c_int]
    lib.vsk_set_tuning_pipe.restype = None
    lib.vsk_set_tuning_pipe.argtypes = [ctypes.c_int]
    lib.vsk_set_tuning_colsplit2.restype = None
    lib.vsk_set_tuning_colsplit2.argtypes = [ctypes.c_int]
    lib.vsk_launches_per_call.restype = ctypes.c_int
    lib.vsk_launches_per_call.argtypes = [ctypes.c_int64] * 6
    lib.vsk_call_form.restype = ctypes.c_char_p
    lib.vsk_call_form.argtypes = [ctypes.c_int64] * 7 + [ctypes.c_int]
    lib.vsk_set_tuning_shape.restype = None
    lib.vsk_set_tuning_shape.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.vsk_last_error.restype = ctypes.c_char_p
    lib.vsk_last_error.argtypes = []
    lib.vsk_version.restype = ctypes.c_char_p
    lib.vsk_version.argtypes = []
    return lib


def lib():
    """The loaded CUDA library; raises if it was not built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"CUDA library {LIB_PATH} is missing: run __graft_entry__.build() "
                        "(there is no CPU fallback)")
                _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def last_error() -> str:
    return lib().vsk_last_error().decode()
