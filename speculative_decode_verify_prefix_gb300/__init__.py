"""Split-KV verify attention for EAGLE target-verify (topk = 1) on GB300.

The computation runs in the CUDA library built from ``csrc/*.cu``
(C ABI: ``include/verify_splitkv.h``); this package is its Python binding.
"""
from .api import (as_vsk, call_form, can_handle, get_workspace, launches_per_call, read_error_flags, set_tuning,
                  set_tuning_cluster, set_tuning_colsplit, set_tuning_colsplit2, set_tuning_pdl, set_tuning_pipe, set_tuning_shape, set_tuning_split_launch, set_tuning_tc,
                  set_tuning_tiles,
                  verify_splitkv_fwd, verify_splitkv_paged_fwd, verify_splitkv_paged_write_fwd,
                  verify_splitkv_write_fwd, version, workspace_size)
from ._native import build, last_error

__all__ = ["as_vsk", "build", "call_form", "can_handle", "get_workspace", "last_error", "launches_per_call", "read_error_flags",
           "set_tuning", "set_tuning_cluster", "set_tuning_colsplit", "set_tuning_colsplit2", "set_tuning_pdl", "set_tuning_pipe", "set_tuning_shape", "set_tuning_split_launch", "set_tuning_tc",
           "set_tuning_tiles", "verify_splitkv_fwd", "verify_splitkv_paged_fwd", "verify_splitkv_paged_write_fwd",
           "verify_splitkv_write_fwd", "version", "workspace_size"]
