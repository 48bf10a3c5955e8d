"""Python binding of the C ABI in include/verify_splitkv.h.

Argument marshalling only: torch tensors become ``vsk_tensor`` views (device
pointer, dtype code, shape, strides) and the call goes straight to the CUDA
library.  Every step of the computation runs in the library's kernel.

``can_handle`` and ``verify_splitkv_fwd`` keep the positional signature of the
sglang "verify_splitkv.py" page (``can_handle``, ``verify_splitkv_fwd``), so a
caller of that module can switch by changing the import.  The workspace cache
mirrors the page's ``_VK_CACHE``: one zero-initialised buffer per (device,
stream), sized by ``max_bs`` and grown only, so its address stays fixed across
batch sizes.  Calls on different streams get different buffers, so they may
overlap on the GPU; calls on one stream are ordered by the stream and share its
buffer.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _native

_DT = {
    torch.bfloat16: _native.DTYPE_BF16,
    torch.float8_e4m3fn: _native.DTYPE_FP8E4M3,
    torch.int32: _native.DTYPE_I32,
    torch.int64: _native.DTYPE_I64,
    torch.uint8: _native.DTYPE_U8,
    torch.bool: _native.DTYPE_U8,
}


def as_vsk(t: torch.Tensor) -> _native.VskTensor:
    """A vsk_tensor view of a torch tensor (no copy)."""
    v = _native.VskTensor()
    v.data = t.data_ptr() if t.numel() else 0
    v.dtype = _DT.get(t.dtype, -1)
    v.ndim = t.dim()
    for i in range(min(3, t.dim())):
        v.shape[i] = t.shape[i]
        v.stride[i] = t.stride(i)
    return v


def _ref(t):
    return ctypes.byref(as_vsk(t))


def _gate(views, is_causal, mle, sliding_window_size, sinks, logit_cap, xai_temperature_len) -> bool:
    sw = -1 if sliding_window_size is None else int(sliding_window_size)
    xai = -1 if xai_temperature_len is None else int(xai_temperature_len)
    cap = float(logit_cap) if logit_cap else 0.0
    return bool(_native.lib().vsk_can_handle(*[ctypes.byref(v) for v in views], int(bool(is_causal)), mle, sw,
                                             int(sinks is not None), cap, xai))


def can_handle(q_extend, k_extend, v_extend, k_buffer, v_buffer, qo_indptr, kv_indptr, kv_indices,
               custom_mask, is_causal, mask_indptr, max_len_extend, sliding_window_size=-1, sinks=None,
               logit_cap=0.0, xai_temperature_len=-1) -> bool:
    """True iff the split-KV verify kernel serves this problem (shape and flag
    checks only; tensor values are never read).  ``custom_mask`` is not
    inspected: the kernel computes pure causal attention, which equals the tree
    mask only at speculative topk == 1, so the caller gates on topk == 1."""
    try:
        mle = int(max_len_extend)
    except (TypeError, ValueError):
        return False
    ts = (q_extend, k_extend, v_extend, k_buffer, v_buffer, qo_indptr, kv_indptr, kv_indices)
    for t in ts:
        if not isinstance(t, torch.Tensor) or t.dtype not in _DT or t.dim() > 3:
            return False
    return _gate([as_vsk(t) for t in ts], is_causal, mle, sliding_window_size, sinks, logit_cap,
                 xai_temperature_len)


_WS = {}
_WS_SIZE = {}  # (device, max_bs, h_q, h_kv, head_dim, v_head_dim, l_ext) -> bytes
_WS_LOCK = threading.Lock()


def workspace_size(max_bs, h_q, h_kv, head_dim, v_head_dim, l_ext) -> int:
    return int(_native.lib().vsk_workspace_size(max_bs, h_q, h_kv, head_dim, v_head_dim, l_ext))


def _stream_key(device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def get_workspace(device, max_bs, h_q, h_kv, head_dim, v_head_dim, l_ext, stream=None) -> torch.Tensor:
    """Zero-filled workspace of ``stream`` (default: the device's current
    stream) on ``device``, grown (never shrunk) to fit max_bs.  One buffer per
    (device, stream): a buffer is never shared by calls that may overlap on the
    GPU.  Growing allocates a new buffer; the old one is released by torch's
    caching allocator on the current stream, after the calls queued on it."""
    device = torch.device(device)
    if device.index is None:
        device = torch.device(device.type, torch.cuda.current_device())
    key = (device, int(max_bs), int(h_q), int(h_kv), int(head_dim), int(v_head_dim), int(l_ext))
    need = _WS_SIZE.get(key)
    if need is None:
        with torch.cuda.device(device):
            need = workspace_size(*key[1:])
        _WS_SIZE[key] = need
    if need == 0:
        raise RuntimeError("workspace size query failed: " + _native.last_error())
    wkey = (device, _stream_key(device, stream))
    with _WS_LOCK:
        ws = _WS.get(wkey)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(need, dtype=torch.uint8, device=device)
            _WS[wkey] = ws
    return ws


def _coerce(x) -> float:
    try:
        return float(x)
    except (TypeError, ValueError):
        return 1.0


def verify_splitkv_fwd(q_extend, k_extend, v_extend, o_extend, k_buffer, v_buffer, qo_indptr, kv_indptr,
                       kv_indices, custom_mask, is_causal, mask_indptr, max_len_extend, k_scale, v_scale,
                       sm_scale=None, logit_cap=0.0, skip_prefix_custom_mask=True, sliding_window_size=-1,
                       sinks=None, window_kv_offsets=None, xai_temperature_len=-1, max_bs=None,
                       workspace=None, stream=None) -> bool:
    """Drop-in for the prefill/extend attention call on the EAGLE target-verify
    shape.  Returns True once the kernel is enqueued on the current stream
    (o_extend will hold the result), False if the case is unsupported
    (nothing was launched; the caller falls back).

    Without ``custom_mask`` the drafts are causal (topk = 1).  With
    ``custom_mask`` / ``mask_indptr`` (the target-verify layout: per sequence
    an l_ext x (prefix + l_ext) uint8 matrix) the draft block follows the
    mask, which serves tree verify (topk > 1); the prefix part of the mask is
    not applied, so ``skip_prefix_custom_mask`` must be True."""
    try:
        mle = int(max_len_extend)
    except (TypeError, ValueError):
        return False
    ts = (q_extend, k_extend, v_extend, k_buffer, v_buffer, qo_indptr, kv_indptr, kv_indices)
    for t in ts:
        if not isinstance(t, torch.Tensor) or t.dtype not in _DT or t.dim() > 3:
            return False
    views = [as_vsk(t) for t in ts]
    if not _gate(views, is_causal, mle, sliding_window_size, sinks, logit_cap, xai_temperature_len):
        return False
    if custom_mask is not None and (not skip_prefix_custom_mask or mask_indptr is None):
        return False  # the prefix part of a tree mask is not applied by this kernel
    bs = qo_indptr.shape[0] - 1
    if stream is None:
        stream = torch.cuda.current_stream(q_extend.device)
    if workspace is None:
        mb = bs if (max_bs is None or max_bs < bs) else int(max_bs)
        workspace = get_workspace(q_extend.device, mb, q_extend.shape[1], k_extend.shape[1],
                                  q_extend.shape[2], v_extend.shape[2], mle, stream)
    sm = 0.0 if sm_scale is None else float(sm_scale)
    if custom_mask is not None:
        cm = custom_mask if custom_mask.dtype == torch.uint8 else custom_mask.view(torch.uint8)
        r = [ctypes.byref(v) for v in views]
        ok = _native.lib().verify_splitkv_tree_fwd(
            r[0], r[1], r[2], _ref(o_extend), r[3], r[4], r[5], r[6], r[7], _ref(cm.reshape(-1)), _ref(mask_indptr), mle,
            _coerce(k_scale), _coerce(v_scale), sm, ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
            ctypes.c_void_p(stream.cuda_stream))
        if not ok:
            raise RuntimeError("verify_splitkv_tree_fwd failed after the gate passed: " + _native.last_error())
        return True
    r = [ctypes.byref(v) for v in views]
    ok = _native.lib().verify_splitkv_fwd(
        r[0], r[1], r[2], _ref(o_extend), r[3], r[4], r[5], r[6], r[7], int(bool(is_causal)), mle,
        _coerce(k_scale), _coerce(v_scale), sm, ctypes.c_void_p(workspace.data_ptr()),
        workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    if not ok:
        raise RuntimeError("verify_splitkv_fwd failed after the gate passed: " + _native.last_error())
    return True


def verify_splitkv_paged_fwd(q, o, k_cache, v_cache, block_table, seq_lens, page_size, max_len_extend,
                             k_scale=1.0, v_scale=1.0, sm_scale=None, max_bs=None, workspace=None,
                             stream=None) -> None:
    """Verify with the drafts already stored in a paged KV cache.

    ``q`` / ``o``: [B*l_ext, h_q, D] bf16; ``k_cache`` / ``v_cache``:
    [n_pages*page_size, h_kv, D] bf16 or fp8 e4m3; ``block_table``: [B,
    max_blocks] int32 page ids; ``seq_lens``: [B] int32 cached tokens before
    the drafts (the drafts occupy cache positions seq_lens[b] ..
    seq_lens[b] + l_ext - 1).  ``k_scale`` / ``v_scale`` apply to every cached
    key and value, drafts included.  Enqueues the kernel on the current stream;
    raises ValueError when the library rejects the arguments."""
    bs = seq_lens.shape[0]
    mle = int(max_len_extend)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if workspace is None:
        mb = bs if (max_bs is None or max_bs < bs) else int(max_bs)
        workspace = get_workspace(q.device, mb, q.shape[1], k_cache.shape[1], q.shape[2], v_cache.shape[2], mle,
                                  stream)
    sm = 0.0 if sm_scale is None else float(sm_scale)
    ok = _native.lib().verify_splitkv_paged_fwd(
        _ref(q), _ref(o), _ref(k_cache), _ref(v_cache), _ref(block_table), _ref(seq_lens), int(page_size), mle,
        _coerce(k_scale), _coerce(v_scale), sm, ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
        ctypes.c_void_p(stream.cuda_stream))
    if not ok:
        raise ValueError("verify_splitkv_paged_fwd: " + _native.last_error())


def verify_splitkv_write_fwd(q_extend, k_extend, v_extend, o_extend, k_buffer, v_buffer, qo_indptr, kv_indptr,
                             kv_indices, out_cache_loc, max_len_extend, k_scale=1.0, v_scale=1.0, sm_scale=None,
                             max_bs=None, workspace=None, stream=None) -> None:
    """``verify_splitkv_fwd`` (causal drafts) that also stores k_extend /
    v_extend into rows ``out_cache_loc`` of k_buffer / v_buffer (quantised
    as x / scale in the pool dtype), in the same launch.  Raises ValueError
    when the library rejects the arguments."""
    bs = qo_indptr.shape[0] - 1
    mle = int(max_len_extend)
    if stream is None:
        stream = torch.cuda.current_stream(q_extend.device)
    if workspace is None:
        mb = bs if (max_bs is None or max_bs < bs) else int(max_bs)
        workspace = get_workspace(q_extend.device, mb, q_extend.shape[1], k_extend.shape[1], q_extend.shape[2],
                                  v_extend.shape[2], mle, stream)
    sm = 0.0 if sm_scale is None else float(sm_scale)
    ok = _native.lib().verify_splitkv_write_fwd(
        _ref(q_extend), _ref(k_extend), _ref(v_extend), _ref(o_extend), _ref(k_buffer), _ref(v_buffer),
        _ref(qo_indptr), _ref(kv_indptr), _ref(kv_indices), _ref(out_cache_loc), mle, _coerce(k_scale),
        _coerce(v_scale), sm, ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
        ctypes.c_void_p(stream.cuda_stream))
    if not ok:
        raise ValueError("verify_splitkv_write_fwd: " + _native.last_error())


def verify_splitkv_paged_write_fwd(q, k_new, v_new, o, k_cache, v_cache, block_table, seq_lens, page_size,
                                   max_len_extend, k_scale=1.0, v_scale=1.0, sm_scale=None, max_bs=None,
                                   workspace=None, stream=None) -> None:
    """``verify_splitkv_paged_fwd`` that first stores the drafts' k_new /
    v_new ([B*l_ext, h_kv, D] bf16) into cache positions seq_lens[b] + t, in
    the same launch; the attention uses the stored values."""
    bs = seq_lens.shape[0]
    mle = int(max_len_extend)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if workspace is None:
        mb = bs if (max_bs is None or max_bs < bs) else int(max_bs)
        workspace = get_workspace(q.device, mb, q.shape[1], k_cache.shape[1], q.shape[2], v_cache.shape[2], mle,
                                  stream)
    sm = 0.0 if sm_scale is None else float(sm_scale)
    ok = _native.lib().verify_splitkv_paged_write_fwd(
        _ref(q), _ref(k_new), _ref(v_new), _ref(o), _ref(k_cache), _ref(v_cache), _ref(block_table), _ref(seq_lens),
        int(page_size), mle, _coerce(k_scale), _coerce(v_scale), sm, ctypes.c_void_p(workspace.data_ptr()),
        workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    if not ok:
        raise ValueError("verify_splitkv_paged_write_fwd: " + _native.last_error())


def read_error_flags(workspace=None, stream=None) -> int:
    """Device error word of a workspace (synchronises; for tests/debugging).
    Default: the cached workspace of ``stream`` (the current stream) on the
    current device."""
    if stream is None:
        stream = torch.cuda.current_stream()
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        with _WS_LOCK:
            workspace = _WS.get((dev, int(stream.cuda_stream)))
    flags = ctypes.c_uint32(0)
    ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    if not _native.lib().vsk_read_error_flags(ptr, ctypes.c_void_p(stream.cuda_stream), ctypes.byref(flags)):
        raise RuntimeError(_native.last_error())
    return int(flags.value)


def set_tuning(num_ctas: int = 0, min_tokens_per_cta: int = 0) -> None:
    """Override the CTA count / minimum tokens per CTA (0 = defaults)."""
    _native.lib().vsk_set_tuning(int(num_ctas), int(min_tokens_per_cta))


def set_tuning_shape(max_ring_stages: int = 0, max_kv_heads_per_cta: int = 0) -> None:
    """Override ring depth / KV heads per CTA (0 = defaults)."""
    _native.lib().vsk_set_tuning_shape(int(max_ring_stages), int(max_kv_heads_per_cta))


def set_tuning_tiles(tiles_per_warp: int = 0) -> None:
    """Override the 16-row query tiles per consumer warp (1 or 2; 0 = default)."""
    _native.lib().vsk_set_tuning_tiles(int(tiles_per_warp))


def set_tuning_tc(mode: int = 3) -> None:
    """Head_dim 256 calls (at most 32 packed rows per KV head) and the
    tensor-memory streams: 3 (the default) the one with the packed query rows
    on the MMAs' M side where it measured faster (by pool dtype, packed rows and
    size), 2 that one wherever it applies, 1 (or ``True``) the one with the keys
    on M wherever it applies, 0 (or ``False``) never (the mma.sync kernels
    only).  For A/B runs and tests."""
    _native.lib().vsk_set_tuning_tc(int(mode))


def set_tuning_colsplit(mode: int = 1) -> None:
    """Head_dim 256 calls (at most 32 packed rows per KV head) that no
    tensor-memory stream takes (``set_tuning_tc``): stream with the
    column-split mma.sync kernel plus a combine launch for small calls (1, the
    default), always (2) or never (0); for A/B runs and tests."""
    _native.lib().vsk_set_tuning_colsplit(int(mode))


def set_tuning_colsplit2(mode: int = 1) -> None:
    """Head_dim 256 calls with 17-32 packed rows per KV head: the column split
    with both tiles in each warp wherever it applies (2) or never (0 and 1, the
    default: the stream-only kernel measured faster); for A/B runs and tests."""
    _native.lib().vsk_set_tuning_colsplit2(int(mode))


def set_tuning_split_launch(mode: int = 1) -> None:
    """Calls with at most 32 drafts: stream-only kernel plus a combine launch
    (head_dim 64 / 128: small and mid-size calls; head_dim 256: from where the
    column split stops up to 2^23 prefix tokens x KV heads, where no
    tensor-memory stream takes the call) by size (1, the default), always (2)
    or never (0); for A/B runs and tests."""
    _native.lib().vsk_set_tuning_split_launch(int(mode))


def set_tuning_cluster(mode: int = 0) -> None:
    """The cluster form (one launch; one thread-block cluster per (sequence,
    KV head) folds its own partials): never (0, the default), for small calls
    (1) or wherever it applies (2); for A/B runs and tests."""
    _native.lib().vsk_set_tuning_cluster(int(mode))


def set_tuning_pdl(mode: int = 1) -> None:
    """The combine kernel of the two-launch forms as a programmatic dependent
    of the prefix stream for small calls (1, the default), always (2) or
    never (0: plain stream order); for A/B runs."""
    _native.lib().vsk_set_tuning_pdl(int(mode))


def set_tuning_pipe(enabled: bool = True) -> None:
    """Head_dim 256 one-launch kernel over e4m3 pools with software-pipelined
    stages (the default) or one stage after the other (bf16 pools always run
    one stage after the other); for A/B runs."""
    _native.lib().vsk_set_tuning_pipe(1 if enabled else 0)


def launches_per_call(batch: int, h_q: int, h_kv: int, head_dim: int, max_len_extend: int,
                      prefix_tokens: int) -> int:
    """Kernel launches one call of these shapes makes (1 or 2; 0 if no entry
    point accepts them); ``prefix_tokens`` = len(kv_indices), or batch x
    block-table columns x page_size for the paged entry points."""
    return int(_native.lib().vsk_launches_per_call(int(batch), int(h_q), int(h_kv), int(head_dim),
                                                   int(max_len_extend), int(prefix_tokens)))


def call_form(batch: int, h_q: int, h_kv: int, head_dim: int, v_head_dim: int, max_len_extend: int,
              prefix_tokens: int, fp8_pool: bool = False) -> str:
    """The form a call of these shapes takes ("one_launch", "cluster",
    "column_split", "column_split_two_tiles", "stream_only", "tensor_memory";
    "" if no entry point accepts them); ``prefix_tokens`` as for
    ``launches_per_call``."""
    return _native.lib().vsk_call_form(int(batch), int(h_q), int(h_kv), int(head_dim), int(v_head_dim),
                                       int(max_len_extend), int(prefix_tokens), 1 if fp8_pool else 0).decode()


def version() -> str:
    return _native.lib().vsk_version().decode()
